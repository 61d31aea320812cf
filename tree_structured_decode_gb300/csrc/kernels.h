// Device-side parameter blocks and kernel launchers (host-callable).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "planner.h"

namespace ta {

// Per group-token record (16 bytes): token id (-1: a filler row of a packed
// unit), visible end inside the group span, the partial-result index of
// chunk 0 (-1: the token's only partial, written straight to the output),
// and pc_slot = the token's number of partials (low 24 bits) | (the page
// slot a packed row sees + 1) << 24 (0: every page of the tile).
struct GroupTok {
  int32_t tok, vis, pbase, pc_slot;
  __host__ __device__ int pcount() const { return pc_slot & 0xFFFFFF; }
  __host__ __device__ int slot() const { return (pc_slot >> 24) - 1; }
};
__host__ __device__ inline int32_t pack_pc_slot(int32_t pcount, int32_t slot) {
  return (pcount & 0xFFFFFF) | ((slot + 1) << 24);
}

// Per merge item: a query token with >= 2 partials.
struct MergeItem {
  int32_t tok, poff, count, pad;
};

// A partial O row whose largest |value| reaches this is stored divided by a
// power of two s (kept beside its lse), so that fp16 never overflows: the
// inputs may hold any bf16 value.
constexpr float kPartialRescaleAt = 32768.f;

// CTAs whose unit ranges travel in the launch parameters (read from the
// constant bank at start-up instead of a dependent global load).
constexpr int kInlineCtas = 320;

struct AttnParams {
  const UnitDesc* units;
  const int2* blocks;        // {page, span_pos * 32 + valid}
  const GroupTok* gtoks;
  const int32_t* cta_off;    // CTA c runs units [cta_off[c], cta_off[c+1])
  const uint16_t* q;         // bf16 bits [nq][hq][d]
  const uint16_t* k;         // bf16 bits [pages][hkv][16][d]
  const uint16_t* v;
  float* out;                // [nq][hq][d]
  float* lse;                // [nq][hq] natural log, or null
  uint16_t* part_o;          // [n_partials][hq][d] fp16 bits: normalised partial O / s
  float2* part_ml;           // [n_partials][hq]: {lse in log2 units, s}; s = 1, or the
                             // power of two that keeps |O| / s inside the fp16 range
  int32_t* err;              // device error word
  int32_t hq, hkv, gqa, n_units;
  float scale_log2;          // softmax scale * log2(e)
  long long wait_timeout_ns;
  int32_t debug_stuck_wait;  // testing aid: wait on a barrier nothing signals
  // fused merge: per (token, q head) arrival counters (zero between runs)
  // and each token's first partial index; merge_fused = 0 leaves the
  // partials to the separate merge kernel
  int32_t* merge_cnt;
  const int32_t* tok_poff;
  int32_t merge_fused;
  // grid <= kInlineCtas: cta_off copied here, cta_inline = 1
  int32_t cta_inline;
  int32_t cta_off_inline[kInlineCtas + 1];
};

struct MergeParams {
  const MergeItem* items;
  int32_t n_items, hq;
  int32_t max_count;         // most partials of any merged token
  const uint16_t* part_o;    // fp16 bits (O / s)
  const float2* part_ml;     // {lse (log2 units), s}
  float* out;
  float* lse;
  // at most kMergeEarlyRows (token, q head) rows: once the partials are
  // visible the kernel lets the stream's next kernel be scheduled
  int32_t early_trigger;
};
constexpr int64_t kMergeEarlyRows = 16384;

// Launch the persistent grouped partial-attention kernel (TMA + tcgen05 /
// CUDA cores), one CTA per schedule entry.  kv_evict: the plan's K/V mostly
// streams once (HostPlan::kv_evict); its copies then carry L2 policies.
cudaError_t launch_tree_attention(const AttnParams& p, int d, int grid, int num_pages,
                                  bool kv_evict, cudaStream_t s);
// Launch the log-sum-exp merge of partial results.
cudaError_t launch_lse_merge(const MergeParams& p, int d, cudaStream_t s);
// Copy each query token's new K and V (bf16 [nq][hkv][d]) into its page slot
// (dst[t] = page * 16 + slot, or -1 to skip) of the paged cache.
cudaError_t launch_append_kv(const uint16_t* k_new, const uint16_t* v_new, const int32_t* dst,
                             int nq, int hkv, int d, uint16_t* k_pages, uint16_t* v_pages,
                             cudaStream_t s);

}  // namespace ta
