// Persistent grouped partial-attention kernel for sm_103a.
//
// Two CTAs per SM each walk their list of work units (group, kv head, query
// tile, chunk).  A unit's KV span is streamed once, 64 tokens (4 pages) per
// tile, by TMA into rings of shared-memory stages (128-byte swizzle; K and V
// have their own rings).  The tile is consumed on one of two paths:
//
//  * tensor cores (stacked query rows; FastTree review page, "高效树结构注意力
//    内核设计": GEMV becomes GEMM once a group's queries are stacked): the
//    group's query tile (128 rows = query tokens x GQA heads; four thin
//    groups, or four kv heads of one, packed one per warp; or a tile of at
//    most 64 rows held once per kv head of a pair) sits in shared memory;
//    S = Q K^T goes to
//    TMEM (double-buffered), the four compute warps read one row per thread,
//    apply the mask and an online softmax (the running max is raised only
//    when it grows by more than 2^8, so O is rarely rescaled), write P as
//    bf16 over S in TMEM, and tcgen05 adds P V (P read from TMEM) into the O
//    accumulator in TMEM.
//  * CUDA cores (groups below the tensor-core row threshold, when it is
//    raised): the compute warps split the tile's pages,
//    lanes split the head dimension, and each warp keeps its own online
//    softmax; the warps' states are combined at the end of the unit.
//
// Each row's result is written as final output when the row has one partial,
// else as a normalised partial (O, lse in base 2) for the merge pass (DeFT
// notes page, "Tree-Topology-Aware Global Reduction Strategy").
//
// Roles: warps 0-3 compute (thread i owns TMEM lane / query row i), warp 4
// streams K and warp 6 streams V by TMA (and zeroes the V rows of unfilled
// page slots), warp 5 owns TMEM and issues tcgen05.mma; the issuing warps
// run converged, one elected lane issuing.  The compute warps' tile loop is
// compiled once per unit form, and rare paths sit in out-of-line functions:
// the speed of this kernel depends on how short its loops' code is.
// Every wait is bounded: if one runs out the CTA records TA_DEVERR_TIMEOUT, stops issuing
// work, waits (bounded) for its copies and MMAs in flight, frees TMEM and
// returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

#include <type_traits>

namespace ta {
namespace {

// Two CTAs per SM, each a full pipeline of two warpgroups: four compute warps
// (thread i owns TMEM lane / query row i) and one warpgroup holding the TMA
// producer warps (K, V), the tcgen05 issuer warp and an idle warp.  The launch gives
// every thread 128 registers; the roles rebalance to 200 (compute) and 56
// (producer/issuer): 128 x 200 + 128 x 56 <= 256 x 128.  The second CTA on
// the SM fills the latency gaps of the first.
constexpr int kThreads = 256;
constexpr int kComputeThreads = 128;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kVProducerWarp = 6;
constexpr int kComputeRegs = 200;
constexpr int kIssueRegs = 56;
static_assert(128 * kComputeRegs + 128 * kIssueRegs <= kThreads * 128, "register split too large");
constexpr int kTileTok = kKvTileTokens;  // KV tokens per tile (4 pages)
constexpr int kBpt = kTileTok / 16;       // pages (blocks) per tile
constexpr float kRescaleLog2 = 8.f;  // lazy-rescale threshold (log2 units)
constexpr float kLn2 = 0.69314718055994530942f;
constexpr uint32_t kTmemCols = 256;  // S0, S1 (64 columns each) and O (128)
constexpr long long kDrainLimitNs = 200000000;  // 200 ms for copies / MMAs already in flight

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kStages = D == 128 ? 2 : 4;
  static constexpr int kQBytes = 128 * D * 2;          // the query tile
  static constexpr int kTileBytes = kTileTok * D * 2;  // K (or V) of one tile
  static constexpr int kScratchBytes = 128 * kTileTok * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffScratch = kOffV + kStages * kTileBytes;
  static constexpr int kOffBar = kOffScratch + kScratchBytes;
  static constexpr int kNumBars = 5 * kStages + 12;
  static constexpr int kOffML = kOffBar + kNumBars * 8 + 16;  // float [4][8][2]
  // the dynamic shared window starts 1024-byte aligned (checked at start)
  static constexpr int kSmem = kOffML + 4 * kSimtTileRows * 2 * 4;
  // two CTAs per SM: 228 KB of shared memory per SM, 1 KB of it reserved per CTA
  static_assert(2 * (kSmem + 1024) <= 228 * 1024, "two CTAs per SM must fit in shared memory");
  // scratch of the CUDA-core path, where its four warps' O are combined
  static_assert(4 * kSimtTileRows * D * 4 <= kScratchBytes, "combine scratch too small");
  // A stage holds K as [64-column half][tile token][128 B] (one box per page
  // and half; QK^T is one N = kTileTok MMA per 16 columns of d) and V as
  // [page][64-column half][16 tokens][128 B] (one box per page-head; P.V is
  // one MMA per page).  Both 128-byte swizzled.
  static constexpr uint32_t kBlockBytes = 16 * D * 2;                // one page-head
  static constexpr uint32_t kIdescQK = ptx::idesc_bf16(128, kTileTok, 0);
  static constexpr uint32_t kIdescPV = ptx::idesc_bf16(128, D, 1);
};

struct Shared {
  uint32_t base;  // 1024-aligned shared address of the layout
  uint8_t* ptr;
  volatile uint32_t* tmem_slot;
  volatile int* abort_flag;
};

// K and V of a stage have their own full / empty barriers: K is released as
// soon as QK^T has read it, V only after P.V, so the next tiles' K streams
// in while the current tile is still in the softmax.
template <int D>
struct Bars {
  static constexpr int S = Cfg<D>::kStages;
  uint32_t b;
  __device__ uint32_t kfull(int s) const { return b + 8 * s; }
  __device__ uint32_t kempty(int s) const { return b + 8 * (S + s); }
  __device__ uint32_t vfull(int s) const { return b + 8 * (2 * S + s); }
  __device__ uint32_t vempty(int s) const { return b + 8 * (3 * S + s); }
  // S buffer i: S ready / its P consumed by P.V / its P written
  __device__ uint32_t s_full(int i) const { return b + 8 * (4 * S + i); }
  __device__ uint32_t pv_done(int i) const { return b + 8 * (4 * S + 2 + i); }
  __device__ uint32_t p_full(int i) const { return b + 8 * (4 * S + 4 + i); }
  __device__ uint32_t o_full() const { return b + 8 * (4 * S + 6); }
  __device__ uint32_t drain() const { return b + 8 * (4 * S + 7); }
  __device__ uint32_t q_full(int i) const { return b + 8 * (4 * S + 8 + i); }
  __device__ uint32_t never() const { return b + 8 * (4 * S + 10); }
  __device__ uint32_t o_empty() const { return b + 8 * (4 * S + 11); }
  // V copies of a tile with unfilled page slots land here; the V producer
  // zeroes those slots' rows and only then completes vfull
  __device__ uint32_t vland(int s) const { return b + 8 * (4 * S + 12 + s); }
};

// Bounded wait.  Returns false (without waiting further) once the CTA has
// aborted; a wait that exceeds the limit aborts the CTA and records the
// error.  A phase that has already completed returns true at once: every
// issue after a wait checks the abort flag itself.
// The polling loop sits out of line: every wait site stays one try_wait and
// a call, which keeps the loops that wait short.  One copy per register
// split (0: compute warps, 1: the issuing warps), as a call must match its
// caller's register count.
template <int kRole>
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int32_t* err, long long limit_ns) {
  if (*abort_flag) return false;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t n = 1;; ++n) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((n & 15) == 0) {
      if (*abort_flag) return false;
      if ((long long)(ptx::globaltimer() - t0) > limit_ns) {
        *abort_flag = 1;
        atomicCAS(err, 0, TA_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}
template <int kRole = 0>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Shared& sh,
                                         int32_t* err, long long limit_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow<kRole>(bar, parity, sh.abort_flag, err, limit_ns);
}

// wait_bar for a whole (converged) warp: true only if every lane's wait
// succeeded, so the warp stays converged.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Shared& sh,
                                          int32_t* err, long long limit_ns) {
  return __all_sync(0xffffffffu, wait_bar<1>(bar, parity, sh, err, limit_ns));
}
__device__ __forceinline__ bool warp_aborted(const Shared& sh) {
  return __any_sync(0xffffffffu, *sh.abort_flag != 0);
}

// Wait used while draining after an abort: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, long long limit_ns) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity))
    if ((long long)(ptx::globaltimer() - t0) > limit_ns) return;
}

// valid slots of a tile's four pages, 5 bits a page, when every page is full
constexpr int kFullTileValid = 16 | 16 << 5 | 16 << 10 | 16 << 15;

__device__ __forceinline__ int unit_tiles(const UnitDesc& u) {
  return (u.blk1 - u.blk0 + kBpt - 1) / kBpt;
}

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// ============================================================== producers
// One warp streams K (kIsV false) or V (true) of every tile of the CTA's
// units into the stage ring.  The whole warp runs the loop (its values stay
// warp-uniform); one elected lane issues each copy.
// kEvict (a plan whose K/V mostly streams once): each unit's copies carry an
// L2 policy, evict-first for a unit whose K/V no other unit reads, else
// evict-last.
template <int D, bool kIsV, bool kEvict>
__device__ void producer(const CUtensorMap* tm, const AttnParams& p, int u0, int u1,
                         const Shared& sh, const Bars<D>& B) {
  using C = Cfg<D>;
  uint32_t g = 0;
  if (!kIsV && p.debug_stuck_wait) warp_wait(B.never(), 0, sh, p.err, p.wait_timeout_ns);
  uint32_t filled[C::kStages];  // 1 + tile index of the last fill issued per stage
  uint32_t land_par = 0;        // V: phase bit of each stage's vland barrier
  // K/V that no other unit reads asks L2 to evict it first; K/V that other
  // units read again asks to be evicted last
  uint64_t pol_once = 0, pol_shared = 0;
  if constexpr (kEvict) {
    pol_once = ptx::policy_evict_first();
    pol_shared = ptx::policy_evict_last();
  }
#pragma unroll
  for (int s = 0; s < C::kStages; ++s) filled[s] = 0;
  UnitDesc un = u0 < u1 ? p.units[u0] : UnitDesc{};
  for (int ui = u0; ui < u1; ++ui) {
    const UnitDesc u = un;
    if (ui + 1 < u1) un = p.units[ui + 1];  // in flight while this unit is issued
    for (int b0 = u.blk0; b0 < u.blk1; b0 += kBpt, ++g) {
      const int s = g % C::kStages;
      const int nb = min(kBpt, u.blk1 - b0);
      int page[kBpt];  // all loads in flight while waiting for the stage
      int nvm = kFullTileValid;  // V: valid slots of the pages
#pragma unroll
      for (int bb = 0; bb < kBpt; ++bb) {
        if constexpr (kIsV) {
          const int2 r = bb < nb ? __ldg(&p.blocks[b0 + bb]) : make_int2(0, 16);
          page[bb] = r.x;
          nvm = (nvm & ~(31 << (5 * bb))) | (r.y & 31) << (5 * bb);
        } else {
          page[bb] = bb < nb ? __ldg(&p.blocks[b0 + bb].x) : 0;
        }
      }
      const uint32_t full = kIsV ? B.vfull(s) : B.kfull(s);
      // V pages with unfilled slots land on vland first (their rows are
      // zeroed below); everything else lands on the stage's full barrier
      const bool zero = kIsV && nvm != kFullTileValid;
      const uint32_t land = zero ? B.vland(s) : full;
      if (g >= (uint32_t)C::kStages &&
          !warp_wait(kIsV ? B.vempty(s) : B.kempty(s), ((g / C::kStages) + 1) & 1, sh, p.err,
                     p.wait_timeout_ns))
        continue;
      if (warp_aborted(sh)) continue;
      const bool leader = ptx::elect_one();
      if (leader) ptx::mbar_arrive_expect_tx(land, (uint32_t)nb * C::kBlockBytes);
      // page bb's kv head: kvh + bb in a unit packed by kv head, kvh + bb / 2
      // in a pair unit, else kvh
      const int kvh = u.kvh, hsh = (u.path & kUnitHeads) ? 0 : (u.path & kUnitPairs) ? 1 : 3;
      const uint64_t pol = (u.path & kUnitReadOnce) ? pol_once : pol_shared;
      const uint32_t dst = sh.base + (kIsV ? C::kOffV : C::kOffK) + s * C::kTileBytes;
#pragma unroll
      for (int bb = 0; bb < kBpt; ++bb) {
        if (bb < nb && leader) {
          if constexpr (!kIsV) {
#pragma unroll
            for (int h = 0; h < C::kHalves; ++h)
              if constexpr (kEvict)
                ptx::tma_load_4d_hint(dst + h * (kTileTok * 128) + bb * 2048, tm, 64 * h, 0,
                                      kvh + (bb >> hsh), page[bb], land, pol);
              else
                ptx::tma_load_4d(dst + h * (kTileTok * 128) + bb * 2048, tm, 64 * h, 0,
                                 kvh + (bb >> hsh), page[bb], land);
          } else if constexpr (D == 128) {  // both 64-column halves of V in one box
            if constexpr (kEvict)
              ptx::tma_load_5d_hint(dst + bb * C::kBlockBytes, tm, 0, 0, 0, kvh + (bb >> hsh), page[bb],
                                    land, pol);
            else
              ptx::tma_load_5d(dst + bb * C::kBlockBytes, tm, 0, 0, 0, kvh + (bb >> hsh), page[bb], land);
          } else {
            if constexpr (kEvict)
              ptx::tma_load_4d_hint(dst + bb * C::kBlockBytes, tm, 0, 0, kvh + (bb >> hsh), page[bb], land,
                                    pol);
            else
              ptx::tma_load_4d(dst + bb * C::kBlockBytes, tm, 0, 0, kvh + (bb >> hsh), page[bb], land);
          }
        }
      }
      if (zero) {
        // A page slot that holds no token may hold anything, NaN included;
        // its P is 0 but 0 * NaN is not 0.  Zero those V rows once the
        // copies have landed, then hand the stage to P.V.
        const uint32_t par = (land_par >> s) & 1;
        land_par ^= 1u << s;
        if (warp_wait(B.vland(s), par, sh, p.err, p.wait_timeout_ns)) {
          uint8_t* vst = sh.ptr + C::kOffV + s * C::kTileBytes;
          const int lane = threadIdx.x & 31;
#pragma unroll
          for (int bb = 0; bb < kBpt; ++bb) {
            const int nv = (nvm >> (5 * bb)) & 31;
            for (int idx = lane; idx < (16 - nv) * 8 * C::kHalves; idx += 32) {
              const int r = nv + idx / (8 * C::kHalves), hh = (idx >> 3) % C::kHalves, ch = idx & 7;
              *reinterpret_cast<uint4*>(vst + bb * C::kBlockBytes + hh * 2048 + r * 128 + ch * 16) =
                  make_uint4(0, 0, 0, 0);
            }
          }
          ptx::fence_proxy_async_smem();
        } else {
          drain_wait(B.vland(s), par, kDrainLimitNs);  // the copies land before the CTA may exit
        }
        __syncwarp();
        if (ptx::elect_one()) ptx::mbar_arrive(full);
      }
#pragma unroll
      for (int t = 0; t < C::kStages; ++t)
        if (t == s) filled[t] = g + 1;
    }
  }
  if (warp_aborted(sh)) {
    // let the last copy issued into every stage land before the CTA exits
#pragma unroll
    for (int s = 0; s < C::kStages; ++s)
      if (filled[s])
        drain_wait(kIsV ? B.vfull(s) : B.kfull(s), ((filled[s] - 1) / C::kStages) & 1, kDrainLimitNs);
  }
}

// ============================================================== MMA issuer
template <int D>
__device__ void mma_issuer(const AttnParams& p, int u0, int u1, const Shared& sh,
                           const Bars<D>& B, uint32_t tmem) {
  using C = Cfg<D>;
  uint32_t g = 0, gm = 0, nu = 0;
  const uint64_t dq = ptx::sdesc_sw128(sh.base + C::kOffQ, 16, 1024);  // the query tile
  bool issued = false;
  UnitDesc un = u0 < u1 ? p.units[u0] : UnitDesc{};
  for (int ui = u0; ui < u1; ++ui) {
    const UnitDesc u = un;
    if (ui + 1 < u1) un = p.units[ui + 1];
    const int T = unit_tiles(u);
    if (!(u.path & kPathMma) || T == 0) {
      g += T;
      continue;
    }
    const bool qok = warp_wait(B.q_full(0), nu & 1, sh, p.err, p.wait_timeout_ns);
    // the query rows were written by the compute warps' cp.async (generic
    // proxy); the tensor cores read them through the async proxy
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_after();
    const uint32_t o_tmem = tmem + 128;
    auto issue_pv = [&](int jj) {
      const int pb = (gm + jj) & 1;  // P(jj) sits in the first 32 columns of S buffer pb
      bool ok = warp_wait(B.p_full(pb), ((gm + jj) >> 1) & 1, sh, p.err, p.wait_timeout_ns);
      // the first P.V of a unit overwrites O: the previous unit's epilogue
      // must have read it
      if (jj == 0 && nu > 0) ok = warp_wait(B.o_empty(), (nu - 1) & 1, sh, p.err, p.wait_timeout_ns) && ok;
      const int s = (g + jj) % C::kStages;
      ok = ok && warp_wait(B.vfull(s), ((g + jj) / C::kStages) & 1, sh, p.err, p.wait_timeout_ns);
      ptx::tc_fence_after();
      const int nbk = min(kBpt, u.blk1 - (u.blk0 + kBpt * jj));
      if (ok && !warp_aborted(sh) && ptx::elect_one()) {
        // descriptors: the 14-bit start address field (16-byte units) of the
        // stage's base descriptor plus the page offset (no carry: the shared
        // window is below 256 KB)
        const uint64_t dv = ptx::sdesc_sw128(sh.base + C::kOffV + s * C::kTileBytes, 2048, 1024);
        for (int kk = 0; kk < nbk; ++kk)  // one page (16 tokens = 8 columns of P) per MMA
          ptx::mma_bf16_ts(o_tmem, tmem + pb * kTileTok + kk * 8, dv + kk * (C::kBlockBytes >> 4),
                           C::kIdescPV, (jj > 0 || kk > 0) ? 1u : 0u);
        issued = true;
      }
      if (ptx::elect_one()) {
        ptx::mma_commit(B.vempty(s));
        ptx::mma_commit(B.pv_done(pb));
      }
    };
    // QK^T of tile j, then P.V of tile j - 1 (its softmax overlaps QK^T(j));
    // one more pass issues the last P.V
    for (int j = 0; j <= T; ++j) {
      if (j < T) {
        const int s = (g + j) % C::kStages;
        const int sb = (gm + j) & 1;
        bool ok = qok && warp_wait(B.kfull(s), ((g + j) / C::kStages) & 1, sh, p.err, p.wait_timeout_ns);
        // S buffer sb holds P of the tile two back until that P.V has completed
        ok = ok && warp_wait(B.pv_done(sb), (((gm + j) >> 1) + 1) & 1, sh, p.err, p.wait_timeout_ns);
        ptx::tc_fence_after();
        if (ok && !warp_aborted(sh) && ptx::elect_one()) {
          const uint64_t dk = ptx::sdesc_sw128(sh.base + C::kOffK + s * C::kTileBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t qoff = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
            const uint32_t koff = (kk >> 2) * (kTileTok * 128) + (kk & 3) * 32;
            ptx::mma_bf16(tmem + sb * kTileTok, dq + (qoff >> 4), dk + (koff >> 4), C::kIdescQK,
                          kk > 0 ? 1u : 0u);
          }
          issued = true;
        }
        if (ptx::elect_one()) {
          ptx::mma_commit(B.s_full(sb));
          ptx::mma_commit(B.kempty(s));
        }
      }
      if (j > 0) issue_pv(j - 1);
    }
    if (ptx::elect_one()) ptx::mma_commit(B.o_full());
    g += T;
    gm += T;
    ++nu;
  }
  if (warp_aborted(sh) && __any_sync(0xffffffffu, issued)) {
    if (ptx::elect_one()) ptx::mma_commit(B.drain());
    drain_wait(B.drain(), 0, kDrainLimitNs);
  }
}

// ============================================================== compute warps
// Shared-memory offset of element [row][col] (col in 0..63 of one 128-byte
// swizzled half) for 8-element chunk granularity.
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return row * 128 + ((chunk ^ (row & 7)) << 4);
}

// ---------------------------------------------------------- fused merge
// After a row's partial (O normalised and stored as O / s, lse in base 2) is
// written, its writer counts it in; the writer of the row's last partial
// folds all of them:
//   m = max lse_i, w_i = 2^(lse_i - m), O = sum w_i s_i (O_i / s_i) / sum w_i,
//   lse = m + log2 sum w_i
// (DeFT notes page, "Tree-Topology-Aware Global Reduction Strategy"), writes
// the output row and resets the counter for the next run.  Release: a fence
// before the count; acquire: a fence after observing the last count; the
// partials are read through L2 (other SMs wrote them).

// One thread folds row (tok, h).  Returns nothing; no-op unless last.
template <int D>
__device__ __noinline__ void merge_row_thread(const AttnParams& p, const GroupTok& gt, int h) {
  const int idx = gt.tok * p.hq + h;
  __threadfence();
  if (atomicAdd(p.merge_cnt + idx, 1) != gt.pcount() - 1) return;
  __threadfence();
  const int poff = __ldcg(p.tok_poff + gt.tok);
  float m = -INFINITY;
  for (int k = 0; k < gt.pcount(); ++k) m = fmaxf(m, __ldcg(p.part_ml + (size_t)(poff + k) * p.hq + h).x);
  float* dst = p.out + (size_t)idx * D;
  float den = 0.f;
  if (m == -INFINITY) {
    for (int c = 0; c < D; c += 4) *reinterpret_cast<float4*>(dst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
  } else {
    for (int k = 0; k < gt.pcount(); ++k)
      den += ptx::ex2(__ldcg(p.part_ml + (size_t)(poff + k) * p.hq + h).x - m);
    const float inv = 1.f / den;
#pragma unroll 1
    for (int c0 = 0; c0 < D; c0 += 32) {
      float4 acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int k = 0; k < gt.pcount(); ++k) {
        const size_t slot = (size_t)(poff + k) * p.hq + h;
        const float2 ml = __ldcg(p.part_ml + slot);
        const float w = ptx::ex2(ml.x - m) * ml.y;
        const uint4* src = reinterpret_cast<const uint4*>(p.part_o + slot * D + c0);  // fp16
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint4 v = __ldcg(src + e);
          const float2 a = ptx::unpack_f16(v.x), b = ptx::unpack_f16(v.y);
          const float2 c = ptx::unpack_f16(v.z), dd = ptx::unpack_f16(v.w);
          acc[2 * e].x = fmaf(w, a.x, acc[2 * e].x);
          acc[2 * e].y = fmaf(w, a.y, acc[2 * e].y);
          acc[2 * e].z = fmaf(w, b.x, acc[2 * e].z);
          acc[2 * e].w = fmaf(w, b.y, acc[2 * e].w);
          acc[2 * e + 1].x = fmaf(w, c.x, acc[2 * e + 1].x);
          acc[2 * e + 1].y = fmaf(w, c.y, acc[2 * e + 1].y);
          acc[2 * e + 1].z = fmaf(w, dd.x, acc[2 * e + 1].z);
          acc[2 * e + 1].w = fmaf(w, dd.y, acc[2 * e + 1].w);
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e)
        *reinterpret_cast<float4*>(dst + c0 + 4 * e) =
            make_float4(acc[e].x * inv, acc[e].y * inv, acc[e].z * inv, acc[e].w * inv);
    }
  }
  if (p.lse) p.lse[idx] = m == -INFINITY ? -INFINITY : (m + __log2f(den)) * kLn2;
  p.merge_cnt[idx] = 0;
}

// A warp folds row (tok, h), lanes over d (lane holds EPL columns).
template <int D>
__device__ __noinline__ void merge_row_warp(const AttnParams& p, const GroupTok& gt, int h, int lane) {
  constexpr int EPL = D / 32;
  const int idx = gt.tok * p.hq + h;
  int last = 0;
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    last = atomicAdd(p.merge_cnt + idx, 1) == gt.pcount() - 1;
  }
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __threadfence();
  const int poff = __ldcg(p.tok_poff + gt.tok);
  float m = -INFINITY;
  for (int k = 0; k < gt.pcount(); ++k) m = fmaxf(m, __ldcg(p.part_ml + (size_t)(poff + k) * p.hq + h).x);
  float acc[EPL], den = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  if (m != -INFINITY) {
    for (int k = 0; k < gt.pcount(); ++k) {
      const size_t slot = (size_t)(poff + k) * p.hq + h;
      const float2 ml = __ldcg(p.part_ml + slot);
      const float w = ptx::ex2(ml.x - m);
      den += w;
      const float wo = w * ml.y;
      const uint32_t* src = reinterpret_cast<const uint32_t*>(p.part_o + slot * D + lane * EPL);
#pragma unroll
      for (int e = 0; e < EPL; e += 2) {
        const float2 v = ptx::unpack_f16(__ldcg(src + e / 2));
        acc[e] = fmaf(wo, v.x, acc[e]);
        acc[e + 1] = fmaf(wo, v.y, acc[e + 1]);
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) p.out[(size_t)idx * D + lane * EPL + e] = acc[e] * inv;
  if (lane == 0) {
    if (p.lse) p.lse[idx] = den > 0.f ? (m + __log2f(den)) * kLn2 : -INFINITY;
    p.merge_cnt[idx] = 0;
  }
}

template <int EPL>
__device__ __forceinline__ void load_slice(const uint8_t* ptr, float (&f)[EPL]) {
  if constexpr (EPL == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(ptr);
    f[0] = bf16_lo(w.x);
    f[1] = bf16_hi(w.x);
    f[2] = bf16_lo(w.y);
    f[3] = bf16_hi(w.y);
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(ptr);
    f[0] = bf16_lo(w);
    f[1] = bf16_hi(w);
  }
}

// Sum of v[t] over the 32 lanes for 16 values t at once (16 shuffles instead
// of 16 x 5): after halving steps over lane bits 4..1 and a final exchange
// over bit 0, lane L holds the total for t = L >> 1.
__device__ __forceinline__ float transpose_sum16(float (&v)[16], int lane) {
  {
    const bool up = lane & 16;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float send = up ? v[k] : v[k + 8];
      const float keep = up ? v[k + 8] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
  }
  {
    const bool up = lane & 8;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float send = up ? v[k] : v[k + 4];
      const float keep = up ? v[k + 4] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
  }
  {
    const bool up = lane & 4;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float send = up ? v[k] : v[k + 2];
      const float keep = up ? v[k + 2] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
  }
  {
    const bool up = lane & 2;
    const float send = up ? v[0] : v[1];
    const float keep = up ? v[1] : v[0];
    v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// CUDA-core consumer for a thin unit (<= 8 rows).  Like the fused-merge
// folds, kept out of line (about half of the kernel's code), so that the
// tensor-core tile loop of the compute warps stays compact in the
// instruction caches.
template <int D>
__device__ __noinline__ void simt_unit(const AttnParams& p, const UnitDesc& u, uint32_t g, int T,
                                       const Shared& sh, const Bars<D>& B) {
  using C = Cfg<D>;
  constexpr int EPL = D / 32;
  constexpr int RB = kSimtTileRows;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nr = min(RB, u.nrows);
  float qv[RB][EPL], o[RB][EPL], m[RB], l[RB];
  int vis[RB], slot[RB];
#pragma unroll
  for (int i = 0; i < RB; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
    vis[i] = 0;
    slot[i] = -1;
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[i][e] = qv[i][e] = 0.f;
    const GroupTok gt = i < nr ? p.gtoks[u.tok_off + (u.row0 + i) / p.gqa]
                               : GroupTok{-1, 0, -1, 0};
    if (gt.tok >= 0) {  // filler rows of a packed unit see nothing
      const int grow = u.row0 + i;
      const int h = u.kvh * p.gqa + grow % p.gqa;
      vis[i] = gt.vis;
      slot[i] = gt.slot();
      const uint16_t* src = p.q + ((size_t)gt.tok * p.hq + h) * D + lane * EPL;
      if constexpr (EPL == 4) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
        qv[i][0] = bf16_lo(w.x) * p.scale_log2;
        qv[i][1] = bf16_hi(w.x) * p.scale_log2;
        qv[i][2] = bf16_lo(w.y) * p.scale_log2;
        qv[i][3] = bf16_hi(w.y) * p.scale_log2;
      } else {
        const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(src));
        qv[i][0] = bf16_lo(w) * p.scale_log2;
        qv[i][1] = bf16_hi(w) * p.scale_log2;
      }
    }
  }
  // lane's slice inside a swizzled 128-byte row
  const int half = (EPL == 4) ? (lane >> 4) : 0;
  const int chunk = (EPL == 4) ? ((lane & 15) >> 1) : (lane >> 2);
  const int inb = (EPL == 4) ? (lane & 1) * 8 : (lane & 3) * 4;
  int mt_next = warp < min(kBpt, u.blk1 - u.blk0) ? __ldg(&p.blocks[u.blk0 + warp].y) : 0;
  for (int j = 0; j < T; ++j) {
    const int s = (g + j) % C::kStages;
    const int nb = min(kBpt, u.blk1 - (u.blk0 + kBpt * j));
    // warp w takes page w of the tile; the next tile's record is loaded now
    const int mt_w = mt_next;
    if (j + 1 < T) {
      const int nbn = min(kBpt, u.blk1 - (u.blk0 + kBpt * (j + 1)));
      mt_next = warp < nbn ? __ldg(&p.blocks[u.blk0 + kBpt * (j + 1) + warp].y) : 0;
    }
    const uint32_t ph = ((g + j) / C::kStages) & 1;
    const bool ok = __all_sync(0xffffffffu, wait_bar(B.kfull(s), ph, sh, p.err, p.wait_timeout_ns) &&
                                                wait_bar(B.vfull(s), ph, sh, p.err, p.wait_timeout_ns));
    const uint8_t* kst = sh.ptr + C::kOffK + s * C::kTileBytes + half * (kTileTok * 128) + inb;
    const uint8_t* vst = sh.ptr + C::kOffV + s * C::kTileBytes + half * 2048 + inb;
    static_assert(kBpt == kComputeThreads / 32, "one page per compute warp");
    if (ok && warp < nb) {
      {
        const int bb = warp;
        const int pos = mt_w >> 5, nvalid = mt_w & 31;
#pragma unroll
        for (int i = 0; i < RB; ++i) {
          // a packed row sees only its own slot's page (warp bb reads page bb)
          const int lim = (i < nr && (slot[i] < 0 || slot[i] == bb)) ? max(0, min(nvalid, vis[i] - pos)) : 0;
          if (lim == 0) continue;  // warp-uniform
          // 16 independent partial dots, then one transposed reduction:
          // lane L ends with the score of token L >> 1 of the block.
          float d[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            float kf[EPL];
            load_slice<EPL>(kst + sw128(bb * 16 + t, chunk), kf);
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc = fmaf(qv[i][e], kf[e], acc);
            d[t] = acc;
          }
          const float sc = transpose_sum16(d, lane);
          const bool valid = (lane >> 1) < lim;
          float bm = valid ? sc : -INFINITY;
#pragma unroll
          for (int off = 16; off > 1; off >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
          const float m_new = fmaxf(m[i], bm);
          const float alpha = ptx::ex2(m[i] - m_new);
          const float pl = valid ? ptx::ex2(sc - m_new) : 0.f;
          float ps = pl;
#pragma unroll
          for (int off = 16; off > 1; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
          l[i] = fmaf(l[i], alpha, ps);
          m[i] = m_new;
#pragma unroll
          for (int e = 0; e < EPL; ++e) o[i][e] *= alpha;
          for (int t = 0; t < lim; ++t) {
            const float pt = __shfl_sync(0xffffffffu, pl, 2 * t);
            float vf[EPL];
            load_slice<EPL>(vst + bb * C::kBlockBytes + sw128(t, chunk), vf);
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[i][e] = fmaf(pt, vf[e], o[i][e]);
          }
        }
      }
    }
    ptx::named_bar_sync(1, kComputeThreads);
    if (tid == 0) {
      ptx::mbar_arrive(B.kempty(s));
      ptx::mbar_arrive(B.vempty(s));
    }
  }
  // combine the four warps' states in the scratch area
  float* sm_o = reinterpret_cast<float*>(sh.ptr + C::kOffScratch);  // [4][RB][D]
  float* sm_ml = reinterpret_cast<float*>(sh.ptr + C::kOffML);  // [4][RB][2]
  if (warp < 4) {  // only warps 0-3 take blocks (4 per tile); 4-7 help write rows
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      if (lane == 0) {
        sm_ml[(warp * RB + i) * 2 + 0] = m[i];
        sm_ml[(warp * RB + i) * 2 + 1] = l[i];
      }
#pragma unroll
      for (int e = 0; e < EPL; ++e) sm_o[(warp * RB + i) * D + lane * EPL + e] = o[i][e];
    }
  }
  ptx::named_bar_sync(1, kComputeThreads);
  for (int i = warp; i < nr; i += kComputeThreads / 32) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, sm_ml[(w * RB + i) * 2]);
    float L = 0.f, O[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) O[e] = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float sc = ptx::ex2(sm_ml[(w * RB + i) * 2] - M);
        L = fmaf(sm_ml[(w * RB + i) * 2 + 1], sc, L);
#pragma unroll
        for (int e = 0; e < EPL; ++e) O[e] = fmaf(sm_o[(w * RB + i) * D + lane * EPL + e], sc, O[e]);
      }
    }
    const GroupTok gt = p.gtoks[u.tok_off + (u.row0 + i) / p.gqa];
    // warp-uniform: the abort flag is read once per warp; filler rows of a
    // packed unit write nothing
    if (__shfl_sync(0xffffffffu, *sh.abort_flag == 0, 0) && gt.tok >= 0) {
      const int grow = u.row0 + i;
      const int h = u.kvh * p.gqa + grow % p.gqa;
      const float inv = L > 0.f ? 1.f / L : 0.f;
      const float lse2 = L > 0.f ? M + __log2f(L) : -INFINITY;
      if (gt.pbase < 0) {
        float* dst = p.out + ((size_t)gt.tok * p.hq + h) * D;
        if (lane == 0 && p.lse) p.lse[(size_t)gt.tok * p.hq + h] = lse2 * kLn2;
#pragma unroll
        for (int e = 0; e < EPL; ++e) dst[lane * EPL + e] = O[e] * inv;
      } else {
        const size_t ps = (size_t)(gt.pbase + u.chunk) * p.hq + h;
        uint32_t* dst = reinterpret_cast<uint32_t*>(p.part_o + ps * D + lane * EPL);
        float am = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) am = fmaxf(am, fabsf(O[e] * inv));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
        const float s_o = ptx::partial_scale(am, kPartialRescaleAt);
        const float inv_s = inv / s_o;
        if (lane == 0) p.part_ml[ps] = make_float2(lse2, s_o);
#pragma unroll
        for (int e = 0; e < EPL; e += 2) dst[e / 2] = ptx::pack_f16(O[e] * inv_s, O[e + 1] * inv_s);
      }
      if (gt.pbase >= 0 && p.merge_fused) merge_row_warp<D>(p, gt, h, lane);
    }
  }
  ptx::named_bar_sync(1, kComputeThreads);
}

// Next unit (list index >= k) that runs on tensor cores and has KV; -1 if none.
__device__ __forceinline__ int next_mma_unit(const AttnParams& p, int k, int u1) {
  for (; k < u1; ++k) {
    const UnitDesc u = p.units[k];
    if ((u.path & kPathMma) && u.blk1 > u.blk0) return k;
  }
  return -1;
}

// q head of row `row` (= row0 + tile row) of a unit; in a unit packed by kv
// head, 32-row slot k belongs to kv head kvh + k, in a pair unit 64-row slot k.
__device__ __forceinline__ int unit_head(const AttnParams& p, const UnitDesc& u, int row) {
  const int slot = (u.path & kUnitHeads) ? row / kPackMmaRows : (u.path & kUnitPairs) ? row / kPairRows : 0;
  return (u.kvh + slot) * p.gqa + row % p.gqa;
}

// Row tid of unit k's query tile: its record (token, visible end, partial
// slot; token -1 past the unit's rows and for filler rows of a packed unit)
// and the start of its query row.  Looked up a unit ahead: the tables are
// usually out of L2 by then.
struct QRow {
  GroupTok gt;
  const uint16_t* src;
};
template <int D>
__device__ __forceinline__ QRow q_row(const AttnParams& p, int k, int tid) {
  const UnitDesc u = p.units[k];
  QRow r{GroupTok{-1, 0, -1, 0}, p.q};
  if (tid < u.nrows) r.gt = p.gtoks[u.tok_off + (u.row0 + tid) / p.gqa];
  if (r.gt.tok >= 0) {
    const int h = unit_head(p, u, u.row0 + tid);
    r.src = p.q + ((size_t)r.gt.tok * p.hq + h) * D;
  }
  return r;
}

// Start copying the query rows into the swizzled buffer at qb (zeros for a
// row without a token; thread tid looked up row tid).  Each warp copies its
// own 32 rows a few at a time: lane l takes 16-byte chunk l % (d / 8) of
// row l / (d / 8) of the group, so one instruction reads whole 256-byte rows
// (d = 128: two rows) instead of one chunk of 32 scattered rows.
// Completion: cp_async_mbar_arrive_noinc() on the buffer's barrier.
template <int D>
__device__ __forceinline__ void load_q(const QRow& r, uint32_t qb, int tid) {
  constexpr int kChunks = D / 8;          // 16-byte chunks per row
  constexpr int kRows = 32 / kChunks;     // rows per instruction
  const int lane = tid & 31, c = lane % kChunks;
  const unsigned long long src = reinterpret_cast<unsigned long long>(r.src);
  const int has = r.gt.tok >= 0;
#pragma unroll
  for (int k = 0; k < 32 / kRows; ++k) {
    const int rr = k * kRows + lane / kChunks;  // row within the warp's 32
    const unsigned long long s = __shfl_sync(0xffffffffu, src, rr);
    const int h = __shfl_sync(0xffffffffu, has, rr);
    ptx::cp_async16(qb + (c >> 3) * (128 * 128) + sw128((tid & ~31) + rr, c & 7),
                    reinterpret_cast<const uint16_t*>(s) + c * 8, h ? 16u : 0u);
  }
  ptx::cp_async_commit();
}

// Write columns [c0, c0 + N) of row `grow`'s result, normalised O times
// `inv`, to the output (fp32, and its lse when with_lse) or to its partial
// slot (fp16).  For a partial row, amax accumulates the largest |O| written,
// so that the caller can tell when fp16 overflowed.
template <int D, int N>
__device__ __forceinline__ void write_row_cols(const AttnParams& p, const UnitDesc& u, int grow,
                                               const GroupTok& gt, const float* o, int c0, float inv,
                                               float lse2, bool with_lse, float& amax) {
  const int h = unit_head(p, u, grow);
  if (gt.pbase < 0) {
    float* dst = p.out + ((size_t)gt.tok * p.hq + h) * D;
    if (with_lse && p.lse) p.lse[(size_t)gt.tok * p.hq + h] = lse2 * kLn2;
    // 32-byte stores: one per sector
#pragma unroll
    for (int c = 0; c < N; c += 8)
      ptx::st_global_v8(dst + c0 + c, __float_as_uint(o[c] * inv), __float_as_uint(o[c + 1] * inv),
                        __float_as_uint(o[c + 2] * inv), __float_as_uint(o[c + 3] * inv),
                        __float_as_uint(o[c + 4] * inv), __float_as_uint(o[c + 5] * inv),
                        __float_as_uint(o[c + 6] * inv), __float_as_uint(o[c + 7] * inv));
  } else {
    const size_t slot = (size_t)(gt.pbase + u.chunk) * p.hq + h;
    uint16_t* dst = p.part_o + slot * D;
#pragma unroll
    for (int c = 0; c < N; c += 2) amax = ptx::max3(amax, fabsf(o[c]), fabsf(o[c + 1]));
#pragma unroll
    for (int c = 0; c < N; c += 16)
      ptx::st_global_v8(dst + c0 + c, ptx::pack_f16(o[c] * inv, o[c + 1] * inv),
                        ptx::pack_f16(o[c + 2] * inv, o[c + 3] * inv),
                        ptx::pack_f16(o[c + 4] * inv, o[c + 5] * inv),
                        ptx::pack_f16(o[c + 6] * inv, o[c + 7] * inv),
                        ptx::pack_f16(o[c + 8] * inv, o[c + 9] * inv),
                        ptx::pack_f16(o[c + 10] * inv, o[c + 11] * inv),
                        ptx::pack_f16(o[c + 12] * inv, o[c + 13] * inv),
                        ptx::pack_f16(o[c + 14] * inv, o[c + 15] * inv));
  }
}

// A partial row whose normalised O reached kPartialRescaleAt is written again
// from TMEM (O is still there) divided by its scale s, which the caller
// stores beside the lse.  Called by the whole warp (the TMEM loads are
// warp-wide); only rows with `mine` write.  Rare: kept out of line.
template <int D>
__device__ __noinline__ void rewrite_scaled_partial(const AttnParams& p, const UnitDesc& u, int grow,
                                                    const GroupTok& gt, uint32_t o_tmem, float inv_s,
                                                    bool mine) {
#pragma unroll 1
  for (int c = 0; c < D; c += 32) {
    float o[32];
    ptx::tmem_ld32(o_tmem + c, o);
    ptx::tmem_wait_ld();
    if (mine) {
      const int h = unit_head(p, u, grow);
      uint16_t* dst = p.part_o + ((size_t)(gt.pbase + u.chunk) * p.hq + h) * D;
#pragma unroll
      for (int e = 0; e < 32; e += 8)
        *reinterpret_cast<uint4*>(dst + c + e) = make_uint4(
            ptx::pack_f16(o[e] * inv_s, o[e + 1] * inv_s), ptx::pack_f16(o[e + 2] * inv_s, o[e + 3] * inv_s),
            ptx::pack_f16(o[e + 4] * inv_s, o[e + 5] * inv_s), ptx::pack_f16(o[e + 6] * inv_s, o[e + 7] * inv_s));
    }
  }
}

// One online-softmax step over N scores of this row (the ones it may not see
// already -inf): the running max m_run is raised (to m_new, with the factor
// alpha for what was summed before) only when the tile's max exceeds it by
// more than 2^kRescaleLog2; P goes to pk as N / 2 bf16 pairs and the tile's
// row sum of exponentials is returned (exact, in fp32).
template <int N>
__device__ __forceinline__ float softmax_step(const float (&sv)[N], float scale_log2, bool wact,
                                              float m_run, float& m_new, float& alpha,
                                              uint32_t* pk) {
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int c = 0; c < N; c += 2) m4[(c >> 1) & 3] = ptx::max3(m4[(c >> 1) & 3], sv[c], sv[c + 1]);
  const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * scale_log2;
  if (wact && mx > m_run + kRescaleLog2) {
    m_new = mx;
    alpha = ptx::ex2(m_run - m_new);
  }
  if (!wact) return 0.f;
  // a row that has seen no key yet has only -inf scores here: any finite
  // offset keeps their exponentials at 0 (and not NaN)
  const float nm = m_new == -INFINITY ? 0.f : -m_new;
  const uint64_t sc2 = ptx::f2(scale_log2, scale_log2), nm2 = ptx::f2(nm, nm);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};  // (0.f, 0.f) pairs
#pragma unroll
  for (int c = 0; c < N; c += 2) {
    float xa, xb;
    ptx::f2_split(ptx::fma_f32x2(ptx::f2(sv[c], sv[c + 1]), sc2, nm2), xa, xb);
    const float a = ptx::ex2(xa), b = ptx::ex2(xb);
    pk[c >> 1] = ptx::pack_bf16(a, b);
    acc[(c >> 1) & 3] = ptx::add_f32x2(acc[(c >> 1) & 3], ptx::f2(a, b));
  }
  float e8[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) ptx::f2_split(acc[k], e8[2 * k], e8[2 * k + 1]);
  return ((e8[0] + e8[1]) + (e8[2] + e8[3])) + ((e8[4] + e8[5]) + (e8[6] + e8[7]));
}

// O *= alpha for this thread's row (a lazy rescale: rare, so out of line,
// which keeps the tile loop short)
template <int D>
__device__ __noinline__ void rescale_o(uint32_t o_tmem, float alpha) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    float t32[32];
    ptx::tmem_ld32(o_tmem + c * 32, t32);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) t32[e] *= alpha;
    ptx::tmem_st32(o_tmem + c * 32, t32);
  }
  ptx::tmem_wait_st();
}

// A unit whose span holds no page: each of its rows gets out = 0 and
// lse = -inf (or that partial).  Rare, so out of line.
template <int D>
__device__ __noinline__ void empty_unit(const AttnParams& p, const UnitDesc& u, const Shared& sh) {
  const int tid = threadIdx.x;
  const GroupTok gt = tid < u.nrows ? p.gtoks[u.tok_off + (u.row0 + tid) / p.gqa]
                                    : GroupTok{-1, 0, -1, 0};
  if (gt.tok < 0 || *sh.abort_flag) return;
  const int h = unit_head(p, u, u.row0 + tid);
  if (gt.pbase < 0) {
    float* dst = p.out + ((size_t)gt.tok * p.hq + h) * D;
    if (p.lse) p.lse[(size_t)gt.tok * p.hq + h] = -INFINITY;
    for (int c = 0; c < D; c += 4)
      *reinterpret_cast<float4*>(dst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
  } else {
    const size_t slot = (size_t)(gt.pbase + u.chunk) * p.hq + h;
    uint16_t* dst = p.part_o + slot * D;
    p.part_ml[slot] = make_float2(-INFINITY, 1.f);
    for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(dst + c) = make_uint4(0, 0, 0, 0);
    if (p.merge_fused) merge_row_thread<D>(p, gt, h);
  }
}

// The four compute warps: thread i owns TMEM lane / query row i.
template <int D>
__device__ void compute_warps(const AttnParams& p, int u0, int u1, const Shared& sh,
                              const Bars<D>& B, uint32_t tmem) {
  using C = Cfg<D>;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t qbuf = sh.base + C::kOffQ;
  const uint32_t o_tmem = tmem + lane_base + 128;
  uint32_t g = 0, gm = 0, nu = 0;
  GroupTok gt_next{-1, 0, -1, 0};  // this thread's row in the next tensor-core unit
  {
    const int first = next_mma_unit(p, u0, u1);
    if (first >= 0) {
      const QRow r = q_row<D>(p, first, tid);
      load_q<D>(r, qbuf, tid);
      gt_next = r.gt;
      ptx::cp_async_mbar_arrive_noinc(B.q_full(0));
    }
  }
  UnitDesc un = u0 < u1 ? p.units[u0] : UnitDesc{};
  for (int ui = u0; ui < u1; ++ui) {
    const UnitDesc u = un;
    if (ui + 1 < u1) un = p.units[ui + 1];
    const int T = unit_tiles(u);
    if (T == 0) {  // empty span: every row sees nothing
      empty_unit<D>(p, u, sh);
      continue;
    }
    if (!(u.path & kPathMma)) {
      simt_unit<D>(p, u, g, T, sh, B);
      g += T;
      continue;
    }
    const GroupTok gt_row = gt_next;
    const int vis = gt_row.vis;
    const int nxt = next_mma_unit(p, ui + 1, u1);
    const QRow q_next = nxt >= 0 ? q_row<D>(p, nxt, tid) : QRow{GroupTok{-1, 0, -1, 0}, p.q};
    const bool row_ok = tid < u.nrows && gt_row.tok >= 0;
    const bool wact = warp * 32 < u.nrows;  // warps of padding rows keep the barriers only
    const bool packed = gt_row.slot() >= 0;  // warp w holds slot w's rows (same in a warp)
    float m_run = -INFINITY, l_run = 0.f;
    // the tiles' page records (span position * 32 + valid slots), each
    // loaded one tile ahead; packed tiles always hold kBpt pages
    int mt[kBpt], mt_p;
    auto load_records = [&](int jt) {
      const int nbt = min(kBpt, u.blk1 - (u.blk0 + kBpt * jt));
      const int2* blk = p.blocks + u.blk0 + kBpt * jt;
#pragma unroll
      for (int bb = 0; bb < kBpt; ++bb) mt[bb] = bb < nbt ? __ldg(&blk[bb].y) : 16;
      mt_p = packed ? __ldg(&blk[warp].y) : 0;
    };
    load_records(0);
    // The tile loop in three forms, each compiled on its own so that the
    // loop a unit runs holds only its own: 0 a plain tile (64 columns per
    // row), 1 a packed unit (a warp's 16 columns), 2 a pair unit (warps 2k,
    // 2k + 1 hold kv head kvh + k and see S columns [32k, 32k + 32), pages
    // 2k and 2k + 1 of every tile).
    auto tile_loop = [&](auto form_c) {
      constexpr int kForm = decltype(form_c)::value;
      constexpr bool kPacked = kForm == 1;
      for (int j = 0; j < T; ++j) {
        const int sb = (gm + j) & 1;
        const int nb = min(kBpt, u.blk1 - (u.blk0 + kBpt * j));
        // Visible columns of this row in each page of the tile (decoded while
        // QK^T may still run).  In a packed unit warp w is slot w and sees
        // only page w of every tile.
        int lim[kBpt];
        bool full = nb == kBpt;
#pragma unroll
        for (int bb = 0; bb < kBpt; ++bb) {
          lim[bb] = 0;
          if (bb < nb) {
            if (row_ok && !kPacked) lim[bb] = max(0, min(mt[bb] & 31, vis - (mt[bb] >> 5)));
          }
          full = full && (!row_ok || lim[bb] == 16);
        }
        // in a unit packed in two phases a row sees only its phase's tiles
        // (phase 0 in lanes 0-15, phase 1 in lanes 16-31 of each slot)
        const bool my_phase =
            !(u.path & kUnitPhases) || ((mt_p >> kPhaseShift) & 1) == ((tid & 31) >> 4);
        const int lim_p = kPacked && row_ok && my_phase
                              ? max(0, min(mt_p & 31, vis - ((mt_p & kPosMask) >> 5)))
                              : 0;
        if (j + 1 < T) load_records(j + 1);
        bool ok = wait_bar(B.s_full(sb), ((gm + j) >> 1) & 1, sh, p.err, p.wait_timeout_ns);
        ok = __all_sync(0xffffffffu, ok);
        ptx::tc_fence_after();
        float m_new = m_run, alpha = 1.f, lsum = 0.f;
        uint32_t pk[kTileTok / 2];
        // P rounds to bf16 for the tensor cores; the row sum is kept exact in
        // fp32 and normalises both O and the lse.
        if constexpr (kPacked) {
          float sv[16];
          if (ok && wact) {
            ptx::tmem_ld16(tmem + lane_base + sb * kTileTok + warp * 16, sv);
            ptx::tmem_wait_ld();
          } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) sv[c] = 0.f;
          }
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < 16; ++c) m4[c & 3] = fmaxf(m4[c & 3], c < lim_p ? sv[c] : -INFINITY);
          const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.scale_log2;
          if (wact && mx > m_run + kRescaleLog2) {
            m_new = mx;
            alpha = ptx::ex2(m_run - m_new);
          }
          float e4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int c = 0; c < 16; c += 2) {
            const float a = ptx::ex2(c < lim_p ? fmaf(sv[c], p.scale_log2, -m_new) : -INFINITY);
            const float b = ptx::ex2(c + 1 < lim_p ? fmaf(sv[c + 1], p.scale_log2, -m_new) : -INFINITY);
            pk[c >> 1] = ptx::pack_bf16(a, b);
            e4[(c >> 1) & 3] += a + b;
          }
          lsum = (e4[0] + e4[1]) + (e4[2] + e4[3]);
        } else if constexpr (kForm == 2) {
          const int sl = warp >> 1;
          float sv[32];
          if (ok && wact) {
            ptx::tmem_ld32(tmem + lane_base + sb * kTileTok + sl * 32, sv);
            ptx::tmem_wait_ld();
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) sv[c] = 0.f;
          }
          const int l0 = sl ? lim[2] : lim[0], l1 = sl ? lim[3] : lim[1];
          if (!__all_sync(0xffffffffu, !row_ok || (l0 == 16 && l1 == 16))) {
#pragma unroll
            for (int c = 0; c < 32; ++c) sv[c] = (c & 15) < (c < 16 ? l0 : l1) ? sv[c] : -INFINITY;
          }
          lsum = softmax_step<32>(sv, p.scale_log2, wact, m_run, m_new, alpha, pk);
        } else {
          float sv[kTileTok];
          if (ok && wact) {
#pragma unroll
            for (int c = 0; c < kTileTok / 32; ++c) {
              float t32[32];
              ptx::tmem_ld32(tmem + lane_base + sb * kTileTok + c * 32, t32);
#pragma unroll
              for (int e = 0; e < 32; ++e) sv[c * 32 + e] = t32[e];
            }
            ptx::tmem_wait_ld();
          } else {
#pragma unroll
            for (int c = 0; c < kTileTok; ++c) sv[c] = 0.f;
          }
          // Scores this row may not see become -inf (exp2 then gives exactly
          // 0); a warp whose rows all see the whole tile skips the selects.
          // One exponentiation body then serves every tile, which keeps the
          // compute warps' loop short.
          if (!__all_sync(0xffffffffu, full)) {
#pragma unroll
            for (int c = 0; c < kTileTok; ++c) sv[c] = (c & 15) < lim[c >> 4] ? sv[c] : -INFINITY;
          }
          lsum = softmax_step<kTileTok>(sv, p.scale_log2, wact, m_run, m_new, alpha, pk);
        }
        l_run = fmaf(l_run, alpha, lsum);
        m_run = m_new;
        // a rescale of O waits until O holds the previous tile's P.V
        if (ok && wact && j > 0 && __any_sync(0xffffffffu, alpha != 1.f) &&
            __all_sync(0xffffffffu, wait_bar(B.pv_done((gm + j - 1) & 1), ((gm + j - 1) >> 1) & 1, sh,
                                             p.err, p.wait_timeout_ns))) {
          ptx::tc_fence_after();
          rescale_o<D>(o_tmem, alpha);
        }
        // P (bf16 pairs, 32 columns) replaces S in the first half of its TMEM
        // buffer; the S values were read above
        if (ok && wact) {
          const uint32_t pt = tmem + lane_base + sb * kTileTok;
          if constexpr (kPacked) {
            // this warp's page is P columns [8w, 8w + 8); the rest is zero
            uint32_t pw[kTileTok / 2];
#pragma unroll
            for (int c = 0; c < kTileTok / 2; ++c) pw[c] = (c >> 3) == warp ? pk[c & 7] : 0u;
            ptx::tmem_st32u(pt, pw);
          } else if constexpr (kForm == 2) {
            // this slot's pages are P columns [16k, 16k + 16); the rest is zero
            const int sl = warp >> 1;
            uint32_t pw[kTileTok / 2];
#pragma unroll
            for (int c = 0; c < kTileTok / 2; ++c) pw[c] = (c >> 4) == sl ? pk[c & 15] : 0u;
            ptx::tmem_st32u(pt, pw);
          } else {
            ptx::tmem_st32u(pt, pk);
          }
          ptx::tmem_wait_st();
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(B.p_full(sb));
      }
    };
    if (u.path & kUnitPairs)
      tile_loop(std::integral_constant<int, 2>{});
    else if (packed)
      tile_loop(std::integral_constant<int, 1>{});
    else
      tile_loop(std::integral_constant<int, 0>{});
    // Every QK^T of this unit has completed (its last S was ready): the
    // query buffer is free.  The next unit's query tile streams in while
    // the last P.V runs; its copies arrive on q_full by themselves, so the
    // compute warps go straight on to the epilogue and the next unit's first
    // QK^T overlaps it.
    if (nxt >= 0) {
      load_q<D>(q_next, qbuf, tid);
      gt_next = q_next.gt;
      ptx::cp_async_mbar_arrive_noinc(B.q_full(0));
    }
    // ---- epilogue: O / l, 32 columns at a time; then O is free again
    bool ok = wait_bar(B.o_full(), nu & 1, sh, p.err, p.wait_timeout_ns);
    ok = __all_sync(0xffffffffu, ok);
    ptx::tc_fence_after();
    if (ok && wact) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const float lse2 = l_run > 0.f ? m_run + __log2f(l_run) : -INFINITY;
      const bool wr = row_ok && !*sh.abort_flag;
      float amax = 0.f;
      // O in 64-column halves: one TMEM round trip per half
#pragma unroll
      for (int c = 0; c < D / 32; c += 2) {
        float o0[32], o1[32];
        ptx::tmem_ld32(o_tmem + c * 32, o0);
        ptx::tmem_ld32(o_tmem + c * 32 + 32, o1);
        ptx::tmem_wait_ld();
        if (wr) {
          write_row_cols<D, 32>(p, u, u.row0 + tid, gt_row, o0, c * 32, inv, lse2, c == 0, amax);
          write_row_cols<D, 32>(p, u, u.row0 + tid, gt_row, o1, c * 32 + 32, inv, lse2, false, amax);
        }
      }
      // a partial row out of fp16's range is stored again, divided by s
      const bool part = wr && gt_row.pbase >= 0;
      const float s_o = part ? ptx::partial_scale(amax * inv, kPartialRescaleAt) : 1.f;
      if (__any_sync(0xffffffffu, s_o != 1.f))
        rewrite_scaled_partial<D>(p, u, u.row0 + tid, gt_row, o_tmem, inv / s_o, s_o != 1.f);
      if (part)
        p.part_ml[(size_t)(gt_row.pbase + u.chunk) * p.hq + unit_head(p, u, u.row0 + tid)] =
            make_float2(lse2, s_o);
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(B.o_empty());  // O is free before the (rare, slow) merge
    if (ok && row_ok && gt_row.pbase >= 0 && p.merge_fused && !*sh.abort_flag)
      merge_row_thread<D>(p, gt_row, unit_head(p, u, u.row0 + tid));
    g += T;
    gm += T;
    ++nu;
  }
  ptx::cp_async_wait_all();  // no copy of this thread is in flight when the CTA ends
}

template <int D, bool kEvict>
__global__ void __launch_bounds__(kThreads, 2)
    tree_attn_kernel(const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, const AttnParams p) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Shared sh;
  sh.base = ptx::smem_u32(smem_raw);
  sh.ptr = smem_raw;
  if (sh.base & 1023) {  // the swizzled layouts need a 1024-byte aligned window
    if (threadIdx.x == 0) atomicCAS(p.err, 0, TA_DEVERR_BOUNDS);
    return;
  }
  Bars<D> B{sh.base + C::kOffBar};
  sh.tmem_slot = reinterpret_cast<volatile uint32_t*>(sh.ptr + C::kOffBar + C::kNumBars * 8);
  sh.abort_flag = reinterpret_cast<volatile int*>(sh.ptr + C::kOffBar + C::kNumBars * 8 + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the merge kernel (a programmatic dependent) may be scheduled from now on;
  // it waits for this grid's completion before reading any partial
  asm volatile("griddepcontrol.launch_dependents;");
  const int u0 = p.cta_inline ? p.cta_off_inline[blockIdx.x] : p.cta_off[blockIdx.x];
  const int u1 = p.cta_inline ? p.cta_off_inline[blockIdx.x + 1] : p.cta_off[blockIdx.x + 1];

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(B.kfull(s), 1);
      ptx::mbar_init(B.kempty(s), 1);
      ptx::mbar_init(B.vfull(s), 1);
      ptx::mbar_init(B.vempty(s), 1);
      ptx::mbar_init(B.vland(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(B.s_full(i), 1);
      ptx::mbar_init(B.pv_done(i), 1);
      // one per S buffer: a warp may arrive for tile t + 1 before the others
      // arrive for tile t, and only tile t + 2 (same buffer) waits for P.V(t)
      ptx::mbar_init(B.p_full(i), kComputeThreads);
    }
    ptx::mbar_init(B.q_full(0), kComputeThreads);
    ptx::mbar_init(B.q_full(1), kComputeThreads);
    ptx::mbar_init(B.o_full(), 1);
    ptx::mbar_init(B.drain(), 1);
    ptx::mbar_init(B.never(), 1);  // nothing arrives here
    ptx::mbar_init(B.o_empty(), kComputeThreads);
    *sh.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    ptx::prefetch_tmap(&tmk);
    ptx::prefetch_tmap(&tmv);
  }
  // Warm L2 with this CTA's tables (unit records, their block lists and row
  // records): the roles then find them in L2 instead of DRAM.
  for (int k = u0 + (int)threadIdx.x; k < u1; k += kThreads) {
    const UnitDesc u = p.units[k];
    for (int b = u.blk0; b < u.blk1; b += 16) ptx::prefetch_l2(&p.blocks[b]);
    const int t0 = u.tok_off + u.row0 / p.gqa, t1 = u.tok_off + (u.row0 + u.nrows - 1) / p.gqa;
    for (int t = t0; t <= t1; t += 8) ptx::prefetch_l2(&p.gtoks[t]);
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(sh.base + C::kOffBar + C::kNumBars * 8, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *sh.tmem_slot;
  // This grid is launched as a programmatic dependent of the stream's
  // previous kernel (often the previous layer's merge): the set-up above
  // reads only this plan's tables, and the queries, pages, outputs and
  // partials are touched only once that grid has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp < kComputeThreads / 32) {
    ptx::setmaxnreg_inc<kComputeRegs>();
    compute_warps<D>(p, u0, u1, sh, B, tmem);
  } else {
    ptx::setmaxnreg_dec<kIssueRegs>();
    if (warp == kProducerWarp) {
      producer<D, false, kEvict>(&tmk, p, u0, u1, sh, B);
    } else if (warp == kMmaWarp) {
      mma_issuer<D>(p, u0, u1, sh, B, tmem);
    } else if (warp == kVProducerWarp) {
      producer<D, true, kEvict>(&tmv, p, u0, u1, sh, B);
    }  // warp 7 only completes the warpgroup
    __syncwarp();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Page pool [pages][hkv][16][d] bf16 as a 4-D tensor (d, slot, head, page)
// whose box is one 64-column half of a page-head; or, for whole_page_head
// with d = 128, a 5-D tensor (64 columns, slot, column half, head, page) whose
// half dimension (stride 128 B) sits outside the slot dimension (stride
// 256 B), so one box lands a whole page-head as [half][16 slots][64 columns].
// 128-byte swizzle in both cases.
cudaError_t make_page_map(CUtensorMap* m, const void* base, int d, int hkv, int num_pages,
                          bool whole_page_head) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  CUresult r;
  if (d == 128 && whole_page_head) {
    cuuint64_t dims[5] = {64, 16, 2, (cuuint64_t)hkv, (cuuint64_t)num_pages};
    cuuint64_t strides[4] = {256, 128, 4096, (cuuint64_t)hkv * 4096};
    cuuint32_t box[5] = {64, 16, 2, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[4] = {(cuuint64_t)d, 16, (cuuint64_t)hkv, (cuuint64_t)num_pages};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)16 * d * 2, (cuuint64_t)hkv * 16 * d * 2};
    cuuint32_t box[4] = {64, 16, 1, 1};  // one 64-column half of a page-head
    cuuint32_t estr[4] = {1, 1, 1, 1};
    r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, bool kEvict>
cudaError_t launch_d(const AttnParams& p, int grid, int num_pages, cudaStream_t s) {
  // The shared-memory limit is an attribute of the kernel in the current
  // device's context: set on every launch (a host-side call of a few
  // microseconds), so a second device, or a context created anew, gets it too.
  cudaError_t e = cudaFuncSetAttribute(tree_attn_kernel<D, kEvict>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmem);
  if (e != cudaSuccess) return e;
  CUtensorMap mk, mv;
  memset(&mk, 0, sizeof mk);
  memset(&mv, 0, sizeof mv);
  if (num_pages > 0) {
    e = make_page_map(&mk, p.k, D, p.hkv, num_pages, false);
    if (e != cudaSuccess) return e;
    e = make_page_map(&mv, p.v, D, p.hkv, num_pages, true);
    if (e != cudaSuccess) return e;
  }
  // a programmatic dependent launch: the CTAs may be scheduled, and run their
  // set-up, while the previous kernel in the stream finishes
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<D>::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tree_attn_kernel<D, kEvict>, mk, mv, p);
}

}  // namespace

cudaError_t launch_tree_attention(const AttnParams& p, int d, int grid, int num_pages,
                                  bool kv_evict, cudaStream_t s) {
  if (p.n_units == 0 || grid == 0) return cudaSuccess;
  if (d == 128)
    return kv_evict ? launch_d<128, true>(p, grid, num_pages, s)
                    : launch_d<128, false>(p, grid, num_pages, s);
  return kv_evict ? launch_d<64, true>(p, grid, num_pages, s) : launch_d<64, false>(p, grid, num_pages, s);
}

}  // namespace ta
