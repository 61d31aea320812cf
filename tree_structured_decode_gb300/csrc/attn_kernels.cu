// Log-sum-exp merge kernel (sm_103a).
//
// merge pass: per (query token, q head), fold its partials (O_i stored in
// fp16 as O_i / s_i, with lse_i and s_i in fp32):
//   m = max lse_i, w_i = 2^(lse_i - m), O = sum w_i s_i (O_i / s_i) / sum w_i,
//   lse = m + log2 sum w_i   (partials keep lse in base 2).
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace ta {
namespace {

constexpr float kLn2 = 0.69314718055994530942f;

// RPW (merge token, q head) rows per warp (two, or one for tokens with many
// partials): a lane holds D * RPW / 32 columns (one 16- or 8-byte fp16 load
// per partial row).  The partials
// are read G at a time (lse and the lane's columns of G partial rows in
// flight together, kept as packed fp16 until folded) and folded online: the
// running max M only grows, and the sums kept so far are scaled by
// 2^(M_old - M_new) when it does.  The launch picks G from the plan's
// largest partial count (4, 8 or 24) so that a token takes one round of
// loads where possible, with as few registers as that allows.
template <int D, int G, int kMinBlocks, int RPW = 2>
__global__ void __launch_bounds__(256, kMinBlocks) lse_merge_kernel(const MergeParams p) {
  constexpr int LPR = 32 / RPW;  // lanes per row
  constexpr int EPL = D / LPR;   // columns per lane
  constexpr int NW = EPL / 2;    // fp16 pairs per lane
  static_assert(EPL == 4 || EPL == 8, "a lane holds 4 or 8 columns");
  const int lane = threadIdx.x & 31, sub = lane / LPR, l16 = lane % LPR;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int total = p.n_items * p.hq;
  // The merge items are plan tables, in place before the partial-attention
  // kernel started: this warp's first one is read before the dependency wait.
  MergeItem it_first = {};
  if (RPW * gw + sub < total) it_first = p.items[(RPW * gw + sub) / p.hq];
  // launched as a programmatic dependent of the partial-attention kernel:
  // wait here until that grid has completed and its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // a small merge lets the stream's next kernel (a programmatic dependent, as
  // the next partial-attention kernel is) be scheduled while it folds; a
  // large one keeps the SMs to itself
  if (p.early_trigger) asm volatile("griddepcontrol.launch_dependents;");
  for (int r0 = RPW * gw; r0 < total; r0 += RPW * nw) {
    const int idx = r0 + sub;
    if (idx >= total) continue;
    const MergeItem it = r0 == RPW * gw ? it_first : p.items[idx / p.hq];
    const int h = idx % p.hq;
    const float2* ml_h = p.part_ml + (size_t)it.poff * p.hq + h;  // partial k at ml_h[k * hq]
    const uint16_t* o_h = p.part_o + ((size_t)it.poff * p.hq + h) * D + l16 * EPL;  // fp16
    float M = -INFINITY, den = 0.f, acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    for (int k0 = 0; k0 < it.count; k0 += G) {
      float w[G], osc[G];
      uint32_t v[G][NW];
#pragma unroll
      for (int q = 0; q < G; ++q) {
        const int k = k0 + q;
        w[q] = -INFINITY;
        osc[q] = 1.f;
#pragma unroll
        for (int e = 0; e < NW; ++e) v[q][e] = 0u;
        if (k < it.count) {
          const float2 ml = __ldcg(ml_h + (size_t)k * p.hq);
          w[q] = ml.x;
          osc[q] = ml.y;
          const uint16_t* src = o_h + (size_t)k * p.hq * D;
          if constexpr (NW == 4) {
            const uint4 t = __ldcg(reinterpret_cast<const uint4*>(src));
            v[q][0] = t.x, v[q][1] = t.y, v[q][2] = t.z, v[q][3] = t.w;
          } else {
            const uint2 t = __ldcg(reinterpret_cast<const uint2*>(src));
            v[q][0] = t.x, v[q][1] = t.y;
          }
        }
      }
      float mr = w[0];
#pragma unroll
      for (int q = 1; q < G; ++q) mr = fmaxf(mr, w[q]);
      const float m_new = fmaxf(M, mr);
      if (m_new == -INFINITY) continue;  // nothing visible so far
      const float sc = ptx::ex2(M - m_new);  // 0 while M is still -inf
      den *= sc;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] *= sc;
#pragma unroll
      for (int q = 0; q < G; ++q) {
        const float wq = ptx::ex2(w[q] - m_new);  // 0 for absent or empty partials
        den += wq;
        const float wo = wq * osc[q];
#pragma unroll
        for (int e = 0; e < NW; ++e) {
          const float2 f = ptx::unpack_f16(v[q][e]);
          acc[2 * e] = fmaf(wo, f.x, acc[2 * e]);
          acc[2 * e + 1] = fmaf(wo, f.y, acc[2 * e + 1]);
        }
      }
      M = m_new;
    }
    const float inv = den > 0.f ? __frcp_rn(den) : 0.f;
    float* dst = p.out + ((size_t)it.tok * p.hq + h) * D + l16 * EPL;
#pragma unroll
    for (int e = 0; e < EPL; e += 4)
      *reinterpret_cast<float4*>(dst + e) = make_float4(acc[e] * inv, acc[e + 1] * inv, acc[e + 2] * inv, acc[e + 3] * inv);
    if (l16 == 0 && p.lse)
      p.lse[(size_t)it.tok * p.hq + h] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
  }
}

// Tokens with at most G partials (one round of loads per row), software-
// pipelined: a warp issues the loads of its next row before it folds the
// current one, and the merge item of the row after that is read one row
// further ahead, so that more loads are in flight per register.
template <int D, int G, int kMinBlocks, int RPW = 2>
__global__ void __launch_bounds__(256, kMinBlocks) lse_merge_pipelined_kernel(const MergeParams p) {
  constexpr int LPR = 32 / RPW;
  constexpr int EPL = D / LPR;
  constexpr int NW = EPL / 2;
  static_assert(EPL == 4 || EPL == 8, "a lane holds 4 or 8 columns");
  const int lane = threadIdx.x & 31, sub = lane / LPR, l16 = lane % LPR;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int hq = p.hq;
  // rows (item, q head) = divmod(RPW * gw + sub + k * stride, hq), k = 0, 1, ...:
  // one division here, then an add and a carry per row
  const int stride = RPW * nw;
  const int s_item = stride / hq, s_h = stride % hq;
  auto advance = [&](int& item, int& h) {
    h += s_h;
    item += s_item;
    if (h >= hq) {
      h -= hq;
      ++item;
    }
  };
  int item0 = (RPW * gw + sub) / hq, h0 = (RPW * gw + sub) % hq;  // this row
  int item1 = item0, h1 = h0;
  advance(item1, h1);  // the next
  int item2 = item1, h2 = h1;
  advance(item2, h2);  // the one after
  // plan tables, in place before the partial-attention kernel started
  MergeItem it = {}, it_next = {};
  if (item0 < p.n_items) it = p.items[item0];
  if (item1 < p.n_items) it_next = p.items[item1];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // a small merge lets the stream's next kernel (a programmatic dependent, as
  // the next partial-attention kernel is) be scheduled while it folds; a
  // large one keeps the SMs to itself
  if (p.early_trigger) asm volatile("griddepcontrol.launch_dependents;");
  auto load = [&](int item, int h, const MergeItem& m, float (&wq)[G], float (&oq)[G],
                  uint32_t (&vq)[G][NW]) {
    const float2* ml_h = p.part_ml + (size_t)m.poff * hq + h;
    const uint16_t* o_h = p.part_o + ((size_t)m.poff * hq + h) * D + l16 * EPL;
#pragma unroll
    for (int q = 0; q < G; ++q) {
      wq[q] = -INFINITY;
      oq[q] = 1.f;
#pragma unroll
      for (int e = 0; e < NW; ++e) vq[q][e] = 0u;
      if (item < p.n_items && q < m.count) {
        const float2 ml = __ldcg(ml_h + (size_t)q * hq);
        wq[q] = ml.x;
        oq[q] = ml.y;
        const uint16_t* src = o_h + (size_t)q * hq * D;
        if constexpr (NW == 4) {
          const uint4 t = __ldcg(reinterpret_cast<const uint4*>(src));
          vq[q][0] = t.x, vq[q][1] = t.y, vq[q][2] = t.z, vq[q][3] = t.w;
        } else {
          const uint2 t = __ldcg(reinterpret_cast<const uint2*>(src));
          vq[q][0] = t.x, vq[q][1] = t.y;
        }
      }
    }
  };
  float w[G], osc[G];
  uint32_t v[G][NW];
  load(item0, h0, it, w, osc, v);
  while (item0 < p.n_items) {
    // the next row's partials, and the item of the row after it
    float w2[G], osc2[G];
    uint32_t v2[G][NW];
    load(item1, h1, it_next, w2, osc2, v2);
    MergeItem it_after = {};
    if (item2 < p.n_items) it_after = p.items[item2];
    // fold this row: m = max lse_i, w_i = 2^(lse_i - m)
    float m = w[0];
#pragma unroll
    for (int q = 1; q < G; ++q) m = fmaxf(m, w[q]);
    float den = 0.f, acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    if (m != -INFINITY) {
#pragma unroll
      for (int q = 0; q < G; ++q) {
        const float wq = ptx::ex2(w[q] - m);  // 0 for absent or empty partials
        den += wq;
        const float wo = wq * osc[q];
#pragma unroll
        for (int e = 0; e < NW; ++e) {
          const float2 f = ptx::unpack_f16(v[q][e]);
          acc[2 * e] = fmaf(wo, f.x, acc[2 * e]);
          acc[2 * e + 1] = fmaf(wo, f.y, acc[2 * e + 1]);
        }
      }
    }
    const float inv = den > 0.f ? __frcp_rn(den) : 0.f;
    float* dst = p.out + ((size_t)it.tok * hq + h0) * D + l16 * EPL;
#pragma unroll
    for (int e = 0; e < EPL; e += 4)
      *reinterpret_cast<float4*>(dst + e) = make_float4(acc[e] * inv, acc[e + 1] * inv, acc[e + 2] * inv, acc[e + 3] * inv);
    if (l16 == 0 && p.lse)
      p.lse[(size_t)it.tok * hq + h0] = den > 0.f ? (m + log2f(den)) * kLn2 : -INFINITY;
    it = it_next;
    it_next = it_after;
    item0 = item1, h0 = h1;
    item1 = item2, h1 = h2;
    advance(item2, h2);
#pragma unroll
    for (int q = 0; q < G; ++q) {
      w[q] = w2[q];
      osc[q] = osc2[q];
#pragma unroll
      for (int e = 0; e < NW; ++e) v[q][e] = v2[q][e];
    }
  }
}

// One thread per 16 bytes of a (token, kv head) row of K or V: the row of
// token t, head h goes to page dst[t] / 16, slot dst[t] % 16, head h.
__global__ void __launch_bounds__(256) append_kv_kernel(const uint4* k_new, const uint4* v_new,
                                                        const int32_t* dst, int nq, int hkv,
                                                        int chunks, uint4* k_pages,
                                                        uint4* v_pages) {
  const long long per_tok = (long long)hkv * chunks;  // 16-byte chunks of one token's K (or V)
  const long long n = 2 * (long long)nq * per_tok;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const bool is_v = i >= (long long)nq * per_tok;
    const long long j = is_v ? i - (long long)nq * per_tok : i;
    const int t = (int)(j / per_tok);
    const int h = (int)((j / chunks) % hkv), c = (int)(j % chunks);
    const int where = __ldg(dst + t);
    if (where < 0) continue;
    const long long row = ((long long)(where >> 4) * hkv + h) * 16 + (where & 15);
    (is_v ? v_pages : k_pages)[row * chunks + c] = __ldg((is_v ? v_new : k_new) + j);
  }
}

}  // namespace

cudaError_t launch_append_kv(const uint16_t* k_new, const uint16_t* v_new, const int32_t* dst,
                             int nq, int hkv, int d, uint16_t* k_pages, uint16_t* v_pages,
                             cudaStream_t s) {
  if (nq == 0) return cudaSuccess;
  const int chunks = d * 2 / 16;
  const long long n = 2LL * nq * hkv * chunks;
  const int blocks = (int)((n + 255) / 256 < 152 * 8 ? (n + 255) / 256 : 152 * 8);
  append_kv_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const uint4*>(k_new),
                                          reinterpret_cast<const uint4*>(v_new), dst, nq, hkv,
                                          chunks, reinterpret_cast<uint4*>(k_pages),
                                          reinterpret_cast<uint4*>(v_pages));
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(const MergeParams& params, int d, cudaStream_t s) {
  if (params.n_items == 0) return cudaSuccess;
  MergeParams p = params;
  p.early_trigger = (int64_t)p.n_items * p.hq <= kMergeEarlyRows ? 1 : 0;
  // two rows per warp, or one (each lane then holds 4 columns) when tokens
  // have many partials: more warps share the same loads
  const int rpw = (d == 128 && p.max_count > 8) ? 1 : 2;
  const long long warps = ((long long)p.n_items * p.hq + rpw - 1) / rpw;
  const int blocks = (int)((warps + 7) / 8 < 152 * 16 ? (warps + 7) / 8 : 152 * 16);
  // A programmatic dependent launch: the merge grid may be scheduled while
  // the partial-attention kernel finishes (it waits in griddepcontrol.wait
  // for that grid's completion), so its launch latency leaves the step.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // one round of loads per token where possible; fewer partials per round
  // leave registers for more resident warps.  At d = 128, plans whose tokens
  // have at most four partials take the software-pipelined form.
  if (d == 128) {
    if (p.max_count > 8) return cudaLaunchKernelEx(&cfg, lse_merge_kernel<128, 24, 1, 1>, p);
    if (p.max_count > 4) return cudaLaunchKernelEx(&cfg, lse_merge_kernel<128, 8, 3>, p);
    if (p.max_count > 3) return cudaLaunchKernelEx(&cfg, lse_merge_pipelined_kernel<128, 4, 3>, p);
    return cudaLaunchKernelEx(&cfg, lse_merge_pipelined_kernel<128, 3, 4>, p);
  }
  if (p.max_count > 8) return cudaLaunchKernelEx(&cfg, lse_merge_kernel<64, 24, 1>, p);
  if (p.max_count > 4) return cudaLaunchKernelEx(&cfg, lse_merge_kernel<64, 8, 3>, p);
  return cudaLaunchKernelEx(&cfg, lse_merge_kernel<64, 4, 6>, p);
}

}  // namespace ta
