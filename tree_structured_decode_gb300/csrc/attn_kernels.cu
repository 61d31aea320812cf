// Log-sum-exp merge kernel (sm_103a).
//
// merge pass: per (query token, q head), fold its partials:
//   m = max lse_i, w_i = 2^(lse_i - m), O = sum w_i O_i / sum w_i,
//   lse = m + log2 sum w_i   (partials keep lse in base 2).
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace ta {
namespace {

constexpr float kLn2 = 0.69314718055994530942f;

// One warp per (merge token, q head).  Lane k reads lse of partial k (the
// common case has fewer than 32 partials), then the partials' rows are read
// four at a time so their loads are in flight together.
template <int D>
__global__ void __launch_bounds__(256) lse_merge_kernel(const MergeParams p) {
  constexpr int EPL = D / 32;  // 4 or 2 columns per lane
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int total = p.n_items * p.hq;
  for (int idx = gw; idx < total; idx += nw) {
    const MergeItem it = p.items[idx / p.hq];
    const int h = idx % p.hq;
    const float* lse_h = p.part_lse + (size_t)it.poff * p.hq + h;  // partial k at lse_h[k * hq]
    float M = -INFINITY;
    for (int k = lane; k < it.count; k += 32) M = fmaxf(M, __ldcg(lse_h + (size_t)k * p.hq));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float acc[EPL], den = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    if (M != -INFINITY) {
      const float* o_h = p.part_o + ((size_t)it.poff * p.hq + h) * D + lane * EPL;
      for (int k0 = 0; k0 < it.count; k0 += 4) {
        float w[4], v[4][EPL];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int k = k0 + q;
          w[q] = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) v[q][e] = 0.f;
          if (k < it.count) {
            w[q] = __ldcg(lse_h + (size_t)k * p.hq);
            const float* src = o_h + (size_t)k * p.hq * D;
            if constexpr (EPL == 4) {
              const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
              v[q][0] = t.x, v[q][1] = t.y, v[q][2] = t.z, v[q][3] = t.w;
            } else {
              const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
              v[q][0] = t.x, v[q][1] = t.y;
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (k0 + q < it.count) {
            const float wq = exp2f(w[q] - M);
            den += wq;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] = fmaf(wq, v[q][e], acc[e]);
          }
        }
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    float* dst = p.out + ((size_t)it.tok * p.hq + h) * D + lane * EPL;
    if constexpr (EPL == 4)
      *reinterpret_cast<float4*>(dst) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    else
      *reinterpret_cast<float2*>(dst) = make_float2(acc[0] * inv, acc[1] * inv);
    if (lane == 0 && p.lse)
      p.lse[(size_t)it.tok * p.hq + h] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_lse_merge(const MergeParams& p, int d, cudaStream_t s) {
  if (p.n_items == 0) return cudaSuccess;
  const long long warps = (long long)p.n_items * p.hq;
  const int blocks = (int)((warps + 7) / 8 < 152 * 16 ? (warps + 7) / 8 : 152 * 16);
  if (d == 128)
    lse_merge_kernel<128><<<blocks, 256, 0, s>>>(p);
  else
    lse_merge_kernel<64><<<blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace ta
