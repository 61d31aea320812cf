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

// One warp per (merge token, q head).
template <int D>
__global__ void __launch_bounds__(256) lse_merge_kernel(const MergeParams p) {
  constexpr int EPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int total = p.n_items * p.hq;
  for (int idx = gw; idx < total; idx += nw) {
    const MergeItem it = p.items[idx / p.hq];
    const int h = idx % p.hq;
    float M = -INFINITY;
    for (int k = 0; k < it.count; ++k)
      M = fmaxf(M, p.part_lse[(size_t)(it.poff + k) * p.hq + h]);
    float acc[EPL], den = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    if (M != -INFINITY) {
      for (int k = 0; k < it.count; ++k) {
        const size_t slot = (size_t)(it.poff + k) * p.hq + h;
        const float w = exp2f(p.part_lse[slot] - M);
        den += w;
        const float* src = p.part_o + slot * D + lane * EPL;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = fmaf(w, src[e], acc[e]);
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    float* dst = p.out + ((size_t)it.tok * p.hq + h) * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) dst[e] = acc[e] * inv;
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
