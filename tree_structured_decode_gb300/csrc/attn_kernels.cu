// Partial attention and log-sum-exp merge kernels (sm_103a).
//
// partial pass: every work unit (group, kv head, query tile, chunk) computes,
// for each of its query rows, attention over the chunk's KV with an online
// softmax, and writes either the final output (a row with one partial) or a
// normalised partial O plus its log-sum-exp (DeFT notes page, "Attention
// Calculation" and "Tree-Topology-Aware Global Reduction Strategy": one
// thread block per QKV group, flash-attention style, partials mapped back to
// their queries and reduced globally).
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

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// EPL = D/32 consecutive bf16 elements -> float.
template <int D>
__device__ __forceinline__ void load_row_slice(const uint16_t* ptr, float (&f)[D / 32]) {
  if constexpr (D == 128) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(ptr));
    f[0] = bf16_lo(u.x);
    f[1] = bf16_hi(u.x);
    f[2] = bf16_lo(u.y);
    f[3] = bf16_hi(u.y);
  } else {
    const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(ptr));
    f[0] = bf16_lo(u);
    f[1] = bf16_hi(u);
  }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// CUDA-core unit kernel: one CTA (4 warps) per unit.  Warps take the chunk's
// 16-token blocks round-robin; lanes split the head dimension; each warp
// keeps an online-softmax state per row; the four states are combined at the
// end of each batch of up to 8 rows.
template <int D>
__global__ void __launch_bounds__(128) simt_unit_kernel(const AttnParams p) {
  constexpr int EPL = D / 32;
  constexpr int RB = kSimtTileRows;
  __shared__ float sm_m[4][RB], sm_l[4][RB];
  __shared__ float sm_o[4][RB][D];

  const UnitDesc u = p.units[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int rb = 0; rb < u.nrows; rb += RB) {
    const int nr = min(RB, u.nrows - rb);
    float qv[RB][EPL], o[RB][EPL], m[RB], l[RB];
    int vis[RB];
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      m[i] = -INFINITY;
      l[i] = 0.f;
      vis[i] = 0;
#pragma unroll
      for (int e = 0; e < EPL; ++e) o[i][e] = qv[i][e] = 0.f;
      if (i < nr) {
        const int row = u.row0 + rb + i;
        const GroupTok gt = p.gtoks[u.tok_off + row / p.gqa];
        const int h = u.kvh * p.gqa + row % p.gqa;
        vis[i] = gt.vis;
        load_row_slice<D>(p.q + ((size_t)gt.tok * p.hq + h) * D + lane * EPL, qv[i]);
#pragma unroll
        for (int e = 0; e < EPL; ++e) qv[i][e] *= p.scale_log2;
      }
    }
    for (int b = u.blk0 + warp; b < u.blk1; b += 4) {
      const int2 bl = p.blocks[b];
      const int pos = bl.y >> 5, nvalid = bl.y & 31;
      const size_t base = ((size_t)bl.x * p.hkv + u.kvh) * 16 * D + lane * EPL;
      for (int s = 0; s < nvalid; ++s) {
        float kf[EPL], vf[EPL];
        load_row_slice<D>(p.k + base + (size_t)s * D, kf);
        load_row_slice<D>(p.v + base + (size_t)s * D, vf);
#pragma unroll
        for (int i = 0; i < RB; ++i) {
          if (i < nr && pos + s < vis[i]) {  // warp-uniform
            float dot = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) dot = fmaf(qv[i][e], kf[e], dot);
            dot = warp_sum(dot);
            const float mn = fmaxf(m[i], dot);
            const float alpha = exp2f(m[i] - mn);
            const float pr = exp2f(dot - mn);
            l[i] = fmaf(l[i], alpha, pr);
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[i][e] = fmaf(o[i][e], alpha, pr * vf[e]);
            m[i] = mn;
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      if (lane == 0) {
        sm_m[warp][i] = m[i];
        sm_l[warp][i] = l[i];
      }
#pragma unroll
      for (int e = 0; e < EPL; ++e) sm_o[warp][i][lane * EPL + e] = o[i][e];
    }
    __syncthreads();
    for (int i = warp; i < nr; i += 4) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) M = fmaxf(M, sm_m[w][i]);
      float L = 0.f, O[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) O[e] = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float sc = exp2f(sm_m[w][i] - M);
          L = fmaf(sm_l[w][i], sc, L);
#pragma unroll
          for (int e = 0; e < EPL; ++e) O[e] = fmaf(sm_o[w][i][lane * EPL + e], sc, O[e]);
        }
      }
      const int row = u.row0 + rb + i;
      const GroupTok gt = p.gtoks[u.tok_off + row / p.gqa];
      const int h = u.kvh * p.gqa + row % p.gqa;
      const float inv = L > 0.f ? 1.f / L : 0.f;
      const float lse2 = L > 0.f ? M + log2f(L) : -INFINITY;
      float* dst;
      if (gt.pbase < 0) {
        dst = p.out + ((size_t)gt.tok * p.hq + h) * D;
        if (lane == 0 && p.lse) p.lse[(size_t)gt.tok * p.hq + h] = lse2 * kLn2;
      } else {
        const size_t slot = (size_t)(gt.pbase + u.chunk) * p.hq + h;
        dst = p.part_o + slot * D;
        if (lane == 0) p.part_lse[slot] = lse2;
      }
#pragma unroll
      for (int e = 0; e < EPL; ++e) dst[lane * EPL + e] = O[e] * inv;
    }
    __syncthreads();
  }
}

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

cudaError_t launch_partial_attention(const AttnParams& p, int d, int grid, cudaStream_t s) {
  (void)grid;
  if (p.n_units == 0) return cudaSuccess;
  if (d == 128)
    simt_unit_kernel<128><<<p.n_units, 128, 0, s>>>(p);
  else
    simt_unit_kernel<64><<<p.n_units, 128, 0, s>>>(p);
  return cudaGetLastError();
}

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
