// Split-key attention partials, head_dim 128, and their merge.
//
// A split covers kAttnKeys consecutive keys of one kv head. For every query
// qi (block row qi / G, query head g * G + qi % G) it leaves an unnormalised
// partial: o[128] = sum_j exp(s_j - m) v_j, then m = max_j s_j and
// l = sum_j exp(s_j - m), in a row of kAttnPartStride floats (528 bytes, a
// multiple of 16 so o can be read with float4 loads). The layout is
// partial[g][split][qi][kAttnPartStride].
#pragma once

#include "common.cuh"

namespace dfl {

constexpr int kAttnHd = 128;
constexpr int kAttnKeys = 128;
constexpr int kAttnPartStride = kAttnHd + 4;

// Splits covering n keys.
__host__ __device__ __forceinline__ int attn_splits(long long n) {
  return static_cast<int>((n + kAttnKeys - 1) / kAttnKeys);
}

// One warp merges the first ns splits (layout stride nsplit) of query qi of kv
// head g, in split order, and writes the normalised bf16 output row.
__device__ __forceinline__ void attn_combine_warp(const float* partial, int nsplit, int ns, int Qn,
                                                  int G, int g, int qi, bf16* out, int ldo,
                                                  int lane) {
  const size_t pstride = kAttnPartStride;
  const float* base = partial + (size_t)g * nsplit * Qn * pstride + (size_t)qi * pstride;
  const size_t sstride = (size_t)Qn * pstride;
  float M = -INFINITY;
  for (int sp = lane; sp < ns; sp += 32) M = fmaxf(M, __ldcg(base + sp * sstride + kAttnHd));
  M = warp_max(M);
  float L = 0.f;
  for (int sp = lane; sp < ns; sp += 32) {
    const float ms = __ldcg(base + sp * sstride + kAttnHd);
    if (ms != -INFINITY) L += expf(ms - M) * __ldcg(base + sp * sstride + kAttnHd + 1);
  }
  L = warp_sum(L);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const int d4 = lane * 4;
  for (int s0 = 0; s0 < ns; s0 += 32) {
    const int sp_l = s0 + lane;
    const float ms_l = sp_l < ns ? __ldcg(base + sp_l * sstride + kAttnHd) : -INFINITY;
    const float f_l = ms_l == -INFINITY ? 0.f : expf(ms_l - M);
    const int n = ns - s0 < 32 ? ns - s0 : 32;
    int j = 0;
    for (; j + 8 <= n; j += 8) {
      float4 ov[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        ov[u] = __ldcg(reinterpret_cast<const float4*>(base + (s0 + j + u) * sstride + d4));
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float f = __shfl_sync(0xffffffffu, f_l, j + u);
        acc[0] += f * ov[u].x; acc[1] += f * ov[u].y; acc[2] += f * ov[u].z; acc[3] += f * ov[u].w;
      }
    }
    for (; j < n; ++j) {
      const float4 ov = __ldcg(reinterpret_cast<const float4*>(base + (s0 + j) * sstride + d4));
      const float f = __shfl_sync(0xffffffffu, f_l, j);
      acc[0] += f * ov.x; acc[1] += f * ov.y; acc[2] += f * ov.z; acc[3] += f * ov.w;
    }
  }
  const float inv = 1.0f / L;
  bf16* dst = out + (size_t)(qi / G) * ldo + (size_t)(g * G + qi % G) * kAttnHd + d4;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(dst) = pk;
}

}  // namespace dfl
