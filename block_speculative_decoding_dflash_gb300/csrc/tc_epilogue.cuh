// Pieces shared by the tensor-core GEMM kernels: the warp layout (warp 0 TMA
// producer, warp 1 MMA issuer, warps 2-5 epilogue on named barrier 1), and
// epilogue helpers.
#pragma once

#include "common.cuh"

namespace dfl {

constexpr int kThreads = 192;
constexpr int kEpiBarrier = 1;
constexpr int kABytes = 128 * 128;     // 128 rows x 64 bf16

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }
__device__ __forceinline__ float rnd_bf(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync %0, %1;" ::"r"(kEpiBarrier), "r"(128) : "memory");
}

// Per-head RMSNorm over a 128-row tile (head_dim 128: one dim per epilogue
// thread) followed by RoPE, for every block row m < M of the tile's BN
// columns; the value is normalised in fp32 and rotated before the single
// rounding the caller applies. All 128 epilogue threads must call it.
template <int BN>
__device__ __forceinline__ void head_norm_rope_tile(float* val, float g, const float2* rope, int M,
                                                    int neox, float eps, int row, int lane, int q,
                                                    float (*ss_sm)[BN], float* x_sm) {
#pragma unroll
  for (int m = 0; m < BN; ++m) {
    const float ss = warp_sum(val[m] * val[m]);
    if (lane == 0) ss_sm[q][m] = ss;
  }
  epi_sync();
#pragma unroll
  for (int m = 0; m < BN; ++m) {
    const float ss = ss_sm[0][m] + ss_sm[1][m] + ss_sm[2][m] + ss_sm[3][m];
    val[m] = val[m] * rsqrtf(ss / 128.0f + eps) * g;
  }
  if (neox) {
#pragma unroll
    for (int m = 0; m < BN; ++m) x_sm[row * BN + m] = val[m];
    epi_sync();
    const int i = row & 63;
    const bool lo = row < 64;
    const int partner = lo ? row + 64 : row - 64;
#pragma unroll
    for (int m = 0; m < BN; ++m) {
      if (m < M) {
        const float2 cs = rope[m * 64 + i];
        const float other = x_sm[partner * BN + m];
        val[m] = lo ? val[m] * cs.x - other * cs.y : other * cs.y + val[m] * cs.x;
      }
    }
    epi_sync();
  } else {
    const int i = row >> 1;
    const bool ev = (row & 1) == 0;
#pragma unroll
    for (int m = 0; m < BN; ++m) {
      const float other = __shfl_xor_sync(0xffffffffu, val[m], 1);
      if (m < M) {
        const float2 cs = rope[m * 64 + i];
        val[m] = ev ? val[m] * cs.x - other * cs.y : other * cs.y + val[m] * cs.x;
      }
    }
  }
}

// CTA owning unit u when U units are split into G contiguous ranges
// [floor(b*U/G), floor((b+1)*U/G)).
__device__ __forceinline__ int owner_of(long long u, long long U, int G) {
  return static_cast<int>((u * G + G - 1) / U);
}

}  // namespace dfl
