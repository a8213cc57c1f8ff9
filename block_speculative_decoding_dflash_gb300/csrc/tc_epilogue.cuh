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

// This thread's RoPE entries for block rows [m0, m1): the (cos, sin) of its
// rotation pair (row & 63 in the half-split layout, row / 2 in the
// interleaved one) at each row's position; rope[m * 64 + i]. They do not
// depend on the tile, so an epilogue can load them once.
template <int BN>
__device__ __forceinline__ void rope_entries(float2 (&cs)[BN], const float2* rope, int M, int neox,
                                             int row, int m0 = 0, int m1 = BN) {
  const int i = neox ? (row & 63) : (row >> 1);
#pragma unroll
  for (int m = 0; m < BN; ++m)
    cs[m] = (m >= m0 && m < m1 && m < M) ? rope[m * 64 + i] : make_float2(1.f, 0.f);
}

// Per-head RMSNorm over a 128-row tile (head_dim 128: one dim per epilogue
// thread) followed by RoPE with the entries cs_at(m) (rope_entries), for the
// block rows m in [m0, m1) of the tile's BN columns (m1 <= M; the bounds are
// the same for all threads); the value is normalised in fp32 and rotated
// before the single rounding the caller applies. All 128 epilogue threads
// must call it.
template <int BN, class CsAt>
__device__ __forceinline__ void head_norm_rope_cs(float* val, float g, CsAt cs_at, int M, int neox,
                                                  float eps, int row, int lane, int q,
                                                  float (*ss_sm)[BN], float* x_sm, int m0 = 0,
                                                  int m1 = BN) {
  if (m1 > M) m1 = M;
#pragma unroll
  for (int m = 0; m < BN; ++m) {
    if (m < m0 || m >= m1) continue;
    const float ss = warp_sum(val[m] * val[m]);
    if (lane == 0) ss_sm[q][m] = ss;
  }
  epi_sync();
#pragma unroll
  for (int m = 0; m < BN; ++m) {
    if (m < m0 || m >= m1) continue;
    const float ss = ss_sm[0][m] + ss_sm[1][m] + ss_sm[2][m] + ss_sm[3][m];
    val[m] = val[m] * rsqrtf(ss / 128.0f + eps) * g;
  }
  if (neox) {
#pragma unroll
    for (int m = 0; m < BN; ++m)
      if (m >= m0 && m < m1) x_sm[row * BN + m] = val[m];
    epi_sync();
    const bool lo = row < 64;
    const int partner = lo ? row + 64 : row - 64;
#pragma unroll
    for (int m = 0; m < BN; ++m) {
      if (m >= m0 && m < m1) {
        const float other = x_sm[partner * BN + m];
        const float2 cs = cs_at(m);
        val[m] = lo ? val[m] * cs.x - other * cs.y : other * cs.y + val[m] * cs.x;
      }
    }
    epi_sync();
  } else {
    const bool ev = (row & 1) == 0;
#pragma unroll
    for (int m = 0; m < BN; ++m) {
      if (m < m0 || m >= m1) continue;
      const float other = __shfl_xor_sync(0xffffffffu, val[m], 1);
      const float2 cs = cs_at(m);
      val[m] = ev ? val[m] * cs.x - other * cs.y : other * cs.y + val[m] * cs.x;
    }
    epi_sync();                                   // ss_sm is free for the next call
  }
}

// The same with the entries read from the table: up to 16 block rows they
// are loaded first (the loads overlap the norm's reduction), beyond that
// where they are used, to save registers.
template <int BN>
__device__ __forceinline__ void head_norm_rope_tile(float* val, float g, const float2* rope, int M,
                                                    int neox, float eps, int row, int lane, int q,
                                                    float (*ss_sm)[BN], float* x_sm, int m0 = 0,
                                                    int m1 = BN) {
  if (BN <= 16) {
    float2 cs[BN];
    rope_entries<BN>(cs, rope, M, neox, row, m0, m1);
    head_norm_rope_cs<BN>(val, g, [&](int m) { return cs[m]; }, M, neox, eps, row, lane, q, ss_sm, x_sm,
                          m0, m1);
  } else {
    const int i = neox ? (row & 63) : (row >> 1);
    head_norm_rope_cs<BN>(val, g, [&](int m) { return rope[m * 64 + i]; }, M, neox, eps, row, lane, q,
                          ss_sm, x_sm, m0, m1);
  }
}

// Split-tile partials: CTA b's fp32 partial of a tile sits in slot 0 (its
// first tile) or 1 (its last) of partials[b][2][128][NV * BN], row-major, so
// a thread moves its row's values as float4. Only the first mq float4 groups
// of each NV block (the block rows m < M) are written and read.
template <int NV, int BN>
__device__ __forceinline__ void put_partial(float* partials, int b, int slot, int row, int mq,
                                            const float (&acc)[NV][BN]) {
  float4* mine = reinterpret_cast<float4*>(partials + ((size_t)b * 2 + slot) * NV * BN * 128 +
                                           (size_t)row * NV * BN);
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int j = 0; j < BN / 4; ++j)
      if (j < mq)
        mine[v * (BN / 4) + j] = make_float4(acc[v][4 * j], acc[v][4 * j + 1], acc[v][4 * j + 2], acc[v][4 * j + 3]);
}

// acc = sum of the partials of CTAs bf..bl in CTA order (deterministic),
// issuing the loads of KB contributors before adding them: L2 latency, not
// bandwidth, bounds this loop, so fewer groups per contributor (MQC) allow a
// deeper batch. The tile is the first one of every contributor after bf
// (slot 0); s_bf is bf's slot for it.
template <int NV, int BN, int MQC, int KB>
__device__ __forceinline__ void sum_partials(float (&acc)[NV][BN], const float* partials, int row, int bf,
                                             int bl, int mq, int s_bf) {
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int m = 0; m < BN; ++m) acc[v][m] = 0.f;
  for (int b0 = bf; b0 <= bl; b0 += KB) {
    float4 pv[KB][NV * MQC];
#pragma unroll
    for (int q = 0; q < KB; ++q) {
      const int bb = b0 + q;
      if (bb > bl) break;
      const float4* p = reinterpret_cast<const float4*>(
          partials + ((size_t)bb * 2 + (bb == bf ? s_bf : 0)) * NV * BN * 128 + (size_t)row * NV * BN);
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int j = 0; j < MQC; ++j)
          pv[q][v * MQC + j] = j < mq ? __ldcg(p + v * (BN / 4) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int q = 0; q < KB; ++q) {
      if (b0 + q > bl) break;
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int j = 0; j < MQC; ++j) {
          float* dst = &acc[v][4 * j];
          const float4 x = pv[q][v * MQC + j];
          dst[0] += x.x; dst[1] += x.y; dst[2] += x.z; dst[3] += x.w;
        }
    }
  }
}

// acc[v][4g .. 4g+3] = the sum of float4 group g of the partials of CTAs
// bf..bl in CTA order, KB contributors' loads in flight at a time (the other
// columns of acc are left zero).
template <int NV, int BN, int KB>
__device__ __forceinline__ void sum_group(float (&acc)[NV][BN], const float* partials, int row, int g,
                                          int bf, int bl, int s_bf) {
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int m = 0; m < BN; ++m) acc[v][m] = 0.f;
  float4 sum[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) sum[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int b0 = bf; b0 <= bl; b0 += KB) {
    float4 pv[KB][NV];
#pragma unroll
    for (int qq = 0; qq < KB; ++qq) {
      const int bb = b0 + qq;
      if (bb > bl) break;
      const float4* p = reinterpret_cast<const float4*>(
          partials + ((size_t)bb * 2 + (bb == bf ? s_bf : 0)) * NV * BN * 128 + (size_t)row * NV * BN);
#pragma unroll
      for (int v = 0; v < NV; ++v) pv[qq][v] = __ldcg(p + v * (BN / 4) + g);
    }
#pragma unroll
    for (int qq = 0; qq < KB; ++qq) {
      if (b0 + qq > bl) break;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        sum[v].x += pv[qq][v].x; sum[v].y += pv[qq][v].y; sum[v].z += pv[qq][v].z; sum[v].w += pv[qq][v].w;
      }
    }
  }
  // g is warp-uniform; the static selection below keeps acc in registers
#pragma unroll
  for (int j = 0; j < BN / 4; ++j)
    if (j == g) {
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        acc[v][4 * j] = sum[v].x; acc[v][4 * j + 1] = sum[v].y;
        acc[v][4 * j + 2] = sum[v].z; acc[v][4 * j + 3] = sum[v].w;
      }
    }
}

// CTA owning unit u when U units are split into G contiguous ranges
// [floor(b*U/G), floor((b+1)*U/G)).
__device__ __forceinline__ int owner_of(long long u, long long U, int G) {
  return static_cast<int>((u * G + G - 1) / U);
}
// The same in 32-bit arithmetic, for U * G < 2^32 (a 64-bit division is a
// long software sequence on the GPU).
__device__ __forceinline__ int owner_of_u32(unsigned u, unsigned U, unsigned G) {
  return static_cast<int>((u * G + G - 1) / U);
}

}  // namespace dfl
