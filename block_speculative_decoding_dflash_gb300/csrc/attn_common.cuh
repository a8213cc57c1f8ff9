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
#include "kernels.h"
#include "ptx.cuh"

namespace dfl {

constexpr int kAttnHd = 128;
constexpr int kAttnKeys = 128;
constexpr int kAttnPartStride = kAttnHd + 4;

// Splits covering n keys.
__host__ __device__ __forceinline__ int attn_splits(long long n) {
  return static_cast<int>((n + kAttnKeys - 1) / kAttnKeys);
}

// Before a kernel waits on the ones still running: asks L2 for the context
// keys (thread 0) and values (thread 1) of key split s of kv head g. The ring
// state read here may be older than the one the kernel then uses (a round
// old at worst, always a valid state, so the range stays inside the ring);
// that only costs the hint.
__device__ __forceinline__ void attn_prefetch_context(const AttnArgs& a, int s, int g) {
  if (threadIdx.x >= 2) return;
  const volatile RingState* rs = a.ring;
  const long long p = rs->offset;
  long long kstart = rs->base;
  if (a.window > 0 && p - a.window > kstart) kstart = p - a.window;
  const long long j0 = (long long)s * kAttnKeys;
  long long n = p - kstart - j0;
  if (n <= 0 || a.cap <= 0) return;
  if (n > kAttnKeys) n = kAttnKeys;
  const long long slot = ring_slot(kstart + j0, a.cap);
  const long long first = n < a.cap - slot ? n : a.cap - slot;
  const char* base = static_cast<const char*>(threadIdx.x == 0 ? a.ring_k : a.ring_v) +
                     (size_t)g * a.cap * kAttnHd * 2;
  l2_prefetch_bulk(base + (size_t)slot * kAttnHd * 2, static_cast<uint32_t>(first * kAttnHd * 2));
  if (n > first) l2_prefetch_bulk(base, static_cast<uint32_t>((n - first) * kAttnHd * 2));
}

// One warp merges the first ns splits (layout stride nsplit) of query qi of kv
// head g, in split order, and writes the normalised bf16 output row. Each
// lane owns 4 output dims; the splits' maxima, sums and output slices of a
// batch of up to 32 splits are requested together, so a merge of up to 32
// splits is one round trip to L2.
__device__ __forceinline__ void attn_combine_warp(const float* partial, int nsplit, int ns, int Qn,
                                                  int G, int g, int qi, bf16* out, int ldo,
                                                  int lane) {
  constexpr int kB = 32;
  const size_t pstride = kAttnPartStride;
  const float* base = partial + (size_t)g * nsplit * Qn * pstride + (size_t)qi * pstride;
  const size_t sstride = (size_t)Qn * pstride;
  const int d4 = lane * 4;
  float M = -INFINITY, L = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int s0 = 0; s0 < ns; s0 += kB) {
    const int n = ns - s0 < kB ? ns - s0 : kB;
    // lane j < n holds split s0 + j's (max, sum); every lane its dims of all n
    float2 ml = make_float2(-INFINITY, 0.f);
    if (lane < n) ml = __ldcg(reinterpret_cast<const float2*>(base + (s0 + lane) * sstride + kAttnHd));
    float4 ov[kB];
#pragma unroll
    for (int j = 0; j < kB; ++j)
      ov[j] = j < n ? __ldcg(reinterpret_cast<const float4*>(base + (s0 + j) * sstride + d4))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    const float Mb = warp_max(ml.x);
    const float Mn = fmaxf(M, Mb);
    // rescale what was merged so far to the new maximum
    const float r = (M == -INFINITY) ? 0.f : expf(M - Mn);
    L *= r;
    acc[0] *= r; acc[1] *= r; acc[2] *= r; acc[3] *= r;
    const float f_l = ml.x == -INFINITY ? 0.f : expf(ml.x - Mn);
    L += warp_sum(f_l * ml.y);
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const float f = __shfl_sync(0xffffffffu, f_l, j);
      acc[0] += f * ov[j].x; acc[1] += f * ov[j].y; acc[2] += f * ov[j].z; acc[3] += f * ov[j].w;
    }
    M = Mn;
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
