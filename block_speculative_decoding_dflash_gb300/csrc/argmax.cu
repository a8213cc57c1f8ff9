// Argmax-producing kernels: the split-vocabulary lm_head + softcap + argmax,
// the target-logit argmax + greedy prefix accept, and the Markov chain step.
//
// All three reduce (value, index) pairs first inside a CTA and then across
// CTAs with the "last CTA done" pattern: every CTA writes its partial, fences,
// and takes a ticket from an atomic counter; the CTA that draws the last
// ticket reduces all partials and resets the counter. No CTA ever waits on
// another. The (larger value, then lower index) rule does not depend on the
// order partials arrive in, so results are deterministic.
#include <math.h>

#include "kernels.h"
#include "mma_sync.cuh"
#include "ptx.cuh"
#include "launch.cuh"

namespace dfl {
namespace {

constexpr int kLmWarps = 8;
constexpr int kLmNR = 4;       // vocab rows per warp step

// True in every thread of the CTA that drew the last ticket.
__device__ __forceinline__ bool last_cta(unsigned* counter, unsigned total) {
  __shared__ bool is_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(counter, 1u) == total - 1);
  __syncthreads();
  if (is_last) __threadfence();
  return is_last;
}

template <typename T, int MT>
__global__ void __launch_bounds__(kLmWarps * 32) lmhead_kernel(LmHeadArgs a) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char lm_smem[];
  T* xs = reinterpret_cast<T*>(lm_smem);                  // [MT][H]
  __shared__ float best_v[kLmWarps][MT];
  __shared__ int best_i[kLmWarps][MT];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x;
  const long long v0 = (long long)a.V * b / a.grid;
  const long long v1 = (long long)a.V * (b + 1) / a.grid;
  const T* W = reinterpret_cast<const T*>(a.w);
  const T* X = reinterpret_cast<const T*>(a.x);
  const float cap = a.softcap;
  const float inv_cap = cap > 0.f ? 1.0f / cap : 0.f;

  for (int m0 = 0; m0 < a.R; m0 += MT) {
    const int mr = min(MT, a.R - m0);
    for (int e = threadIdx.x * 8; e < MT * a.H; e += blockDim.x * 8) {
      const int m = e / a.H, k = e % a.H;
      if (m < mr) {
        const uint4* src = reinterpret_cast<const uint4*>(X + (size_t)(m0 + m) * a.ldx + k);
        uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)m * a.H + k);
        dst[0] = src[0];
        if (sizeof(T) == 4) dst[1] = src[1];
      }
    }
    __syncthreads();
    float bv[MT];
    int bi[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) { bv[m] = -INFINITY; bi[m] = 0x7fffffff; }

    for (long long v = v0 + (long long)warp * kLmNR; v < v1; v += kLmWarps * kLmNR) {
      const int nr = static_cast<int>(min((long long)kLmNR, v1 - v));
      float acc[kLmNR][MT];
#pragma unroll
      for (int r = 0; r < kLmNR; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;
      for (int k = lane * 8; k < a.H; k += 32 * 8) {
        float w[kLmNR][8];
#pragma unroll
        for (int r = 0; r < kLmNR; ++r) {
          if (r < nr) {
            load8_stream(W + (size_t)(v + r) * a.H + k, w[r]);
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) w[r][q] = 0.f;
          }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < mr) {
            float xv[8];
            load8(xs + (size_t)m * a.H + k, xv);
#pragma unroll
            for (int r = 0; r < kLmNR; ++r) {
              float s = acc[r][m];
#pragma unroll
              for (int q = 0; q < 8; ++q) s = fmaf(w[r][q], xv[q], s);
              acc[r][m] = s;
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kLmNR; ++r) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          float z = warp_sum(acc[r][m]);
          if (r < nr && m < mr) {
            if (cap > 0.f) z = cap * tanhf(z * inv_cap);
            const int vi = static_cast<int>(v + r);
            if (a.logits != nullptr && lane == 0) a.logits[(size_t)(m0 + m) * a.V + vi] = z;
            if (better(z, vi, bv[m], bi[m])) { bv[m] = z; bi[m] = vi; }
          }
        }
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int m = 0; m < MT; ++m) { best_v[warp][m] = bv[m]; best_i[warp][m] = bi[m]; }
    }
    __syncthreads();
    if (threadIdx.x < mr) {
      const int m = threadIdx.x;
      float v = best_v[0][m];
      int i = best_i[0][m];
      for (int w = 1; w < kLmWarps; ++w)
        if (better(best_v[w][m], best_i[w][m], v, i)) { v = best_v[w][m]; i = best_i[w][m]; }
      a.part_v[(size_t)b * a.R + m0 + m] = v;
      a.part_i[(size_t)b * a.R + m0 + m] = i;
    }
    __syncthreads();
  }

  if (last_cta(a.counter, gridDim.x)) {
    for (int m = threadIdx.x; m < a.R; m += blockDim.x) {
      float v = -INFINITY;
      int i = 0x7fffffff;
      for (int c = 0; c < a.grid; ++c) {
        const float cv = __ldcg(a.part_v + (size_t)c * a.R + m);
        const int ci = __ldcg(a.part_i + (size_t)c * a.R + m);
        if (better(cv, ci, v, i)) { v = cv; i = ci; }
      }
      a.ids[m] = i;
      if (a.ids2) a.ids2[m] = i;
      a.maxv[m] = v;
    }
    if (threadIdx.x == 0) *a.counter = 0u;
  }
}

template <typename T, int MT>
cudaError_t lm_launch(const LmHeadArgs& a, cudaStream_t st) {
  const size_t smem = (size_t)MT * a.H * sizeof(T);
  launch_pdl(lmhead_kernel<T, MT>, dim3(a.grid), dim3(kLmWarps * 32), smem, st, a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t lm_dispatch(const LmHeadArgs& a, cudaStream_t st) {
  if (a.R <= 1) return lm_launch<T, 1>(a, st);
  if (a.R <= 2) return lm_launch<T, 2>(a, st);
  if (a.R <= 4) return lm_launch<T, 4>(a, st);
  if (a.R <= 8) return lm_launch<T, 8>(a, st);
  return lm_launch<T, 16>(a, st);
}

template <typename T, int MT>
cudaError_t lm_attr(int H) {
  return cudaFuncSetAttribute(lmhead_kernel<T, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)((size_t)MT * H * sizeof(T)));
}

// ---- verify: target argmax per row + greedy accept ------------------------------------
constexpr int kVerifyChunk = 8192;
constexpr int kMaxVerifyRows = 1024;

template <typename T>
__global__ void __launch_bounds__(256) verify_kernel(VerifyArgs a) {
  if (threadIdx.x == 0) ktrace_mark(a.trace, 0);
  pdl_enter();
  if (threadIdx.x == 0) ktrace_mark(a.trace, 1);
  __shared__ float sv[8];
  __shared__ int si[8];
  __shared__ int t_s[kMaxVerifyRows];
  // sequence blockIdx.z of a batch: its own logits, drafts, outputs, state,
  // partials and ticket
  {
    const int sq = blockIdx.z;
    a.L = static_cast<const char*>(a.L) + (size_t)sq * a.B * a.V * sizeof(T);
    a.d += (size_t)sq * (a.B - 1);
    a.tokens += (size_t)sq * a.B;
    a.n += sq;
    a.rs += sq;
    a.part_v += (size_t)sq * a.B * a.chunks;
    a.part_i += (size_t)sq * a.B * a.chunks;
    a.counter += sq;
  }
  const int i = blockIdx.y, c = blockIdx.x;
  const T* row = reinterpret_cast<const T*>(a.L) + (size_t)i * a.V;
  const int v0 = c * kVerifyChunk;
  const int v1 = min(a.V, v0 + kVerifyChunk);
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  // 8 consecutive logits per load (16 bytes for bf16) when the row is
  // 16-byte aligned; the chunk's 1024 groups are all requested up front.
  if ((a.V & 7) == 0 && (reinterpret_cast<uintptr_t>(a.L) & 15) == 0 && sizeof(T) == 2) {
    float z[4][8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int v = v0 + (threadIdx.x + k * 256) * 8;
      if (v < v1) load8(row + v, z[k]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int v = v0 + (threadIdx.x + k * 256) * 8;
      if (v < v1) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (better(z[k][e], v + e, bv, bi)) { bv = z[k][e]; bi = v + e; }
      }
    }
  } else {
    for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
      const float z = to_f(row[v]);
      if (better(z, v, bv, bi)) { bv = z; bi = v; }
    }
  }
  warp_argmax(bv, bi);
  if ((threadIdx.x & 31) == 0) { sv[threadIdx.x >> 5] = bv; si[threadIdx.x >> 5] = bi; }
  __syncthreads();
  if (threadIdx.x == 0) {
    bv = sv[0];
    bi = si[0];
    for (int w = 1; w < 8; ++w)
      if (better(sv[w], si[w], bv, bi)) { bv = sv[w]; bi = si[w]; }
    a.part_v[(size_t)i * a.chunks + c] = bv;
    a.part_i[(size_t)i * a.chunks + c] = bi;
  }
  if (last_cta(a.counter, gridDim.x * gridDim.y)) {
    // warp w reduces rows w, w + 8, ...: lane q takes chunks q, q + 32, ...
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int r = warp; r < a.B; r += 8) {
      float v = -INFINITY;
      int idx = 0x7fffffff;
      for (int q = lane; q < a.chunks; q += 32) {
        const float cv = __ldcg(a.part_v + (size_t)r * a.chunks + q);
        const int ci = __ldcg(a.part_i + (size_t)r * a.chunks + q);
        if (better(cv, ci, v, idx)) { v = cv; idx = ci; }
      }
      warp_argmax(v, idx);
      if (lane == 0) t_s[r] = idx;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int acc = 0;
      while (acc < a.B - 1 && a.d[acc] == t_s[acc]) ++acc;
      for (int q = 0; q < a.B; ++q) a.tokens[q] = q < acc ? a.d[q] : (q == acc ? t_s[acc] : -1);
      *a.n = acc + 1;
      a.rs->n = acc + 1;
      a.rs->a = acc;
      a.rs->bonus = t_s[acc];
      *a.counter = 0u;
      ktrace_mark(a.trace, 2);
    }
  }
}

// ---- Markov chain step ---------------------------------------------------------------------
// One launch per chain step (step j needs step j-1's argmax). A step reads
// all of W2 (33.6 MB for the DSpark head, resident in L2 after the first
// step) and is bound by how many of those bytes are in flight: a CTA takes
// kMkCols vocabulary columns with 16 groups of 8 columns x kMkParts slices
// of the rank, and each thread requests all of its slice's rows (16 at r =
// 256) before it uses any, so about the whole matrix is requested at once
// (512 CTAs at V = 65536). The slices are summed in shared memory in slice
// order. Each CTA folds its best (value, column) into one 64-bit key per step
// with an atomic maximum (the order-preserving value bits above the inverted
// column); the last CTA decodes it into out[j] and clears it.
constexpr int kMkThreads = 256;
constexpr int kMkParts = 16;
constexpr int kMkGroups = kMkThreads / kMkParts;
constexpr int kMkCols = kMkGroups * 8;
constexpr int kMkBatch = 16;                  // W2 rows a thread has in flight at once

__device__ __forceinline__ unsigned long long mk_key(float v, int i) {
  const uint32_t u = __float_as_uint(v + 0.0f);
  const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(ord) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(i));
}

template <typename T>
__global__ void __launch_bounds__(kMkThreads) markov_step_kernel(MarkovArgs a, int j) {
  const KTrace tr{a.trace.p, a.trace.slot + j};
  if (threadIdx.x == 0) ktrace_mark(tr, 0);
  pdl_enter();
  if (threadIdx.x == 0) ktrace_mark(tr, 1);
  extern __shared__ float w1s[];               // [r]
  __shared__ float part[kMkParts][kMkGroups][8];
  int prev;
  if (j == 0) prev = a.anchor_host >= 0 ? a.anchor_host : a.rs->anchor;
  else prev = a.out[j - 1];
  if (prev < 0 || prev >= a.V) prev = 0;
  const T* w1 = reinterpret_cast<const T*>(a.w1) + (size_t)prev * a.r;
  for (int q = threadIdx.x; q < a.r; q += blockDim.x) w1s[q] = to_f(w1[q]);
  __syncthreads();
  const int grp = threadIdx.x % kMkGroups, pt = threadIdx.x / kMkGroups;
  const int c = blockIdx.x * kMkCols + grp * 8;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (c < a.V) {
    const T* w2 = reinterpret_cast<const T*>(a.w2) + c;
    // rows pt, pt + kMkParts, ...: kMkBatch of them requested before use
    for (int q0 = pt; q0 < a.r; q0 += kMkBatch * kMkParts) {
      if constexpr (sizeof(T) == 2) {
        // kept as packed bf16 until used: 4 registers a row
        uint4 raw[kMkBatch];
#pragma unroll
        for (int b = 0; b < kMkBatch; ++b) {
          const int q = q0 + b * kMkParts;
          raw[b] = q < a.r ? __ldg(reinterpret_cast<const uint4*>(w2 + (size_t)q * a.V)) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int b = 0; b < kMkBatch; ++b) {
          const int q = q0 + b * kMkParts;
          const float sc = q < a.r ? w1s[q] : 0.f;
          const bf16* e8 = reinterpret_cast<const bf16*>(&raw[b]);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[e] = fmaf(sc, __bfloat162float(e8[e]), acc[e]);
        }
      } else {
        float wv[kMkBatch / 2][8];
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int b = 0; b < kMkBatch / 2; ++b) {
            const int q = q0 + (h * kMkBatch / 2 + b) * kMkParts;
            if (q < a.r) load8(w2 + (size_t)q * a.V, wv[b]);
          }
#pragma unroll
          for (int b = 0; b < kMkBatch / 2; ++b) {
            const int q = q0 + (h * kMkBatch / 2 + b) * kMkParts;
            if (q < a.r) {
              const float sc = w1s[q];
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[e] = fmaf(sc, wv[b][e], acc[e]);
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) part[pt][grp][e] = acc[e];
  __syncthreads();
  if (threadIdx.x < 32) {
    // threads 0..15 sum their group's slices in slice order; the warp folds
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    const int cc = blockIdx.x * kMkCols + threadIdx.x * 8;
    if (threadIdx.x < kMkGroups && cc < a.V) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float z = 0.f;
        for (int p = 0; p < kMkParts; ++p) z += part[p][threadIdx.x][e];
        if (a.z) z = a.z[(size_t)j * a.ldz + cc + e] + z;
        if (cc + e < a.V && better(z, cc + e, bv, bi)) { bv = z; bi = cc + e; }
      }
    }
    warp_argmax(bv, bi);
    if (threadIdx.x == 0) atomicMax(a.key + j, mk_key(bv, bi));
  }
  if (last_cta(a.counter, gridDim.x) && threadIdx.x == 0) {
    const unsigned long long key = atomicExch(a.key + j, 0ull);
    const int idx = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key));
    a.out[j] = idx;
    if (a.out2) a.out2[j] = idx;
    *a.counter = 0u;
    ktrace_mark(tr, 2);
  }
}

// ---- the whole chain in one cooperative launch ------------------------------------------
// CTA b holds W2's columns [b * cols, (b + 1) * cols) of every rank row in
// shared memory (221 KB for the DSpark head on 152 SMs), loaded once before
// the dependency resolves (W2 is a weight). Per step every CTA scores its
// columns against W1[prev]: a warp takes 4 column groups of 8 x 8 slices of
// the rank and sums the slices with shuffles (a fixed order); it folds its
// best into key[j] with an atomic maximum; a grid barrier (all CTAs are
// resident: cooperative launch; the wait is bounded and reports bit 64 in
// err) makes the step's winner the next prev of every CTA.
constexpr int kMkcThreads = 448;              // 14 warps x 4 groups = 56 groups of 8 columns
constexpr int kMkcGroups = kMkcThreads / 32 * 4;
constexpr int kMkcParts = 8;
constexpr unsigned kMkcSpins = 1u << 22;

__device__ __forceinline__ bool mkc_barrier(unsigned* count, unsigned* gen, unsigned nb, unsigned& g, int* err) {
  __shared__ bool s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    bool ok = true;
    const unsigned target = g + 1;
    __threadfence();
    if (atomicAdd(count, 1u) == nb - 1) {
      atomicExch(count, 0u);
      __threadfence();
      atomicExch(gen, target);
    } else {
      unsigned spins = 0;
      while (ld_acquire(gen) != target) {
        if (++spins > kMkcSpins) { atomicOr(err, 64); ok = false; break; }
        __nanosleep(64);
      }
    }
    __threadfence();
    s_ok = ok;
  }
  g += 1;
  __syncthreads();
  return s_ok;
}

__global__ void __launch_bounds__(kMkcThreads, 1) markov_chain_coop_kernel(MarkovArgs a, int cols) {
  extern __shared__ __align__(16) uint8_t mk_smem[];
  bf16* w2s = reinterpret_cast<bf16*>(mk_smem);                         // [r][cols]
  float* w1s = reinterpret_cast<float*>(mk_smem + (size_t)a.r * cols * 2);  // [r]
  __shared__ float sv[kMkcThreads / 32];
  __shared__ int si[kMkcThreads / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c0 = blockIdx.x * cols;
  const int ngran = cols / 8;
  const bf16* w2 = reinterpret_cast<const bf16*>(a.w2);
  for (int e = tid; e < a.r * ngran; e += blockDim.x) {
    const int q = e / ngran, gcol = c0 + (e % ngran) * 8;
    const bool valid = gcol < a.V;
    cp_async16(w2s + (size_t)q * cols + (e % ngran) * 8, w2 + (size_t)q * a.V + (valid ? gcol : 0), valid);
  }
  unsigned g = ld_acquire(a.bar + 1);          // barrier generation at entry
  if (threadIdx.x == 0) ktrace_mark(a.trace, 0);
  pdl_enter();
  if (threadIdx.x == 0) ktrace_mark(a.trace, 1);
  cp_async_wait_all();
  // warp w: groups 4w .. 4w + 3; lane = group-in-warp + 4 * slice
  const int gw = lane & 3, part = lane >> 2;
  const int grp = warp * 4 + gw;
  const int lc = grp * 8;                      // local column of this group
  const bf16* w1 = reinterpret_cast<const bf16*>(a.w1);
  int prev = a.anchor_host >= 0 ? a.anchor_host : a.rs->anchor;
  for (int j = 0; j < a.gamma; ++j) {
    if (prev < 0 || prev >= a.V) prev = 0;
    for (int q = tid; q < a.r; q += blockDim.x) w1s[q] = __bfloat162float(w1[(size_t)prev * a.r + q]);
    __syncthreads();
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (lc < cols) {
      for (int q = part; q < a.r; q += kMkcParts) {
        const uint4 raw = *reinterpret_cast<const uint4*>(w2s + (size_t)q * cols + lc);
        const bf16* e8 = reinterpret_cast<const bf16*>(&raw);
        const float sc = w1s[q];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(sc, __bfloat162float(e8[e]), acc[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 4);
      acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 8);
      acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 16);
    }
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    const int cc = c0 + lc;
    if (part == 0 && lc < cols) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (cc + e >= a.V) continue;
        float z = acc[e];
        if (a.z) z = a.z[(size_t)j * a.ldz + cc + e] + z;
        if (better(z, cc + e, bv, bi)) { bv = z; bi = cc + e; }
      }
    }
    warp_argmax(bv, bi);
    if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
    __syncthreads();
    if (tid == 0) {
      bv = sv[0];
      bi = si[0];
      for (int w = 1; w < kMkcThreads / 32; ++w)
        if (better(sv[w], si[w], bv, bi)) { bv = sv[w]; bi = si[w]; }
      atomicMax(a.key + j, mk_key(bv, bi));
    }
    mkc_barrier(a.bar, a.bar + 1, gridDim.x, g, a.err);
    const unsigned long long key = __ldcg(a.key + j);
    prev = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key));
    if (blockIdx.x == 0 && tid == 0) {
      a.out[j] = prev;
      if (a.out2) a.out2[j] = prev;
    }
  }
  // every CTA has read every key: clear them for the next chain
  mkc_barrier(a.bar, a.bar + 1, gridDim.x, g, a.err);
  if (blockIdx.x == 0)
    for (int j = tid; j < a.gamma; j += blockDim.x) a.key[j] = 0ull;
  if (blockIdx.x == 0 && tid == 0) ktrace_mark(a.trace, 2);
}

}  // namespace

static int mkc_cols(int V, int grid) { return ((V + grid - 1) / grid + 7) / 8 * 8; }
static size_t mkc_smem(int V, int r, int grid) { return (size_t)r * mkc_cols(V, grid) * 2 + (size_t)r * 4; }

bool markov_coop_ok(int dtype, int V, int r, int grid) {
  if (dtype != 1 || V % 8 || r < 1 || grid < 1) return false;
  if (mkc_cols(V, grid) / 8 > kMkcGroups) return false;
  const size_t smem = mkc_smem(V, r, grid);
  if (smem > 227 * 1024) return false;
  if (cudaFuncSetAttribute(markov_chain_coop_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return false;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, markov_chain_coop_kernel, kMkcThreads, smem) !=
      cudaSuccess)
    return false;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return per_sm >= 1 && grid <= per_sm * sms;
}

cudaError_t launch_markov_chain_coop(int dtype, const MarkovArgs& a, int grid, cudaStream_t st) {
  if (dtype != 1 || a.V % 8 || !a.bar || !a.err) return cudaErrorNotSupported;
  const int cols = mkc_cols(a.V, grid);
  if (cols / 8 > kMkcGroups) return cudaErrorNotSupported;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMkcThreads);
  cfg.dynamicSmemBytes = mkc_smem(a.V, a.r, grid);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, markov_chain_coop_kernel, a, cols);
}

// Batch read-out: ids of every block row [nseq][rows] -> draft ids [nseq]
// [rows - read0] (and the same for a second copy and the maxima).
__global__ void split_ids_kernel(const int* ids_all, const float* maxv_all, int rows, int read0, int nseq,
                                 int* ids, int* ids2, float* maxv) {
  pdl_enter();
  const int per = rows - read0;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= nseq * per) return;
  const int src = (e / per) * rows + read0 + e % per;
  ids[e] = ids_all[src];
  if (ids2) ids2[e] = ids_all[src];
  if (maxv) maxv[e] = maxv_all[src];
}

cudaError_t launch_split_ids(const int* ids_all, const float* maxv_all, int rows, int read0, int nseq, int* ids,
                             int* ids2, float* maxv, cudaStream_t st) {
  const int n = nseq * (rows - read0);
  launch_pdl(split_ids_kernel, dim3((n + 127) / 128), dim3(128), 0, st, ids_all, maxv_all, rows, read0, nseq, ids,
             ids2, maxv);
  return cudaGetLastError();
}

int lmhead_grid(int V) {
  const int g = (V + 63) / 64;
  return g < 608 ? g : 608;
}

int verify_chunks(int V) { return (V + kVerifyChunk - 1) / kVerifyChunk; }

int markov_grid(int V) { return (V + kMkCols - 1) / kMkCols; }

cudaError_t init_lmhead_attrs(int H) {
  cudaError_t e;
  if ((e = lm_attr<bf16, 1>(H)) != cudaSuccess) return e;
  if ((e = lm_attr<bf16, 2>(H)) != cudaSuccess) return e;
  if ((e = lm_attr<bf16, 4>(H)) != cudaSuccess) return e;
  if ((e = lm_attr<bf16, 8>(H)) != cudaSuccess) return e;
  if ((e = lm_attr<bf16, 16>(H)) != cudaSuccess) return e;
  if ((e = lm_attr<float, 1>(H)) != cudaSuccess) return e;
  if ((e = lm_attr<float, 2>(H)) != cudaSuccess) return e;
  if ((e = lm_attr<float, 4>(H)) != cudaSuccess) return e;
  if ((e = lm_attr<float, 8>(H)) != cudaSuccess) return e;
  return lm_attr<float, 16>(H);
}

cudaError_t launch_lmhead_argmax(int dtype, const LmHeadArgs& a, cudaStream_t st) {
  return dtype ? lm_dispatch<bf16>(a, st) : lm_dispatch<float>(a, st);
}

cudaError_t launch_verify(int dtype, const VerifyArgs& a, cudaStream_t st) {
  dim3 grid(a.chunks, a.B, a.nseq > 1 ? a.nseq : 1);
  if (dtype) launch_pdl(verify_kernel<bf16>, dim3(grid), dim3(256), 0, st, a);
  else launch_pdl(verify_kernel<float>, dim3(grid), dim3(256), 0, st, a);
  return cudaGetLastError();
}

cudaError_t launch_markov_chain(int dtype, const MarkovArgs& a, cudaStream_t st) {
  if (a.V % 8) return cudaErrorInvalidValue;   // 8-column loads of W2 rows
  const size_t smem = sizeof(float) * a.r;
  for (int j = 0; j < a.gamma; ++j) {
    if (dtype) launch_pdl(markov_step_kernel<bf16>, dim3(a.grid), dim3(kMkThreads), smem, st, a, j);
    else launch_pdl(markov_step_kernel<float>, dim3(a.grid), dim3(kMkThreads), smem, st, a, j);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dfl
