// Two steps beside the greedy round:
//
// * Speculative-sampling verify at temperature T > 0 ("Load Meta's
//   Muse-Glimmer-30B-assistant DFlash head", "Measured": the sampled-
//   acceptance run). The drafter proposes its argmaxes, so its proposal
//   distribution is a point mass on d_{i+1}, and the standard acceptance
//   min(1, p/q) becomes: row i accepts d_{i+1} iff u[i] < p_i(d_{i+1}) with
//   p_i = softmax(c tanh(L[i] / c) / T). After a rejection at row a the bonus
//   is drawn from the residual (p_a without d_{a+1}), after a full accept
//   from p_{B-1}, by inverse CDF in vocabulary order with u[B-1]. One CTA per
//   row computes the row's maximum, its sums and the row's own accept test
//   and bonus candidate; the last CTA to finish picks the first rejection.
//
// * The LFM2 short convolution and its partial-accept rollback ("LFM2 /
//   LFM2.5 DSpark drafter on the DFlash loop", "Short-conv rollback"): a
//   conv state cannot be trimmed like a KV cache, so the committed state is
//   recomputed as the last L - 1 rows of concat(previous state or zeros,
//   Bx[:n]), with n read on the device from the verify.
#include <math.h>

#include "kernels.h"
#include "launch.cuh"

namespace dfl {
namespace {

constexpr int kSampThreads = 1024;

__device__ __forceinline__ bool sampled_last_cta(unsigned* counter, unsigned total) {
  __shared__ bool is_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(counter, 1u) == total - 1);
  __syncthreads();
  if (is_last) __threadfence();
  return is_last;
}

template <typename T>
__global__ void __launch_bounds__(kSampThreads) verify_sampled_kernel(SampledVerifyArgs a) {
  pdl_enter();
  __shared__ float red[kSampThreads / 32];
  __shared__ float wsum[kSampThreads / 32];
  __shared__ float s_M, s_ed, s_tot;
  __shared__ int s_tok, s_thr;
  const int i = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = a.V;
  const T* L = reinterpret_cast<const T*>(a.L) + (size_t)i * V;
  const bool last_row = i == a.B - 1;
  const int d = last_row ? -1 : a.d[i];                 // the draft this row checks
  const float invT = 1.0f / a.temperature;
  const float cap = a.softcap;
  auto zval = [&](int v) {
    float x = to_f(L[v]);
    if (cap > 0.f) x = cap * tanhf(x / cap);
    return x * invT;
  };
  const int seg = (V + kSampThreads - 1) / kSampThreads;
  const int v0 = min(tid * seg, V), v1 = min(v0 + seg, V);
  // row maximum
  float m = -INFINITY;
  for (int v = v0; v < v1; ++v) m = fmaxf(m, zval(v));
  m = warp_max(m);
  if (lane == 0) red[warp] = m;
  if (tid == 0) { s_ed = 0.f; s_tok = -1; s_thr = kSampThreads; }
  __syncthreads();
  if (warp == 0) {
    float x = lane < kSampThreads / 32 ? red[lane] : -INFINITY;
    x = warp_max(x);
    if (lane == 0) s_M = x;
  }
  __syncthreads();
  const float M = s_M;
  // this thread's sum of exp(z - M) in vocabulary order, the row's draft
  // kept apart (the residual after a rejection leaves it out)
  float s = 0.f;
  for (int v = v0; v < v1; ++v) {
    const float e = expf(zval(v) - M);
    if (v == d) s_ed = e;
    else s += e;
  }
  // exclusive prefix of the per-thread sums, in thread order
  float incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    float w = lane < kSampThreads / 32 ? wsum[lane] : 0.f;
    float wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < kSampThreads / 32) wsum[lane] = wi - w;   // exclusive warp offsets
    if (lane == 31) s_tot = wi;
  }
  __syncthreads();
  const float excl = wsum[warp] + incl - s;              // sum of the earlier threads
  const float tot = s_tot;                               // residual mass (without d)
  // inverse CDF: the first vocabulary entry whose running sum exceeds t. The
  // thread whose range [its prefix, the next thread's prefix) holds t scans
  // its entries; rounding can make two ranges overlap, so the lowest such
  // thread wins.
  const float t = a.u[a.B - 1] * tot;
  float hi = __shfl_down_sync(0xffffffffu, excl, 1);
  if (lane == 31) hi = warp + 1 < kSampThreads / 32 ? wsum[warp + 1] : tot;
  if (excl <= t && t < hi) atomicMin(&s_thr, tid);
  __syncthreads();
  if (tid == s_thr) {
    float run = excl;
    int tok = -1, last_pos = -1;
    for (int v = v0; v < v1 && tok < 0; ++v) {
      if (v == d) continue;
      const float e = expf(zval(v) - M);
      if (e > 0.f) last_pos = v;
      run += e;
      if (run > t) tok = v;
    }
    s_tok = tok >= 0 ? tok : last_pos;
  }
  __syncthreads();
  if (tid == 0) {
    int tok = s_tok;
    if (tok < 0) {
      // t at or past the total by rounding: the last entry of positive mass
      for (int v = V - 1; v >= 0 && tok < 0; --v)
        if (v != d && expf(zval(v) - M) > 0.f) tok = v;
      if (tok < 0) tok = 0;
    }
    a.cand[i] = tok;
    const float pd = last_row ? 0.f : s_ed / (tot + s_ed);
    a.acc[i] = (!last_row && a.u[i] < pd) ? 1 : 0;
    a.pd[i] = pd;
  }
  if (sampled_last_cta(a.counter, gridDim.x) && tid == 0) {
    int acc = 0;
    while (acc < a.B - 1 && __ldcg(a.acc + acc)) ++acc;
    const int bonus = __ldcg(a.cand + acc);
    for (int q = 0; q < a.B; ++q) a.tokens[q] = q < acc ? a.d[q] : (q == acc ? bonus : -1);
    *a.n = acc + 1;
    if (a.rs) {
      a.rs->n = acc + 1;
      a.rs->a = acc;
      a.rs->bonus = bonus;
    }
    *a.counter = 0u;
  }
}

// y[l][t][c] = sum_k w[l][c][k] x[l][t + k][c], x = concat(state or zeros,
// bx); state_after = the last L - 1 rows of x. One thread per (layer,
// channel), rows in order.
template <typename T>
__global__ void short_conv_kernel(const T* state, const T* bx, const T* w, int layers, int lc,
                                  int C, int block, T* y, T* state_after) {
  pdl_enter();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= layers * C) return;
  const int l = idx / C, c = idx % C;
  float win[kShortConvMaxL];
  float wk[kShortConvMaxL];
  for (int k = 0; k < lc; ++k) wk[k] = to_f(w[((size_t)l * C + c) * lc + k]);
  for (int k = 0; k < lc - 1; ++k) win[k] = state ? to_f(state[((size_t)l * (lc - 1) + k) * C + c]) : 0.f;
  for (int t = 0; t < block; ++t) {
    win[lc - 1] = to_f(bx[((size_t)l * block + t) * C + c]);
    float acc = 0.f;
    for (int k = 0; k < lc; ++k) acc = fmaf(wk[k], win[k], acc);
    y[((size_t)l * block + t) * C + c] = from_f<T>(acc);
    for (int k = 0; k < lc - 1; ++k) win[k] = win[k + 1];
  }
  if (state_after)
    for (int k = 0; k < lc - 1; ++k) state_after[((size_t)l * (lc - 1) + k) * C + c] = from_f<T>(win[k]);
}

// out = the last L - 1 rows of concat(prev or zeros, bx[:n]), n = *n_dev
// (clamped to [0, block]). Each thread reads all of its channel's rows before
// writing, so out may alias prev.
template <typename T>
__global__ void short_conv_rollback_kernel(const T* prev, const T* bx, const int* n_dev, int layers,
                                           int lc, int C, int block, T* out) {
  pdl_enter();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= layers * C) return;
  const int l = idx / C, c = idx % C;
  int n = *n_dev;
  n = n < 0 ? 0 : (n > block ? block : n);
  T row[kShortConvMaxL];
  for (int j = 0; j < lc - 1; ++j) {
    const int src = n + j;                                // index into concat(prev, bx[:n])
    if (src < lc - 1) row[j] = prev ? prev[((size_t)l * (lc - 1) + src) * C + c] : from_f<T>(0.f);
    else row[j] = bx[((size_t)l * block + (src - (lc - 1))) * C + c];
  }
  for (int j = 0; j < lc - 1; ++j) out[((size_t)l * (lc - 1) + j) * C + c] = row[j];
}

}  // namespace

cudaError_t launch_verify_sampled(int dtype, const SampledVerifyArgs& a, cudaStream_t st) {
  if (dtype) launch_pdl(verify_sampled_kernel<bf16>, dim3(a.B), dim3(kSampThreads), 0, st, a);
  else launch_pdl(verify_sampled_kernel<float>, dim3(a.B), dim3(kSampThreads), 0, st, a);
  return cudaGetLastError();
}

cudaError_t launch_short_conv(int dtype, const void* state, const void* bx, const void* w, int layers,
                              int lc, int C, int block, void* y, void* state_after, cudaStream_t st) {
  const int n = layers * C;
  const dim3 grid((n + 127) / 128), blk(128);
  if (dtype)
    launch_pdl(short_conv_kernel<bf16>, grid, blk, 0, st, (const bf16*)state, (const bf16*)bx, (const bf16*)w,
               layers, lc, C, block, (bf16*)y, (bf16*)state_after);
  else
    launch_pdl(short_conv_kernel<float>, grid, blk, 0, st, (const float*)state, (const float*)bx,
               (const float*)w, layers, lc, C, block, (float*)y, (float*)state_after);
  return cudaGetLastError();
}

cudaError_t launch_short_conv_rollback(int dtype, const void* prev, const void* bx, const int* n_dev,
                                       int layers, int lc, int C, int block, void* out, cudaStream_t st) {
  const int n = layers * C;
  const dim3 grid((n + 127) / 128), blk(128);
  if (dtype)
    launch_pdl(short_conv_rollback_kernel<bf16>, grid, blk, 0, st, (const bf16*)prev, (const bf16*)bx, n_dev,
               layers, lc, C, block, (bf16*)out);
  else
    launch_pdl(short_conv_rollback_kernel<float>, grid, blk, 0, st, (const float*)prev, (const float*)bx,
               n_dev, layers, lc, C, block, (float*)out);
  return cudaGetLastError();
}

}  // namespace dfl
