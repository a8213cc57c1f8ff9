// Sliding-window grouped-query attention of a block of rows (the drafter's
// bidirectional mask, or a causal one for the target's verify forward)
// over the ring cache plus the block's own K/V.
//
// Keys are addressed by absolute position: the ring holds position q in slot
// q mod cap, and query row i (position p + i) sees key position k iff
// |p + i - k| <= W (W <= 0: every key). The key list -- context positions
// [kstart, p) followed by the block's rows -- is cut into splits of kKS
// keys; one CTA per (split, kv head) scores all rows*G queries of that kv
// head against its keys (each K/V byte is read once) and writes an
// online-softmax partial (max, sum, o[hd]); a combine kernel merges them.
// This CUDA-core version serves fp32 and head dims other than 128; bf16 with
// head_dim 128 goes to the tensor-core version in attention_mma.cu.
#include <math.h>

#include "kernels.h"
#include "launch.cuh"

namespace dfl {
namespace {

constexpr int kKS = 64;        // keys per split
constexpr int kWarps = 8;

template <typename T>
__global__ void __launch_bounds__(kWarps * 32) attn_partial_kernel(AttnArgs a, int nsplit) {
  pdl_enter();
  attn_select_seq(a, blockIdx.z, nsplit, sizeof(T), a.hd + 2);
  extern __shared__ float smem[];
  const int hd = a.hd, hdp = hd + 1;
  float* Ks = smem;                       // [kKS][hd+1]
  float* Vs = Ks + kKS * hdp;             // [kKS][hd+1]
  float* qs = Vs + kKS * hdp;             // [kWarps][hd]
  float* ps = qs + kWarps * hd;           // [kWarps][kKS]

  const int s = blockIdx.x, g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.nq / a.nkv;
  const int Qn = a.rows * G;
  const long long p = a.ring->offset;
  long long kstart = a.ring->base;
  if (a.window > 0 && p - a.window > kstart) kstart = p - a.window;
  const int nctx = static_cast<int>(p - kstart);
  const int nk = nctx + a.rows;
  const int j0 = s * kKS;
  float* part = a.partial + ((size_t)g * nsplit + s) * Qn * (hd + 2);

  if (j0 >= nk) {
    for (int qi = threadIdx.x; qi < Qn; qi += blockDim.x) {
      part[(size_t)qi * (hd + 2) + hd] = -INFINITY;
      part[(size_t)qi * (hd + 2) + hd + 1] = 0.f;
    }
    return;
  }
  const T* rk = reinterpret_cast<const T*>(a.ring_k) + (size_t)g * a.cap * hd;
  const T* rv = reinterpret_cast<const T*>(a.ring_v) + (size_t)g * a.cap * hd;
  const T* kb = reinterpret_cast<const T*>(a.kb);
  const T* vb = reinterpret_cast<const T*>(a.vb);
  for (int e = threadIdx.x; e < kKS * hd; e += blockDim.x) {
    const int j = e / hd, d = e % hd;
    const int kj = j0 + j;
    float kv = 0.f, vv = 0.f;
    if (kj < nctx) {
      const long long slot = ring_slot(kstart + kj, a.cap);
      kv = to_f(rk[slot * hd + d]);
      vv = to_f(rv[slot * hd + d]);
    } else if (kj < nk) {
      const int jb = kj - nctx;
      kv = to_f(kb[(size_t)jb * a.ldkv + (size_t)g * hd + d]);
      vv = to_f(vb[(size_t)jb * a.ldkv + (size_t)g * hd + d]);
    }
    Ks[j * hdp + d] = kv;
    Vs[j * hdp + d] = vv;
  }
  __syncthreads();

  const float scale = rsqrtf(static_cast<float>(hd));
  const T* qg = reinterpret_cast<const T*>(a.q);
  float* q = qs + warp * hd;
  float* pw = ps + warp * kKS;
  for (int qi = warp; qi < Qn; qi += kWarps) {
    const int r = qi / G, h = g * G + qi % G;
    for (int d = lane; d < hd; d += 32) q[d] = to_f(qg[(size_t)r * a.ldq + (size_t)h * hd + d]);
    __syncwarp();
    const long long qpos = p + r;
    float sc[kKS / 32];
    float mx = -INFINITY;
#pragma unroll
    for (int t = 0; t < kKS / 32; ++t) {
      const int j = lane + 32 * t;
      const int kj = j0 + j;
      float v = -INFINITY;
      if (kj < nk) {
        const long long kpos = kj < nctx ? kstart + kj : p + (kj - nctx);
        const long long dd = qpos - kpos;
        const bool vis = a.causal ? (dd >= 0 && (a.window <= 0 || dd <= a.window))
                                  : (a.window <= 0 || (dd < 0 ? -dd : dd) <= a.window);
        if (vis) {
          float acc = 0.f;
          const float* kr = Ks + j * hdp;
          for (int d = 0; d < hd; ++d) acc = fmaf(q[d], kr[d], acc);
          v = acc * scale;
        }
      }
      sc[t] = v;
      mx = fmaxf(mx, v);
    }
    mx = warp_max(mx);
    float l = 0.f;
#pragma unroll
    for (int t = 0; t < kKS / 32; ++t) {
      const float e = (mx == -INFINITY || sc[t] == -INFINITY) ? 0.f : expf(sc[t] - mx);
      pw[lane + 32 * t] = e;
      l += e;
    }
    l = warp_sum(l);
    __syncwarp();
    float* out = part + (size_t)qi * (hd + 2);
    for (int d = lane; d < hd; d += 32) {
      float o = 0.f;
      for (int j = 0; j < kKS; ++j) o = fmaf(pw[j], Vs[j * hdp + d], o);
      out[d] = o;
    }
    if (lane == 0) { out[hd] = mx; out[hd + 1] = l; }
    __syncwarp();
  }
}

template <typename T>
__global__ void attn_combine_kernel(AttnArgs a, int nsplit) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.nq / a.nkv;
  const int Qn = a.rows * G;
  int item = blockIdx.x * (blockDim.x >> 5) + warp;         // over nseq * nkv * Qn
  if (item >= (a.nseq > 1 ? a.nseq : 1) * a.nkv * Qn) return;
  attn_select_seq(a, item / (a.nkv * Qn), nsplit, sizeof(T), a.hd + 2);
  item %= a.nkv * Qn;
  const int g = item / Qn, qi = item % Qn;
  const int r = qi / G, h = g * G + qi % G;
  const int hd = a.hd;
  const float* base = a.partial + (size_t)g * nsplit * Qn * (hd + 2) + (size_t)qi * (hd + 2);
  const size_t sstride = (size_t)Qn * (hd + 2);
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, base[s * sstride + hd]);
  float L = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float ms = base[s * sstride + hd];
    if (ms != -INFINITY) L += expf(ms - M) * base[s * sstride + hd + 1];
  }
  T* out = reinterpret_cast<T*>(a.out) + (size_t)r * a.ldo + (size_t)h * hd;
  for (int d = lane; d < hd; d += 32) {
    float o = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float ms = base[s * sstride + hd];
      if (ms != -INFINITY) o += expf(ms - M) * base[s * sstride + d];
    }
    out[d] = from_f<T>(o / L);
  }
}

int num_splits(int rows, int max_ctx) { return (max_ctx + rows + kKS - 1) / kKS; }

size_t partial_smem(int hd) {
  return sizeof(float) * (2 * kKS * (hd + 1) + kWarps * hd + kWarps * kKS);
}

}  // namespace

size_t attention_scratch_floats(int rows, int nq, int nkv, int hd, int max_ctx) {
  return (size_t)nkv * num_splits(rows, max_ctx) * rows * (nq / nkv) * (hd + 2);
}

cudaError_t init_attention_attrs(int hd) {
  cudaError_t e = init_attention_mma_attrs();
  if (e != cudaSuccess) return e;
  const int smem = static_cast<int>(partial_smem(hd));
  e = cudaFuncSetAttribute(attn_partial_kernel<bf16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attn_partial_kernel<float>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

cudaError_t launch_attention(int dtype, const AttnArgs& a, cudaStream_t st) {
  if (attention_mma_ok(dtype, a.hd)) return launch_attention_mma(a, st);
  const int nsplit = num_splits(a.rows, a.max_ctx);
  const size_t smem = partial_smem(a.hd);
  const int ns = a.nseq > 1 ? a.nseq : 1;
  dim3 grid(nsplit, a.nkv, ns);
  if (dtype) launch_pdl(attn_partial_kernel<bf16>, dim3(grid), dim3(kWarps * 32), smem, st, a, nsplit);
  else launch_pdl(attn_partial_kernel<float>, dim3(grid), dim3(kWarps * 32), smem, st, a, nsplit);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int items = ns * a.nkv * a.rows * (a.nq / a.nkv);
  const int cgrid = (items + 3) / 4;
  if (dtype) launch_pdl(attn_combine_kernel<bf16>, dim3(cgrid), dim3(128), 0, st, a, nsplit);
  else launch_pdl(attn_combine_kernel<float>, dim3(cgrid), dim3(128), 0, st, a, nsplit);
  return cudaGetLastError();
}

}  // namespace dfl
