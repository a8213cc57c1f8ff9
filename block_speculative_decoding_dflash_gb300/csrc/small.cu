// Per-row kernels of the round: block embedding + RoPE table, RMSNorm,
// per-head q/k RMSNorm + RoPE, the K/V -> ring write, ring bookkeeping, the
// commit, and the stand-in target.
#include "kernels.h"
#include "launch.cuh"

namespace dfl {
namespace {

template <typename T>
__device__ __forceinline__ void copy8(const T* src, T* dst) {
  if (sizeof(T) == 2) {
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  } else {
    reinterpret_cast<float4*>(dst)[0] = reinterpret_cast<const float4*>(src)[0];
    reinterpret_cast<float4*>(dst)[1] = reinterpret_cast<const float4*>(src)[1];
  }
}

// Block input rows [anchor, mask, ..., mask] from the raw embedding table, and
// the RoPE table of the block positions p .. p+tab_rows-1.
template <typename T>
__global__ void embed_block_kernel(const T* E, int H, int vocab, RoundState* rs,
                                   int mask_id, int rows, T* x,
                                   const RingState* ring, const double* inv_freq,
                                   int half, int tab_rows, float2* rope,
                                   int anchor_host, long long expect_pos, int nseq) {
  pdl_enter();
  // sequence s of a batch takes rows s * rows .. and table rows s * tab_rows ..
  const int per = gridDim.x / nseq;
  const int sq = blockIdx.x / per, r = blockIdx.x % per;
  rs += sq;
  ring += sq;
  x += (size_t)sq * rows * H;
  rope += (size_t)sq * tab_rows * half;
  if (r == 0 && threadIdx.x == 0) {
    // A host-given anchor replaces the device-resident one (the Markov chain
    // that may follow seeds from it); a host-given position is checked
    // against the committed context length, which stays authoritative.
    if (anchor_host >= 0) rs->anchor = anchor_host;
    if (expect_pos >= 0 && ring->offset != expect_pos) atomicOr(&rs->error, kErrPos);
  }
  if (r < rows) {
    int tok = (r == 0) ? (anchor_host >= 0 ? anchor_host : rs->anchor) : mask_id;
    if (tok < 0 || tok >= vocab) {
      if (threadIdx.x == 0) atomicOr(&rs->error, kErrRange);
      tok = 0;
    }
    const T* src = E + (size_t)tok * H;
    T* dst = x + (size_t)r * H;
    for (int i = threadIdx.x * 8; i < H; i += blockDim.x * 8) copy8(src + i, dst + i);
  }
  if (r < tab_rows) {
    const long long pos = ring->offset + r;
    for (int i = threadIdx.x; i < half; i += blockDim.x)
      rope[(size_t)r * half + i] = rope_entry(inv_freq, i, pos);
  }
}

__global__ void rope_table_kernel(const double* inv_freq, int half, const RingState* ring,
                                  long long pos0, int rows, float2* rope) {
  pdl_enter();
  // table row blockIdx.x is row r of sequence s (rows per sequence)
  const int sq = blockIdx.x / rows, r = blockIdx.x % rows;
  const long long base = ring ? ring[sq].offset : pos0;
  for (int i = threadIdx.x; i < half; i += blockDim.x)
    rope[(size_t)blockIdx.x * half + i] = rope_entry(inv_freq, i, base + r);
}

template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const T* x, int ldx, const T* g,
                                                     T* y, int ldy, int H, float eps, KTrace tr) {
  if (threadIdx.x == 0) ktrace_mark(tr, 0);
  pdl_enter();
  if (threadIdx.x == 0) ktrace_mark(tr, 1);
  __shared__ float red[8];
  const int r = blockIdx.x;
  const T* xr = x + (size_t)r * ldx;
  float ss = 0.f;
  for (int i = threadIdx.x * 8; i < H; i += blockDim.x * 8) {
    float v[8];
    load8(xr + i, v);
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(v[e], v[e], ss);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    t = warp_sum(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float inv = rsqrtf(red[0] / static_cast<float>(H) + eps);
  T* yr = y + (size_t)r * ldy;
  for (int i = threadIdx.x * 8; i < H; i += blockDim.x * 8) {
    float v[8], gv[8];
    load8(xr + i, v);
    load8(g + i, gv);
#pragma unroll
    for (int e = 0; e < 8; ++e) yr[i + e] = from_f<T>(v[e] * inv * gv[e]);
  }
  if (tr.p) {
    __syncthreads();
    if (threadIdx.x == 0) ktrace_mark(tr, 2);
  }
}

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// The finish of a split-K GEMM whose CTAs added their fp32 partial sums into
// acc (bf16 path): per row, h = rnd(x + rnd(acc)) (or rnd(acc) when x is
// NULL), stored back into x, acc cleared for the next GEMM, then y =
// rnd(h / rms(h) * g). One CTA per row; each thread keeps its 8-element
// groups in registers between the passes (H <= 256 * 8 * kResidGroups).
constexpr int kResidGroups = 4;
__global__ void __launch_bounds__(256) resid_rmsnorm_kernel(bf16* x, int ldx, float* acc, int ldacc,
                                                           const bf16* g, bf16* y, int ldy, int H,
                                                           float eps, KTrace tr) {
  if (threadIdx.x == 0) ktrace_mark(tr, 0);
  // the gains are weights, written by no earlier kernel: load them before
  // waiting for the GEMM whose sums this kernel finishes
  float gv[kResidGroups][8];
#pragma unroll
  for (int q = 0; q < kResidGroups; ++q) {
    const int i = (threadIdx.x + q * blockDim.x) * 8;
    if (i < H) load8(g + i, gv[q]);
  }
  pdl_enter();
  if (threadIdx.x == 0) ktrace_mark(tr, 1);
  __shared__ float red[8];
  const int r = blockIdx.x;
  bf16* xr = x ? x + (size_t)r * ldx : nullptr;
  float* ar = acc + (size_t)r * ldacc;
  float h[kResidGroups][8];
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < kResidGroups; ++q) {
    const int i = (threadIdx.x + q * blockDim.x) * 8;
    if (i >= H) break;
    float xv[8];
    if (xr) load8(xr + i, xv);
    const float4 a0 = __ldcg(reinterpret_cast<const float4*>(ar + i));
    const float4 a1 = __ldcg(reinterpret_cast<const float4*>(ar + i + 4));
    const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    uint4 pk;
    uint32_t* w32 = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const float o0 = __bfloat162float(__float2bfloat16_rn(av[e]));
      const float o1 = __bfloat162float(__float2bfloat16_rn(av[e + 1]));
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(xr ? xv[e] + o0 : o0, xr ? xv[e + 1] + o1 : o1);
      h[q][e] = __low2float(b2);
      h[q][e + 1] = __high2float(b2);
      w32[e >> 1] = *reinterpret_cast<const uint32_t*>(&b2);
      ss = fmaf(h[q][e], h[q][e], ss);
      ss = fmaf(h[q][e + 1], h[q][e + 1], ss);
    }
    if (xr) *reinterpret_cast<uint4*>(xr + i) = pk;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    reinterpret_cast<float4*>(ar + i)[0] = z;
    reinterpret_cast<float4*>(ar + i)[1] = z;
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    t = warp_sum(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float inv = rsqrtf(red[0] / static_cast<float>(H) + eps);
  bf16* yr = y + (size_t)r * ldy;
#pragma unroll
  for (int q = 0; q < kResidGroups; ++q) {
    const int i = (threadIdx.x + q * blockDim.x) * 8;
    if (i >= H) break;
    uint4 pk;
    uint32_t* w32 = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const __nv_bfloat162 b2 =
          __floats2bfloat162_rn(h[q][e] * inv * gv[q][e], h[q][e + 1] * inv * gv[q][e + 1]);
      w32[e >> 1] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    *reinterpret_cast<uint4*>(yr + i) = pk;
  }
  if (tr.p) {
    __syncthreads();
    if (threadIdx.x == 0) ktrace_mark(tr, 2);
  }
}

// SwiGLU finish of a kEpiRedPair GEMM: blockIdx.y is the row, each thread
// one group of 8 columns.
__global__ void __launch_bounds__(256) swiglu_finish_kernel(float* acc, int ldacc, bf16* sout, int lds,
                                                           int I, KTrace tr) {
  if (threadIdx.x == 0) ktrace_mark(tr, 0);
  pdl_enter();
  if (threadIdx.x == 0) ktrace_mark(tr, 1);
  float* ar = acc + (size_t)blockIdx.y * ldacc;
  bf16* sr = sout + (size_t)blockIdx.y * lds;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  const int i = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (i < I) {
    const float4 g0 = __ldcg(reinterpret_cast<const float4*>(ar + i));
    const float4 g1 = __ldcg(reinterpret_cast<const float4*>(ar + i + 4));
    const float4 u0 = __ldcg(reinterpret_cast<const float4*>(ar + I + i));
    const float4 u1 = __ldcg(reinterpret_cast<const float4*>(ar + I + i + 4));
    const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const float u[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    uint4 pk;
    uint32_t* w32 = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      float o[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float gr = __bfloat162float(__float2bfloat16_rn(g[e + k]));
        const float ur = __bfloat162float(__float2bfloat16_rn(u[e + k]));
        o[k] = gr / (1.0f + expf(-gr)) * ur;
      }
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(o[0], o[1]);
      w32[e >> 1] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    *reinterpret_cast<uint4*>(sr + i) = pk;
    reinterpret_cast<float4*>(ar + i)[0] = z;
    reinterpret_cast<float4*>(ar + i)[1] = z;
    reinterpret_cast<float4*>(ar + I + i)[0] = z;
    reinterpret_cast<float4*>(ar + I + i)[1] = z;
  }
  if (tr.p) {
    __syncthreads();
    if (threadIdx.x == 0) ktrace_mark(tr, 2);
  }
}

// One warp per (row, head): RMSNorm over hd with gain g[hd], then RoPE with
// the row's (cos, sin) table; the result is rounded once. src may equal dst.
template <typename T>
__device__ __forceinline__ void norm_rope_warp(const T* src, T* dst, int hd,
                                               const T* g, float eps,
                                               const float2* rope_row, int neox,
                                               float* sm) {
  const int lane = threadIdx.x & 31;
  float ss = 0.f;
  for (int d = lane; d < hd; d += 32) {
    const float v = to_f(src[d]);
    sm[d] = v;
    ss = fmaf(v, v, ss);
  }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / static_cast<float>(hd) + eps);
  __syncwarp();
  for (int d = lane; d < hd; d += 32) sm[d] = sm[d] * inv * to_f(g[d]);
  __syncwarp();
  const int half = hd >> 1;
  for (int i = lane; i < half; i += 32) {
    const int ia = neox ? i : 2 * i;
    const int ib = neox ? i + half : 2 * i + 1;
    const float2 cs = rope_row[i];
    const float a = sm[ia], b = sm[ib];
    dst[ia] = from_f<T>(a * cs.x - b * cs.y);
    dst[ib] = from_f<T>(a * cs.y + b * cs.x);
  }
  __syncwarp();
}

constexpr int kMaxHd = 256;

template <typename T>
__global__ void __launch_bounds__(128) head_norm_rope_kernel(T* buf, int ld, int rows,
                                                             int heads, int hd, const T* g,
                                                             float eps, const float2* rope,
                                                             int neox) {
  pdl_enter();
  __shared__ float sm[4][kMaxHd];
  const int warp = threadIdx.x >> 5;
  const int item = blockIdx.x * 4 + warp;
  if (item >= rows * heads) return;
  const int r = item / heads, h = item % heads;
  T* p = buf + (size_t)r * ld + (size_t)h * hd;
  norm_rope_warp(p, p, hd, g, eps, rope + (size_t)r * (hd >> 1), neox, sm[warp]);
}

// kv [rows, 2*nkv*hd]: K heads then V heads. K: norm + RoPE into the ring; V:
// copied into the ring. Ring layout [nkv][cap][hd].
template <typename T>
__global__ void __launch_bounds__(128) kv_to_ring_kernel(const T* kv, int ld, int rows,
                                                         int nkv, int hd, const T* kg,
                                                         float eps, const float2* rope,
                                                         int neox, T* ring_k, T* ring_v,
                                                         long long cap, int append_only,
                                                         RingState* ring, int use_dev,
                                                         long long pos_host, int rows_per_seq,
                                                         long long seq_kv) {
  pdl_enter();
  __shared__ float sm[4][kMaxHd];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x * 4 + warp;
  if (item >= rows * nkv) return;
  const int r = item / nkv, h = item % nkv;
  const int sq = r / rows_per_seq;
  ring += sq;
  ring_k += (size_t)sq * seq_kv;
  ring_v += (size_t)sq * seq_kv;
  const long long pos = (use_dev ? ring->offset : pos_host) + r % rows_per_seq;
  if (append_only && pos - ring->base >= cap) {
    if (lane == 0) atomicOr(&ring->error, kErrFull);
    return;
  }
  const long long slot = ring_slot(pos, cap);
  const T* ksrc = kv + (size_t)r * ld + (size_t)h * hd;
  const T* vsrc = kv + (size_t)r * ld + (size_t)(nkv + h) * hd;
  T* kdst = ring_k + ((size_t)h * cap + slot) * hd;
  T* vdst = ring_v + ((size_t)h * cap + slot) * hd;
  norm_rope_warp(ksrc, kdst, hd, kg, eps, rope + (size_t)r * (hd >> 1), neox, sm[warp]);
  for (int d = lane; d < hd; d += 32) vdst[d] = vsrc[d];
}

// Finish of the append's K/V GEMM (kEpiRed, head_dim 128): the fp32 sums of
// block row r for layer l are acc[r][l * 2 kvdim + (K heads | V heads)];
// each K head is rounded (the GEMM's output rounding), RMS-normalised with
// the layer's k-norm gain and rotated at position ring->offset + r, each V
// head rounded, both stored into the ring slot; the sums are cleared. One
// warp per (row, layer, kv head), four dims a lane.
__global__ void __launch_bounds__(128) kv_acc_to_ring_kernel(float* acc, int ldacc, int rows, int L,
                                                            int nkv, const void* const* kgain, float eps,
                                                            const float2* rope, int neox, bf16* ring_k,
                                                            bf16* ring_v, long long cap, int append_only,
                                                            RingState* ring, int rows_per_seq,
                                                            long long seq_kv) {
  pdl_enter();
  __shared__ float sm[4][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x * 4 + warp;
  if (item >= rows * L * nkv) return;
  const int r = item / (L * nkv), l = (item / nkv) % L, h = item % nkv;
  const int kvdim = nkv * 128;
  float* kacc = acc + (size_t)r * ldacc + (size_t)l * 2 * kvdim + h * 128;
  float* vacc = kacc + kvdim;
  const float4 k4 = __ldcg(reinterpret_cast<const float4*>(kacc) + lane);
  const float4 v4 = __ldcg(reinterpret_cast<const float4*>(vacc) + lane);
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  reinterpret_cast<float4*>(kacc)[lane] = z;
  reinterpret_cast<float4*>(vacc)[lane] = z;
  // row r of the batch is row r % rows_per_seq of sequence r / rows_per_seq
  const int sq = r / rows_per_seq;
  ring += sq;
  ring_k += (size_t)sq * seq_kv;
  ring_v += (size_t)sq * seq_kv;
  const long long pos = ring->offset + r % rows_per_seq;
  if (append_only && pos - ring->base >= cap) {
    if (lane == 0) atomicOr(&ring->error, kErrFull);
    return;
  }
  const long long slot = ring_slot(pos, cap);
  const size_t head = (((size_t)l * nkv + h) * cap + slot) * 128;
  // V: rounded and stored
  {
    uint2 pk;
    pk.x = pack_bf2(v4.x, v4.y);
    pk.y = pack_bf2(v4.z, v4.w);
    reinterpret_cast<uint2*>(ring_v + head)[lane] = pk;
  }
  // K: rounded, head RMSNorm, gain, RoPE, rounded once more
  const float kv[4] = {rnd<bf16>(k4.x), rnd<bf16>(k4.y), rnd<bf16>(k4.z), rnd<bf16>(k4.w)};
  float ss = kv[0] * kv[0] + kv[1] * kv[1] + kv[2] * kv[2] + kv[3] * kv[3];
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / 128.0f + eps);
  const bf16* g = reinterpret_cast<const bf16*>(kgain[l]);
#pragma unroll
  for (int e = 0; e < 4; ++e) sm[warp][lane * 4 + e] = kv[e] * inv * __bfloat162float(g[lane * 4 + e]);
  __syncwarp();
  const float2* rr = rope + (size_t)r * 64;
  bf16* kd = ring_k + head;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int i = lane + 32 * q;                         // rotation pair i of 64
    const int ia = neox ? i : 2 * i, ib = neox ? i + 64 : 2 * i + 1;
    const float2 cs = rr[i];
    const float a = sm[warp][ia], b = sm[warp][ib];
    kd[ia] = __float2bfloat16_rn(a * cs.x - b * cs.y);
    kd[ib] = __float2bfloat16_rn(a * cs.y + b * cs.x);
  }
}

// Finish of the QKV GEMM's fp32 sums (bf16, head_dim 128): one warp per
// (row, head) of the nq + 2 nkv heads, four dims a lane; every value rounded
// (the GEMM's output rounding); q and k heads then the per-head RMSNorm (gains
// qn / kn) and RoPE (rope[r][64]), rounded once more; the sums cleared. It
// waits for the GEMM before it lets the attention launch, so everything
// before the GEMM is complete once the attention runs: the attention may read
// the ring's context rows before its own dependency resolves.
__global__ void __launch_bounds__(128) qkv_finish_kernel(float* acc, int ldacc, bf16* out, int ldo, int rows,
                                                        int nq, int nkv, const bf16* qn, const bf16* kn,
                                                        float eps, const float2* rope, int neox, KTrace tr) {
  if (threadIdx.x == 0) ktrace_mark(tr, 0);
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) ktrace_mark(tr, 1);
  __shared__ float sm[4][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int heads = nq + 2 * nkv;
  const int item = blockIdx.x * 4 + warp;
  if (item < rows * heads) {
    const int r = item / heads, h = item % heads;
    float* src = acc + (size_t)r * ldacc + (size_t)h * 128;
    const float4 v4 = __ldcg(reinterpret_cast<const float4*>(src) + lane);
    reinterpret_cast<float4*>(src)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
    const float x[4] = {rnd<bf16>(v4.x), rnd<bf16>(v4.y), rnd<bf16>(v4.z), rnd<bf16>(v4.w)};
    bf16* dst = out + (size_t)r * ldo + (size_t)h * 128;
    if (h >= nq + nkv) {                               // V: rounded
      uint2 pk;
      pk.x = pack_bf2(x[0], x[1]);
      pk.y = pack_bf2(x[2], x[3]);
      reinterpret_cast<uint2*>(dst)[lane] = pk;
    } else {                                           // q or k: head RMSNorm, gain, RoPE
      const bf16* g = h < nq ? qn : kn;
      float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
      ss = warp_sum(ss);
      const float inv = rsqrtf(ss / 128.0f + eps);
#pragma unroll
      for (int e = 0; e < 4; ++e) sm[warp][lane * 4 + e] = x[e] * inv * __bfloat162float(g[lane * 4 + e]);
      __syncwarp();
      const float2* rr = rope + (size_t)r * 64;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int i = lane + 32 * q;                   // rotation pair i of 64
        const int ia = neox ? i : 2 * i, ib = neox ? i + 64 : 2 * i + 1;
        const float2 cs = rr[i];
        const float a = sm[warp][ia], b = sm[warp][ib];
        dst[ia] = __float2bfloat16_rn(a * cs.x - b * cs.y);
        dst[ib] = __float2bfloat16_rn(a * cs.y + b * cs.x);
      }
    }
  }
  if (tr.p) {
    __syncthreads();
    if (threadIdx.x == 0) ktrace_mark(tr, 2);
  }
}

// ---- the synthetic target's verify forward --------------------------------------
// x[r] = E[tokens[r]]; a token outside the vocabulary reads row 0 and sets
// kErrRange in rs.
template <typename T>
__global__ void embed_tokens_kernel(const T* E, int H, int vocab, const int* tokens, T* x, RoundState* rs) {
  pdl_enter();
  const int r = blockIdx.x;
  int tok = tokens[r];
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0) atomicOr(&rs->error, kErrRange);
    tok = 0;
  }
  const T* src = E + (size_t)tok * H;
  T* dst = x + (size_t)r * H;
  for (int i = threadIdx.x * 8; i < H; i += blockDim.x * 8) copy8(src + i, dst + i);
}

// The verify block [anchor, d_1 .. d_{block-1}] from the drafter's round
// state; the drafter's committed length must be the target's (kErrPos in trs
// otherwise).
__global__ void verify_tokens_kernel(const RoundState* drs, const RingState* dring, const int* d, int block,
                                     int* tokens, const RingState* tring, RoundState* trs) {
  pdl_enter();
  for (int i = threadIdx.x; i < block; i += blockDim.x) tokens[i] = i == 0 ? drs->anchor : d[i - 1];
  if (threadIdx.x == 0 && dring->offset != tring->offset) atomicOr(&trs->error, kErrPos);
}

// K and V of `rows` block rows (the finished QKV output: K at column kofs, V
// at vofs of each row, nkv heads of hd) into the ring slots of positions
// ring->offset + r; an append-only ring refuses rows past its capacity.
template <typename T>
__global__ void kv_rows_to_ring_kernel(const T* qkv, int ld, int kofs, int vofs, int rows, int nkv, int hd,
                                       T* ring_k, T* ring_v, long long cap, int append_only, RingState* ring) {
  pdl_enter();
  const int chunks = hd / 8;
  const int item = blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= rows * nkv * chunks) return;
  const int r = item / (nkv * chunks), h = (item / chunks) % nkv, c = item % chunks;
  const long long pos = ring->offset + r;
  if (append_only && pos - ring->base >= cap) {
    if (c == 0) atomicOr(&ring->error, kErrFull);
    return;
  }
  const long long slot = ring_slot(pos, cap);
  const size_t src = (size_t)r * ld + (size_t)h * hd + c * 8;
  const size_t dst = ((size_t)h * cap + slot) * hd + c * 8;
  copy8(qkv + kofs + src, ring_k + dst);
  copy8(qkv + vofs + src, ring_v + dst);
}

// The trim after a verify of `block` rows: every layer drops the last
// block - n rows, n = *n_dev (the verify's accepted + 1); a and b are the
// sliding and full layers' ring states (b may be NULL).
__global__ void target_trim_kernel(RingState* a, RingState* b, const int* n_dev, int block, RoundState* trs) {
  pdl_enter();
  if (threadIdx.x != 0) return;
  const int d = block - *n_dev;
  RingState* rr[2] = {a, b};
  for (int i = 0; i < 2; ++i) {
    RingState* r = rr[i];
    if (!r) continue;
    if (d < 0 || d >= block || d > r->appended) {
      atomicOr(&trs->error, kErrTrim);
      continue;
    }
    r->offset -= d;
    r->appended = 0;
  }
}

// ---- ring bookkeeping ------------------------------------------------------------
__global__ void ring_advance_kernel(RingState* ring, int d, int mode) {
  pdl_enter();
  ring += threadIdx.x;                         // one thread per sequence
  if (mode == 1) {
    ring->offset -= d;
    ring->appended = 0;
  } else {
    ring->offset += d;
    if (ring->offset - 1 > ring->hw) ring->hw = ring->offset - 1;
    ring->appended = (mode == 0) ? ring->appended + d : 0;
  }
}

__global__ void ring_reset_kernel(RingState* ring, long long base) {
  pdl_enter();
  ring->offset = base;
  ring->base = base;
  ring->hw = base - 1;
  ring->appended = 0;
  ring->error = 0;
}

__global__ void set_anchor_kernel(RoundState* rs, int anchor) {
  pdl_enter(); rs->anchor = anchor; }

// Partial-accept rollback: the block's `block` rows were appended (offset
// advanced by block); keep the first `keep` (keep < 0: the verify's n).
__global__ void commit_kernel(RoundState* rs, RingState* ring, int block, int keep) {
  pdl_enter();
  rs += threadIdx.x;                           // one thread per sequence
  ring += threadIdx.x;
  const int k = keep >= 0 ? keep : rs->n;
  ring->offset -= (block - k);
  ring->appended = 0;
  rs->anchor = rs->bonus;
  rs->rounds += 1;
  rs->proposed += block - 1;
  rs->accepted += rs->a;
  rs->emitted += rs->a + 1;
}

template <typename T>
__global__ void ring_append_kernel(const T* k, const T* v, int L, int n, int nkv,
                                   int hd, T* ring_k, T* ring_v, long long cap,
                                   const RingState* ring) {
  pdl_enter();
  const long long total = (long long)L * n * nkv;
  for (long long it = blockIdx.x; it < total; it += gridDim.x) {
    const int h = static_cast<int>(it % nkv);
    const int j = static_cast<int>((it / nkv) % n);
    const int l = static_cast<int>(it / ((long long)nkv * n));
    const long long slot = ring_slot(ring->offset + j, cap);
    const size_t src = (((size_t)l * n + j) * nkv + h) * hd;
    const size_t dst = (((size_t)l * nkv + h) * cap + slot) * hd;
    for (int d = threadIdx.x; d < hd; d += blockDim.x) {
      ring_k[dst + d] = k[src + d];
      ring_v[dst + d] = v[src + d];
    }
  }
}

template <typename T>
__global__ void ring_gather_kernel(const T* ring_k, const T* ring_v, int L,
                                   long long cap, int nkv, int hd, long long pos0,
                                   int count, T* k_out, T* v_out) {
  pdl_enter();
  const long long total = (long long)L * count * nkv;
  for (long long it = blockIdx.x; it < total; it += gridDim.x) {
    const int h = static_cast<int>(it % nkv);
    const int j = static_cast<int>((it / nkv) % count);
    const int l = static_cast<int>(it / ((long long)nkv * count));
    const long long slot = ring_slot(pos0 + j, cap);
    const size_t dst = (((size_t)l * count + j) * nkv + h) * hd;
    const size_t src = (((size_t)l * nkv + h) * cap + slot) * hd;
    for (int d = threadIdx.x; d < hd; d += blockDim.x) {
      k_out[dst + d] = ring_k[src + d];
      v_out[dst + d] = ring_v[src + d];
    }
  }
}

// ---- stand-in target -------------------------------------------------------------
template <typename T>
__global__ void synth_target_kernel(SynthArgs a) {
  if (threadIdx.x == 0) ktrace_mark(a.trace, 0);
  pdl_enter();
  if (threadIdx.x == 0) ktrace_mark(a.trace, 1);
  // sequence blockIdx.z of a batch draws pool entry r * nseq + s
  const int sq = blockIdx.z;
  const long long r = a.rs[sq].rounds * a.nseq + sq;
  const int kl = static_cast<int>(r % a.n_logit);
  const int kc = static_cast<int>(r % a.n_coin);
  const int kr = static_cast<int>(r % a.n_resid);
  a.d += (size_t)sq * (a.block - 1);
  a.logits_out = static_cast<char*>(a.logits_out) + (size_t)sq * a.block * a.V * sizeof(T);
  a.resid_out = static_cast<char*>(a.resid_out) + (size_t)sq * a.block * a.kin * sizeof(T);
  // block row i = blockIdx.y; this thread's 8 consecutive elements of the
  // row's logits and of its residual row (16-byte copies when both rows are
  // 16-byte aligned, element by element otherwise)
  const int i = blockIdx.y;
  const int v = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  const T* L = reinterpret_cast<const T*>(a.logit_pool) + ((size_t)kl * a.block_max + i) * a.V;
  const T* R = reinterpret_cast<const T*>(a.resid_pool) + ((size_t)kr * a.block_max + i) * a.kin;
  T* Lo = reinterpret_cast<T*>(a.logits_out) + (size_t)i * a.V;
  T* Ro = reinterpret_cast<T*>(a.resid_out) + (size_t)i * a.kin;
  const bool plant = i < a.block - 1 && a.coins[(size_t)kc * a.block_max + i];
  const int di = plant ? a.d[i] : -1;
  const T pv = plant ? reinterpret_cast<const T*>(a.plant)[(size_t)kl * a.block_max + i] : T{};
  const bool vec = a.vec != 0;
  if (v < a.V) {
    if (vec && v + 8 <= a.V) {
      uint4 u[sizeof(T) / 2];
#pragma unroll
      for (int k = 0; k < (int)(sizeof(T) / 2); ++k) u[k] = reinterpret_cast<const uint4*>(L + v)[k];
      T* ue = reinterpret_cast<T*>(u);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (v + e == di) ue[e] = pv;
#pragma unroll
      for (int k = 0; k < (int)(sizeof(T) / 2); ++k) reinterpret_cast<uint4*>(Lo + v)[k] = u[k];
    } else {
      for (int e = v; e < v + 8 && e < a.V; ++e) Lo[e] = e == di ? pv : L[e];
    }
  }
  if (v < a.kin) {
    if (vec && v + 8 <= a.kin) {
#pragma unroll
      for (int k = 0; k < (int)(sizeof(T) / 2); ++k)
        reinterpret_cast<uint4*>(Ro + v)[k] = reinterpret_cast<const uint4*>(R + v)[k];
    } else {
      for (int e = v; e < v + 8 && e < a.kin; ++e) Ro[e] = R[e];
    }
  }
  if (a.trace.p) {
    __syncthreads();
    if (threadIdx.x == 0) ktrace_mark(a.trace, 2);
  }
}

}  // namespace

cudaError_t launch_embed_block(int dtype, const void* embed, int H, int vocab, RoundState* rs,
                               int mask_id, int rows, void* x, const RingState* ring,
                               const double* inv_freq, int half, int tab_rows, float2* rope,
                               int anchor_host, long long expect_pos, cudaStream_t st, int nseq) {
  const int grid = (rows > tab_rows ? rows : tab_rows) * nseq;
  if (dtype)
    launch_pdl(embed_block_kernel<bf16>, dim3(grid), dim3(256), 0, st, (const bf16*)embed, H, vocab, rs, mask_id,
                                                   rows, (bf16*)x, ring, inv_freq, half,
                                                   tab_rows, rope, anchor_host, expect_pos, nseq);
  else
    launch_pdl(embed_block_kernel<float>, dim3(grid), dim3(256), 0, st, (const float*)embed, H, vocab, rs, mask_id,
                                                    rows, (float*)x, ring, inv_freq, half,
                                                    tab_rows, rope, anchor_host, expect_pos, nseq);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(const double* inv_freq, int half, const RingState* ring,
                              long long pos0, int rows, float2* rope, cudaStream_t st, int nseq) {
  if (rows <= 0) return cudaSuccess;
  launch_pdl(rope_table_kernel, dim3(rows * nseq), dim3(64), 0, st, inv_freq, half, ring, pos0, rows, rope);
  return cudaGetLastError();
}

cudaError_t launch_resid_rmsnorm(void* x, int ldx, float* acc, int ldacc, const void* g, void* y,
                                 int ldy, int rows, int H, float eps, cudaStream_t st, KTrace tr) {
  if (rows <= 0) return cudaSuccess;
  if (H % 8 || H > 256 * 8 * kResidGroups || ldacc % 4 || (x && ldx % 8) || ldy % 8)
    return cudaErrorInvalidValue;
  launch_pdl(resid_rmsnorm_kernel, dim3(rows), dim3(256), 0, st, (bf16*)x, ldx, acc, ldacc,
             (const bf16*)g, (bf16*)y, ldy, H, eps, tr);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_finish(float* acc, int ldacc, void* sout, int lds, int rows, int I,
                                 cudaStream_t st, KTrace tr) {
  if (rows <= 0) return cudaSuccess;
  if (I % 8 || ldacc % 4 || lds % 8) return cudaErrorInvalidValue;
  launch_pdl(swiglu_finish_kernel, dim3((I / 8 + 255) / 256, rows), dim3(256), 0, st, acc, ldacc,
             (bf16*)sout, lds, I, tr);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(int dtype, const void* x, int ldx, const void* g, void* y,
                           int ldy, int rows, int H, float eps, cudaStream_t st, KTrace tr) {
  if (rows <= 0) return cudaSuccess;
  if (dtype)
    launch_pdl(rmsnorm_kernel<bf16>, dim3(rows), dim3(256), 0, st, (const bf16*)x, ldx, (const bf16*)g, (bf16*)y,
                                               ldy, H, eps, tr);
  else
    launch_pdl(rmsnorm_kernel<float>, dim3(rows), dim3(256), 0, st, (const float*)x, ldx, (const float*)g,
                                                (float*)y, ldy, H, eps, tr);
  return cudaGetLastError();
}

cudaError_t launch_head_norm_rope(int dtype, void* buf, int ld, int rows, int heads, int hd,
                                  const void* g, float eps, const float2* rope, int neox,
                                  cudaStream_t st) {
  const int items = rows * heads;
  if (items <= 0) return cudaSuccess;
  const int grid = (items + 3) / 4;
  if (dtype)
    launch_pdl(head_norm_rope_kernel<bf16>, dim3(grid), dim3(128), 0, st, (bf16*)buf, ld, rows, heads, hd,
                                                      (const bf16*)g, eps, rope, neox);
  else
    launch_pdl(head_norm_rope_kernel<float>, dim3(grid), dim3(128), 0, st, (float*)buf, ld, rows, heads, hd,
                                                       (const float*)g, eps, rope, neox);
  return cudaGetLastError();
}

cudaError_t launch_kv_to_ring(int dtype, const void* kv, int ld, int rows, int nkv, int hd,
                              const void* kg, float eps, const float2* rope, int neox,
                              void* ring_k, void* ring_v, long long cap, int append_only,
                              RingState* ring, int use_dev, long long pos_host,
                              cudaStream_t st, int rows_per_seq, long long seq_kv) {
  const int items = rows * nkv;
  if (items <= 0) return cudaSuccess;
  const int grid = (items + 3) / 4;
  if (dtype)
    launch_pdl(kv_to_ring_kernel<bf16>, dim3(grid), dim3(128), 0, st, (const bf16*)kv, ld, rows, nkv, hd,
                                                  (const bf16*)kg, eps, rope, neox,
                                                  (bf16*)ring_k, (bf16*)ring_v, cap,
                                                  append_only, ring, use_dev, pos_host, rows_per_seq, seq_kv);
  else
    launch_pdl(kv_to_ring_kernel<float>, dim3(grid), dim3(128), 0, st, (const float*)kv, ld, rows, nkv, hd,
                                                   (const float*)kg, eps, rope, neox,
                                                   (float*)ring_k, (float*)ring_v, cap,
                                                   append_only, ring, use_dev, pos_host, rows_per_seq, seq_kv);
  return cudaGetLastError();
}

cudaError_t launch_kv_acc_to_ring(float* acc, int ldacc, int rows, int L, int nkv,
                                  const void* const* kgain, float eps, const float2* rope, int neox,
                                  void* ring_k, void* ring_v, long long cap, int append_only,
                                  RingState* ring, cudaStream_t st, KTrace tr, int rows_per_seq,
                                  long long seq_kv) {
  (void)tr;
  const int items = rows * L * nkv;
  if (items <= 0) return cudaSuccess;
  if (ldacc % 4 || rows_per_seq < 1) return cudaErrorInvalidValue;
  launch_pdl(kv_acc_to_ring_kernel, dim3((items + 3) / 4), dim3(128), 0, st, acc, ldacc, rows, L, nkv, kgain,
             eps, rope, neox, (bf16*)ring_k, (bf16*)ring_v, cap, append_only, ring, rows_per_seq, seq_kv);
  return cudaGetLastError();
}

cudaError_t launch_qkv_finish(float* acc, int ldacc, void* out, int ldo, int rows, int nq, int nkv,
                              const void* qn, const void* kn, float eps, const float2* rope, int neox,
                              cudaStream_t st, KTrace tr) {
  const int items = rows * (nq + 2 * nkv);
  if (items <= 0) return cudaSuccess;
  if (ldacc % 4 || ldo % 4) return cudaErrorInvalidValue;
  launch_pdl(qkv_finish_kernel, dim3((items + 3) / 4), dim3(128), 0, st, acc, ldacc, (bf16*)out, ldo, rows, nq,
             nkv, (const bf16*)qn, (const bf16*)kn, eps, rope, neox, tr);
  return cudaGetLastError();
}

cudaError_t launch_embed_tokens(int dtype, const void* embed, int H, int vocab, const int* tokens, int rows,
                                void* x, RoundState* rs, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (dtype)
    launch_pdl(embed_tokens_kernel<bf16>, dim3(rows), dim3(256), 0, st, (const bf16*)embed, H, vocab, tokens,
               (bf16*)x, rs);
  else
    launch_pdl(embed_tokens_kernel<float>, dim3(rows), dim3(256), 0, st, (const float*)embed, H, vocab, tokens,
               (float*)x, rs);
  return cudaGetLastError();
}

cudaError_t launch_verify_tokens(const RoundState* drs, const RingState* dring, const int* d, int block,
                                 int* tokens, const RingState* tring, RoundState* trs, cudaStream_t st) {
  launch_pdl(verify_tokens_kernel, dim3(1), dim3(128), 0, st, drs, dring, d, block, tokens, tring, trs);
  return cudaGetLastError();
}

cudaError_t launch_kv_rows_to_ring(int dtype, const void* qkv, int ld, int kofs, int vofs, int rows, int nkv,
                                   int hd, void* ring_k, void* ring_v, long long cap, int append_only,
                                   RingState* ring, cudaStream_t st) {
  const int items = rows * nkv * (hd / 8);
  if (items <= 0) return cudaSuccess;
  if (hd % 8 || ld % 8 || kofs % 8 || vofs % 8) return cudaErrorInvalidValue;
  const dim3 grid((items + 127) / 128), blk(128);
  if (dtype)
    launch_pdl(kv_rows_to_ring_kernel<bf16>, grid, blk, 0, st, (const bf16*)qkv, ld, kofs, vofs, rows, nkv, hd,
               (bf16*)ring_k, (bf16*)ring_v, cap, append_only, ring);
  else
    launch_pdl(kv_rows_to_ring_kernel<float>, grid, blk, 0, st, (const float*)qkv, ld, kofs, vofs, rows, nkv, hd,
               (float*)ring_k, (float*)ring_v, cap, append_only, ring);
  return cudaGetLastError();
}

cudaError_t launch_target_trim(RingState* a, RingState* b, const int* n_dev, int block, RoundState* trs,
                               cudaStream_t st) {
  launch_pdl(target_trim_kernel, dim3(1), dim3(32), 0, st, a, b, n_dev, block, trs);
  return cudaGetLastError();
}

cudaError_t launch_commit(RoundState* rs, RingState* ring, int block, int keep,
                          cudaStream_t st, int nseq) {
  launch_pdl(commit_kernel, dim3(1), dim3(nseq), 0, st, rs, ring, block, keep);
  return cudaGetLastError();
}

cudaError_t launch_ring_advance(RingState* ring, int d, int mode, cudaStream_t st, int nseq) {
  launch_pdl(ring_advance_kernel, dim3(1), dim3(nseq), 0, st, ring, d, mode);
  return cudaGetLastError();
}

cudaError_t launch_ring_reset(RingState* ring, long long base, cudaStream_t st) {
  launch_pdl(ring_reset_kernel, dim3(1), dim3(1), 0, st, ring, base);
  return cudaGetLastError();
}

cudaError_t launch_set_anchor(RoundState* rs, int anchor, cudaStream_t st) {
  launch_pdl(set_anchor_kernel, dim3(1), dim3(1), 0, st, rs, anchor);
  return cudaGetLastError();
}

cudaError_t launch_ring_append(int dtype, const void* k, const void* v, int L, int n, int nkv,
                               int hd, void* ring_k, void* ring_v, long long cap,
                               RingState* ring, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const long long items = (long long)L * n * nkv;
  const int grid = static_cast<int>(items < 4096 ? items : 4096);
  if (dtype)
    launch_pdl(ring_append_kernel<bf16>, dim3(grid), dim3(128), 0, st, (const bf16*)k, (const bf16*)v, L, n, nkv,
                                                   hd, (bf16*)ring_k, (bf16*)ring_v, cap, ring);
  else
    launch_pdl(ring_append_kernel<float>, dim3(grid), dim3(128), 0, st, (const float*)k, (const float*)v, L, n, nkv,
                                                    hd, (float*)ring_k, (float*)ring_v, cap,
                                                    ring);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_ring_advance(ring, n, 0, st);
}

cudaError_t launch_ring_gather(int dtype, const void* ring_k, const void* ring_v, int L,
                               long long cap, int nkv, int hd, long long pos0, int count,
                               void* k_out, void* v_out, cudaStream_t st) {
  if (count <= 0) return cudaSuccess;
  const long long items = (long long)L * count * nkv;
  const int grid = static_cast<int>(items < 4096 ? items : 4096);
  if (dtype)
    launch_pdl(ring_gather_kernel<bf16>, dim3(grid), dim3(128), 0, st, (const bf16*)ring_k, (const bf16*)ring_v, L,
                                                   cap, nkv, hd, pos0, count, (bf16*)k_out,
                                                   (bf16*)v_out);
  else
    launch_pdl(ring_gather_kernel<float>, dim3(grid), dim3(128), 0, st, (const float*)ring_k, (const float*)ring_v,
                                                    L, cap, nkv, hd, pos0, count,
                                                    (float*)k_out, (float*)v_out);
  return cudaGetLastError();
}

cudaError_t launch_synth_target(int dtype, const SynthArgs& a, cudaStream_t st) {
  if (a.block <= 0) return cudaSuccess;
  SynthArgs b = a;
  const size_t esz = dtype ? 2 : 4;
  const auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  b.vec = (a.V * esz) % 16 == 0 && (a.kin * esz) % 16 == 0 && al16(a.logit_pool) && al16(a.resid_pool) &&
          al16(a.logits_out) && al16(a.resid_out);
  const int n = a.V > a.kin ? a.V : a.kin;
  if (b.nseq < 1) b.nseq = 1;
  const dim3 grid((n + 8 * 256 - 1) / (8 * 256), a.block, b.nseq);
  if (dtype) launch_pdl(synth_target_kernel<bf16>, grid, dim3(256), 0, st, b);
  else launch_pdl(synth_target_kernel<float>, grid, dim3(256), 0, st, b);
  return cudaGetLastError();
}

}  // namespace dfl
