// Linear layers of the drafter on CUDA cores.
//
// linear_rows_kernel: the M = block-rows case. Every weight byte is read once
// from HBM with 16-byte streaming loads; the few activation rows come from
// L1/L2. A CTA owns 4 output features and its 4 warps split K, so an
// N = 2048 layer already spreads over 512 CTAs. More than 16 rows are done in
// passes of 16 (later passes re-read the CTA's weight rows from L2).
//
// linear_tiled_kernel: the many-rows case (context ingest), a 64x64 fp32
// register-tiled GEMM.
//
// Both accumulate in fp32 and round once to the storage type at the
// epilogue (plus the residual / SwiGLU rounding points).
#include "kernels.h"
#include "launch.cuh"

namespace dfl {
namespace {

constexpr int kRowsNR = 4;       // output features per CTA
constexpr int kRowsWarps = 4;

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

template <typename T, int MT, int EPI>
__global__ void __launch_bounds__(kRowsWarps * 32)
linear_rows_kernel(LinearArgs a) {
  pdl_enter();
  constexpr int NR = kRowsNR;
  constexpr int NV = (EPI == kEpiSwiglu) ? 2 : 1;
  __shared__ float red[kRowsWarps][NV * NR * MT];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * NR;
  if (n0 >= a.N) return;
  int seg = 0;
  while (seg < a.nseg - 1 && n0 >= a.seg_end[seg]) ++seg;
  const int seg_start = seg ? a.seg_end[seg - 1] : 0;
  const int nrows = min(NR, a.seg_end[seg] - n0);
  const T* W = reinterpret_cast<const T*>(a.w[seg]) + (size_t)(n0 - seg_start) * a.K;
  const T* W2 = (EPI == kEpiSwiglu) ? reinterpret_cast<const T*>(a.w2) + (size_t)n0 * a.K : nullptr;
  const T* X = reinterpret_cast<const T*>(a.x);

  for (int m0 = 0; m0 < a.M; m0 += MT) {
    float acc[NV][NR][MT];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[v][r][m] = 0.f;

    for (int k = (warp * 32 + lane) * 8; k < a.K; k += kRowsWarps * 32 * 8) {
      float w[NV][NR][8];
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        if (r < nrows) {
          load8_stream(W + (size_t)r * a.K + k, w[0][r]);
          if (EPI == kEpiSwiglu) load8_stream(W2 + (size_t)r * a.K + k, w[NV - 1][r]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) { w[0][r][e] = 0.f; w[NV - 1][r][e] = 0.f; }
        }
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m0 + m < a.M) {
          float xv[8];
          load8(X + (size_t)(m0 + m) * a.ldx + k, xv);
#pragma unroll
          for (int v = 0; v < NV; ++v)
#pragma unroll
            for (int r = 0; r < NR; ++r) {
              float s = acc[v][r][m];
#pragma unroll
              for (int e = 0; e < 8; ++e) s = fmaf(w[v][r][e], xv[e], s);
              acc[v][r][m] = s;
            }
        }
      }
    }
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          float s = warp_sum(acc[v][r][m]);
          if (lane == 0) red[warp][(v * NR + r) * MT + m] = s;
        }
    __syncthreads();
    for (int t = threadIdx.x; t < NR * MT; t += blockDim.x) {
      const int r = t / MT, m = t % MT;
      if (r < nrows && m0 + m < a.M) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int w = 0; w < kRowsWarps; ++w) {
          s0 += red[w][(0 * NR + r) * MT + m];
          if (EPI == kEpiSwiglu) s1 += red[w][((NV - 1) * NR + r) * MT + m];
        }
        const int n = n0 + r, row = m0 + m;
        T* Y = reinterpret_cast<T*>(a.y) + (size_t)row * a.ldy + n;
        float out;
        if (EPI == kEpiStore) {
          out = s0;
        } else if (EPI == kEpiResid) {
          const T* R = reinterpret_cast<const T*>(a.r) + (size_t)row * a.ldr + n;
          out = to_f(*R) + rnd<T>(s0);
        } else {
          const float g = rnd<T>(s0), u = rnd<T>(s1);
          out = silu_f(g) * u;
        }
        *Y = from_f<T>(out);
      }
    }
    __syncthreads();
  }
}

template <typename T, int EPI>
cudaError_t rows_dispatch(const LinearArgs& a, cudaStream_t st) {
  dim3 grid((a.N + kRowsNR - 1) / kRowsNR), block(kRowsWarps * 32);
  const int mt = a.M;
  if (mt <= 1) launch_pdl(linear_rows_kernel<T, 1, EPI>, dim3(grid), dim3(block), 0, st, a);
  else if (mt <= 2) launch_pdl(linear_rows_kernel<T, 2, EPI>, dim3(grid), dim3(block), 0, st, a);
  else if (mt <= 4) launch_pdl(linear_rows_kernel<T, 4, EPI>, dim3(grid), dim3(block), 0, st, a);
  else if (mt <= 8) launch_pdl(linear_rows_kernel<T, 8, EPI>, dim3(grid), dim3(block), 0, st, a);
  else launch_pdl(linear_rows_kernel<T, 16, EPI>, dim3(grid), dim3(block), 0, st, a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t rows_epi(const LinearArgs& a, cudaStream_t st) {
  switch (a.epi) {
    case kEpiStore: return rows_dispatch<T, kEpiStore>(a, st);
    case kEpiResid: return rows_dispatch<T, kEpiResid>(a, st);
    default: return rows_dispatch<T, kEpiSwiglu>(a, st);
  }
}

// ---------------------------------------------------------------------------
// Tiled GEMM for the context side (many rows), store epilogue only.
// ---------------------------------------------------------------------------
constexpr int TB = 64, TK = 16;

template <typename T>
__global__ void __launch_bounds__(256) linear_tiled_kernel(LinearArgs a) {
  pdl_enter();
  __shared__ float As[TK][TB + 4];
  __shared__ float Bs[TK][TB + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * TB, n0 = blockIdx.x * TB;
  const T* A = reinterpret_cast<const T*>(a.x);
  float acc[4][4] = {};
  for (int k0 = 0; k0 < a.K; k0 += TK) {
    for (int e = threadIdx.x; e < TB * TK; e += 256) {
      const int row = e / TK, kk = e % TK;
      const int m = m0 + row, k = k0 + kk;
      As[kk][row] = (m < a.M && k < a.K) ? to_f(A[(size_t)m * a.ldx + k]) : 0.f;
      const int n = n0 + row;
      float bv = 0.f;
      if (n < a.N && k < a.K) {
        int s = 0;
        while (s < a.nseg - 1 && n >= a.seg_end[s]) ++s;
        const int ss = s ? a.seg_end[s - 1] : 0;
        bv = to_f(reinterpret_cast<const T*>(a.w[s])[(size_t)(n - ss) * a.K + k]);
      }
      Bs[kk][row] = bv;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { av[i] = As[kk][ty * 4 + i]; bv[i] = Bs[kk][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  T* Y = reinterpret_cast<T*>(a.y);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < a.N) Y[(size_t)m * a.ldy + n] = from_f<T>(acc[i][j]);
    }
  }
}

}  // namespace

cudaError_t launch_linear_rows(int dtype, const LinearArgs& a, cudaStream_t st) {
  if (a.M <= 0 || a.N <= 0) return cudaSuccess;
  return dtype ? rows_epi<bf16>(a, st) : rows_epi<float>(a, st);
}

cudaError_t launch_linear_tiled(int dtype, const LinearArgs& a, cudaStream_t st) {
  if (a.M <= 0 || a.N <= 0) return cudaSuccess;
  dim3 grid((a.N + TB - 1) / TB, (a.M + TB - 1) / TB);
  if (dtype) launch_pdl(linear_tiled_kernel<bf16>, dim3(grid), dim3(256), 0, st, a);
  else launch_pdl(linear_tiled_kernel<float>, dim3(grid), dim3(256), 0, st, a);
  return cudaGetLastError();
}

}  // namespace dfl
