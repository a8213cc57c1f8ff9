// Sliding-window GQA attention of a block of rows (the drafter's
// bidirectional mask, or a causal one for the target's verify forward), bf16,
// head_dim 128, on tensor cores, one CTA per (split of kKeys = 128 keys, kv
// head g); the queries of g are the block rows x its G query heads.
//
// One 16-query tile at a time (attn_mma_kernel, mma.sync m16n8k16, fp32
// accumulate): each of the 8 warps scores the tile against 16 keys (S = Q
// K^T, mask |q - k| <= W by absolute positions) into shared memory; each warp
// then takes two query rows' softmax over the split (P as a high and a low
// bf16 part); each warp finally computes P V for 16 of the 128 output dims
// over all the split's keys and writes them to the CTA's partial (the tile
// loop serves any number of tiles; it runs for one). Two or more tiles:
// attn_tc_kernel (tcgen05.mma, below). A combine kernel (one warp per (query, head)) then
// merges the splits in split order and writes the bf16 output; nothing waits
// on another CTA and the result is deterministic.
//
// Keys are addressed by absolute position (ring slot = position mod cap), the
// context keys [kstart, p) followed by the block's own rows.
#include <math.h>

#include "attn_common.cuh"
#include "kernels.h"
#include "mma_sync.cuh"
#include "launch.cuh"

namespace dfl {
namespace {

constexpr int kHd = kAttnHd;
constexpr int kKeys = kAttnKeys;
constexpr int kWarps = 8;
constexpr int kPad = 8;                    // bf16 elements of row padding (conflict-free ldmatrix)
constexpr int kPartStride = kAttnPartStride;
constexpr int kQChunk = 64;

// Phase marks of the kernel trace (last CTA through each phase): slot + 2
// (k 1, 2) and slot + 3 (k 1, 2); slot + 1 is the merge kernel's.
__device__ __forceinline__ void attn_phase(const KTrace& t, int n) {
  if (t.p && threadIdx.x == 0) ktrace_mark(KTrace{t.p, t.slot + 2 + (n >> 1)}, 1 + (n & 1));
}

// This CTA's share of the two weights in a.l2_next (equal slices of their
// concatenation, in 4 KB multiples), asked into L2 in pieces of at most 1 MB.
__device__ __forceinline__ void attn_l2_prefetch_next(const AttnArgs& a) {
  if (!a.l2_next[0] || threadIdx.x != 0) return;
  const long long nct = (long long)gridDim.x * gridDim.y * gridDim.z;
  const long long id = blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z);
  const long long each = a.l2_next_bytes, total = 2 * each;
  const long long per = ((total + nct - 1) / nct + 4095) & ~4095LL;
  long long b0 = id * per;
  const long long b1 = b0 + per < total ? b0 + per : total;
  while (b0 < b1) {
    const int w = b0 >= each ? 1 : 0;
    const long long end = w ? b1 : (b1 < each ? b1 : each);
    const long long n = end - b0 < (1 << 20) ? end - b0 : (1 << 20);
    l2_prefetch_bulk(static_cast<const char*>(a.l2_next[w]) + (b0 - w * each), static_cast<uint32_t>(n));
    b0 += n;
  }
}

struct MmaSmem {
  bf16 k[kKeys][kHd + kPad];
  bf16 v[kKeys][kHd + kPad];
  bf16 q[kQChunk][kHd + kPad];            // up to 64 query rows, loaded with K/V
  float s[16][kKeys + 4];                  // scaled, masked scores of one query tile
  bf16 ph[16][kKeys + kPad];               // P = exp(S - M): high bf16 part
  bf16 pl[16][kKeys + kPad];               //                 low bf16 part
  float rm[16];                            // per query row: maximum score
  float rl[16];                            //                sum of P
};

__global__ void __launch_bounds__(kWarps * 32) attn_mma_kernel(AttnArgs a, int nsplit) {
  attn_select_seq(a, blockIdx.z, nsplit, 2, kPartStride);
  if (threadIdx.x == 0) ktrace_mark(a.trace, 0);
  extern __shared__ __align__(16) uint8_t smem_raw[];
  MmaSmem& S = *reinterpret_cast<MmaSmem*>(smem_raw);
  if (!a.early_ctx) {
    // (Measured: 3 us per draft faster at 4 block rows.)
    attn_prefetch_context(a, blockIdx.x, blockIdx.y);
    pdl_enter();
    if (threadIdx.x == 0) ktrace_mark(a.trace, 1);
  }
  const int s = blockIdx.x, g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.nq / a.nkv;
  const int Qn = a.rows * G;
  const long long p = a.ring->offset;
  long long kstart = a.ring->base;
  if (a.window > 0 && p - a.window > kstart) kstart = p - a.window;
  const int nctx = static_cast<int>(p - kstart);
  const int nk = nctx + a.rows;
  const int j0 = s * kKeys;
  const int cap = static_cast<int>(a.cap);
  const int slot0 = static_cast<int>(ring_slot(kstart, a.cap));
  const size_t pstride = kPartStride;     // 16-byte aligned rows for float4 reads
  float* part = a.partial + ((size_t)g * nsplit + s) * Qn * pstride;
  const bf16* rk = reinterpret_cast<const bf16*>(a.ring_k) + (size_t)g * a.cap * kHd;
  const bf16* rv = reinterpret_cast<const bf16*>(a.ring_v) + (size_t)g * a.cap * kHd;
  const bf16* kb = reinterpret_cast<const bf16*>(a.kb);
  const bf16* vb = reinterpret_cast<const bf16*>(a.vb);
  const bf16* qg = reinterpret_cast<const bf16*>(a.q);

  auto load_q = [&](int q0) {
    const int rows = Qn - q0 < kQChunk ? Qn - q0 : kQChunk;
    for (int e = threadIdx.x; e < kQChunk * (kHd / 8); e += blockDim.x) {
      const int r = e >> 4, ch = e & 15;
      const int qi = q0 + r;
      const bool valid = r < rows;
      const size_t off = valid ? (size_t)(qi / G) * a.ldq + (size_t)(g * G + qi % G) * kHd + ch * 8 : 0;
      cp_async16(&S.q[r][ch * 8], qg + off, valid);
    }
  };
  // K and V tiles: 128 keys x 16 chunks of 16 bytes each; the context rows
  // (and zeros past the keys) first, before the dependency resolves when the
  // ring may be read then (a.early_ctx), the block's own rows after it.
  if (j0 < nk) {
    for (int e = threadIdx.x; e < kKeys * (kHd / 8); e += blockDim.x) {
      const int j = e >> 4, ch = e & 15;
      const int kj = j0 + j;
      if (kj >= nctx && kj < nk) continue;
      const bool valid = kj < nctx;
      int slot = slot0 + kj;                       // = ring_slot(kstart + kj, cap)
      if (slot >= cap) slot -= cap;
      const size_t off = valid ? (size_t)slot * kHd + ch * 8 : 0;
      cp_async16(&S.k[j][ch * 8], rk + off, valid);
      cp_async16(&S.v[j][ch * 8], rv + off, valid);
    }
  }
  if (a.early_ctx) {
    pdl_enter();
    if (threadIdx.x == 0) ktrace_mark(a.trace, 1);
  }
  if (j0 < nk) {
    const int kb0 = nctx > j0 ? nctx - j0 : 0;
    const int kb1 = nk - j0 < kKeys ? nk - j0 : kKeys;
    for (int e = threadIdx.x; e < (kb1 - kb0) * (kHd / 8); e += blockDim.x) {
      const int j = kb0 + (e >> 4), ch = e & 15;
      const size_t off = (size_t)(j0 + j - nctx) * a.ldkv + (size_t)g * kHd + ch * 8;
      cp_async16(&S.k[j][ch * 8], kb + off, true);
      cp_async16(&S.v[j][ch * 8], vb + off, true);
    }
  }
  load_q(0);
  cp_async_wait_all();
  __syncthreads();
  attn_phase(a.trace, 0);                          // K, V, q loaded
  attn_l2_prefetch_next(a);

  const int grp = lane >> 2, tig = lane & 3;
  const float scale = rsqrtf(static_cast<float>(kHd));
  for (int qt = 0; qt * 16 < Qn; ++qt) {
    const int qr = (qt * 16) % kQChunk;           // row of this tile in the Q chunk
    if (qt > 0 && qr == 0) {                      // next chunk of 64 queries
      load_q(qt * 16);
      cp_async_wait_all();
      __syncthreads();
    }
    // S = Q K^T: warp w scores the 16 queries of this tile against its 16
    // keys (two 8-key n-tiles), masks |q - k| <= W by absolute positions and
    // scales; the scores go to shared memory.
    {
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if (j0 < nk) {
#pragma unroll
        for (int ks = 0; ks < kHd / 16; ++ks) {
          uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
          const int mi = lane >> 3;
          ldsm_x4(&S.q[qr + (lane & 7) + (mi & 1) * 8][ks * 16 + (mi >> 1) * 8], a0, a1, a2, a3);
          ldsm_x4(&S.k[warp * 16 + (mi >> 1) * 8 + (lane & 7)][ks * 16 + (mi & 1) * 8], b0, b1, b2, b3);
          mma16816(sc[0], a0, a1, a2, a3, b0, b1);
          mma16816(sc[1], a0, a1, a2, a3, b2, b3);
        }
      }
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int qi = qt * 16 + grp + hr * 8;
        const long long qpos = p + (qi < Qn ? qi / G : 0);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int kk = warp * 16 + nt * 8 + tig * 2 + c;
            const int kj = j0 + kk;
            bool vis = qi < Qn && kj < nk;
            if (vis && (a.window > 0 || a.causal)) {
              const long long kpos = kj < nctx ? kstart + kj : p + (kj - nctx);
              const long long d = qpos - kpos;
              vis = a.causal ? (d >= 0 && (a.window <= 0 || d <= a.window)) : (d < 0 ? -d : d) <= a.window;
            }
            S.s[grp + hr * 8][kk] = vis ? sc[nt][hr * 2 + c] * scale : -INFINITY;
          }
      }
    }
    __syncthreads();
    if (qt == 0) attn_phase(a.trace, 1);            // first tile scored
    // Softmax rows: warp w takes query rows 2w and 2w + 1, four keys a lane;
    // P is kept as a high and a low bf16 part (about 16 significant bits).
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int r = warp * 2 + rr;
      const float4 v4 = *reinterpret_cast<const float4*>(&S.s[r][lane * 4]);
      const float v[4] = {v4.x, v4.y, v4.z, v4.w};
      float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
      mx = warp_max(mx);
      float pe[4], l = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pe[e] = (mx == -INFINITY || v[e] == -INFINITY) ? 0.f : expf(v[e] - mx);
        l += pe[e];
      }
      l = warp_sum(l);
      *reinterpret_cast<uint2*>(&S.ph[r][lane * 4]) = make_uint2(pack_bf16(pe[0], pe[1]), pack_bf16(pe[2], pe[3]));
      *reinterpret_cast<uint2*>(&S.pl[r][lane * 4]) =
          make_uint2(pack_bf16_residue(pe[0], pe[1]), pack_bf16_residue(pe[2], pe[3]));
      if (lane == 0) { S.rm[r] = mx; S.rl[r] = l; }
    }
    __syncthreads();
    if (qt == 0) attn_phase(a.trace, 2);            // first tile's softmax
    // O = P V: warp w owns output dims 16w .. 16w + 15 over all keys of the
    // split (eight 16-key steps, high and low parts of P)
    float o[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if (j0 < nk) {
#pragma unroll
      for (int ks = 0; ks < kKeys / 16; ++ks) {
        uint32_t h0, h1, h2, h3, l0, l1, l2, l3, b0, b1, b2, b3;
        const int mi = lane >> 3;
        ldsm_x4(&S.ph[(lane & 7) + (mi & 1) * 8][ks * 16 + (mi >> 1) * 8], h0, h1, h2, h3);
        ldsm_x4(&S.pl[(lane & 7) + (mi & 1) * 8][ks * 16 + (mi >> 1) * 8], l0, l1, l2, l3);
        ldsm_x4_t(&S.v[ks * 16 + (mi & 1) * 8 + (lane & 7)][warp * 16 + (mi >> 1) * 8], b0, b1, b2, b3);
        mma16816(o[0], h0, h1, h2, h3, b0, b1);
        mma16816(o[1], h0, h1, h2, h3, b2, b3);
        mma16816(o[0], l0, l1, l2, l3, b0, b1);
        mma16816(o[1], l0, l1, l2, l3, b2, b3);
      }
    }
    // the split's partial: unnormalised O, then the row's maximum and sum
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = grp + hr * 8;
      const int qi = qt * 16 + r;
      if (qi >= Qn) continue;
      float* out = part + (size_t)qi * pstride;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
        *reinterpret_cast<float2*>(out + warp * 16 + nt * 8 + tig * 2) = make_float2(o[nt][hr * 2], o[nt][hr * 2 + 1]);
      if (warp == 0 && tig == 0) { out[kHd] = S.rm[r]; out[kHd + 1] = S.rl[r]; }
    }
  }
  if (threadIdx.x == 0) ktrace_mark(a.trace, 2);
}

// One warp per (query, kv head): merge the splits' partials in split order.
__global__ void __launch_bounds__(128) attn_mma_combine_kernel(AttnArgs a, int nsplit) {
  const KTrace tr{a.trace.p, a.trace.slot + 1};
  if (threadIdx.x == 0) ktrace_mark(tr, 0);
  pdl_enter();
  if (threadIdx.x == 0) ktrace_mark(tr, 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.nq / a.nkv;
  const int Qn = a.rows * G;
  const int ns = a.nseq > 1 ? a.nseq : 1;
  const int item = blockIdx.x * 4 + warp;
  if (item < ns * a.nkv * Qn) {
    attn_select_seq(a, item / (a.nkv * Qn), nsplit, 2, kPartStride);
    const int it = item % (a.nkv * Qn);
    attn_combine_warp(a.partial, nsplit, nsplit, Qn, G, it / Qn, it % Qn,
                      reinterpret_cast<bf16*>(a.out), a.ldo, lane);
  }
  if (tr.p) {
    __syncthreads();
    if (threadIdx.x == 0) ktrace_mark(KTrace{tr.p, tr.slot + 3}, 1);   // merged
  }
  if (tr.p && threadIdx.x == 0) ktrace_mark(tr, 2);
}

constexpr int kTileQ = 64;                 // queries per kv head of the tensor-core kernel

// ---------------------------------------------------------------------------
// Up to 64 queries per kv head on the 5th-generation tensor cores. Per key
// split: S = Q K^T and then O = P V, 128 x 128 x 128 products issued as
// tcgen05.mma (kind::f16, fp32 accumulators in TMEM); P V is two products,
// of P's high and low bf16 parts, so P keeps about 16 significant bits. Operands are
// K-major shared-memory tiles in the 128-byte swizzled layout: Q and K as
// loaded, V transposed in shared memory (keys along K), P written by the
// softmax threads into Q's place once S is done.
//
// The 64 queries fill operand rows 0-63 and again 64-127, so that all eight
// warps can read S back (a warp reads the TMEM lanes of its quarter): row R
// holds query R mod 64, and its P row carries only the keys of its half
// (R < 64: keys 0-63, else 64-127; zeros elsewhere), so O = P V leaves two
// partial products per query, added when O is read back. Each thread takes
// 32 keys of one row for the softmax (the row's maximum and sum combine four
// threads through shared memory). Same partial format as the kernel above;
// the separate merge kernel combines the splits (folding the merge into this
// kernel, with every split of a head waiting for the others, measured 12 us
// per draft slower at 16 block rows: it keeps the 131 KB CTAs resident while
// the next GEMM's CTAs wait for their shared memory).
// ---------------------------------------------------------------------------
constexpr int kTcTileB = 128 * 128;                  // one 128-row x 64-column bf16 tile
constexpr int kTcQ = 0, kTcK = 2 * kTcTileB, kTcVt = 4 * kTcTileB, kTcVs = 6 * kTcTileB;
constexpr int kTcVsRow = kHd * 2 + 16;               // padded staging rows of V
constexpr int kTcBars = kTcVs + kKeys * kTcVsRow;
constexpr size_t kTcAttnSmem = (size_t)kTcBars + 64 + 1024;
constexpr int kTcOStride = kHd + 4;                  // O staging rows (floats), over K and V^T
static_assert(kTileQ * kTcOStride * 4 <= 4 * kTcTileB, "O staging must fit in the K and V^T tiles");
constexpr int kTileQWide = 128;            // queries per kv head of the wide variant

// Byte offset of element (row, col) of a 128-row x 128-column bf16 operand
// stored as two K-major 64-column tiles with 16-byte granules swizzled by row.
__device__ __forceinline__ uint32_t tc_sw128(int row, int col) {
  return (col >> 6) * kTcTileB + row * 128 + ((((col >> 3) & 7) ^ (row & 7)) << 4) + (col & 7) * 2;
}

// WIDE: more than 64 queries, in chunks of 128 over the same K and V^T, one
// operand row per query (row R = query R of the chunk, P rows over all 128
// keys), 16 warps: warps w, w + 4, w + 8, w + 12 read the same TMEM lanes and
// take keys 0-31, ..., 96-127 of those rows for the softmax; O needs no pair
// sum and each thread stores 32 dims of its row's partial directly.
template <bool WIDE>
__global__ void __launch_bounds__((WIDE ? 2 : 1) * kWarps * 32) attn_tc_kernel(AttnArgs a, int nsplit) {
  constexpr int TQ = WIDE ? kTileQWide : kTileQ;     // queries held
  constexpr int KPT = 32;                             // keys a thread takes in the softmax
  attn_select_seq(a, blockIdx.z, nsplit, 2, kPartStride);
  if (threadIdx.x == 0) ktrace_mark(a.trace, 0);
  if (!a.early_ctx) {
    pdl_enter();
    if (threadIdx.x == 0) ktrace_mark(a.trace, 1);
  }
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023) & ~1023u) - raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kTcBars);     // [0] S ready, [1] O ready
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar + 2);
  __shared__ float red_m[4][TQ], red_l[4][TQ];
  const int s = blockIdx.x, g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.nq / a.nkv;
  const int Qn = a.rows * G;
  const long long p = a.ring->offset;
  long long kstart = a.ring->base;
  const int window = a.window;
  if (window > 0 && p - window > kstart) kstart = p - window;
  const int nctx = static_cast<int>(p - kstart);
  const int nk = nctx + a.rows;
  const int j0 = s * kKeys;
  const int cap = static_cast<int>(a.cap);
  const int slot0 = static_cast<int>(ring_slot(kstart, a.cap));
  const int ldkv = a.ldkv, ldq = a.ldq;
  float* part = a.partial + ((size_t)g * nsplit + s) * Qn * kPartStride;
  const bf16* rk = reinterpret_cast<const bf16*>(a.ring_k) + (size_t)g * a.cap * kHd;
  const bf16* rv = reinterpret_cast<const bf16*>(a.ring_v) + (size_t)g * a.cap * kHd;
  const bf16* kb = reinterpret_cast<const bf16*>(a.kb) + (size_t)g * kHd;
  const bf16* vb = reinterpret_cast<const bf16*>(a.vb) + (size_t)g * kHd;
  const bf16* qg = reinterpret_cast<const bf16*>(a.q) + (size_t)g * G * kHd;

  // K into its tile, V into padded staging rows: the context rows and zeros
  // past the keys first (before the dependency resolves with a.early_ctx),
  // the block's own rows after it
  if (j0 < nk) {
    for (int e = threadIdx.x; e < kKeys * (kHd / 8); e += blockDim.x) {
      const int j = e >> 4, ch = e & 15;
      const int kj = j0 + j;
      if (kj >= nctx && kj < nk) continue;
      const bool valid = kj < nctx;
      int slot = slot0 + kj;
      if (slot >= cap) slot -= cap;
      const size_t off = valid ? (size_t)slot * kHd + ch * 8 : 0;
      cp_async16(sm + kTcK + tc_sw128(j, ch * 8), rk + off, valid);
      cp_async16(sm + kTcVs + j * kTcVsRow + ch * 16, rv + off, valid);
    }
  }
  if (a.early_ctx) {
    pdl_enter();
    if (threadIdx.x == 0) ktrace_mark(a.trace, 1);
  }
  if (j0 >= nk) {
    // a split past the keys: an empty partial (weight 0 in the merge)
    for (int e = threadIdx.x; e < Qn * kPartStride; e += blockDim.x) {
      const int d = e % kPartStride;
      part[e] = d == kHd ? -INFINITY : 0.f;
    }
    attn_l2_prefetch_next(a);
    if (a.trace.p) { __syncthreads(); if (threadIdx.x == 0) ktrace_mark(a.trace, 2); }
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_holder, 256);

  // the block's own keys and values, each query into rows r and r + 64
  {
    const int kb0 = nctx > j0 ? nctx - j0 : 0;
    const int kb1 = nk - j0 < kKeys ? nk - j0 : kKeys;
    for (int e = threadIdx.x; e < (kb1 - kb0) * (kHd / 8); e += blockDim.x) {
      const int j = kb0 + (e >> 4), ch = e & 15;
      const size_t off = (size_t)(j0 + j - nctx) * ldkv + ch * 8;
      cp_async16(sm + kTcK + tc_sw128(j, ch * 8), kb + off, true);
      cp_async16(sm + kTcVs + j * kTcVsRow + ch * 16, vb + off, true);
    }
  }
  for (int e = threadIdx.x; e < 2 * kTileQ * (kHd / 8); e += blockDim.x) {
    const int r = e >> 4, ch = e & 15, qr = WIDE ? r : (r & (kTileQ - 1));
    const bool valid = qr < Qn;
    const size_t off = valid ? (size_t)(qr / G) * ldq + (size_t)(qr % G) * kHd + ch * 8 : 0;
    cp_async16(sm + kTcQ + tc_sw128(r, ch * 8), qg + off, valid);
  }
  cp_async_wait_all();
  fence_proxy_async_shared();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  attn_phase(a.trace, 0);                          // K, V, q loaded
  attn_l2_prefetch_next(a);
  const uint32_t tmem = *tmem_holder;
  constexpr uint32_t idesc = idesc_bf16(128, 128);
  const uint32_t sbase = smem_u32(sm);
  // WIDE: the queries in chunks of 128 over the same K and V^T; P's low part
  // then goes into V's staging rows (free once V^T is built) so that K stays
  // for the next chunk's scores.
  const int nqc = WIDE ? (Qn + kTileQWide - 1) / kTileQWide : 1;
  const int plo = WIDE ? kTcVs : kTcK;
  static_assert(2 * kTcTileB <= kTcBars - kTcVs, "P's low part must fit in V's staging rows");
  const int quad = warp & 3, half = warp >> 2;          // half: 0-1 (WIDE: 0-3)
  const int R = quad * 32 + lane, rh = R >> 6;
  const int grp = WIDE ? half : rh * 2 + half;         // which quarter of the keys
  const int kc0 = grp * KPT;
  const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  const float sl2 = rsqrtf(static_cast<float>(kHd)) * 1.4426950408889634f;   // scale * log2(e)
  bool ok = true;
  for (int qc = 0; qc < nqc; ++qc) {
    if (qc > 0) {
      // the next 128 queries into Q's tiles (the last P V is done with them)
      for (int e = threadIdx.x; e < kTileQWide * (kHd / 8); e += blockDim.x) {
        const int r = e >> 4, ch = e & 15, qr = qc * kTileQWide + r;
        const bool valid = qr < Qn;
        const size_t off = valid ? (size_t)(qr / G) * ldq + (size_t)(qr % G) * kHd + ch * 8 : 0;
        cp_async16(sm + kTcQ + tc_sw128(r, ch * 8), qg + off, valid);
      }
      cp_async_wait_all();
      fence_proxy_async_shared();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
    if (threadIdx.x == 0) {
#pragma unroll
      for (int kc = 0; kc < 2; ++kc)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_bf16(tmem, smem_desc_sw128(sbase + kTcQ + kc * kTcTileB + kk * 32),
                      smem_desc_sw128(sbase + kTcK + kc * kTcTileB + kk * 32), idesc, (kc | kk) ? 1u : 0u);
      tc_commit(&bar[0]);
    }
    if (qc == 0) {
      // V^T while S is computed: the lanes of a warp take consecutive keys of
      // one 8-dim granule, so each of its stores fills part of one row (fenced
      // for the tensor cores with P below)
      for (int e = threadIdx.x; e < kKeys * (kHd / 8); e += blockDim.x) {
        const int j = e & (kKeys - 1), ch = e >> 7;
        const uint4 u = *reinterpret_cast<const uint4*>(sm + kTcVs + j * kTcVsRow + ch * 16);
        const bf16* h = reinterpret_cast<const bf16*>(&u);
#pragma unroll
        for (int t = 0; t < 8; ++t) *reinterpret_cast<bf16*>(sm + kTcVt + tc_sw128(ch * 8 + t, j)) = h[t];
      }
    }

    // thread: operand row R (TMEM lane), query qi = R mod 64, keys kc0 .. kc0 + 31
    // (WIDE: query qc * 128 + R)
    const int qi = WIDE ? qc * kTileQWide + R : (R & (kTileQ - 1));
    const int qs = WIDE ? R : qi;                        // its slot in red_m / red_l
    // visible keys of this query: kpos = kstart + kj within the window of its
    // position, kj < nk (0 <= lo, hi < nk)
    int lo = 0, hi = nk - 1;
    if (qi >= Qn) {
      lo = 1; hi = 0;
    } else {
      const long long rel = p + qi / G - kstart;           // query position - kstart
      if (window > 0 && rel - window > lo) lo = static_cast<int>(rel - window);
      if (a.causal) {
        if (rel < hi) hi = static_cast<int>(rel);
      } else if (window > 0 && rel + window < hi) {
        hi = static_cast<int>(rel + window);
      }
    }
    ok = mbar_wait(&bar[0], static_cast<unsigned>(qc & 1)) && ok;
    tc_fence_after();
    float sv[KPT];
#pragma unroll
    for (int i = 0; i < KPT / 16; ++i) tmem_ld16(trow + kc0 + i * 16, &sv[i * 16]);
    tmem_ld_wait();
    float mrow = -INFINITY;
#pragma unroll
    for (int c = 0; c < KPT; ++c) {
      const int kj = j0 + kc0 + c;
      sv[c] = (kj >= lo && kj <= hi) ? sv[c] * sl2 : -INFINITY;
      mrow = fmaxf(mrow, sv[c]);
    }
    red_m[grp][qs] = mrow;
    __syncthreads();
    if (qc == 0) attn_phase(a.trace, 1);             // S read back

    const float M = fmaxf(fmaxf(red_m[0][qs], red_m[1][qs]), fmaxf(red_m[2][qs], red_m[3][qs]));
    float l = 0.f;
    uint32_t pk[KPT / 2], pr[KPT / 2];
#pragma unroll
    for (int c = 0; c < KPT; c += 2) {
      const float p0 = (M == -INFINITY || sv[c] == -INFINITY) ? 0.f : exp2f(sv[c] - M);
      const float p1 = (M == -INFINITY || sv[c + 1] == -INFINITY) ? 0.f : exp2f(sv[c + 1] - M);
      l += p0 + p1;
      pk[c >> 1] = pack_bf16(p0, p1);
      pr[c >> 1] = pack_bf16_residue(p0, p1);
    }
    red_l[grp][qs] = l;
    // P row R: this thread's 32 keys (tile rh, granules half*4 ..), and zeros
    // over the same granules of the other tile; the high bf16 part in Q's
    // tiles, the low part in K's (K is no longer read once S is done). WIDE:
    // only its own 32 keys (tile grp / 2, granules (grp % 2) * 4 ..) in row R,
    // every key of the row being some thread's; the low part in V's staging
    // rows.
    if (WIDE) {
#pragma unroll
      for (int gi = 0; gi < 4; ++gi) {
        const int gg = (grp & 1) * 4 + gi;
        const int at = R * 128 + ((gg ^ (R & 7)) << 4);
        *reinterpret_cast<uint4*>(sm + kTcQ + (grp >> 1) * kTcTileB + at) =
            make_uint4(pk[4 * gi], pk[4 * gi + 1], pk[4 * gi + 2], pk[4 * gi + 3]);
        *reinterpret_cast<uint4*>(sm + plo + (grp >> 1) * kTcTileB + at) =
            make_uint4(pr[4 * gi], pr[4 * gi + 1], pr[4 * gi + 2], pr[4 * gi + 3]);
      }
    } else {
#pragma unroll
      for (int gi = 0; gi < 4; ++gi) {
        const int gg = half * 4 + gi;
        const int at = R * 128 + ((gg ^ (R & 7)) << 4);
        *reinterpret_cast<uint4*>(sm + kTcQ + rh * kTcTileB + at) =
            make_uint4(pk[4 * gi], pk[4 * gi + 1], pk[4 * gi + 2], pk[4 * gi + 3]);
        *reinterpret_cast<uint4*>(sm + kTcQ + (rh ^ 1) * kTcTileB + at) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(sm + plo + rh * kTcTileB + at) =
            make_uint4(pr[4 * gi], pr[4 * gi + 1], pr[4 * gi + 2], pr[4 * gi + 3]);
        *reinterpret_cast<uint4*>(sm + plo + (rh ^ 1) * kTcTileB + at) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    fence_proxy_async_shared();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (qc == 0) attn_phase(a.trace, 2);             // P written
    if (threadIdx.x == 0) {
#pragma unroll
      for (int kc = 0; kc < 2; ++kc)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_bf16(tmem + 128, smem_desc_sw128(sbase + kTcQ + kc * kTcTileB + kk * 32),
                      smem_desc_sw128(sbase + kTcVt + kc * kTcTileB + kk * 32), idesc, (kc | kk) ? 1u : 0u);
#pragma unroll
      for (int kc = 0; kc < 2; ++kc)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_bf16(tmem + 128, smem_desc_sw128(sbase + plo + kc * kTcTileB + kk * 32),
                      smem_desc_sw128(sbase + kTcVt + kc * kTcTileB + kk * 32), idesc, 1u);
      tc_commit(&bar[1]);
    }
    // O: rows R and R + 64 hold the two halves of query qi's sum; each thread
    // reads 64 dims of its row, the low rows store them, the high rows add
    // (WIDE: row R is query qi's whole sum)
    ok = mbar_wait(&bar[1], static_cast<unsigned>(qc & 1)) && ok;
    tc_fence_after();
    float ov[64];
    if (WIDE) {
      // its 32 dims straight into the partial, with the row's maximum
      // (natural-log units) and sum
#pragma unroll
      for (int i = 0; i < 2; ++i) tmem_ld16(trow + 128 + grp * 32 + i * 16, &ov[i * 16]);
      tmem_ld_wait();
      if (qi < Qn) {
        float* out = part + (size_t)qi * kPartStride;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<float4*>(out + grp * 32 + 4 * i) =
              make_float4(ov[4 * i], ov[4 * i + 1], ov[4 * i + 2], ov[4 * i + 3]);
        if (grp == 0) {
          out[kHd] = M == -INFINITY ? -INFINITY : M * 0.6931471805599453f;
          out[kHd + 1] = (red_l[0][qs] + red_l[1][qs]) + (red_l[2][qs] + red_l[3][qs]);
        }
      }
      // S, O and Q's tiles, red_m and red_l free for the next chunk
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      continue;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) tmem_ld16(trow + 128 + half * 64 + i * 16, &ov[i * 16]);
    tmem_ld_wait();
    float* ost = reinterpret_cast<float*>(sm + kTcK) + qi * kTcOStride + half * 64;
    if (rh == 0) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        *reinterpret_cast<float4*>(ost + 4 * i) = make_float4(ov[4 * i], ov[4 * i + 1], ov[4 * i + 2], ov[4 * i + 3]);
    }
    __syncthreads();
    attn_phase(a.trace, 3);                        // O read back
    if (rh == 1) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float4 x = *reinterpret_cast<float4*>(ost + 4 * i);
        x.x += ov[4 * i]; x.y += ov[4 * i + 1]; x.z += ov[4 * i + 2]; x.w += ov[4 * i + 3];
        *reinterpret_cast<float4*>(ost + 4 * i) = x;
      }
    }
  }
  if (!ok && lane == 0) atomicOr(a.err, 32);
  tc_fence_before();
  __syncthreads();
  if (WIDE) attn_phase(a.trace, 3);                // O read back (every chunk)
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
  if (!WIDE) {
    // the split's partial, one query row per warp pass (coalesced)
    const float* osm = reinterpret_cast<const float*>(sm + kTcK);
    for (int e = threadIdx.x; e < Qn * (kHd / 4); e += blockDim.x) {
      const int q = e / (kHd / 4), d4 = (e % (kHd / 4)) * 4;
      float* out = part + (size_t)q * kPartStride;
      *reinterpret_cast<float4*>(out + d4) = *reinterpret_cast<const float4*>(osm + q * kTcOStride + d4);
      if (d4 == 0) {
        // the row's maximum in natural-log units, as the merge expects
        const float Mq = fmaxf(fmaxf(red_m[0][q], red_m[1][q]), fmaxf(red_m[2][q], red_m[3][q]));
        out[kHd] = Mq == -INFINITY ? -INFINITY : Mq * 0.6931471805599453f;
        out[kHd + 1] = (red_l[0][q] + red_l[1][q]) + (red_l[2][q] + red_l[3][q]);
      }
    }
  }
  if (a.trace.p) { __syncthreads(); if (threadIdx.x == 0) ktrace_mark(a.trace, 2); }
}

}  // namespace

int attention_mma_splits(int rows, int max_ctx) { return (max_ctx + rows + kKeys - 1) / kKeys; }

size_t attention_mma_scratch_floats(int rows, int nq, int nkv, int max_ctx) {
  return (size_t)nkv * attention_mma_splits(rows, max_ctx) * rows * (nq / nkv) * kPartStride;
}

bool attention_mma_ok(int dtype, int hd) { return dtype == 1 && hd == kHd; }

cudaError_t init_attention_mma_attrs() {
  // the largest shared-memory carveout, as the GEMMs around them
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kTcAttnSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_tc_kernel<false>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcAttnSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_tc_kernel<true>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(MmaSmem));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_mma_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  return e;
}

cudaError_t launch_attention_mma(const AttnArgs& a, cudaStream_t st) {
  const int nsplit = attention_mma_splits(a.rows, a.max_ctx);
  const int ns = a.nseq > 1 ? a.nseq : 1;
  dim3 grid(nsplit, a.nkv, ns);
  const int Qn = a.rows * (a.nq / a.nkv);
  // Two to four 16-query tiles per kv head: the tensor-core kernel (A/B on
  // one GB300 at 64 queries per kv head: 16 us per draft faster than an
  // mma.sync kernel with the split merge folded in); five or more: its
  // one-row-per-query variant, 128 queries at a time. One tile: mma.sync.
  if (Qn > 16 && Qn <= kTileQ) {
    cudaError_t e = launch_pdl(attn_tc_kernel<false>, grid, dim3(kWarps * 32), kTcAttnSmem, st, a, nsplit);
    if (e != cudaSuccess) return e;
  } else if (Qn > kTileQ) {
    cudaError_t e = launch_pdl(attn_tc_kernel<true>, grid, dim3(2 * kWarps * 32), kTcAttnSmem, st, a, nsplit);
    if (e != cudaSuccess) return e;
  } else {
    cudaError_t e = launch_pdl(attn_mma_kernel, grid, dim3(kWarps * 32), sizeof(MmaSmem), st, a, nsplit);
    if (e != cudaSuccess) return e;
  }
  const int items = ns * a.nkv * a.rows * (a.nq / a.nkv);
  return launch_pdl(attn_mma_combine_kernel, dim3((items + 3) / 4), dim3(128), 0, st, a, nsplit);
}

}  // namespace dfl
