// Bidirectional sliding-window GQA attention of the drafter block, bf16,
// head_dim 128, on tensor cores (mma.sync m16n8k16, fp32 accumulate).
//
// One CTA per (split of kKeys = 128 keys, kv head g); its 8 warps each own 16
// keys. For every 16-query tile (queries = block rows x the G query heads of
// g): S = Q K^T for the warp's keys (mask |q - k| <= W by absolute
// positions), the warp's online-softmax partial (max, sum, P V), a merge of
// the 8 warps in shared memory in warp order, and the CTA's partial written
// to global scratch. A combine kernel (one warp per (query, head)) merges the
// splits in split order and writes the bf16 output; nothing waits on another
// CTA and the result is deterministic.
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
constexpr int kPad = 8;                    // bf16 elements of row padding
constexpr int kRowB = (kHd + kPad) * 2;    // 272-byte rows: conflict-free ldmatrix
constexpr int kPartStride = kAttnPartStride;
constexpr int kQChunk = 64;

struct MmaSmem {
  bf16 k[kKeys][kHd + kPad];
  bf16 v[kKeys][kHd + kPad];
  bf16 q[kQChunk][kHd + kPad];            // up to 64 query rows, loaded with K/V
  float o[kWarps][16][kHd];                // per-warp unnormalised P V
  float m[kWarps][16];
  float l[kWarps][16];
  float f[kWarps][16];                     // exp(m_w - M) per (warp, row)
  float L[16];                             // merged sum per row
  float M[16];                             // merged max per row
};

__global__ void __launch_bounds__(kWarps * 32) attn_mma_kernel(AttnArgs a, int nsplit) {
  if (threadIdx.x == 0) ktrace_mark(a.trace, 0);
  // (Measured: 3 us per draft faster at 4 block rows; at 16, where the query
  // tile kernel runs, the hint's traffic costs the QKV GEMM about as much.)
  attn_prefetch_context(a, blockIdx.x, blockIdx.y);
  pdl_enter();
  if (threadIdx.x == 0) ktrace_mark(a.trace, 1);
  extern __shared__ __align__(16) uint8_t smem_raw[];
  MmaSmem& S = *reinterpret_cast<MmaSmem*>(smem_raw);
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
    for (int e = threadIdx.x; e < kQChunk * (kHd / 8); e += blockDim.x) {
      const int r = e >> 4, ch = e & 15;
      const int qi = q0 + r;
      const bool valid = qi < Qn;
      const bf16* src = qg;
      if (valid) src = qg + (size_t)(qi / G) * a.ldq + (size_t)(g * G + qi % G) * kHd + ch * 8;
      cp_async16(&S.q[r][ch * 8], src, valid);
    }
  };
  if (j0 < nk) {
    // K and V tiles: 128 keys x 16 chunks of 16 bytes each.
    for (int e = threadIdx.x; e < kKeys * (kHd / 8); e += blockDim.x) {
      const int j = e >> 4, ch = e & 15;
      const int kj = j0 + j;
      const bf16* ks = kb;
      const bf16* vs = vb;
      bool valid = kj < nk;
      if (kj < nctx) {
        int slot = slot0 + kj;                     // = ring_slot(kstart + kj, cap)
        if (slot >= cap) slot -= cap;
        ks = rk + (size_t)slot * kHd + ch * 8;
        vs = rv + (size_t)slot * kHd + ch * 8;
      } else if (valid) {
        const size_t off = (size_t)(kj - nctx) * a.ldkv + (size_t)g * kHd + ch * 8;
        ks = kb + off;
        vs = vb + off;
      }
      cp_async16(&S.k[j][ch * 8], ks, valid);
      cp_async16(&S.v[j][ch * 8], vs, valid);
    }
  }
  load_q(0);
  cp_async_wait_all();
  __syncthreads();

  const int grp = lane >> 2, tig = lane & 3;
  const float scale = rsqrtf(static_cast<float>(kHd));
  for (int qt = 0; qt * 16 < Qn; ++qt) {
    const int qr = (qt * 16) % kQChunk;           // row of this tile in the Q chunk
    if (qt > 0 && qr == 0) {                      // next chunk of 64 queries
      load_q(qt * 16);
      cp_async_wait_all();
      __syncthreads();
    }
    float m_row[2] = {-INFINITY, -INFINITY}, l_row[2] = {0.f, 0.f};
    float o[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

    if (j0 < nk) {
      // S = Q K^T over the warp's 16 keys (two 8-key n-tiles).
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < kHd / 16; ++ks) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        const int mi = lane >> 3;
        ldsm_x4(&S.q[qr + (lane & 7) + (mi & 1) * 8][ks * 16 + (mi >> 1) * 8], a0, a1, a2, a3);
        ldsm_x4(&S.k[warp * 16 + (mi >> 1) * 8 + (lane & 7)][ks * 16 + (mi & 1) * 8], b0, b1, b2, b3);
        mma16816(sc[0], a0, a1, a2, a3, b0, b1);
        mma16816(sc[1], a0, a1, a2, a3, b2, b3);
      }
      // mask, scale, per-row max over the warp's keys
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int qi = qt * 16 + grp + hr * 8;
        const long long qpos = p + (qi < Qn ? qi / G : 0);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int kj = j0 + warp * 16 + nt * 8 + tig * 2 + c;
            bool vis = qi < Qn && kj < nk;
            if (vis && a.window > 0) {
              const long long kpos = kj < nctx ? kstart + kj : p + (kj - nctx);
              const long long d = qpos > kpos ? qpos - kpos : kpos - qpos;
              vis = d <= a.window;
            }
            float& v = sc[nt][hr * 2 + c];
            v = vis ? v * scale : -INFINITY;
            m_row[hr] = fmaxf(m_row[hr], v);
          }
        m_row[hr] = fmaxf(m_row[hr], __shfl_xor_sync(0xffffffffu, m_row[hr], 1));
        m_row[hr] = fmaxf(m_row[hr], __shfl_xor_sync(0xffffffffu, m_row[hr], 2));
      }
      // P = exp(S - m) (bf16 for the MMA), row sums, O = P V
      uint32_t pa[4];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        float pv[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const float v = sc[nt][hr * 2 + c];
            pv[nt][c] = (m_row[hr] == -INFINITY || v == -INFINITY) ? 0.f : expf(v - m_row[hr]);
            l_row[hr] += pv[nt][c];
          }
        pa[hr] = pack_bf16(pv[0][0], pv[0][1]);        // keys 0..7 of this row
        pa[2 + hr] = pack_bf16(pv[1][0], pv[1][1]);    // keys 8..15
        l_row[hr] += __shfl_xor_sync(0xffffffffu, l_row[hr], 1);
        l_row[hr] += __shfl_xor_sync(0xffffffffu, l_row[hr], 2);
      }
#pragma unroll
      for (int dt = 0; dt < kHd / 16; ++dt) {
        uint32_t b0, b1, b2, b3;
        const int mi = lane >> 3;
        ldsm_x4_t(&S.v[warp * 16 + (mi & 1) * 8 + (lane & 7)][dt * 16 + (mi >> 1) * 8], b0, b1, b2, b3);
        mma16816(o[dt * 2], pa[0], pa[1], pa[2], pa[3], b0, b1);
        mma16816(o[dt * 2 + 1], pa[0], pa[1], pa[2], pa[3], b2, b3);
      }
    }
    // publish the warp's partial, then merge the 8 warps in warp order
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        S.o[warp][grp + hr * 8][nt * 8 + tig * 2] = o[nt][hr * 2];
        S.o[warp][grp + hr * 8][nt * 8 + tig * 2 + 1] = o[nt][hr * 2 + 1];
      }
    if (tig == 0) {
      S.m[warp][grp] = m_row[0]; S.m[warp][grp + 8] = m_row[1];
      S.l[warp][grp] = l_row[0]; S.l[warp][grp + 8] = l_row[1];
    }
    __syncthreads();
    // per-row merge weights of the 8 warps: one thread per (row, warp)
    if (threadIdx.x < 16 * kWarps) {
      const int r = threadIdx.x >> 3, w = threadIdx.x & 7;
      float M = -INFINITY;
#pragma unroll
      for (int x = 0; x < kWarps; ++x) M = fmaxf(M, S.m[x][r]);
      const float mw = S.m[w][r];
      const float f = (M == -INFINITY || mw == -INFINITY) ? 0.f : expf(mw - M);
      S.f[w][r] = f;
      float lw = f * S.l[w][r];
#pragma unroll
      for (int o2 = 4; o2 > 0; o2 >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o2);
      if (w == 0) { S.L[r] = lw; S.M[r] = M; }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < 16 * kHd; e += blockDim.x) {
      const int r = e / kHd, d = e % kHd;
      const int qi = qt * 16 + r;
      if (qi >= Qn) continue;
      float O = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) O = fmaf(S.f[w][r], S.o[w][r][d], O);
      float* out = part + (size_t)qi * pstride;
      out[d] = O;
      if (d == 0) { out[kHd] = S.M[r]; out[kHd + 1] = S.L[r]; }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) ktrace_mark(a.trace, 2);
}

// ---------------------------------------------------------------------------
// Up to 64 queries per kv head (block rows x query heads per kv head): the 8
// warps split (16-query tile) x (key group) — 1 tile x 8 groups of 16 keys,
// 2 x 4 of 32, or 4 x 2 of 64 — and each runs an online softmax over its keys.
// Once every warp is done with K and V their shared memory holds the warps'
// partials, which are merged per query in group order and written out. 87 KB
// of shared memory, so the next GEMM's CTAs fit beside it and start streaming
// their weights.
// ---------------------------------------------------------------------------
constexpr int kTileQ = 64;

// Phase stamps of the tile kernel in the two trace slots after its own
// (latest CTA; allotted only when the split merge is folded in): slot + 1 gets
// [1] loads landed, [2] per-warp attention done; slot + 2 gets [1] partials
// written, [2] the head's splits all present.
__device__ __forceinline__ void attn_phase(const KTrace& t, int slot_off, int k) {
  if (t.p && threadIdx.x == 0) ktrace_mark(KTrace{t.p, t.slot + slot_off}, k);
}

// The split merge inside the attention kernel, for grids of at most one CTA
// per SM (all resident, so waiting on the other splits of a head cannot
// block them): split s of kv head g arrives on the head's counter after
// writing its partial, waits for the head's other splits (bounded), then its
// warps merge queries s, s + nsplit, ... of that head (in split order, as the
// standalone merge kernel does). The last split to leave rearms the counters.
__device__ __noinline__ void merge_splits(const AttnArgs& a, int nsplit, int s, int g, int G, int Qn) {
  unsigned* arrive = a.head_ctr + g;
  unsigned* depart = a.head_ctr + a.nkv + g;
  __shared__ int s_ok;
  __syncthreads();
  const bool mine = s < Qn;
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(arrive, 1u);
    int ok = 1;
    if (mine) {
      unsigned spins = 0;
      while (*reinterpret_cast<volatile unsigned*>(arrive) < static_cast<unsigned>(nsplit)) {
        if (++spins > (1u << 24)) { atomicOr(a.err, 16); ok = 0; break; }
        __nanosleep(64);
      }
      __threadfence();
      if (a.trace.p) ktrace_mark(KTrace{a.trace.p, a.trace.slot + 2}, 2);
    }
    s_ok = ok;
  }
  __syncthreads();
  if (mine && s_ok) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int qi = s + nsplit * warp; qi < Qn; qi += nsplit * kWarps)
      attn_combine_warp(a.partial, nsplit, nsplit, Qn, G, g, qi, reinterpret_cast<bf16*>(a.out), a.ldo, lane);
  }
  __syncthreads();
  if (threadIdx.x == 0 && atomicAdd(depart, 1u) == static_cast<unsigned>(nsplit - 1)) {
    *arrive = 0u;                     // every split of the head is past its wait
    *depart = 0u;
  }
}

struct TileSmem {
  union {
    struct {
      bf16 k[kKeys][kHd + kPad];
      bf16 v[kKeys][kHd + kPad];
    } kv;
    struct {
      float o[kWarps][16][kHd];
      float m[kWarps][16];
      float l[kWarps][16];
      float f[kTileQ][kWarps];
      float M[kTileQ];
      float L[kTileQ];
    } mg;
  };
  bf16 q[kTileQ][kHd + kPad];
};
static_assert(sizeof(TileSmem) <= 90 * 1024, "attention tile too large to share an SM with a GEMM CTA");

__global__ void __launch_bounds__(kWarps * 32) attn_tile_kernel(AttnArgs a, int nsplit, int merge) {
  if (threadIdx.x == 0) ktrace_mark(a.trace, 0);
  pdl_enter();
  if (threadIdx.x == 0) ktrace_mark(a.trace, 1);
  extern __shared__ __align__(16) uint8_t smem_raw[];
  TileSmem& S = *reinterpret_cast<TileSmem*>(smem_raw);
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

  if (j0 >= nk) {
    // a split past the keys: an empty partial (weight 0 in the merge)
    for (int e = threadIdx.x; e < Qn * kPartStride; e += blockDim.x) {
      const int d = e % kPartStride;
      part[e] = d == kHd ? -INFINITY : 0.f;
    }
    if (merge) merge_splits(a, nsplit, s, g, G, Qn);
    if (a.trace.p) { __syncthreads(); if (threadIdx.x == 0) ktrace_mark(a.trace, 2); }
    return;
  }
  for (int e = threadIdx.x; e < kKeys * (kHd / 8); e += blockDim.x) {
    const int j = e >> 4, ch = e & 15;
    const int kj = j0 + j;
    const bf16* ks = kb;
    const bf16* vs = vb;
    const bool valid = kj < nk;
    if (kj < nctx) {
      int slot = slot0 + kj;
      if (slot >= cap) slot -= cap;
      ks = rk + (size_t)slot * kHd + ch * 8;
      vs = rv + (size_t)slot * kHd + ch * 8;
    } else if (valid) {
      const size_t off = (size_t)(kj - nctx) * ldkv + ch * 8;
      ks = kb + off;
      vs = vb + off;
    }
    cp_async16(&S.kv.k[j][ch * 8], ks, valid);
    cp_async16(&S.kv.v[j][ch * 8], vs, valid);
  }
  const int nqt = (Qn + 15) / 16;
  for (int e = threadIdx.x; e < nqt * 16 * (kHd / 8); e += blockDim.x) {
    const int r = e >> 4, ch = e & 15;
    const bool valid = r < Qn;
    const bf16* src = qg;
    if (valid) src = qg + (size_t)(r / G) * ldq + (size_t)(r % G) * kHd + ch * 8;
    cp_async16(&S.q[r][ch * 8], src, valid);
  }
  cp_async_wait_all();
  __syncthreads();
  if (merge) attn_phase(a.trace, 1, 1);

  const int kg = nqt == 1 ? 8 : nqt == 2 ? 4 : 2;   // key groups per query tile
  const int span = kKeys / kg;                        // keys per warp
  const int qt = warp / kg, gk = warp % kg;
  const bool busy = qt < nqt;
  const int grp = lane >> 2, tig = lane & 3, mi = lane >> 3;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  if (busy) {
    const float scale = rsqrtf(static_cast<float>(kHd));
    int qrel[2];
    bool qok[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int qi = qt * 16 + grp + hr * 8;
      qok[hr] = qi < Qn;
      qrel[hr] = qok[hr] ? qi / G : 0;
    }
    // the warp's 16 queries as MMA A fragments, loaded once for all its keys
    uint32_t qa[kHd / 16][4];
#pragma unroll
    for (int ks = 0; ks < kHd / 16; ++ks)
      ldsm_x4(&S.q[qt * 16 + (lane & 7) + (mi & 1) * 8][ks * 16 + (mi >> 1) * 8], qa[ks][0], qa[ks][1],
              qa[ks][2], qa[ks][3]);
    for (int kb0 = gk * span; kb0 < (gk + 1) * span; kb0 += 16) {
      const int kj0 = j0 + kb0;
      if (kj0 >= nk) break;
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < kHd / 16; ++ks) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(&S.kv.k[kb0 + (mi >> 1) * 8 + (lane & 7)][ks * 16 + (mi & 1) * 8], b0, b1, b2, b3);
        mma16816(sc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
        mma16816(sc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
      }
      float mb[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int kj = kj0 + nt * 8 + tig * 2 + c;
            bool vis = qok[hr] && kj < nk;
            if (window > 0) {
              const int d = qrel[hr] - (kj - nctx);          // positions relative to the block
              vis = vis && (d < 0 ? -d : d) <= window;
            }
            float& v = sc[nt][hr * 2 + c];
            v = vis ? v * scale : -INFINITY;
            mb[hr] = fmaxf(mb[hr], v);
          }
        mb[hr] = fmaxf(mb[hr], __shfl_xor_sync(0xffffffffu, mb[hr], 1));
        mb[hr] = fmaxf(mb[hr], __shfl_xor_sync(0xffffffffu, mb[hr], 2));
      }
      uint32_t pa[4];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const float m_new = fmaxf(m_run[hr], mb[hr]);
        const float alpha = m_run[hr] == -INFINITY ? 0.f : expf(m_run[hr] - m_new);
        float pv[2][2];
        float ls = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const float v = sc[nt][hr * 2 + c];
            pv[nt][c] = (m_new == -INFINITY || v == -INFINITY) ? 0.f : expf(v - m_new);
            ls += pv[nt][c];
          }
        ls += __shfl_xor_sync(0xffffffffu, ls, 1);
        ls += __shfl_xor_sync(0xffffffffu, ls, 2);
        l_run[hr] = l_run[hr] * alpha + ls;
        m_run[hr] = m_new;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) { o[nt][hr * 2] *= alpha; o[nt][hr * 2 + 1] *= alpha; }
        pa[hr] = pack_bf16(pv[0][0], pv[0][1]);
        pa[2 + hr] = pack_bf16(pv[1][0], pv[1][1]);
      }
#pragma unroll
      for (int dt = 0; dt < kHd / 16; ++dt) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(&S.kv.v[kb0 + (mi & 1) * 8 + (lane & 7)][dt * 16 + (mi >> 1) * 8], b0, b1, b2, b3);
        mma16816(o[dt * 2], pa[0], pa[1], pa[2], pa[3], b0, b1);
        mma16816(o[dt * 2 + 1], pa[0], pa[1], pa[2], pa[3], b2, b3);
      }
    }
  }
  __syncthreads();                                    // K and V are no longer read
  if (merge) attn_phase(a.trace, 1, 2);
  if (busy) {
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr)
        *reinterpret_cast<float2*>(&S.mg.o[warp][grp + hr * 8][nt * 8 + tig * 2]) =
            make_float2(o[nt][hr * 2], o[nt][hr * 2 + 1]);
    if (tig == 0) {
      S.mg.m[warp][grp] = m_run[0]; S.mg.m[warp][grp + 8] = m_run[1];
      S.mg.l[warp][grp] = l_run[0]; S.mg.l[warp][grp + 8] = l_run[1];
    }
  }
  __syncthreads();
  // merge weights: one thread per query
  if (threadIdx.x < Qn) {
    const int qi = threadIdx.x, t = qi >> 4, r = qi & 15;
    float M = -INFINITY;
    for (int x = 0; x < kg; ++x) M = fmaxf(M, S.mg.m[t * kg + x][r]);
    float L = 0.f;
    for (int x = 0; x < kg; ++x) {
      const float mw = S.mg.m[t * kg + x][r];
      const float f = (M == -INFINITY || mw == -INFINITY) ? 0.f : expf(mw - M);
      S.mg.f[qi][x] = f;
      L += f * S.mg.l[t * kg + x][r];
    }
    S.mg.M[qi] = M;
    S.mg.L[qi] = L;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < Qn * (kHd / 4); e += blockDim.x) {
    const int qi = e / (kHd / 4), d4 = (e % (kHd / 4)) * 4;
    const int t = qi >> 4, r = qi & 15;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int x = 0; x < kg; ++x) {
      const float f = S.mg.f[qi][x];
      const float4 ov = *reinterpret_cast<const float4*>(&S.mg.o[t * kg + x][r][d4]);
      acc.x += f * ov.x; acc.y += f * ov.y; acc.z += f * ov.z; acc.w += f * ov.w;
    }
    float* out = part + (size_t)qi * kPartStride;
    *reinterpret_cast<float4*>(out + d4) = acc;
    if (d4 == 0) { out[kHd] = S.mg.M[qi]; out[kHd + 1] = S.mg.L[qi]; }
  }
  if (merge) {
    __syncthreads();
    attn_phase(a.trace, 2, 1);
    merge_splits(a, nsplit, s, g, G, Qn);
  }
  if (a.trace.p) { __syncthreads(); if (threadIdx.x == 0) ktrace_mark(a.trace, 2); }
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
  const int item = blockIdx.x * 4 + warp;
  if (item < a.nkv * Qn)
    attn_combine_warp(a.partial, nsplit, nsplit, Qn, G, item / Qn, item % Qn,
                      reinterpret_cast<bf16*>(a.out), a.ldo, lane);
  if (tr.p) { __syncthreads(); if (threadIdx.x == 0) ktrace_mark(tr, 2); }
}

}  // namespace

int attention_mma_splits(int rows, int max_ctx) { return (max_ctx + rows + kKeys - 1) / kKeys; }

size_t attention_mma_scratch_floats(int rows, int nq, int nkv, int max_ctx) {
  return (size_t)nkv * attention_mma_splits(rows, max_ctx) * rows * (nq / nkv) * kPartStride;
}

bool attention_mma_ok(int dtype, int hd) { return dtype == 1 && hd == kHd; }

cudaError_t init_attention_mma_attrs() {
  cudaError_t e = cudaFuncSetAttribute(attn_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(TileSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attn_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sizeof(MmaSmem));
}

cudaError_t launch_attention_mma(const AttnArgs& a, unsigned*, cudaStream_t st) {
  const int nsplit = attention_mma_splits(a.rows, a.max_ctx);
  dim3 grid(nsplit, a.nkv);
  const int Qn = a.rows * (a.nq / a.nkv);
  // The 87 KB tile kernel with the split merge folded in pays from two query
  // tiles on (A/B on one GB300: -12 us per draft at 64 queries per kv head);
  // at one tile the 8-warp key split with its separate merge is faster (-6 us).
  if (Qn > 16 && Qn <= kTileQ) {
    const int merge = (a.head_ctr && a.err && nsplit * a.nkv <= a.sms) ? 1 : 0;
    cudaError_t e = launch_pdl(attn_tile_kernel, grid, dim3(kWarps * 32), sizeof(TileSmem), st, a, nsplit, merge);
    if (e != cudaSuccess || merge) return e;
  } else {
    cudaError_t e = launch_pdl(attn_mma_kernel, grid, dim3(kWarps * 32), sizeof(MmaSmem), st, a, nsplit);
    if (e != cudaSuccess) return e;
  }
  const int items = a.nkv * a.rows * (a.nq / a.nkv);
  return launch_pdl(attn_mma_combine_kernel, dim3((items + 3) / 4), dim3(128), 0, st, a, nsplit);
}

}  // namespace dfl
