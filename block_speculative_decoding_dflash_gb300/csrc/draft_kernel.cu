// The drafter block forward as one persistent, cooperative launch (one CTA
// per SM), for bf16 drafters with head_dim 128 and at most 16 block rows:
//
//   embed -> [ rmsnorm -> QKV (+ q/k head norm + RoPE) -> attention partials
//              -> split merge -> O (+ residual) -> rmsnorm -> gate/up (SwiGLU)
//              -> down (+ residual) ] x layers -> rmsnorm -> lm_head
//              (+ softcap + argmax)
//
// which is the drafter of "DFlash: Block Diffusion for Flash Speculative
// Decoding" (drafter architecture: encoder.fc output normalised, sliding
// attention layers with per-head q/k RMSNorm, untied lm_head with the final
// logit softcap) at batch 1. Decoding at batch 1 streams every weight byte
// once per block, so the kernel is built to keep HBM busy from the first
// weight tile to the last:
//
// * Phases run in order; phase p starts on a CTA once every CTA has counted
//   itself done with phase p - 1 (a per-phase counter in global memory).
//   Each GEMM's (128-row weight tile, 64-wide K chunk) units are split into
//   one contiguous range per CTA, as in the standalone weight-streaming GEMM,
//   with the same deterministic split-tile fixup by the last contributor.
// * Warp 0 streams weight tiles through a shared-memory ring with TMA. Weight
//   loads never wait for a phase boundary: the ring fills with the next
//   phase's tiles while the current phase finishes; only the loads of an
//   activation operand wait until the phase that writes it is complete.
// * RMSNorm is not a phase of its own: before a GEMM whose input is a
//   normalised row, every CTA normalises the (at most 16) rows itself and
//   writes them into shared memory in the 128-byte-swizzled layout the MMA
//   reads, so that operand never round-trips global memory.
// * Warp 1 issues tcgen05.mma (128 x 16 x 16, fp32 accumulators in TMEM, two
//   accumulator buffers); warps 2-5 run the epilogues and every non-GEMM
//   phase (attention on mma.sync, the split merge, the embedding gather).
// * Every wait is bounded (time and polls). A CTA that gives up raises a
//   shared abort flag that ends every other wait, drains its own copies and
//   MMAs in flight, frees its TMEM and returns; the error word records it.
//
// Rounding points are those of the one-kernel-per-operation path: the
// normalised rows, each GEMM output, the residual sums and the SwiGLU product
// are rounded to bf16 where they are stored.
#include <cudaTypedefs.h>

#include "attn_common.cuh"
#include "kernels.h"
#include "mma_sync.cuh"
#include "ptx.cuh"
#include "tc_epilogue.cuh"

namespace dfl {
namespace {

constexpr int BN = 16;                                 // block rows per MMA
constexpr int kStages = 6;
constexpr int kStageBytes = kABytes + BN * 128;        // weight tile + activation tile
constexpr int kRingBytes = kStages * kStageBytes;
constexpr int kMaxNormK = 2048;                        // widest normalised operand
constexpr int kXnBytes = (kMaxNormK / 64) * BN * 128;  // 64 KB

// Attention tiles (one split of 128 keys of one kv head, up to 64 queries).
constexpr int kPad = 8;
constexpr int kRow = kAttnHd + kPad;                   // 272-byte rows: conflict-free ldmatrix
constexpr int kMaxQ = 64;
struct AttnTile {
  bf16 k[kAttnKeys][kRow];
  bf16 v[kAttnKeys][kRow];
  bf16 q[kMaxQ][kRow];
};
constexpr int kUnionBytes = (int)(sizeof(AttnTile) > (size_t)kXnBytes ? sizeof(AttnTile) : kXnBytes);
constexpr int kNumBars = 2 * kStages + 4 + 3;
constexpr size_t kSmemBytes = 1024 + (size_t)kRingBytes + kUnionBytes + kNumBars * 8 + 16;

constexpr unsigned long long kWaitNs = 2000000000ull;  // no legitimate wait comes near this
constexpr int kTraceSlots = kMegaTraceSlots;
constexpr int kMaxPhases = kMegaMaxPhases;
constexpr int kDoneStride = kMegaDoneStride;            // one 128-byte line per phase counter

__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ unsigned ld_volatile(const unsigned* p) {
  return *reinterpret_cast<const volatile unsigned*>(p);
}

// Trace stamp k of phase p on this CTA (tracing on only).
__device__ __forceinline__ void stamp(unsigned long long* trace, int p, int k) {
  if (trace) trace[((size_t)p * gridDim.x + blockIdx.x) * kTraceSlots + k] = gtimer();
}

// Bound on one wait: false once the abort flag is up (when given), after
// kWaitNs of wall time, or after kSpinLimit polls. The clock is first read
// after 64 polls, so a short wait costs no timer read.
struct Bound {
  unsigned long long t0 = 0;
  unsigned n = 0;
  __device__ __forceinline__ bool ok(const unsigned* abort_flag) {
    if ((++n & 63) != 0) return true;
    if (n >= kSpinLimit) return false;
    if (abort_flag && ld_volatile(abort_flag)) return false;
    const unsigned long long t = gtimer();
    if (t0 == 0) t0 = t;
    return t - t0 < kWaitNs;
  }
};

__device__ __forceinline__ bool mbar_try(uint64_t* bar, unsigned parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return done != 0;
}
// Waits with a growing sleep between polls after the first few: a thread
// spinning on an mbarrier competes for the shared-memory pipe with the warps
// that do the work.
__device__ __forceinline__ bool mwait(uint64_t* bar, unsigned parity, const unsigned* abort_flag) {
  Bound bd;
  unsigned ns = 0;
  while (!mbar_try(bar, parity)) {
    if (!bd.ok(abort_flag)) return false;
    if (bd.n > 4) {
      ns = ns ? (ns < 256 ? 2 * ns : 256) : 32;
      __nanosleep(ns);
    }
  }
  return true;
}

// Named-barrier vote of the 128 worker threads: true iff every one passes
// true. Every worker reaches it, so a wait that ended differently on
// different threads still leaves them all on the same path.
__device__ __forceinline__ bool epi_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.and.pred q, %2, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r) : "r"(static_cast<uint32_t>(v)), "r"(kEpiBarrier) : "memory");
  return r != 0;
}


__device__ __forceinline__ void raise_abort(const MegaArgs& a, int bit) {
  atomicOr(a.err, bit);
  atomicExch(a.abort_flag, 1u);
}

// Units of a GEMM phase owned by CTA b of G.
struct Range { long long u0, u1, U; };
__device__ __forceinline__ Range unit_range(const MegaPhase& ph, int b, int G) {
  const long long U = (long long)ph.tiles * ph.kchunks;
  return {U * b / G, U * (b + 1) / G, U};
}
__device__ __forceinline__ int nv_of(const MegaPhase& ph) { return ph.epi == kEpiSwiglu ? 2 : 1; }

// Item cursor of the producer: (phase, unit, sub-item) over the GEMM phases.
// A SwiGLU unit has two items (gate tile, up tile) in consecutive stages.
struct Cursor {
  int p;
  long long u, u1;
  int v, nv;
  bool valid;
};
__device__ __forceinline__ void cursor_seek(Cursor& c, const MegaPhase* phs, int nphase, int from, int b, int G) {
  for (int p = from; p < nphase; ++p) {
    const MegaPhase& ph = phs[p];
    if (ph.kind != kPhGemm) continue;
    const Range r = unit_range(ph, b, G);
    if (r.u1 > r.u0) {
      c.p = p; c.u = r.u0; c.u1 = r.u1; c.v = 0; c.nv = nv_of(ph); c.valid = true;
      return;
    }
  }
  c.valid = false;
}
__device__ __forceinline__ void cursor_next(Cursor& c, const MegaPhase* phs, int nphase, int b, int G) {
  if (++c.v < c.nv) return;
  c.v = 0;
  if (++c.u < c.u1) return;
  cursor_seek(c, phs, nphase, c.p + 1, b, G);
}

// ---------------------------------------------------------------------------
// Worker-side pieces (warps 2-5, 128 threads, worker index wt = 0..127). The
// large ones are out of line: each then gets its own register allocation
// instead of adding to the kernel's, at the price of a call per phase.
// ---------------------------------------------------------------------------

// xn[m] = rnd(x[m] * rsqrt(mean(x^2) + eps) * gain) for m < Mr, zero rows up
// to BN, written as the MMA's B operand: 64-wide K chunks of BN rows x 128
// bytes, 16-byte groups swizzled by row (the TMA SWIZZLE_128B layout). When
// out is given the rows are also stored there, row-major [Mr][K].
//
// Latency, not bandwidth, decides this step (the rows are 64 KB at most and
// sit in L2 while weight tiles stream in), so every load is issued at once:
// the rows go into xn unswizzled and the gain into gsm with cp.async (rows
// past Mr zero-filled), the row sums come from shared memory, and each
// thread then rewrites whole 128-byte blocks of a row in place, normalised
// and swizzled.
__device__ __noinline__ void build_norm_operand(const MegaArgs& a, int pidx, uint8_t* xn, const bf16* x, int ldx, int Mr,
                                   const bf16* gain, int K, float eps, bf16* out, bf16* gsm,
                                   float* inv_sm, int wt) {
  const int w = wt >> 5, lane = wt & 31;
  const int kg = K >> 3;                            // 16-byte granules per row
  for (int i = wt; i < BN * kg; i += 128) {
    const int m = i / kg, g8 = i - m * kg;
    const int k = g8 * 8;
    const bool valid = m < Mr;
    const bf16* src = valid ? x + (size_t)m * ldx + k : x;
    cp_async16(xn + (size_t)(k >> 6) * (BN * 128) + m * 128 + ((g8 & 7) << 4), src, valid);
  }
  for (int i = wt; i < kg; i += 128) cp_async16(gsm + i * 8, gain + i * 8, true);
  cp_async_wait_all();
  epi_sync();
  if (wt == 0) stamp(a.trace, pidx, 8);
  for (int m = w; m < BN; m += 4) {
    float ss = 0.f;
    if (m < Mr) {
      for (int g8 = lane; g8 < kg; g8 += 32) {
        float v[8];
        load8(reinterpret_cast<const bf16*>(xn + (size_t)(g8 >> 3) * (BN * 128) + m * 128 + ((g8 & 7) << 4)), v);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(v[e], v[e], ss);
      }
      ss = warp_sum(ss);
    }
    if (lane == 0) inv_sm[m] = rsqrtf(ss / static_cast<float>(K) + eps);
  }
  epi_sync();
  if (wt == 0) stamp(a.trace, pidx, 9);
  const int nblk = BN * (K >> 6);
  for (int bi = wt; bi < nblk; bi += 128) {
    const int m = bi % BN, c = bi / BN;
    uint8_t* blk = xn + (size_t)c * (BN * 128) + m * 128;
    uint4 raw[8];                                     // static indexing only: stays in registers
#pragma unroll
    for (int j = 0; j < 8; ++j) raw[j] = *reinterpret_cast<const uint4*>(blk + (j << 4));
    const float inv = inv_sm[m];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float v[8], g[8];
      load8(reinterpret_cast<const bf16*>(&raw[j]), v);
      load8(gsm + c * 64 + j * 8, g);
      uint4 pk;
      uint32_t* w32 = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * e] * inv * g[2 * e], v[2 * e + 1] * inv * g[2 * e + 1]);
        w32[e] = *reinterpret_cast<uint32_t*>(&b2);
      }
      raw[j] = pk;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(blk + ((j ^ (m & 7)) << 4)) = raw[j];
    if (out && m < Mr) {
      uint4* o = reinterpret_cast<uint4*>(out + (size_t)m * K + c * 64);
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j] = raw[j];
    }
  }
}

struct AttnGeom {
  long long p, kstart;
  int nctx, nk, ns, Qn, G;
};
__device__ __forceinline__ AttnGeom attn_geom(const MegaArgs& a) {
  AttnGeom g;
  g.p = a.ring->offset;
  g.kstart = a.ring->base;
  if (a.window > 0 && g.p - a.window > g.kstart) g.kstart = g.p - a.window;
  g.nctx = static_cast<int>(g.p - g.kstart);
  g.nk = g.nctx + a.M;
  g.ns = attn_splits(g.nk);
  if (g.ns > a.nsplit) {
    // More keys than the scratch was sized for (an append-only ring pushed
    // past max_context): attend to the first nsplit splits and flag it.
    g.ns = a.nsplit;
    if (blockIdx.x == 0 && threadIdx.x == 64) atomicOr(a.err, 8);
  }
  g.G = a.nq / a.nkv;
  g.Qn = a.M * g.G;
  return g;
}

// One split (128 keys from key index j0) of one kv head: each warp owns 16
// queries and runs an online softmax over the split's keys in blocks of 16
// (S = Q K^T and O += P V on mma.sync, P rounded to bf16), then writes its
// queries' partials. Keys 0 .. nctx-1 are the context (ring slots slot0 + j,
// wrapping at cap), keys nctx .. nk-1 the block's own rows; positions are
// taken relative to the block's first row, so the window test is |q - k| <=
// window on small integers. Everything the loops touch is in registers or
// shared memory.
__device__ __noinline__ void attn_split(const bf16* rk, const bf16* rv, const bf16* qb, const bf16* kb,
                                        const bf16* vb, int ldq, float* part, int slot0, int cap,
                                        int nctx, int nk, int Qn, int G, int window, int j0,
                                        AttnTile& S, int wt, unsigned long long* issued_at) {
  const int w = wt >> 5, lane = wt & 31;
  for (int e = wt; e < kAttnKeys * (kAttnHd / 8); e += 128) {
    const int j = e >> 4, ch = e & 15;
    const int kj = j0 + j;
    const bf16* ks = qb;
    const bf16* vs = qb;
    const bool valid = kj < nk;
    if (kj < nctx) {
      int slot = slot0 + kj;
      if (slot >= cap) slot -= cap;
      ks = rk + (size_t)slot * kAttnHd + ch * 8;
      vs = rv + (size_t)slot * kAttnHd + ch * 8;
    } else if (valid) {
      const size_t off = (size_t)(kj - nctx) * ldq + ch * 8;
      ks = kb + off;
      vs = vb + off;
    }
    cp_async16(&S.k[j][ch * 8], ks, valid);
    cp_async16(&S.v[j][ch * 8], vs, valid);
  }
  const int qrows = (Qn + 15) & ~15;
  for (int e = wt; e < qrows * (kAttnHd / 8); e += 128) {
    const int r = e >> 4, ch = e & 15;
    const bool valid = r < Qn;
    const bf16* src = qb;
    if (valid) src = qb + (size_t)(r / G) * ldq + (size_t)(r % G) * kAttnHd + ch * 8;
    cp_async16(&S.q[r][ch * 8], src, valid);
  }
  if (issued_at && wt == 0) *issued_at = gtimer();
  cp_async_wait_all();
  epi_sync();

  if (w * 16 < Qn) {
    const int qt = w;
    const int grp = lane >> 2, tig = lane & 3;
    const int mi = lane >> 3;
    const float scale = rsqrtf(static_cast<float>(kAttnHd));
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float o[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    int qrel[2];                           // query row positions relative to the block start
    bool qok[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int qi = qt * 16 + grp + hr * 8;
      qok[hr] = qi < Qn;
      qrel[hr] = qok[hr] ? qi / G : 0;
    }
    for (int kb0 = 0; kb0 < kAttnKeys; kb0 += 16) {
      const int kj0 = j0 + kb0;
      if (kj0 >= nk) break;
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < kAttnHd / 16; ++ks) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(&S.q[qt * 16 + (lane & 7) + (mi & 1) * 8][ks * 16 + (mi >> 1) * 8], a0, a1, a2, a3);
        ldsm_x4(&S.k[kb0 + (mi >> 1) * 8 + (lane & 7)][ks * 16 + (mi & 1) * 8], b0, b1, b2, b3);
        mma16816(sc[0], a0, a1, a2, a3, b0, b1);
        mma16816(sc[1], a0, a1, a2, a3, b2, b3);
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
              const int d = qrel[hr] - (kj - nctx);          // >= -(M - 1)
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
        pa[hr] = pack_bf16(pv[0][0], pv[0][1]);        // keys 0..7 of this row
        pa[2 + hr] = pack_bf16(pv[1][0], pv[1][1]);    // keys 8..15
      }
#pragma unroll
      for (int dt = 0; dt < kAttnHd / 16; ++dt) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(&S.v[kb0 + (mi & 1) * 8 + (lane & 7)][dt * 16 + (mi >> 1) * 8], b0, b1, b2, b3);
        mma16816(o[dt * 2], pa[0], pa[1], pa[2], pa[3], b0, b1);
        mma16816(o[dt * 2 + 1], pa[0], pa[1], pa[2], pa[3], b2, b3);
      }
    }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int qi = qt * 16 + grp + hr * 8;
      if (!qok[hr]) continue;
      float* out = part + (size_t)qi * kAttnPartStride;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt)
        *reinterpret_cast<float2*>(out + nt * 8 + tig * 2) = make_float2(o[nt][hr * 2], o[nt][hr * 2 + 1]);
      if (tig == 0) { out[kAttnHd] = m_run[hr]; out[kAttnHd + 1] = l_run[hr]; }
    }
  }
  epi_sync();   // the tile is reused by the next split
}

struct EpiSmem {
  float best_v[BN];
  int best_i[BN];
  float red_v[4][BN];
  int red_i[4][BN];
  float kv_ss[4][BN];
  float kv_x[128 * BN];
  bf16 gain[kMaxNormK];          // RMSNorm gain of the normalised operand
  float inv[BN];                 // its per-row 1 / rms
  volatile int ready;            // latest phase every CTA has finished (seen by one poller)
  int flag;
};

// Epilogues of this CTA's tiles of GEMM phase ph (Mr block rows). seg counts
// accumulator segments across phases (it selects the TMEM buffer and its
// parity); returns the count after this phase, or -1 if a wait gave up.
template <int EPI>
__device__ __noinline__ int gemm_epilogue(const MegaArgs& a, const MegaPhase& ph, int pidx, int Mr, uint32_t tmem,
                              uint64_t* acc_full, uint64_t* acc_empty, int seg, EpiSmem& E,
                              int wt) {
  constexpr int NV = EPI == kEpiSwiglu ? 2 : 1;
  const int warp = (wt >> 5) + 2, lane = wt & 31;
  const int q = warp & 3;                   // TMEM lane quarter this warp may read
  const int row = q * 32 + lane;            // output feature within the tile
  const int G = gridDim.x, b = blockIdx.x;
  // Everything the tile loop reads, in registers (a and ph live in memory).
  const int KC = ph.kchunks, N = ph.N, ldy = ph.ldy, nq_tiles = ph.nq_tiles;
  bf16* const Yp = reinterpret_cast<bf16*>(ph.y);
  const bf16* const qn = reinterpret_cast<const bf16*>(ph.qn);
  const bf16* const kn = reinterpret_cast<const bf16*>(ph.kn);
  float* const partials = a.partials;
  unsigned* const tile_ctr = a.tile_ctr;
  const unsigned* const abort_flag = a.abort_flag;
  const float softcap = a.softcap, eps = a.eps;
  const int nkv = a.nkv, read0 = a.read0, neox = a.neox;
  const float2* const rope = a.rope;
  const Range rg = unit_range(ph, b, G);
  const int first_tile = static_cast<int>(rg.u0 / KC);
  for (long long u = rg.u0; u < rg.u1; ++seg) {
    const int t = static_cast<int>(u / KC);
    const int c0 = static_cast<int>(u % KC);
    const int c1 = static_cast<int>(c0 + (rg.u1 - u < KC - c0 ? rg.u1 - u : KC - c0));
    const int buf = seg & 1;
    // The residual of this tile (final only after the previous phase), read
    // while the accumulator is still being produced.
    float res[BN];
    if (EPI == kEpiResid) {
      const bf16* Y = Yp;
      const int n = t * 128 + row;
#pragma unroll
      for (int m = 0; m < BN; ++m)
        res[m] = (m < Mr && n < N) ? __bfloat162float(Y[(size_t)m * ldy + n]) : 0.f;
    }
    // One thread waits; the vote hands its outcome to the other 127.
    if (!epi_all(wt != 0 || mwait(&acc_full[buf], static_cast<unsigned>((seg / 2) & 1), abort_flag))) return -1;
    if (wt == 0 && u == rg.u0) stamp(a.trace, pidx, 2);
    tc_fence_after();
    float acc[NV][BN];
#pragma unroll
    for (int v = 0; v < NV; ++v)
      tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * 32 + v * BN, &acc[v][0]);
    tmem_ld_wait();
    tc_fence_before();
    mbar_arrive(&acc_empty[buf]);
    u += c1 - c0;

    bool finish = (c0 == 0 && c1 == KC);
    if (!finish) {
      const int slot = (t == first_tile) ? 0 : 1;
      const int mq = (Mr + 3) / 4;
      put_partial<NV, BN>(partials, b, slot, row, mq, acc);
      epi_sync();
      const int bf = owner_of((long long)t * KC, rg.U, G);
      const int bl = owner_of((long long)t * KC + KC - 1, rg.U, G);
      if (wt == 0) {
        __threadfence();
        const unsigned ticket = atomicAdd(&tile_ctr[t], 1u);
        E.flag = (ticket == static_cast<unsigned>(bl - bf));
      }
      epi_sync();
      finish = E.flag != 0;
      if (finish) {
        __threadfence();
        const int s_bf = t == static_cast<int>((rg.U * bf / G) / KC) ? 0 : 1;
        if (mq == 1) sum_partials<NV, BN, 1, 4 / NV>(acc, partials, row, bf, bl, mq, s_bf);
        else sum_partials<NV, BN, BN / 4, (NV == 1 ? 4 : 2)>(acc, partials, row, bf, bl, mq, s_bf);
        if (wt == 0) tile_ctr[t] = 0u;
      }
    }
    if (!finish) continue;

    const int n = t * 128 + row;
    const bool valid = n < N;
    if (EPI == kEpiArgmax) {
      const float cap = softcap;
#pragma unroll
      for (int m = 0; m < BN; ++m) {
        float z = acc[0][m];
        if (cap > 0.f) z = cap * tanhf(z / cap);
        float bv = (valid && m >= read0 && m < Mr) ? z : -INFINITY;
        int bi = valid ? n : 0x7fffffff;
        warp_argmax(bv, bi);
        if (lane == 0) { E.red_v[q][m] = bv; E.red_i[q][m] = bi; }
      }
      epi_sync();
      if (wt < BN) {
        const int m = wt;
        float bv = E.best_v[m];
        int bi = E.best_i[m];
#pragma unroll
        for (int w = 0; w < 4; ++w)
          if (better(E.red_v[w][m], E.red_i[w][m], bv, bi)) { bv = E.red_v[w][m]; bi = E.red_i[w][m]; }
        E.best_v[m] = bv;
        E.best_i[m] = bi;
      }
      epi_sync();
    } else if (EPI == kEpiQKV) {
      float val[BN];
#pragma unroll
      for (int m = 0; m < BN; ++m) val[m] = rnd_bf(acc[0][m]);
      const bool isq = t < nq_tiles;
      const bool isk = !isq && t < nq_tiles + nkv;
      if (isq || isk) {
        const float g = __bfloat162float((isq ? qn : kn)[row]);
        head_norm_rope_tile<BN>(val, g, rope, Mr, neox, eps, row, lane, q, E.kv_ss, E.kv_x);
      }
      bf16* Y = Yp;
#pragma unroll
      for (int m = 0; m < BN; ++m)
        if (m < Mr && valid) Y[(size_t)m * ldy + n] = __float2bfloat16_rn(val[m]);
    } else if (valid) {
      bf16* Y = Yp;
#pragma unroll
      for (int m = 0; m < BN; ++m) {
        if (m < Mr) {
          float out;
          if (EPI == kEpiResid)
            out = res[m] + rnd_bf(acc[0][m]);
          else
            out = silu_f(rnd_bf(acc[0][m])) * rnd_bf(acc[NV - 1][m]);
          Y[(size_t)m * ldy + n] = __float2bfloat16_rn(out);
        }
      }
    }
  }
  return seg;
}

// Shared-memory layout: the weight ring, the union of the normalised operand
// and the attention tile, then the mbarriers and the TMEM address.
struct Lay {
  uint8_t* ring;
  uint8_t* uni;
  uint64_t *full, *empty, *acc_full, *acc_empty, *bready, *bfree, *drain;
  uint32_t* tmem_holder;
};
__device__ __forceinline__ Lay smem_layout() {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  Lay L;
  L.ring = smem_raw + (((raw + 1023) & ~1023u) - raw);
  L.uni = L.ring + kRingBytes;
  L.full = reinterpret_cast<uint64_t*>(L.uni + kUnionBytes);
  L.empty = L.full + kStages;
  L.acc_full = L.empty + kStages;
  L.acc_empty = L.acc_full + 2;
  L.bready = L.acc_empty + 2;                         // normalised operand written
  L.bfree = L.bready + 1;                             // ... and no longer read by MMAs
  L.drain = L.bfree + 1;
  L.tmem_holder = reinterpret_cast<uint32_t*>(L.drain + 1);
  return L;
}
__shared__ EpiSmem g_epi;
__shared__ MegaPhase g_phases[kMaxPhases];            // the phase list, read per weight tile

// Each role is a function of its own, so that each gets its own register
// allocation and the producer's per-tile loop keeps its state in registers.

// Warp 0, lane 0: TMA producer.
__device__ __noinline__ void producer_role(const MegaArgs& a) {
  const Lay L = smem_layout();
  uint8_t* const ring = L.ring;
  uint64_t* const full = L.full;
  uint64_t* const empty = L.empty;
  EpiSmem& E = g_epi;
  const MegaPhase* const sph = g_phases;
  const int nph = a.nphase, G = gridDim.x, b = blockIdx.x;
  const CUtensorMap* const maps = a.maps;
  const unsigned* const abort_flag = a.abort_flag;
  unsigned long long* const trace = a.trace;
  const uint64_t pol = policy_evict_first();
  Cursor ca, cb;
  cursor_seek(ca, sph, nph, 0, b, G);
  cb = ca;
  long long ia = 0, ib = 0;
  int ready = -1;                     // latest phase whose activation input is complete
  int last_pa = -1, last_pb = -1;     // trace: phases whose first loads were stamped
  bool ok = true;
  Bound bd;
  while (ok) {
    bool prog = false;
    while (ib < ia) {
      const MegaPhase& ph = sph[cb.p];
      if (!ph.norm) {
        if (ready < cb.p) {
          // The worker that polls the phase counters publishes here what
          // every CTA has finished (after its own acquire fence).
          if (cb.p > 0 && E.ready < cb.p - 1) break;
          __threadfence_block();
          fence_proxy_async_global(); // ... for the TMA reads that follow
          ready = cb.p;
        }
        const int st = static_cast<int>(ib % kStages);
        const int c = static_cast<int>(cb.u % ph.kchunks);
        if (cb.p != last_pb) { stamp(trace, cb.p, 7); last_pb = cb.p; }
        tma_load_2d(ring + (size_t)st * kStageBytes + kABytes, &maps[ph.b_map], c * 64, 0, &full[st]);
      }
      cursor_next(cb, sph, nph, b, G);
      ++ib;
      prog = true;
    }
    if (ca.valid) {
      const int st = static_cast<int>(ia % kStages);
      if (ia < kStages || mbar_test(&empty[st], static_cast<unsigned>((ia / kStages - 1) & 1))) {
        const MegaPhase& ph = sph[ca.p];
        const int t = static_cast<int>(ca.u / ph.kchunks), c = static_cast<int>(ca.u % ph.kchunks);
        const CUtensorMap* map;
        int row0;
        if (ca.v == 0) {
          int s = 0;
          while (s < ph.nseg - 1 && t >= ph.seg_tiles[s]) ++s;
          map = &maps[ph.a_map[s]];
          row0 = (t - (s ? ph.seg_tiles[s - 1] : 0)) * 128;
        } else {
          map = &maps[ph.a2_map];
          row0 = t * 128;
        }
        if (ca.p != last_pa) { stamp(trace, ca.p, 6); last_pa = ca.p; }
        mbar_expect_tx(&full[st], kABytes + (ph.norm ? 0 : BN * 128));
        tma_load_2d_hint(ring + (size_t)st * kStageBytes, map, c * 64, row0, &full[st], pol);
        cursor_next(ca, sph, nph, b, G);
        ++ia;
        prog = true;
      }
    } else if (ib == ia) {
      break;                          // every load issued
    }
    if (prog) {
      bd = Bound();
    } else {
      if (!bd.ok(abort_flag)) ok = false;
      __nanosleep(64);
    }
  }
  if (!ok) {
    if (!ld_volatile(a.abort_flag)) raise_abort(a, 1);
    // Complete the operand of every stage whose weight tile is in flight
    // (stale activations are harmless now), then wait for those copies.
    while (ib < ia) {
      const MegaPhase& ph = sph[cb.p];
      if (!ph.norm) {
        const int st = static_cast<int>(ib % kStages);
        const int c = static_cast<int>(cb.u % ph.kchunks);
        tma_load_2d(ring + (size_t)st * kStageBytes + kABytes, &maps[ph.b_map], c * 64, 0, &full[st]);
      }
      cursor_next(cb, sph, nph, b, G);
      ++ib;
    }
    for (long long i = ia > kStages ? ia - kStages : 0; i < ia; ++i)
      mwait(&full[i % kStages], static_cast<unsigned>((i / kStages) & 1), nullptr);
  }
}

// Warp 1, lane 0: tcgen05.mma issuer.
__device__ __noinline__ void mma_role(const MegaArgs& a, uint32_t tmem) {
  const Lay L = smem_layout();
  uint8_t* const ring = L.ring;
  uint8_t* const uni = L.uni;
  uint64_t* const full = L.full;
  uint64_t* const empty = L.empty;
  uint64_t* const acc_full = L.acc_full;
  uint64_t* const acc_empty = L.acc_empty;
  uint64_t* const bready = L.bready;
  uint64_t* const bfree = L.bfree;
  uint64_t* const drain = L.drain;
  const MegaPhase* const sph = g_phases;
  const int nph = a.nphase, G = gridDim.x, b = blockIdx.x;
  constexpr uint32_t idesc = idesc_bf16(128, BN);
  const uint32_t xn_base = smem_u32(uni);
  bool ok = true;
  bool issued = false;
  long long i = 0;
  int seg = 0, kn = 0;
  for (int p = 0; p < nph && ok; ++p) {
    const MegaPhase& ph = sph[p];
    if (ph.kind != kPhGemm) continue;
    const int NV = nv_of(ph);
    const int KC = ph.kchunks;
    const Range rg = unit_range(ph, b, G);
    if (ph.norm) {
      ok = mwait(bready, static_cast<unsigned>(kn & 1), a.abort_flag);
      if (!ok) break;
      tc_fence_after();
    }
    for (long long u = rg.u0; u < rg.u1 && ok; ++seg) {
      const int c0 = static_cast<int>(u % KC);
      const int c1 = static_cast<int>(c0 + (rg.u1 - u < KC - c0 ? rg.u1 - u : KC - c0));
      const int buf = seg & 1;
      if (u == rg.u0) stamp(a.trace, p, 4);
      if (seg >= 2) ok = mwait(&acc_empty[buf], static_cast<unsigned>((seg / 2 - 1) & 1), a.abort_flag);
      if (!ok) break;
      tc_fence_after();
      const uint32_t d = tmem + buf * 32;
      for (int c = c0; c < c1 && ok; ++c) {
        for (int v = 0; v < NV; ++v, ++i) {
          const int st = static_cast<int>(i % kStages);
          ok = mwait(&full[st], static_cast<unsigned>((i / kStages) & 1), a.abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t sa = smem_u32(ring + (size_t)st * kStageBytes);
          const uint32_t sb = ph.norm ? xn_base + c * (BN * 128) : sa + kABytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_bf16(d + v * BN, smem_desc_sw128(sa + kk * 32), smem_desc_sw128(sb + kk * 32), idesc,
                        (c > c0 || kk > 0) ? 1u : 0u);
          tc_commit(&empty[st]);
          issued = true;
        }
      }
      if (!ok) break;
      tc_commit(&acc_full[buf]);
      u += c1 - c0;
      if (u == rg.u1) stamp(a.trace, p, 5);
    }
    if (!ok) break;
    if (ph.norm) {
      if (rg.u1 > rg.u0) tc_commit(bfree);
      else mbar_arrive(bfree);
      ++kn;
    }
  }
  if (!ok) {
    if (!ld_volatile(a.abort_flag)) raise_abort(a, 2);
    if (issued) {
      tc_commit(drain);
      mwait(drain, 0, nullptr);
    }
  }
}

// Warps 2-5: epilogues and every non-GEMM phase.
__device__ __noinline__ void worker_role(const MegaArgs& a, uint32_t tmem) {
  const Lay L = smem_layout();
  uint8_t* const uni = L.uni;
  uint64_t* const acc_full = L.acc_full;
  uint64_t* const acc_empty = L.acc_empty;
  uint64_t* const bready = L.bready;
  uint64_t* const bfree = L.bfree;
  EpiSmem& E = g_epi;
  const MegaPhase* const sph = g_phases;
  const int nph = a.nphase, G = gridDim.x, b = blockIdx.x;
  const int wt = threadIdx.x - 64;
  int seg = 0, kn = 0;
  bool ok = true;

  if (wt < BN) { E.best_v[wt] = -INFINITY; E.best_i[wt] = 0x7fffffff; }
  for (int p = 0; p < nph && ok; ++p) {
    const MegaPhase& ph = sph[p];
    if (p > 0) {
      if (wt == 0) {
        Bound bd;
        bool seen = true;
        while (ld_volatile(&a.done[(size_t)(p - 1) * kDoneStride]) < static_cast<unsigned>(G)) {
          if (!bd.ok(a.abort_flag)) { seen = false; break; }
          __nanosleep(100);
        }
        __threadfence();
        E.flag = seen;
        if (seen) {
          E.ready = p - 1;
          __threadfence_block();
        }
      }
      epi_sync();
      ok = E.flag != 0;
      epi_sync();
      if (!ok) break;
    }
    if (wt == 0) stamp(a.trace, p, 0);
    if (ph.kind == kPhEmbed) {
      for (int r = b; r < a.M; r += G) {
        int tok = (r == 0) ? a.rs->anchor : a.mask_id;
        if (tok < 0 || tok >= a.V) {
          if (wt == 0) atomicOr(&a.rs->error, kErrRange);
          tok = 0;
        }
        const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const bf16*>(a.embed) + (size_t)tok * a.H);
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(a.x) + (size_t)r * a.H);
        for (int i = wt; i < a.H / 8; i += 128) dst[i] = src[i];
        const long long pos = a.ring->offset + r;
        for (int i = wt; i < a.half; i += 128) a.rope[(size_t)r * a.half + i] = rope_entry(a.inv_freq, i, pos);
      }
    } else if (ph.kind == kPhGemm) {
      const int Mr = a.M;
      if (ph.norm) {
        build_norm_operand(a, p, uni, reinterpret_cast<const bf16*>(a.x), a.H, Mr,
                           reinterpret_cast<const bf16*>(ph.gain), ph.K, a.eps,
                           (ph.lm && b == 0) ? reinterpret_cast<bf16*>(a.xf) : nullptr, E.gain, E.inv, wt);
        fence_proxy_async_shared();
        epi_sync();
        if (wt == 0) { mbar_arrive(bready); stamp(a.trace, p, 1); }
      }
      switch (ph.epi) {
        case kEpiQKV: seg = gemm_epilogue<kEpiQKV>(a, ph, p, Mr, tmem, acc_full, acc_empty, seg, E, wt); break;
        case kEpiResid: seg = gemm_epilogue<kEpiResid>(a, ph, p, Mr, tmem, acc_full, acc_empty, seg, E, wt); break;
        case kEpiSwiglu: seg = gemm_epilogue<kEpiSwiglu>(a, ph, p, Mr, tmem, acc_full, acc_empty, seg, E, wt); break;
        default: seg = gemm_epilogue<kEpiArgmax>(a, ph, p, Mr, tmem, acc_full, acc_empty, seg, E, wt); break;
      }
      ok = seg >= 0;
      if (ok && ph.norm) {
        ok = epi_all(wt != 0 || mwait(bfree, static_cast<unsigned>(kn & 1), a.abort_flag));
        ++kn;
      }
      if (!ok) break;
      if (ph.epi == kEpiArgmax) {
        // Per-CTA best of every lm_head row (block column read0 + r); the
        // last CTA to finish reduces them.
        const int Ml = a.Mlm;
        epi_sync();
        if (wt < Ml) {
          a.part_v[(size_t)b * Ml + wt] = E.best_v[a.read0 + wt];
          a.part_i[(size_t)b * Ml + wt] = E.best_i[a.read0 + wt];
        }
        epi_sync();
        if (wt == 0) {
          __threadfence();
          E.flag = (atomicAdd(&a.done[(size_t)p * kDoneStride], 1u) == static_cast<unsigned>(G - 1));
          stamp(a.trace, p, 3);
        }
        epi_sync();
        if (E.flag) {
          __threadfence();
          if (wt < Ml) {
            float v = -INFINITY;
            int idx = 0x7fffffff;
            for (int c = 0; c < G; ++c) {
              const float cv = __ldcg(a.part_v + (size_t)c * Ml + wt);
              const int ci = __ldcg(a.part_i + (size_t)c * Ml + wt);
              if (better(cv, ci, v, idx)) { v = cv; idx = ci; }
            }
            a.ids[wt] = idx;
            if (a.ids2) a.ids2[wt] = idx;
            a.maxv[wt] = v;
          }
          // Every CTA is past its last wait: rearm the phase counters.
          for (int i = wt; i < nph; i += 128) a.done[(size_t)i * kDoneStride] = 0u;
        }
        continue;
      }
    } else if (ph.kind == kPhAttn) {
      const AttnGeom gm = attn_geom(a);
      AttnTile& S = *reinterpret_cast<AttnTile*>(uni);
      const int qdim = a.nq * kAttnHd, kvdim = a.nkv * kAttnHd;
      const bf16* qkv = reinterpret_cast<const bf16*>(a.qkv);
      const size_t lay = (size_t)ph.layer * a.nkv * a.cap * kAttnHd;
      const int slot0 = static_cast<int>(ring_slot(gm.kstart, a.cap));
      for (int it = b; it < gm.ns * a.nkv; it += G) {
        const int sp = it % gm.ns, g = it / gm.ns;
        const size_t head = lay + (size_t)g * a.cap * kAttnHd;
        attn_split(reinterpret_cast<const bf16*>(a.ring_k) + head, reinterpret_cast<const bf16*>(a.ring_v) + head,
                   qkv + (size_t)g * gm.G * kAttnHd, qkv + qdim + (size_t)g * kAttnHd,
                   qkv + qdim + kvdim + (size_t)g * kAttnHd, a.qkv_n,
                   a.attn_part + ((size_t)g * a.nsplit + sp) * gm.Qn * kAttnPartStride, slot0,
                   static_cast<int>(a.cap), gm.nctx, gm.nk, gm.Qn, gm.G, a.window, sp * kAttnKeys, S, wt,
                   (a.trace && it == b) ? a.trace + ((size_t)p * G + b) * kTraceSlots + 11 : nullptr);
        if (wt == 0 && it == b) stamp(a.trace, p, 10);
      }
      if (wt == 0) stamp(a.trace, p, 1);
    } else {  // kPhComb
      const AttnGeom gm = attn_geom(a);
      const int w = wt >> 5;
      for (int it = b * 4 + w; it < a.nkv * gm.Qn; it += G * 4)
        attn_combine_warp(a.attn_part, a.nsplit, gm.ns, gm.Qn, gm.G, it / gm.Qn, it % gm.Qn,
                          reinterpret_cast<bf16*>(a.attn), a.nq * kAttnHd, wt & 31);
    }
    // This CTA is done with phase p; its writes (ordered before wt 0's fence
    // by the barrier) are visible before it counts. Outputs that the next
    // phase reads with TMA (the split merge's rows, the SwiGLU rows) also
    // need the generic-to-async proxy fence.
    if (ph.kind == kPhComb || (ph.kind == kPhGemm && ph.epi == kEpiSwiglu)) fence_proxy_async_global();
    epi_sync();
    if (wt == 0) {
      __threadfence();
      atomicAdd(&a.done[(size_t)p * kDoneStride], 1u);
      stamp(a.trace, p, 3);
    }
  }
  if (!ok && !ld_volatile(a.abort_flag)) {
    if (wt == 0) raise_abort(a, 4);
  }
}

__global__ void __launch_bounds__(kThreads, 1) draft_kernel(const __grid_constant__ MegaArgs a) {
  const Lay L = smem_layout();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nph = a.nphase;
  constexpr uint32_t kTmemCols = 64;                   // 2 buffers x (gate | up) x 16 columns
  {
    const int* src = reinterpret_cast<const int*>(a.phases);
    int* dst = reinterpret_cast<int*>(g_phases);
    for (int i = threadIdx.x; i < nph * (int)(sizeof(MegaPhase) / 4); i += blockDim.x) dst[i] = src[i];
  }
  if (threadIdx.x == 0) {
    g_epi.ready = -1;               // no phase finished yet
    for (int s = 0; s < kStages; ++s) { mbar_init(&L.full[s], 1); mbar_init(&L.empty[s], 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(&L.acc_full[s], 1); mbar_init(&L.acc_empty[s], 128); }
    mbar_init(L.bready, 1);
    mbar_init(L.bfree, 1);
    mbar_init(L.drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(L.tmem_holder, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *L.tmem_holder;

  if (warp == 0) {
    if (lane == 0) producer_role(a);
  } else if (warp == 1) {
    if (lane == 0) mma_role(a, tmem);
  } else {
    worker_role(a, tmem);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t draft_kernel_smem() { return kSmemBytes; }

cudaError_t init_draft_kernel_attrs() {
  return cudaFuncSetAttribute(draft_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
}

int draft_kernel_blocks_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, draft_kernel, kThreads, kSmemBytes) != cudaSuccess)
    return 0;
  return n;
}

cudaError_t launch_draft_kernel(const MegaArgs& a, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, draft_kernel, a);
}

}  // namespace dfl
