// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05 + TMEM,
// operands staged by TMA), for the decode-shaped linear layers of the round:
//
//   D[n, m] = sum_k W[n, k] * X[m, k],   n < N (output features, large),
//                                        m < M <= BN (block rows, small)
//
// W is the MMA's A operand (128-row tiles), X its B operand (BN rows, zero
// filled past M), so one MMA is 128 x BN x 16 and the accumulator is a
// 128-lane x BN-column fp32 tile in TMEM.
//
// Work split: the (tile, 64-wide K chunk) units of the whole GEMM are cut
// into gridDim.x contiguous ranges, one per CTA (one CTA per SM), so every
// SM streams the same number of weight bytes. A tile whose K range spans
// several CTAs is finished cooperatively: each contributor writes its fp32
// partial and arrives on the tile's counter; once all of a CTA's own tiles
// are published, contributor k of n waits (bounded) for the others and
// reduces float4 groups k, k + n, ... of the block rows, summing the partials
// in CTA order (deterministic). Every CTA of the grid is resident (one per
// SM), so these waits cannot block one another. The lm_head's split tiles
// (two contributors) are finished by the later one, which knows it is last
// from a ticket.
//
// Roles: warp 0 issues TMA loads into an S-stage shared-memory ring (the
// weight tiles of the first S units are requested before the programmatic
// launch dependency is resolved, so they stream while the previous kernel
// finishes); warp 1 allocates TMEM and issues tcgen05.mma; warps 2-5 read the
// accumulators back and run the epilogue (store, residual add, SwiGLU, K/V
// with k-norm + RoPE into ring slots, or softcap + argmax for the lm_head).
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.h"
#include "ptx.cuh"
#include "tc_epilogue.cuh"

namespace dfl {
namespace {

constexpr uint32_t tmem_cols(int n) { return n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : n <= 256 ? 256 : 512; }

// A stage holds P consecutive K chunks of one tile (P = 2: each weight row
// is read as 256 contiguous bytes per stage instead of 128, which lets HBM
// stream at ~95% of its copy rate instead of ~65%): the P weight sub-tiles
// (NV each: gate, up), then the P activation sub-tiles.
template <int BN, int NV, int STAGES, int P>
struct Cfg {
  static constexpr int kSub = NV * kABytes;
  static constexpr int kBOff = P * kSub;
  static constexpr int kStage = P * (kSub + BN * 128);
  // accumulator buffers in TMEM: two (the epilogue of one tile overlaps the
  // next tile's MMAs) while they fit the 512 columns, else one
  static constexpr int kBufs = 2 * NV * BN <= 512 ? 2 : 1;
  static constexpr uint32_t kTmem = tmem_cols(kBufs * NV * BN);
  static constexpr size_t kSmem = (size_t)STAGES * kStage + 1024 + 512;
};


// BN block rows: 16 or 32 for a draft block; 64, 128 or 160 for more rows in
// one launch (the fp32-sum and argmax epilogues only; 160 for the sums):
// the B tile is then loaded as BN / 32 boxes of 32 rows, one MMA still covers
// all BN columns, and the epilogue reads the accumulator 32 columns at a time.
template <int BN, int EPI, int STAGES, int P>
__global__ void __launch_bounds__(kThreads, 2) tc_gemm_kernel(const __grid_constant__ TcGemmArgs a) {
  constexpr int NV = (EPI == kEpiSwiglu || EPI == kEpiRedPair) ? 2 : 1;
  using C = Cfg<BN, NV, STAGES, P>;
  constexpr int EC = BN < 32 ? BN : 32;           // block rows an epilogue pass takes (and a TMA box holds)
  constexpr int NCH = BN / EC;
  static_assert(NCH == 1 || EPI == kEpiRed || EPI == kEpiRedPair || EPI == kEpiArgmax,
                "more than 32 block rows only for the fp32-sum and argmax epilogues");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023) & ~1023u) - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)STAGES * C::kStage);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
  __shared__ float best_v[BN];
  __shared__ int best_i[BN];
  __shared__ float red_v[4][BN];
  __shared__ int red_i[4][BN];
  __shared__ int s_last;
  __shared__ float kv_ss[4][BN];
  __shared__ float kv_x[EPI == kEpiKVRing ? 128 * BN : 1];
  // argmax over more than 32 block rows: each epilogue warp's 32 x 32 chunk
  // of softcapped logits, transposed so that a lane scans one block row
  __shared__ float tr_z[(EPI == kEpiArgmax && NCH > 1) ? 4 * 32 * 33 : 1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, b = blockIdx.x;
  // Units (tile, 64-wide K chunk) in 32-bit arithmetic: the host checks
  // that tiles * kchunks * grid fits.
  const unsigned KC = a.kchunks;
  const unsigned U = static_cast<unsigned>(a.tiles) * KC;
  // With a.whole_tiles (the lm_head at more than 8 rows) every CTA takes
  // whole tiles (10 or 11 of the 1579 at the Muse shape): no split tile to
  // finish at the end of its range, whose argmax epilogue grows with the
  // rows, against a ~3% imbalance; otherwise the units are cut evenly.
  const unsigned tb0 = static_cast<unsigned>(a.tiles) * b / G, tb1 = static_cast<unsigned>(a.tiles) * (b + 1) / G;
  const bool whole = EPI == kEpiArgmax && a.whole_tiles;
  const unsigned u0 = whole ? tb0 * KC : U * b / G;
  const unsigned u1 = whole ? tb1 * KC : U * (b + 1) / G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(&acc_full[s], 1); mbar_init(&acc_empty[s], 128); }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_holder, C::kTmem);
  if (threadIdx.x < BN) { best_v[threadIdx.x] = -INFINITY; best_i[threadIdx.x] = 0x7fffffff; }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  pdl_launch_dependents();
  if (threadIdx.x == 0) ktrace_mark(a.trace, 0);

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&a.b_map);
      const uint64_t pol = policy_evict_first();
      bool ok = true;
      // Stage i covers units [u, u + nc): nc = P while the next unit is in the
      // same tile and in this CTA's range (the MMA issuer pairs the same way).
      auto issue_a = [&](int st, unsigned u, int nc) {
        const int t = static_cast<int>(u / KC), c = static_cast<int>(u % KC);
        int s = 0;
        while (s < a.nseg - 1 && t >= a.seg_tiles[s]) ++s;
        const int row0 = (t - (s ? a.seg_tiles[s - 1] : 0)) * 128;
        uint8_t* sa = smem + (size_t)st * C::kStage;
        mbar_expect_tx(&full[st], nc * (C::kSub + BN * 128));
        for (int k = 0; k < nc; ++k) {
          tma_load_2d_hint(sa + k * C::kSub, &a.a_map[s], (c + k) * 64, row0, &full[st], pol);
          if (NV == 2) tma_load_2d_hint(sa + k * C::kSub + kABytes, &a.a2_map, (c + k) * 64, t * 128, &full[st], pol);
        }
      };
      auto issue_b = [&](int st, unsigned u, int nc) {
        const int c = static_cast<int>(u % KC);
        uint8_t* sb = smem + (size_t)st * C::kStage + C::kBOff;
        for (int k = 0; k < nc; ++k)
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch)
            tma_load_2d(sb + k * BN * 128 + ch * EC * 128, &a.b_map, (c + k) * 64, a.b_row0 + ch * EC, &full[st]);
      };
      auto width = [&](unsigned u) {
        return (P == 2 && u + 1 < u1 && (u % KC) + 1 < KC) ? 2 : 1;
      };
      // The weight tiles of the first stages do not depend on earlier
      // kernels: request them before the programmatic launch dependency
      // resolves, and their activations once it has.
      unsigned u = u0;
      int pre = 0;
      for (; pre < STAGES && u < u1; ++pre) {
        const int nc = width(u);
        issue_a(pre, u, nc);
        u += nc;
      }
      pdl_wait();
      {
        unsigned v = u0;
        for (int j = 0; j < pre; ++j) {
          const int nc = width(v);
          issue_b(j, v, nc);
          v += nc;
        }
      }
      for (unsigned i = pre; u < u1 && ok; ++i) {
        const int st = static_cast<int>(i % STAGES);
        ok = mbar_wait(&empty[st], static_cast<unsigned>((i / STAGES - 1) & 1));
        if (!ok) break;
        const int nc = width(u);
        issue_a(st, u, nc);
        issue_b(st, u, nc);
        u += nc;
      }
      if (!ok) atomicOr(a.err, 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, BN);
      bool ok = true;
      unsigned i = 0;
      int seg = 0;
      for (unsigned u = u0; u < u1 && ok; ++seg) {
        const int c0 = static_cast<int>(u % KC);
        const int c1 = static_cast<int>(c0 + (u1 - u < KC - c0 ? u1 - u : KC - c0));
        const int buf = seg % C::kBufs;
        if (seg >= C::kBufs) ok = mbar_wait(&acc_empty[buf], static_cast<unsigned>((seg / C::kBufs - 1) & 1));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * NV * BN;
        for (int c = c0; c < c1; ++i) {
          const int nc = (P == 2 && c + 1 < c1) ? 2 : 1;
          const int st = static_cast<int>(i % STAGES);
          ok = mbar_wait(&full[st], static_cast<unsigned>((i / STAGES) & 1));
          if (!ok) break;
          tc_fence_after();
          const uint32_t s0 = smem_u32(smem + (size_t)st * C::kStage);
          for (int k = 0; k < nc; ++k) {
            const uint32_t sa = s0 + k * C::kSub;
            const uint32_t sb = s0 + C::kBOff + k * BN * 128;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bd = smem_desc_sw128(sb + kk * 32);
              const uint32_t acc = (c + k > c0 || kk > 0) ? 1u : 0u;
              tc_mma_bf16(d, smem_desc_sw128(sa + kk * 32), bd, idesc, acc);
              if (NV == 2) tc_mma_bf16(d + BN, smem_desc_sw128(sa + kABytes + kk * 32), bd, idesc, acc);
            }
          }
          tc_commit(&empty[st]);
          c += nc;
        }
        if (!ok) break;
        tc_commit(&acc_full[buf]);
        u += c1 - c0;
      }
      if (a.trace.p) ktrace_mark(KTrace{a.trace.p, a.trace.slot + 1}, 1);   // last MMA issued
      if (!ok) atomicOr(a.err, 2);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    pdl_wait();
    if (threadIdx.x == 64) ktrace_mark(a.trace, 1);
    const int q = warp & 3;                       // TMEM lane quarter this warp may read
    const int row = q * 32 + lane;                // accumulator row = output feature in tile
    const int first_tile = static_cast<int>(u0 / KC);
    const int mq = (a.M + 3) / 4;                 // float4 groups of block rows
    bool ok = true;
    int seg = 0;

    // Per-tile values the epilogue needs, requested early: the ring offset
    // and base (K/V into the ring) and, per tile, this row's head-norm gain.
    long long ring_off = 0, ring_base = 0;
    int ring_s0 = 0;                              // ring slot of ring_off
    if (EPI == kEpiKVRing) {
      ring_off = a.ring->offset;
      ring_base = a.ring->base;
      ring_s0 = static_cast<int>(ring_slot(ring_off, a.cap));
    }
    // This thread's RoPE entries, the same for every tile (kept in registers
    // for 16 block rows; 32 would crowd out the epilogue's other values).
    constexpr bool kHoistRope = EPI == kEpiKVRing && BN == 16;
    float2 rope_cs[BN];
    if (kHoistRope) rope_entries<BN>(rope_cs, a.rope, a.M, a.neox, row);
    auto gain_of = [&](int t) -> float {
      if (EPI == kEpiKVRing) {
        const int sg = t / a.nkv;
        if (!(sg & 1)) return __bfloat162float(reinterpret_cast<const bf16*>(a.kgain[sg >> 1])[row]);
      }
      return 0.f;
    };
    // Final epilogue of tile t for block rows [m0, m1); gv = gain_of(t).
    // Residuals of tile t's row for the block rows (kEpiResid), requested
    // ahead of the accumulator so the finish has no dependent load.
    // (Kept for 16 block rows; at 32 the registers are better spent elsewhere
    // and the finish loads them.)
    constexpr bool kHoistResid = EPI == kEpiResid && BN == 16;
    auto resid_at = [&](int m, int n) {
      return __bfloat162float(reinterpret_cast<const bf16*>(a.r)[(size_t)m * a.ldr + n]);
    };
    auto resid_of = [&](int t, float (&res)[BN]) {
      const int n = t * 128 + row;
#pragma unroll
      for (int m = 0; m < BN; ++m) res[m] = (kHoistResid && m < a.M && n < a.N) ? resid_at(m, n) : 0.f;
    };
    auto finish_tile = [&](float (&acc)[NV][BN], int t, int m0, int m1, float gv, const float (&res)[BN]) {
      const int n = t * 128 + row;
      const bool valid = n < a.N;
      if (EPI == kEpiArgmax) {
        const float cap = a.softcap;
#pragma unroll
        for (int m = 0; m < BN; ++m) {
          if (m < m0 || m >= m1) continue;        // uniform: only this call's columns
          float z = acc[0][m];
          if (cap > 0.f) z = cap * tanhf(z / cap);
          float bv = valid ? z : -INFINITY;
          int bi = valid ? n : 0x7fffffff;
          warp_argmax(bv, bi);
          if (lane == 0) { red_v[q][m] = bv; red_i[q][m] = bi; }
        }
        epi_sync();
        if (threadIdx.x >= 64 + m0 && threadIdx.x < 64 + m1) {
          const int m = threadIdx.x - 64;
          float bv = best_v[m];
          int bi = best_i[m];
#pragma unroll
          for (int w = 0; w < 4; ++w)
            if (better(red_v[w][m], red_i[w][m], bv, bi)) { bv = red_v[w][m]; bi = red_i[w][m]; }
          best_v[m] = bv;
          best_i[m] = bi;
        }
        epi_sync();
      } else if (EPI == kEpiKVRing) {
        // tile t = kv head h of layer l, K or V (hd = 128 = one tile)
        const int sg = t / a.nkv, h = t % a.nkv;
        const int layer = sg >> 1;
        const bool isv = sg & 1;
        const long long off0 = ring_off;
        const size_t head_base = (((size_t)layer * a.nkv + h) * a.cap) * 128;
        bf16* dst = reinterpret_cast<bf16*>(isv ? a.ring_v : a.ring_k) + head_base;
        float val[BN];
#pragma unroll
        for (int m = 0; m < BN; ++m) val[m] = rnd_bf(acc[0][m]);
        if (!isv) {
          if (kHoistRope) head_norm_rope_cs<BN>(val, gv, [&](int m) { return rope_cs[m]; }, a.M, a.neox, a.eps, row, lane, q, kv_ss, kv_x, m0, m1);
          else head_norm_rope_tile<BN>(val, gv, a.rope, a.M, a.neox, a.eps, row, lane, q, kv_ss, kv_x, m0, m1);
        }
#pragma unroll
        for (int m = 0; m < BN; ++m) {
          if (m < m0 || m >= m1) continue;
          const long long pos = off0 + m;
          if (a.append_only && pos - ring_base >= a.cap) {
            if (row == 0) atomicOr(&a.ring->error, kErrFull);
            continue;
          }
          int slot = ring_s0 + m;                 // = ring_slot(pos, cap)
          while (slot >= a.cap) slot -= static_cast<int>(a.cap);
          dst[(size_t)slot * 128 + row] = __float2bfloat16_rn(val[m]);
        }
      } else if (valid) {
        bf16* Y = reinterpret_cast<bf16*>(a.y);
#pragma unroll
        for (int m = 0; m < BN; ++m) {
          if (m >= m0 && m < m1) {
            float out;
            if (EPI == kEpiStore) {
              out = acc[0][m];
            } else if (EPI == kEpiResid) {
              out = (kHoistResid ? res[m] : resid_at(m, n)) + rnd_bf(acc[0][m]);
            } else {
              out = silu_f(rnd_bf(acc[0][m])) * rnd_bf(acc[NV - 1][m]);
            }
            Y[(size_t)m * a.ldy + n] = __float2bfloat16_rn(out);
          }
        }
      }
    };

    // Whole tiles are finished at once. A tile split across CTAs is finished
    // cooperatively: every contributor publishes its fp32 partial and arrives
    // on the tile's counter; once all of this CTA's tiles are published it
    // waits for the other contributors of its split tiles and reduces one
    // float4 group of block rows each (contributor k of n takes groups k,
    // k + n, ...), summing the partials in CTA order. (The lm_head's split
    // tiles have two contributors; the later one finishes those alone.)
    int split_first = -1, split_last = -1;        // split tiles published (slot 0, slot 1)
    float gv_first = 0.f, gv_last = 0.f;          // and their rows' gains
    float res_first[BN], res_last[BN];            // and residuals
#pragma unroll
    for (int m = 0; m < BN; ++m) res_first[m] = res_last[m] = 0.f;
    unsigned* const arrive = a.tile_ctr;
    unsigned* const depart = a.tile_ctr + kTileDepart;
    for (unsigned u = u0; u < u1 && ok; ++seg) {
      const int t = static_cast<int>(u / KC);
      const int c0 = static_cast<int>(u % KC);
      const int c1 = static_cast<int>(c0 + (u1 - u < KC - c0 ? u1 - u : KC - c0));
      const int buf = seg % C::kBufs;
      const float gv = gain_of(t);
      float res[BN];
      resid_of(t, res);
      ok = mbar_wait(&acc_full[buf], static_cast<unsigned>((seg / C::kBufs) & 1));
      if (!ok) break;
      tc_fence_after();
      if constexpr (NCH > 1) {
        // 32 block rows at a time; every tile here is whole (the argmax) or
        // needs no finish (the fp32 sums)
        const int n = t * 128 + row;
#pragma unroll 1
        for (int ch = 0; ch < NCH; ++ch) {
          const int mo = ch * EC;
          float acc[NV][EC];
#pragma unroll
          for (int v = 0; v < NV; ++v)
#pragma unroll
            for (int j = 0; j < EC / 16; ++j)
              tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * NV * BN + v * BN + mo + j * 16,
                        &acc[v][j * 16]);
          tmem_ld_wait();
          if (ch == NCH - 1) {
            tc_fence_before();
            mbar_arrive(&acc_empty[buf]);
          }
          if (EPI == kEpiRed || EPI == kEpiRedPair) {
            if (n < a.N) {
#pragma unroll
              for (int v = 0; v < NV; ++v) {
                float* dst = a.acc + (size_t)v * a.N + n;
#pragma unroll
                for (int m = 0; m < EC; ++m)
                  if (mo + m < a.M) atomicAdd(dst + (size_t)(mo + m) * a.ldacc, acc[v][m]);
              }
            }
          } else {
            // the warp's 32 vocabulary rows x 32 block rows through shared
            // memory: lane m then scans block row mo + m over the 32 rows in
            // index order (ties keep the lower index)
            const bool valid = n < a.N;
            const float cap = a.softcap;
            float* tz = tr_z + q * 32 * 33;
#pragma unroll
            for (int m = 0; m < EC; ++m) {
              float z = acc[0][m];
              if (cap > 0.f) z = cap * tanhf(z / cap);
              tz[lane * 33 + m] = valid ? z : -INFINITY;
            }
            __syncwarp();
            {
              float bv = -INFINITY;
              int bi = 0x7fffffff;
              const int n0 = t * 128 + q * 32;
              if (mo + lane < a.M) {
#pragma unroll 8
                for (int l = 0; l < 32; ++l) {
                  const float v = tz[l * 33 + lane];
                  if (n0 + l < a.N && better(v, n0 + l, bv, bi)) { bv = v; bi = n0 + l; }
                }
              }
              red_v[q][mo + lane] = bv;
              red_i[q][mo + lane] = bi;
            }
            __syncwarp();
            epi_sync();
            if (threadIdx.x >= 64 && threadIdx.x < 64 + EC && mo + static_cast<int>(threadIdx.x) - 64 < a.M) {
              const int m = mo + static_cast<int>(threadIdx.x) - 64;
              float bv = best_v[m];
              int bi = best_i[m];
#pragma unroll
              for (int w = 0; w < 4; ++w)
                if (better(red_v[w][m], red_i[w][m], bv, bi)) { bv = red_v[w][m]; bi = red_i[w][m]; }
              best_v[m] = bv;
              best_i[m] = bi;
            }
            epi_sync();
          }
        }
        u += c1 - c0;
        continue;
      }
      float acc[NV][BN];
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int j = 0; j < BN / 16; ++j)
          tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * NV * BN + v * BN + j * 16,
                    &acc[v][j * 16]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);
      u += c1 - c0;
      if (EPI == kEpiRed || EPI == kEpiRedPair) {
        // add this CTA's K range of the tile into the fp32 sums (the second
        // weight's at column offset N); the kernel that reads them (after the
        // programmatic dependency) finishes them
        const int n = t * 128 + row;
        if (n < a.N) {
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            float* dst = a.acc + (size_t)v * a.N + n;
#pragma unroll
            for (int m = 0; m < BN; ++m)
              if (m < a.M) atomicAdd(dst + (size_t)m * a.ldacc, acc[v][m]);
          }
        }
        continue;
      }
      if (c0 == 0 && c1 == KC) {
        finish_tile(acc, t, 0, a.M, gv, res);
      } else if (EPI == kEpiArgmax) {
        // lm_head: a split tile has two contributors (each CTA streams many
        // tiles); the later one reads the other's partial and finishes it.
        const int slot = (t == first_tile) ? 0 : 1;
        put_partial<NV, BN>(a.partials, b, slot, row, mq, acc);
        epi_sync();
        const int bf = owner_of_u32(t * KC, U, G);
        const int bl = owner_of_u32(t * KC + KC - 1, U, G);
        if (threadIdx.x == 64) {
          __threadfence();
          s_last = (atomicAdd(&arrive[t], 1u) == static_cast<unsigned>(bl - bf));
        }
        epi_sync();
        if (s_last) {
          __threadfence();
          const int s_bf = U * bf / G == t * KC ? 0 : 1;
          if (mq == 1) sum_partials<NV, BN, 1, 2>(acc, a.partials, row, bf, bl, mq, s_bf);
          else sum_partials<NV, BN, BN / 4, 2>(acc, a.partials, row, bf, bl, mq, s_bf);
          if (threadIdx.x == 64) arrive[t] = 0u;
          finish_tile(acc, t, 0, a.M, gv, res);
        }
      } else {
        const int slot = (t == first_tile) ? 0 : 1;
        put_partial<NV, BN>(a.partials, b, slot, row, mq, acc);
        if (slot == 0) {
          split_first = t; gv_first = gv;
#pragma unroll
          for (int m = 0; m < BN; ++m) res_first[m] = res[m];
        } else {
          split_last = t; gv_last = gv;
#pragma unroll
          for (int m = 0; m < BN; ++m) res_last[m] = res[m];
        }
        epi_sync();
        if (threadIdx.x == 64) {
          __threadfence();
          atomicAdd(&arrive[t], 1u);
        }
      }
    }
    if (a.trace.p && threadIdx.x == 64) ktrace_mark(KTrace{a.trace.p, a.trace.slot + 1}, 2);  // tiles published
    // split tiles (one launch's block rows at most 32)
    if constexpr (NCH == 1) {
    // Contributors whose partial loads are in flight at once: the long-K
    // GEMMs (residual, store) split a tile over about ten CTAs, the others
    // over two to four and need the registers for their epilogue.
    constexpr int kSumBatch = (EPI == kEpiResid || EPI == kEpiStore) ? (NV == 1 ? 16 : 4) : (NV == 1 ? 8 : 4);
    int bfs[2], bls[2];
    bool work[2];
#pragma unroll
    for (int slot = 0; slot < 2; ++slot) {
      const int t = slot == 0 ? split_first : split_last;
      bfs[slot] = t < 0 ? 0 : owner_of_u32(t * KC, U, G);
      bls[slot] = t < 0 ? -1 : owner_of_u32(t * KC + KC - 1, U, G);
      work[slot] = t >= 0 && b - bfs[slot] < mq;
    }
    // Wait for the other contributors of both split tiles before reducing
    // either, so the two waits overlap.
    if (threadIdx.x == 64 && ok) {
#pragma unroll
      for (int slot = 0; slot < 2; ++slot) {
        if (!work[slot]) continue;
        const int t = slot == 0 ? split_first : split_last;
        const unsigned nc = static_cast<unsigned>(bls[slot] - bfs[slot] + 1);
        unsigned spins = 0;
        while (ld_acquire(&arrive[t]) < nc) {
          if (++spins > (1u << 24)) { atomicOr(a.err, 8); break; }
          __nanosleep(64);
        }
      }
      if (a.trace.p && (work[0] || work[1])) ktrace_mark(KTrace{a.trace.p, a.trace.slot + 2}, 1);  // present
    }
    // This CTA no longer reads the arrive counters: depart. The last
    // contributor of a tile to depart clears both of its counters for the
    // next launch; the results are looked at only after the reduction, so the
    // atomics' round trip overlaps it.
    unsigned dep[2] = {0u, 0u};
    if (threadIdx.x == 64 && ok) {
#pragma unroll
      for (int slot = 0; slot < 2; ++slot) {
        const int t = slot == 0 ? split_first : split_last;
        if (t >= 0) dep[slot] = atomicAdd(&depart[t], 1u);
      }
    }
    if (ok && (work[0] || work[1])) {
      epi_sync();
#pragma unroll
      for (int slot = 0; slot < 2; ++slot) {
        if (!work[slot]) continue;
        const int t = slot == 0 ? split_first : split_last;
        const int bf = bfs[slot], bl = bls[slot];
        const int nc = bl - bf + 1;
        const int s_bf = U * bf / G == t * KC ? 0 : 1;
        for (int g = b - bf; g < mq; g += nc) {
          float acc[NV][BN];
          sum_group<NV, BN, kSumBatch>(acc, a.partials, row, g, bf, bl, s_bf);
          finish_tile(acc, t, 4 * g, 4 * g + 4 < a.M ? 4 * g + 4 : a.M, slot == 0 ? gv_first : gv_last,
                      slot == 0 ? res_first : res_last);
        }
      }
      if (a.trace.p && threadIdx.x == 64) ktrace_mark(KTrace{a.trace.p, a.trace.slot + 3}, 1);  // summed
    }
    if (threadIdx.x == 64 && ok) {
#pragma unroll
      for (int slot = 0; slot < 2; ++slot) {
        const int t = slot == 0 ? split_first : split_last;
        if (t >= 0 && dep[slot] == static_cast<unsigned>(bls[slot] - bfs[slot])) {
          arrive[t] = 0u;
          depart[t] = 0u;
        }
      }
    }
    }
    if (a.trace.p && threadIdx.x == 64) ktrace_mark(KTrace{a.trace.p, a.trace.slot + 2}, 2);  // finished
    if (!ok) atomicOr(a.err, 4);

    if (EPI == kEpiArgmax) {
      // Per-CTA best of every row folded into one 64-bit key per row with an
      // atomic maximum: the value's order-preserving bits above the inverted
      // index, so the larger value wins and equal values keep the lower
      // index (-0 is taken as +0). The last CTA to finish decodes the keys and
      // clears them for the next launch.
      epi_sync();
      if (threadIdx.x >= 64 && threadIdx.x < 64 + BN && threadIdx.x - 64 < a.M) {
        const int m = threadIdx.x - 64;
        const uint32_t u = __float_as_uint(best_v[m] + 0.0f);
        const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
        const unsigned long long key =
            (static_cast<unsigned long long>(ord) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(best_i[m]));
        atomicMax(a.best_key + m, key);
      }
      __threadfence();
      epi_sync();
      if (threadIdx.x == 64) s_last = (atomicAdd(a.done_ctr, 1u) == static_cast<unsigned>(G - 1));
      epi_sync();
      if (s_last && threadIdx.x >= 64 && threadIdx.x < 64 + BN && threadIdx.x - 64 < a.M) {
        __threadfence();
        const int m = threadIdx.x - 64;
        const unsigned long long key = atomicExch(a.best_key + m, 0ull);
        const uint32_t ord = static_cast<uint32_t>(key >> 32);
        const uint32_t u = (ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord;
        const int idx = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key));
        a.ids[m] = idx;
        if (a.ids2) a.ids2[m] = idx;
        a.maxv[m] = __uint_as_float(u);
        if (m == 0) *a.done_ctr = 0u;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) ktrace_mark(a.trace, 2);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmem);
  }
}

// Ring depth in paired-chunk stages: the decode-layer GEMMs take four (three
// for the two-weight SwiGLU stages), which at up to 16 block rows holds most
// of a CTA's weight range, requested before the programmatic dependency
// resolves; the lm_head is long and takes a deeper ring.
// With 64, 128 or 160 block rows a stage's X sub-tiles grow to 8, 16 or
// 20 KB: the ring shrinks to what fits (48 / 64 / 72 KB stages; two weights:
// 80 / 96 / 104 KB). Single-chunk stages with deeper rings measured no
// faster for the layer GEMMs and slower for the lm_head.
template <int BN, int EPI>
constexpr int stages_for() {
  if (BN == 64) return (EPI == kEpiSwiglu || EPI == kEpiRedPair) ? 2 : 4;
  if (BN == 128) return (EPI == kEpiSwiglu || EPI == kEpiRedPair) ? 2 : 3;
  if (BN == 160) return (EPI == kEpiSwiglu || EPI == kEpiRedPair) ? 2 : 3;
  return EPI == kEpiArgmax ? (BN == 16 ? 6 : 5) : (EPI == kEpiSwiglu || EPI == kEpiRedPair) ? 3 : 4;
}
template <int BN, int EPI>
constexpr int pairs_for() { return 2; }

template <int BN, int EPI>
cudaError_t launch_tc(const TcGemmArgs& a, int grid, bool pdl, cudaStream_t st) {
  constexpr int S = stages_for<BN, EPI>();
  constexpr int P = pairs_for<BN, EPI>();
  constexpr int NV = (EPI == kEpiSwiglu || EPI == kEpiRedPair) ? 2 : 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<BN, NV, S, P>::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<BN, EPI, S, P>, a);
}

// Every tensor-core kernel asks for the largest shared-memory carveout, so
// that an SM moving from one of them to the next (the GEMMs of a layer take
// 131 to 197 KB) never has to drain to reconfigure its L1 / shared split.
template <int BN, int EPI>
cudaError_t attr_tc() {
  constexpr int S = stages_for<BN, EPI>();
  constexpr int P = pairs_for<BN, EPI>();
  constexpr int NV = (EPI == kEpiSwiglu || EPI == kEpiRedPair) ? 2 : 1;
  const cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<BN, EPI, S, P>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)Cfg<BN, NV, S, P>::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(tc_gemm_kernel<BN, EPI, S, P>, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared);
}

// ---------------------------------------------------------------------------
// Many-row GEMM (context ingest): Y[m, n] = rnd(sum_k X[m, k] W[n, k]) with
// X the A operand (128-row tiles) and W the B operand (256-row tiles), one
// 128 x 256 x 16 MMA per K step, fp32 accumulators in TMEM (two 256-column
// buffers = the whole TMEM), full K per tile, persistent CTAs striding over
// the (m-tile, n-tile) grid. Same warp roles as above.
// ---------------------------------------------------------------------------
constexpr int kWideN = 256;
constexpr int kWideStages = 4;
constexpr int kWideStage = kABytes + kWideN * 128;          // 48 KB
constexpr size_t kWideSmem = (size_t)kWideStages * kWideStage + 1024 + 512;

__global__ void __launch_bounds__(kThreads, 1) tc_gemm_wide_kernel(const __grid_constant__ TcWideArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023) & ~1023u) - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kWideStages * kWideStage);
  uint64_t* empty = full + kWideStages;
  uint64_t* acc_full = empty + kWideStages;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = (a.M + 127) / 128, nt = (a.N + kWideN - 1) / kWideN;
  const int T = mt * nt, KC = a.K / 64;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kWideStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(&acc_full[s], 1); mbar_init(&acc_empty[s], 128); }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      pdl_wait();
      bool ok = true;
      long long i = 0;
      for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
        const int m0 = (t % mt) * 128, n0 = (t / mt) * kWideN;
        int s = 0;
        while (s < a.nseg - 1 && n0 >= a.seg_rows[s]) ++s;
        const int nrow0 = n0 - (s ? a.seg_rows[s - 1] : 0);
        for (int c = 0; c < KC && ok; ++c, ++i) {
          const int st = static_cast<int>(i % kWideStages);
          if (i >= kWideStages) ok = mbar_wait(&empty[st], static_cast<unsigned>((i / kWideStages - 1) & 1));
          if (!ok) break;
          uint8_t* sa = smem + (size_t)st * kWideStage;
          mbar_expect_tx(&full[st], kWideStage);
          tma_load_2d(sa, &a.x_map, c * 64, m0, &full[st]);
          tma_load_2d(sa + kABytes, &a.w_map[s], c * 64, nrow0, &full[st]);
        }
      }
      if (!ok) atomicOr(a.err, 8);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, kWideN);
      bool ok = true;
      long long i = 0;
      int seg = 0;
      for (int t = blockIdx.x; t < T && ok; t += gridDim.x, ++seg) {
        const int buf = seg & 1;
        if (seg >= 2) ok = mbar_wait(&acc_empty[buf], static_cast<unsigned>((seg / 2 - 1) & 1));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * kWideN;
        for (int c = 0; c < KC; ++c, ++i) {
          const int st = static_cast<int>(i % kWideStages);
          ok = mbar_wait(&full[st], static_cast<unsigned>((i / kWideStages) & 1));
          if (!ok) break;
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + (size_t)st * kWideStage);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_bf16(d, smem_desc_sw128(sa + kk * 32), smem_desc_sw128(sa + kABytes + kk * 32), idesc,
                        (c > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&empty[st]);
        }
        tc_commit(&acc_full[buf]);
      }
      if (!ok) atomicOr(a.err, 16);
    }
  } else {
    pdl_wait();
    const int q = warp & 3;
    const int row = q * 32 + lane;
    bool ok = true;
    int seg = 0;
    bf16* Y = reinterpret_cast<bf16*>(a.y);
    for (int t = blockIdx.x; t < T && ok; t += gridDim.x, ++seg) {
      const int m0 = (t % mt) * 128, n0 = (t / mt) * kWideN;
      const int buf = seg & 1;
      ok = mbar_wait(&acc_full[buf], static_cast<unsigned>((seg / 2) & 1));
      if (!ok) break;
      tc_fence_after();
      const int m = m0 + row;
      if (a.ring_k) {
        // Two whole heads of one layer's K or V: the thread holds its row's
        // 128 values of each head, so the head norm and RoPE are thread-local.
        const int per_layer = 2 * a.kvdim;
        const int cin = n0 % per_layer;
        const bool isv = cin >= a.kvdim;
        const int layer = a.l0 + n0 / per_layer;
        const int hbase = (cin % a.kvdim) / 128;
        const long long pos = a.pos0 + m;
        bool store = m < a.M;
        if (store && a.append_only && pos - a.ring->base >= a.cap) {
          atomicOr(&a.ring->error, kErrFull);
          store = false;
        }
        const long long slot = ring_slot(pos, a.cap);
        const bf16* g = reinterpret_cast<const bf16*>(a.kgain[layer]);
        const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * kWideN;
        auto put16 = [&](bf16* dst, const float* v) {
          uint4 pk[2];
          uint32_t* w32 = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
            w32[e] = *reinterpret_cast<uint32_t*>(&b2);
          }
          reinterpret_cast<uint4*>(dst)[0] = pk[0];
          reinterpret_cast<uint4*>(dst)[1] = pk[1];
        };
        for (int hh = 0; hh < kWideN / 128; ++hh) {
          const uint32_t th = tl + hh * 128;
          bf16* dst = reinterpret_cast<bf16*>(isv ? a.ring_v : a.ring_k) +
                      (((size_t)layer * a.nkv + hbase + hh) * a.cap + slot) * 128;
          if (isv) {
            for (int j = 0; j < 8; ++j) {
              float v[16];
              tmem_ld16(th + j * 16, v);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] = rnd_bf(v[e]);
              if (store) put16(dst + j * 16, v);
            }
            continue;
          }
          // K head: the values rounded as stored, their 1/rms, then per piece
          // the gain and RoPE (neox pairs dims i and i + 64: pieces j, j + 4).
          float ss = 0.f;
          for (int j = 0; j < 8; ++j) {
            float v[16];
            tmem_ld16(th + j * 16, v);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) { const float r = rnd_bf(v[e]); ss = fmaf(r, r, ss); }
          }
          const float inv = rsqrtf(ss / 128.0f + a.eps);
          const float2* rr = a.rope + (size_t)(m < a.M ? m : 0) * 64;
          auto scale = [&](float* v, int d0) {
            float gv[16];
            load8(g + d0, gv);
            load8(g + d0 + 8, gv + 8);
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = rnd_bf(v[e]) * inv * gv[e];
          };
          if (a.neox) {
            for (int j = 0; j < 4; ++j) {
              float lo[16], hi[16];
              tmem_ld16(th + j * 16, lo);
              tmem_ld16(th + (j + 4) * 16, hi);
              tmem_ld_wait();
              scale(lo, j * 16);
              scale(hi, (j + 4) * 16);
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const float2 cs = rr[j * 16 + e];
                const float x0 = lo[e], x1 = hi[e];
                lo[e] = x0 * cs.x - x1 * cs.y;
                hi[e] = x0 * cs.y + x1 * cs.x;
              }
              if (store) { put16(dst + j * 16, lo); put16(dst + (j + 4) * 16, hi); }
            }
          } else {
            for (int j = 0; j < 8; ++j) {
              float v[16];
              tmem_ld16(th + j * 16, v);
              tmem_ld_wait();
              scale(v, j * 16);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float2 cs = rr[j * 8 + e];
                const float x0 = v[2 * e], x1 = v[2 * e + 1];
                v[2 * e] = x0 * cs.x - x1 * cs.y;
                v[2 * e + 1] = x0 * cs.y + x1 * cs.x;
              }
              if (store) put16(dst + j * 16, v);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&acc_empty[buf]);
        continue;
      }
      for (int j = 0; j < kWideN / 16; ++j) {
        float v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * kWideN + j * 16, v);
        tmem_ld_wait();
        const int n = n0 + j * 16;
        if (m < a.M && n < a.N) {
          uint4 pk[2];
          uint32_t* w32 = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
            w32[e] = *reinterpret_cast<uint32_t*>(&b2);
          }
          uint4* dst = reinterpret_cast<uint4*>(Y + (size_t)m * a.ldy + n);
          dst[0] = pk[0];
          dst[1] = pk[1];
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);
    }
    if (!ok) atomicOr(a.err, 32);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

}  // namespace

bool tc_encode_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                   uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t init_tc_attrs() {
  cudaError_t e;
  if ((e = attr_tc<16, kEpiStore>()) != cudaSuccess) return e;
  if ((e = attr_tc<16, kEpiResid>()) != cudaSuccess) return e;
  if ((e = attr_tc<16, kEpiSwiglu>()) != cudaSuccess) return e;
  if ((e = attr_tc<16, kEpiArgmax>()) != cudaSuccess) return e;
  if ((e = attr_tc<32, kEpiStore>()) != cudaSuccess) return e;
  if ((e = attr_tc<32, kEpiResid>()) != cudaSuccess) return e;
  if ((e = attr_tc<32, kEpiSwiglu>()) != cudaSuccess) return e;
  if ((e = attr_tc<16, kEpiKVRing>()) != cudaSuccess) return e;
  if ((e = attr_tc<32, kEpiKVRing>()) != cudaSuccess) return e;
  if ((e = attr_tc<16, kEpiRed>()) != cudaSuccess) return e;
  if ((e = attr_tc<32, kEpiRed>()) != cudaSuccess) return e;
  if ((e = attr_tc<16, kEpiRedPair>()) != cudaSuccess) return e;
  if ((e = attr_tc<32, kEpiRedPair>()) != cudaSuccess) return e;
  if ((e = attr_tc<64, kEpiRed>()) != cudaSuccess) return e;
  if ((e = attr_tc<64, kEpiRedPair>()) != cudaSuccess) return e;
  if ((e = attr_tc<64, kEpiArgmax>()) != cudaSuccess) return e;
  if ((e = attr_tc<128, kEpiRed>()) != cudaSuccess) return e;
  if ((e = attr_tc<128, kEpiRedPair>()) != cudaSuccess) return e;
  if ((e = attr_tc<128, kEpiArgmax>()) != cudaSuccess) return e;
  if ((e = attr_tc<160, kEpiRed>()) != cudaSuccess) return e;
  if ((e = attr_tc<160, kEpiRedPair>()) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(tc_gemm_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kWideSmem)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(tc_gemm_wide_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                (int)cudaSharedmemCarveoutMaxShared)) != cudaSuccess) return e;
  return attr_tc<32, kEpiArgmax>();
}

cudaError_t launch_tc_wide(const TcWideArgs& a, int grid, cudaStream_t st) {
  const int T = ((a.M + 127) / 128) * ((a.N + kWideN - 1) / kWideN);
  if (grid > T) grid = T;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kWideSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_gemm_wide_kernel, a);
}

cudaError_t launch_tc_gemm(const TcGemmArgs& a, int bn, int grid, bool pdl, cudaStream_t st) {
  // At least kMinUnits (64-wide K chunks of a 128-row tile, 16 KB of weights
  // each) per CTA: a short GEMM then splits a tile over a few CTAs rather than
  // a dozen.
  constexpr long long kMinUnits = 8;
  if (a.tiles > kTileDepart) return cudaErrorInvalidValue;     // split-tile counters
  const long long U = (long long)a.tiles * a.kchunks;
  const long long want = (U + kMinUnits - 1) / kMinUnits;
  if (grid > want) grid = static_cast<int>(want);
  if (grid < 1) grid = 1;
  if (U * grid >= (1ll << 32)) return cudaErrorInvalidValue;   // 32-bit unit arithmetic
  if (bn == 160) {
    if (a.epi == kEpiRed) return launch_tc<160, kEpiRed>(a, grid, pdl, st);
    if (a.epi == kEpiRedPair) return launch_tc<160, kEpiRedPair>(a, grid, pdl, st);
    return cudaErrorInvalidValue;
  }
  if (bn == 64 || bn == 128) {
    // more than 32 block rows: the fp32-sum and argmax epilogues, whole
    // lm_head tiles
    if (a.epi == kEpiArgmax && !a.whole_tiles) return cudaErrorInvalidValue;
    switch (a.epi) {
      case kEpiRed: return bn == 64 ? launch_tc<64, kEpiRed>(a, grid, pdl, st) : launch_tc<128, kEpiRed>(a, grid, pdl, st);
      case kEpiRedPair:
        return bn == 64 ? launch_tc<64, kEpiRedPair>(a, grid, pdl, st) : launch_tc<128, kEpiRedPair>(a, grid, pdl, st);
      case kEpiArgmax:
        return bn == 64 ? launch_tc<64, kEpiArgmax>(a, grid, pdl, st) : launch_tc<128, kEpiArgmax>(a, grid, pdl, st);
      default: return cudaErrorInvalidValue;
    }
  }
  if (bn == 16) {
    switch (a.epi) {
      case kEpiStore: return launch_tc<16, kEpiStore>(a, grid, pdl, st);
      case kEpiResid: return launch_tc<16, kEpiResid>(a, grid, pdl, st);
      case kEpiSwiglu: return launch_tc<16, kEpiSwiglu>(a, grid, pdl, st);
      case kEpiKVRing: return launch_tc<16, kEpiKVRing>(a, grid, pdl, st);
      case kEpiRed: return launch_tc<16, kEpiRed>(a, grid, pdl, st);
      case kEpiRedPair: return launch_tc<16, kEpiRedPair>(a, grid, pdl, st);
      default: return launch_tc<16, kEpiArgmax>(a, grid, pdl, st);
    }
  }
  switch (a.epi) {
    case kEpiStore: return launch_tc<32, kEpiStore>(a, grid, pdl, st);
    case kEpiResid: return launch_tc<32, kEpiResid>(a, grid, pdl, st);
    case kEpiSwiglu: return launch_tc<32, kEpiSwiglu>(a, grid, pdl, st);
    case kEpiKVRing: return launch_tc<32, kEpiKVRing>(a, grid, pdl, st);
    case kEpiRed: return launch_tc<32, kEpiRed>(a, grid, pdl, st);
    case kEpiRedPair: return launch_tc<32, kEpiRedPair>(a, grid, pdl, st);
    default: return launch_tc<32, kEpiArgmax>(a, grid, pdl, st);
  }
}

}  // namespace dfl
