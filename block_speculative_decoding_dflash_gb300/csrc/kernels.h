// Host-side launchers of the libdflash kernels (one translation unit per
// kernel family). Every launcher enqueues on `st` and returns the launch
// status; none allocates or synchronizes.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace dfl {

// ---- linear layers -------------------------------------------------------------
enum Epi : int {
  kEpiStore = 0,   // Y = rnd(X W^T)
  kEpiResid = 1,   // Y = rnd(R + rnd(X W^T)); R may alias Y
  kEpiSwiglu = 2,  // Y = rnd(silu(rnd(X Wg^T)) * rnd(X Wu^T))
};

// Up to three weight segments stacked along the output dimension: output
// columns [seg_end[s-1], seg_end[s]) come from w[s] (its row 0 is column
// seg_end[s-1]).
struct LinearArgs {
  const void* x; int ldx;           // [M, K]
  const void* w[3]; int seg_end[3]; // [N_s, K] each
  int nseg;
  const void* w2;                   // the up weight of kEpiSwiglu ([N, K])
  const void* r; int ldr;           // residual of kEpiResid
  void* y; int ldy;                 // [M, N]
  int M, N, K;
  int epi;
};
enum : int {
  kEpiArgmax = 3,   // tensor-core GEMM only: softcap + per-row argmax
  kEpiKVRing = 4,   // tensor-core GEMM only: K head-norm + RoPE / V, into ring slots
  kEpiRed = 5,      // tensor-core GEMM only: fp32 sums added into acc (zeroed), no finish;
                    // launch_resid_rmsnorm finishes them
  kEpiRedPair = 6,  // as kEpiRed for the two weights of a SwiGLU (gate sums at acc[m][n],
                    // up sums at acc[m][N + n]); launch_swiglu_finish finishes them
};
constexpr int kTcMaxSeg = 10;
constexpr int kTileDepart = 4096;  // tiles per GEMM at most; departures follow arrivals

// Tensor-core weight-streaming GEMM D[n, m] = sum_k W[n, k] X[m, k] (bf16,
// fp32 accumulate), M <= BN rows of X (BN 16 or 32). Weight rows are stacked
// segments of whole 128-row tiles (seg_tiles = cumulative tile counts); the
// last segment may end in a partial tile (rows past N are zero-filled).
struct TcGemmArgs {
  CUtensorMap a_map[kTcMaxSeg];    // weight segments, box {64, 128}
  CUtensorMap a2_map;              // up weight of kEpiSwiglu, box {64, 128}
  CUtensorMap b_map;               // X, box {64, BN}
  int b_row0;                      // first row of X this launch reads (TMA row coordinate)
  int seg_tiles[kTcMaxSeg];
  int nseg;
  int M, N, K, tiles, kchunks, epi;
  void* y; int ldy;                // output [M, N] (row stride ldy)
  const void* r; int ldr;          // residual of kEpiResid (may alias y)
  float* acc; int ldacc;           // kEpiRed: [M][ldacc] fp32, zero before the launch
  float* partials;                 // [grid][2][NV*BN][128] fp32 split-tile partials
  unsigned* tile_ctr;              // [kTileDepart + tiles]: arrivals, then departures per
                                   // split tile; zero between launches
  int* err;                        // bounded-wait timeouts are reported here
  float softcap;                   // kEpiArgmax
  int* ids; int* ids2; float* maxv;
  unsigned long long* best_key;     // kEpiArgmax: [M] packed (value, index) maxima, zero between launches
  int whole_tiles;                 // kEpiArgmax: whole tiles per CTA (no split-tile finish)
  unsigned* done_ctr;
  // kEpiKVRing: the weight rows are [K_0 | V_0 | K_1 | V_1 | ...], one
  // 128-row tile per kv head (head_dim 128); row m goes to position
  // ring->offset + m.
  void* ring_k; void* ring_v;      // [L][nkv][cap][128]
  long long cap;
  RingState* ring;
  const float2* rope;              // [M][64] (cos, sin)
  const void* const* kgain;        // [L] k_norm gains, device array of pointers
  int nkv, neox, append_only;
  float eps;
  KTrace trace;
};
// Many-row tensor-core GEMM (context ingest): Y[m, n] = rnd(X W^T), X [M, K]
// (box {64, 128}), W stacked segments of rows (box {64, 256}; segment row
// counts multiples of 256), bf16 out with row stride ldy.
struct TcWideArgs {
  CUtensorMap x_map;
  CUtensorMap w_map[kTcMaxSeg];
  int seg_rows[kTcMaxSeg];         // cumulative row ends of the segments
  int nseg;
  int M, N, K;
  void* y; int ldy;
  int* err;
  // K/V into the ring instead of y (ring_k != NULL): the columns are layers
  // l0, l0+1, ... of [K heads | V heads] (kvdim each, kvdim % 256 == 0,
  // head_dim 128); row m is position pos0 + m; K heads get the per-head
  // RMSNorm (kgain[layer]) and RoPE (rope[m][64]) before the ring store.
  void* ring_k; void* ring_v;      // [L][nkv][cap][128]
  long long cap, pos0;
  RingState* ring;
  const float2* rope;
  const void* const* kgain;
  int nkv, kvdim, l0, append_only, neox;
  float eps;
};
cudaError_t launch_tc_wide(const TcWideArgs& a, int grid, cudaStream_t st);

bool tc_encode_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                   uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows);
cudaError_t init_tc_attrs();
cudaError_t launch_tc_gemm(const TcGemmArgs& a, int bn, int grid, bool pdl, cudaStream_t st);

// Block rows (any M; 16 rows per weight pass): weight-streaming kernel.
cudaError_t launch_linear_rows(int dtype, const LinearArgs& a, cudaStream_t st);
// Many rows (context ingest), kEpiStore only: register-tiled GEMM.
cudaError_t launch_linear_tiled(int dtype, const LinearArgs& a, cudaStream_t st);

// ---- small per-row kernels -------------------------------------------------------
// x[r] = E[tok_r] with tok_0 = the anchor and tok_r = mask for r > 0; also
// the RoPE table rope[tab_rows][hd/2] = (cos, sin) at ring->offset + r. The
// anchor is anchor_host when >= 0 (also stored as the device anchor), else
// the device anchor; expect_pos >= 0 is compared with ring->offset (kErrPos).
cudaError_t launch_embed_block(int dtype, const void* embed, int H, int vocab,
                               RoundState* rs, int mask_id, int rows, void* x,
                               const RingState* ring, const double* inv_freq,
                               int half, int tab_rows, float2* rope, int anchor_host,
                               long long expect_pos, cudaStream_t st, int nseq = 1);
// RoPE table at positions base + r, base = ring->offset when ring != NULL,
// else pos0.
cudaError_t launch_rope_table(const double* inv_freq, int half, const RingState* ring,
                              long long pos0, int rows, float2* rope, cudaStream_t st, int nseq = 1);
cudaError_t launch_rmsnorm(int dtype, const void* x, int ldx, const void* g,
                           void* y, int ldy, int rows, int H, float eps,
                           cudaStream_t st, KTrace trace = KTrace{nullptr, 0});
// bf16: finishes a split-K GEMM that added its fp32 sums into acc [rows,
// ldacc] (kEpiRed): h = rnd(x + rnd(acc)) (rnd(acc) when x is NULL) written
// back into x (when not NULL), acc cleared, y = rnd(rmsnorm(h) * g). H % 8 ==
// 0, H <= 8192.
cudaError_t launch_resid_rmsnorm(void* x, int ldx, float* acc, int ldacc, const void* g, void* y,
                                 int ldy, int rows, int H, float eps, cudaStream_t st,
                                 KTrace trace = KTrace{nullptr, 0});
// bf16: finishes a kEpiRedPair gate/up GEMM: s[m][k] = rnd(silu(rnd(g)) *
// rnd(u)) with g = acc[m][k], u = acc[m][I + k] (row stride ldacc), acc
// cleared. I % 8 == 0, I <= 8192.
cudaError_t launch_swiglu_finish(float* acc, int ldacc, void* s, int lds, int rows, int I,
                                 cudaStream_t st, KTrace trace = KTrace{nullptr, 0});
// bf16, head_dim 128: finishes the append's K/V GEMM (kEpiRed over the
// [K_l | V_l] column blocks of L layers, acc row stride ldacc): rounds, k-norm
// (gain kgain[l]) + RoPE (rope[r][64]) for K, stores K and V of row r at
// position ring[s].offset + r % rows_per_seq of sequence s = r / rows_per_seq
// (its ring rows seq_kv elements after sequence s - 1's), clears the sums.
cudaError_t launch_kv_acc_to_ring(float* acc, int ldacc, int rows, int L, int nkv,
                                  const void* const* kgain, float eps, const float2* rope, int neox,
                                  void* ring_k, void* ring_v, long long cap, int append_only,
                                  RingState* ring, cudaStream_t st, KTrace trace, int rows_per_seq,
                                  long long seq_kv);
// bf16, head_dim 128: finishes a kEpiRed QKV GEMM (acc [rows][ldacc] fp32,
// nq q heads, nkv k heads, nkv v heads): out = the rounded values, q and k
// heads with the per-head RMSNorm (gains qn, kn) + RoPE (rope[r][64]); the
// sums cleared. Waits for the GEMM before it lets the next kernel launch.
cudaError_t launch_qkv_finish(float* acc, int ldacc, void* out, int ldo, int rows, int nq, int nkv,
                              const void* qn, const void* kn, float eps, const float2* rope, int neox,
                              cudaStream_t st, KTrace trace = KTrace{nullptr, 0});
// The synthetic target's verify forward: x[r] = embed[tokens[r]] (out-of-
// range ids read row 0, kErrRange in rs); the verify block [drafter anchor,
// d...] (kErrPos in trs unless the drafter's ring offset is the target's);
// K / V rows of the finished QKV output into ring slots at ring->offset + r;
// the trim of block - *n_dev rows on both ring states (kErrTrim in trs when
// longer than the rows appended since the last trim).
cudaError_t launch_embed_tokens(int dtype, const void* embed, int H, int vocab, const int* tokens, int rows,
                                void* x, RoundState* rs, cudaStream_t st);
cudaError_t launch_verify_tokens(const RoundState* drs, const RingState* dring, const int* d, int block,
                                 int* tokens, const RingState* tring, RoundState* trs, cudaStream_t st);
cudaError_t launch_kv_rows_to_ring(int dtype, const void* qkv, int ld, int kofs, int vofs, int rows, int nkv,
                                   int hd, void* ring_k, void* ring_v, long long cap, int append_only,
                                   RingState* ring, cudaStream_t st);
cudaError_t launch_target_trim(RingState* a, RingState* b, const int* n_dev, int block, RoundState* trs,
                               cudaStream_t st);
// In place per-head RMSNorm + RoPE on buf[rows, heads, hd] (row stride ld).
cudaError_t launch_head_norm_rope(int dtype, void* buf, int ld, int rows,
                                  int heads, int hd, const void* g, float eps,
                                  const float2* rope, int neox, cudaStream_t st);
// kv[rows, 2*nkv*hd] = K heads then V heads: K -> head norm + RoPE -> ring K,
// V -> ring V, at positions (use_dev ? ring->offset : pos_host) + r; row r
// belongs to sequence r / rows_per_seq (its ring state ring[s], its rows
// seq_kv elements on).
// append_only: refuse (and flag) positions at or past base + cap.
cudaError_t launch_kv_to_ring(int dtype, const void* kv, int ld, int rows,
                              int nkv, int hd, const void* kg, float eps,
                              const float2* rope, int neox, void* ring_k,
                              void* ring_v, long long cap, int append_only,
                              RingState* ring, int use_dev, long long pos_host,
                              cudaStream_t st, int rows_per_seq, long long seq_kv);

// ---- attention ---------------------------------------------------------------------
struct AttnArgs {
  const void* q; int ldq;      // [rows, nq, hd]
  const void* kb; const void* vb; int ldkv;  // block K/V [rows, nkv, hd]
  const void* ring_k; const void* ring_v;    // [nkv][cap][hd]
  long long cap;
  const RingState* ring;       // offset = position of block row 0
  int window;                  // <= 0: unbounded
  int causal;                  // 0: key visible iff |q - k| <= window (the drafter's bidirectional
                               // sliding mask); 1: iff 0 <= q - k and (window <= 0 or q - k <= window)
  int rows, nq, nkv, hd;
  int max_ctx;                 // most context keys any round can see
  float* partial;              // scratch [nkv][nsplit][rows*G][hd + 2]
  void* out; int ldo;          // [rows, nq, hd]
  int* err;                    // bounded-wait timeouts are reported here (bit 32)
  KTrace trace;                // attention kernel; the separate merge kernel uses slot + 1
                               // (its phase mark slot + 4), the attention's phase marks
                               // slots + 2 and + 3
  // Batch of nseq sequences (0 or 1: one): sequence s (blockIdx.z) has its
  // own ring state ring[s], ring rows seq_kv elements after sequence s - 1's,
  // its rows s * rows .. of q, kb, vb, out and the RoPE table, and its own
  // partials.
  int nseq;
  long long seq_kv;
  // The kernel before the attention waited for its own dependency before it
  // let the attention launch (launch_qkv_finish), so every kernel before that
  // one is complete: the ring's context rows (and the ring state) may be read
  // before the attention's own dependency resolves.
  int early_ctx;
  // The layer's gate and up weights (l2_next_bytes each, or null): every CTA
  // asks L2 for its share of them once its own operands have landed, since
  // HBM otherwise idles through the attention and its merge, and the gate/up
  // GEMM two kernels later then streams them from L2.
  const void* l2_next[2];
  long long l2_next_bytes;
};
// Points a's per-sequence operands at sequence s: q, kb, vb, the ring and out
// hold elements of esz bytes; partial rows are part_stride floats per query.
__device__ __forceinline__ void attn_select_seq(AttnArgs& a, int s, int nsplit, int esz, int part_stride) {
  if (s == 0) return;
  const int Qn = a.rows * (a.nq / a.nkv);
  a.ring += s;
  a.q = static_cast<const char*>(a.q) + (size_t)s * a.rows * a.ldq * esz;
  a.kb = static_cast<const char*>(a.kb) + (size_t)s * a.rows * a.ldkv * esz;
  a.vb = static_cast<const char*>(a.vb) + (size_t)s * a.rows * a.ldkv * esz;
  a.ring_k = static_cast<const char*>(a.ring_k) + (size_t)s * a.seq_kv * esz;
  a.ring_v = static_cast<const char*>(a.ring_v) + (size_t)s * a.seq_kv * esz;
  a.out = static_cast<char*>(a.out) + (size_t)s * a.rows * a.ldo * esz;
  a.partial += (size_t)s * a.nkv * nsplit * Qn * part_stride;
}
cudaError_t launch_attention(int dtype, const AttnArgs& a, cudaStream_t st);
// bf16, head_dim 128: tensor-core attention with the split merge fused in.
bool attention_mma_ok(int dtype, int hd);
size_t attention_mma_scratch_floats(int rows, int nq, int nkv, int max_ctx);
cudaError_t init_attention_mma_attrs();
cudaError_t launch_attention_mma(const AttnArgs& a, cudaStream_t st);
size_t attention_scratch_floats(int rows, int nq, int nkv, int hd, int max_ctx);
cudaError_t init_attention_attrs(int hd);

// ---- lm_head + softcap + argmax ------------------------------------------------------
struct LmHeadArgs {
  const void* x; int ldx;      // [R, H] normed rows to read out
  const void* w;               // [V, H]
  int R, H, V;
  float softcap;
  int* ids;                    // [R] argmax
  int* ids2;                   // optional second copy of ids (NULL)
  float* maxv;                 // [R] selected capped logit
  float* logits;               // optional [R, V] capped fp32 logits (NULL)
  float* part_v; int* part_i;  // scratch [grid * R]
  unsigned* counter;           // scratch, zero between launches
  int grid;
};
cudaError_t launch_lmhead_argmax(int dtype, const LmHeadArgs& a, cudaStream_t st);
int lmhead_grid(int V);
cudaError_t init_lmhead_attrs(int H);

// ---- verify / commit / Markov / stand-in target ---------------------------------------
struct VerifyArgs {
  const void* L;               // [B, V]
  int B, V;
  const int* d;                // [B-1]
  int* tokens;                 // [B]
  int* n;                      // [1]
  RoundState* rs;
  float* part_v; int* part_i;  // scratch [B * chunks]
  unsigned* counter;
  int chunks;
  int nseq;                    // batch (0 or 1: one): sequence s at L + s [B, V], d + s [B-1],
                               // tokens + s [B], n + s, rs + s, partials + s [B * chunks],
                               // counter + s
  KTrace trace;
};
cudaError_t launch_verify(int dtype, const VerifyArgs& a, cudaStream_t st);
// Batch read-out: ids [nseq][rows - read0] = ids_all[s * rows + read0 + i]
// (and a second copy ids2, and maxv from maxv_all, when not NULL).
cudaError_t launch_split_ids(const int* ids_all, const float* maxv_all, int rows, int read0, int nseq, int* ids,
                             int* ids2, float* maxv, cudaStream_t st);
int verify_chunks(int V);
// Text returned by dflash_last_error(NULL).
void set_global_error(const char* msg);

cudaError_t launch_commit(RoundState* rs, RingState* ring, int block, int keep,
                          cudaStream_t st, int nseq = 1);
// mode 0: append d rows; 1: trim d rows; 2: advance d committed rows.
cudaError_t launch_ring_advance(RingState* ring, int d, int mode, cudaStream_t st, int nseq = 1);
cudaError_t launch_ring_reset(RingState* ring, long long base, cudaStream_t st);
cudaError_t launch_set_anchor(RoundState* rs, int anchor, cudaStream_t st);
// Copies rows [L, n, nkv, hd] into ring slots at offset + r, then advances.
cudaError_t launch_ring_append(int dtype, const void* k, const void* v, int L,
                               int n, int nkv, int hd, void* ring_k, void* ring_v,
                               long long cap, RingState* ring, cudaStream_t st);
cudaError_t launch_ring_gather(int dtype, const void* ring_k, const void* ring_v,
                               int L, long long cap, int nkv, int hd,
                               long long pos0, int count, void* k_out,
                               void* v_out, cudaStream_t st);

// Speculative-sampling verify at temperature T > 0 (one CTA per row).
struct SampledVerifyArgs {
  const void* L;               // [B, V]
  int B, V;
  const int* d;                // [B-1]
  const float* u;              // [B] uniforms in [0, 1): B-1 accept tests, the bonus draw
  float temperature, softcap;
  int* tokens;                 // [B]
  int* n;                      // [1]
  RoundState* rs;              // may be NULL
  int* acc; int* cand;         // scratch [B]
  float* pd;                   // [B] p_i(d_{i+1}) (0 for the last row)
  unsigned* counter;           // zero between launches
};
cudaError_t launch_verify_sampled(int dtype, const SampledVerifyArgs& a, cudaStream_t st);
constexpr int kShortConvMaxL = 16;
cudaError_t launch_short_conv(int dtype, const void* state, const void* bx, const void* w, int layers,
                              int lc, int C, int block, void* y, void* state_after, cudaStream_t st);
cudaError_t launch_short_conv_rollback(int dtype, const void* prev, const void* bx, const int* n_dev,
                                       int layers, int lc, int C, int block, void* out, cudaStream_t st);

struct MarkovArgs {
  const void* w1; const void* w2;  // [V, r], [r, V]
  int V, r;
  const RoundState* rs;        // anchor source when anchor_host < 0
  int anchor_host;
  const float* z; int ldz;     // optional [gamma, V] fp32
  int gamma;
  int* out;                    // [gamma]
  int* out2;                   // optional second copy
  unsigned long long* key;     // scratch [gamma] packed per-step maxima, zero between launches
  unsigned* counter;
  int grid;
  KTrace trace;                // gamma slots: step j marks slot + j
  unsigned* bar;               // [2] zeroed: grid barrier count and generation (one-launch chain)
  int* err;                    // a barrier wait that gave up: bit 64
};
cudaError_t launch_markov_chain(int dtype, const MarkovArgs& a, cudaStream_t st);
// The whole chain in one cooperative launch of `grid` CTAs (one per SM), W2
// held in shared memory; cudaErrorNotSupported when W2 does not fit (the
// caller then launches the chain step by step).
cudaError_t launch_markov_chain_coop(int dtype, const MarkovArgs& a, int grid, cudaStream_t st);
// Whether the one-launch chain fits this GPU for vocab V and rank r.
bool markov_coop_ok(int dtype, int V, int r, int grid);
int markov_grid(int V);

struct SynthArgs {
  const void* logit_pool; const void* plant; const uint8_t* coins;
  const void* resid_pool;
  int n_logit, n_coin, n_resid, block_max, block, V, kin;
  const int* d;
  void* logits_out; void* resid_out;
  const RoundState* rs;
  int vec;                     // set by the launcher: rows allow 16-byte copies
  int nseq;                    // batch: sequence s uses rs[s], d + s (block-1), outputs + s block
                               // rows, and pool entry (round * nseq + s)
  KTrace trace;
};
cudaError_t launch_synth_target(int dtype, const SynthArgs& a, cudaStream_t st);

}  // namespace dfl
