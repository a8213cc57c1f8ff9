// libdflash host side: argument checks, the context and ring objects, the
// order of kernel launches that makes one DFlash round, and CUDA-graph
// capture of rounds. Nothing here throws across the C ABI and nothing in the
// round path allocates or synchronizes.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <limits>
#include <string>
#include <vector>

#include "../../include/dflash.h"
#include "kernels.h"

using namespace dfl;

namespace {

thread_local std::string g_create_err;

int fail(std::string& err, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  err = buf;
  return code;
}

int cuda_fail(std::string& err, cudaError_t e, const char* what) {
  return fail(err, DFLASH_ECUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

#define CK(err, call)                                             \
  do {                                                            \
    cudaError_t e_ = (call);                                      \
    if (e_ != cudaSuccess) return cuda_fail((err), e_, #call);    \
  } while (0)

int slack_rule(int block, bool floor) {
  int s = 8 * block;
  if (s < 32) s = 32;
  if (s > 128) s = 128;
  return (floor && s < block) ? block : s;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int64_t kI32Max = std::numeric_limits<int32_t>::max();
constexpr int kIngestChunk = 2048;
constexpr int kMaxBlock = 1024;
constexpr int kTcGrid = 256;      // upper bound of the tensor-core GEMM grid (SM count)
constexpr int kTcTiles = 8192;    // split-tile ticket counters

int check_config(const dflash_config* c, std::string& err) {
  if (!c) return fail(err, DFLASH_EINVAL, "config is NULL");
  if (c->n_layers < 1 || c->hidden < 1 || c->n_q_heads < 1 || c->n_kv_heads < 1 ||
      c->head_dim < 1 || c->intermediate < 1 || c->vocab < 2 || c->k_target_layers < 1 ||
      c->target_hidden < 1)
    return fail(err, DFLASH_EINVAL, "every dimension must be positive (vocab >= 2)");
  if (c->dtype != DFLASH_F32 && c->dtype != DFLASH_BF16)
    return fail(err, DFLASH_EINVAL, "dtype must be DFLASH_F32 or DFLASH_BF16");
  if (c->kind != DFLASH_KIND_DFLASH && c->kind != DFLASH_KIND_DSPARK)
    return fail(err, DFLASH_EINVAL, "kind must be DFLASH_KIND_DFLASH or DFLASH_KIND_DSPARK");
  if (c->rope_neox != 0 && c->rope_neox != 1) return fail(err, DFLASH_EINVAL, "rope_neox must be 0 or 1");
  if (c->n_q_heads % c->n_kv_heads) return fail(err, DFLASH_EINVAL, "n_q_heads %% n_kv_heads != 0");
  if (c->hidden % 8 || c->head_dim % 8 || c->intermediate % 8 ||
      ((int64_t)c->k_target_layers * c->target_hidden) % 8)
    return fail(err, DFLASH_EINVAL, "hidden, head_dim, intermediate and k*target_hidden must be multiples of 8");
  if (c->head_dim > 256) return fail(err, DFLASH_EINVAL, "head_dim must be at most 256");
  if (c->max_block < 2 || c->max_block > kMaxBlock)
    return fail(err, DFLASH_ERANGE, "max_block %d outside [2, %d]", c->max_block, kMaxBlock);
  if (c->mask_token_id < 0 || c->mask_token_id >= c->vocab)
    return fail(err, DFLASH_ERANGE, "mask_token_id %d outside [0, vocab=%d)", c->mask_token_id, c->vocab);
  if (c->markov_rank < 0 || c->markov_rank > 4096)
    return fail(err, DFLASH_EINVAL, "markov_rank %d outside [0, 4096]", c->markov_rank);
  if (c->markov_add != 0 && c->markov_add != 1) return fail(err, DFLASH_EINVAL, "markov_add must be 0 or 1");
  if (c->markov_rank > 0 && c->vocab % 8)
    return fail(err, DFLASH_EINVAL, "a Markov head needs vocab to be a multiple of 8");
  if (c->window <= 0 && c->max_context < 1)
    return fail(err, DFLASH_EINVAL, "an unbounded window needs max_context >= 1");
  if (!(c->rope_theta > 0.f) || !std::isfinite(c->rope_theta) || !(c->rms_eps >= 0.f) ||
      !std::isfinite(c->rms_eps) || !(c->softcap >= 0.f) || !std::isfinite(c->softcap))
    return fail(err, DFLASH_EINVAL, "rope_theta must be > 0, rms_eps and softcap >= 0, all finite");
  // Products the kernels index with 32-bit integers.
  const int64_t prods[] = {
      (int64_t)c->n_q_heads * c->head_dim,
      (int64_t)(c->n_q_heads + 2 * (int64_t)c->n_kv_heads) * c->head_dim,
      (int64_t)c->k_target_layers * c->target_hidden,
      (int64_t)c->window + slack_rule(c->max_block, true),
      (int64_t)c->max_block * c->vocab,
      (int64_t)c->max_block * c->n_q_heads * c->head_dim,
      (int64_t)c->max_block * ((int64_t)c->k_target_layers * c->target_hidden + c->vocab),
      (int64_t)c->n_kv_heads * ((int64_t)(c->window > 0 ? c->window : c->max_context) +
                                c->max_block) * (c->n_q_heads / c->n_kv_heads) * c->max_block,
  };
  for (int64_t p : prods)
    if (p > kI32Max) return fail(err, DFLASH_EINVAL, "a dimension product (%lld) would wrap an int32", (long long)p);
  return DFLASH_OK;
}

enum LayerW { kInNorm, kWq, kWk, kWv, kQNorm, kKNorm, kWo, kPostNorm, kWg, kWu, kWd };

}  // namespace

namespace dfl {
void set_global_error(const char* msg) { g_create_err = msg; }
}  // namespace dfl

// ---------------------------------------------------------------------------
// Objects
// ---------------------------------------------------------------------------
struct ring_cache {
  int L = 0, nkv = 0, hd = 0, window = 0, max_block = 0, dtype = 0, flags = 0;
  long long cap = 0;
  int append_only = 0;
  size_t esz = 4;
  void* k = nullptr;
  void* v = nullptr;
  RingState* st = nullptr;
  cudaStream_t stream = nullptr;
  bool owned_by_ctx = false;
  bool view = false;        // a batch sequence's view into its context's ring storage
  int nseq = 1;             // sequences whose rings this storage holds (a context's batch)
  int host_appended = 0;
  long long pos_hi = 0;     // upper bound of the device offset
  long long host_base = 0;
  std::string err;
};

struct dflash_ctx {
  dflash_config cfg{};
  const void* embed = nullptr;
  const void* fc = nullptr;
  const void* hidden_norm = nullptr;
  const void* final_norm = nullptr;
  const void* lm_head = nullptr;
  const void* w1 = nullptr;
  const void* w2 = nullptr;
  std::vector<const void*> layers;
  cudaStream_t stream = nullptr;
  ring_cache* ring = nullptr;
  int dt = 0;
  size_t esz = 4;
  int H = 0, nq = 0, nkv = 0, hd = 0, half = 0, I = 0, V = 0, kin = 0;
  int qdim = 0, kvdim = 0, qkv_n = 0, rows_max = 0, max_ctx = 0;

  char* arena = nullptr;
  size_t arena_bytes = 0;
  RoundState* rs = nullptr;
  double* inv_freq = nullptr;
  void *x = nullptr, *xn = nullptr, *qkv = nullptr, *attn = nullptr, *sbuf = nullptr, *xf = nullptr;
  float2* rope = nullptr;
  float* attn_part = nullptr;
  size_t attn_part_floats = 0;
  void *app_f = nullptr, *app_c = nullptr, *app_kv = nullptr;
  float2* app_rope = nullptr;
  void *ing_f = nullptr, *ing_c = nullptr, *ing_kv = nullptr;
  float2* ing_rope = nullptr;
  int ing_rows = 0;
  float* lm_pv = nullptr;
  int* lm_pi = nullptr;
  int lm_grid = 0;
  float* vf_pv = nullptr;
  int* vf_pi = nullptr;
  int vf_chunks = 0;
  float* mk_pv = nullptr;
  int* mk_pi = nullptr;
  int mk_grid = 0;
  unsigned* counters = nullptr;  // [0] lm_head, [1] verify, [2] markov, [4..5] markov grid barrier
  bool mk_coop = false;          // the Markov chain in one cooperative launch (W2 fits shared memory)
  bool mk_stepwise = false;      // DFLASH_OPT_MARKOV_STEPWISE
  int mk_coop_grid = 0;
  float* maxv = nullptr;
  int* backbone_ids = nullptr;
  float* zlog = nullptr;
  // batch: nseq sequences per round, each with its own ring (views[s]),
  // round state (rs[s]) and verify ticket; an ingest writes sequence seq_cur
  int nseq = 1;
  int seq_cur = 0;
  std::vector<ring_cache*> views;
  std::vector<char> seq_ctx;
  int* ids_all = nullptr;                      // [R] read-out ids of every block row (batch)
  float* maxv_all = nullptr;                   // [R]
  unsigned* vf_ctr = nullptr;                  // [nseq] verify tickets
  // the synthetic target (dflash_target_create): causal layers, the full
  // layers' append-only cache beside the sliding ring, residual capture
  bool is_target = false;
  ring_cache* ring_full = nullptr;
  std::vector<int> full_idx;                   // per layer: its index in ring_full, -1 if it slides
  std::vector<int> capture;                    // captured layers, in order
  void* cap_out = nullptr;                     // the forward being enqueued: its captured rows
  int* tok = nullptr;                          // [max_block] the verify block's tokens
  void* fc_unused = nullptr;                   // a zeroed stand-in for the drafter-only encoder.fc
  float* acc = nullptr;                        // [R][H] fp32 sums of the kEpiRed GEMMs, zero between uses
  float* qkv_acc = nullptr;                    // [R][qkv_n] fp32 sums of the QKV GEMM, zero between uses
  float* gu_acc = nullptr;                     // [R][2 I] fp32 gate / up sums, zero between uses
  float* kv_acc = nullptr;                     // [R][L 2 kvdim] fp32 sums of the append's K/V GEMM
  int* samp_acc = nullptr;                     // sampled verify: per-row accept, bonus candidate,
  int* samp_cand = nullptr;                    // p(d), ticket
  float* samp_pd = nullptr;
  unsigned* samp_ctr = nullptr;

  bool has_context = false;
  int last_draft_block = 0;
  int last_verify_block = 0;
  int32_t* last_tokens = nullptr;              // the last verify's outputs (dflash_sync_round)
  int32_t* last_n = nullptr;
  int last_tokens_block = 0;
  int appended_block = 0;
  bool capturing = false;
  int saved_flags[4] = {0, 0, 0, 0};
  cudaGraphExec_t graphs[64] = {};
  long long graph_kernels[64] = {};
  // tensor-core path (bf16 with 128-aligned output dims)
  bool use_tc = false;
  int num_sms = 148;
  int R = 0;                                  // rows of every activation buffer
  struct LayerMaps { CUtensorMap wq, wk, wv, wo, wg, wu, wd; };
  std::vector<LayerMaps> lmaps;
  CUtensorMap fc_map{}, lm_map{};
  struct WideMaps { CUtensorMap wk, wv; };
  std::vector<WideMaps> lmaps_wide;          // box {64, 256} for the ingest GEMM
  CUtensorMap fcw_map{};
  CUtensorMap xn_map[2]{}, attn_map[2]{}, sbuf_map[2]{}, appc_map[2]{}, xf_map[2][2]{};
  float* tc_part = nullptr;
  unsigned* tc_tiles = nullptr;
  int* tc_err = nullptr;
  unsigned long long* tc_best = nullptr;       // lm_head: packed per-row argmax keys
  int* tc_lm_pi = nullptr;
  unsigned* tc_done = nullptr;
  const void** kgain_dev = nullptr;            // [n_layers] k_norm gain pointers
  cudaEvent_t lm_ev[2] = {nullptr, nullptr};
  bool lm_timing = false;
  bool lm_recorded = false;
  unsigned long long* ktr = nullptr;           // DFLASH_OPT_KERNEL_TRACE: [3][kKTraceSlots]
  bool ktr_on = false;
  int ktr_n = 0;
  std::vector<std::string> ktr_names;
  cudaEvent_t ing_ev[4] = {nullptr, nullptr, nullptr, nullptr};   // fc GEMM, K/V GEMM brackets
  bool ing_timing = false;
  bool ing_recorded = false;
  std::string err;
};

namespace {

template <typename P>
P* carve(char*& cur, size_t bytes) {
  char* p = cur;
  cur += (bytes + 255) & ~size_t(255);
  return reinterpret_cast<P*>(p);
}

int ring_create_impl(int L, int nkv, int hd, int window, int max_block, int dtype,
                     int max_context, int flags, cudaStream_t st, ring_cache** out,
                     std::string& err, int nseq = 1) {
  if (!out) return fail(err, DFLASH_EINVAL, "out is NULL");
  *out = nullptr;
  if (L < 1 || nkv < 1 || hd < 1) return fail(err, DFLASH_EINVAL, "ring dimensions must be positive");
  if (dtype != DFLASH_F32 && dtype != DFLASH_BF16) return fail(err, DFLASH_EINVAL, "bad dtype");
  if (max_block < 1 || max_block > kMaxBlock)
    return fail(err, DFLASH_ERANGE, "max_block %d outside [1, %d]", max_block, kMaxBlock);
  if (window <= 0 && max_context < 1)
    return fail(err, DFLASH_EINVAL, "an append-only ring needs max_context >= 1");
  ring_cache* r = new (std::nothrow) ring_cache();
  if (!r) return fail(err, DFLASH_ECUDA, "out of host memory");
  r->L = L; r->nkv = nkv; r->hd = hd; r->window = window; r->max_block = max_block;
  r->dtype = dtype; r->flags = flags; r->stream = st;
  r->append_only = window <= 0;
  r->cap = window > 0 ? (long long)window + slack_rule(max_block, !(flags & DFLASH_RING_UNFLOORED))
                      : (long long)max_context;
  r->esz = dtype == DFLASH_BF16 ? 2 : 4;
  r->nseq = nseq;
  const size_t bytes = (size_t)nseq * L * nkv * (size_t)r->cap * hd * r->esz;
  cudaError_t e;
  if ((e = cudaMalloc(&r->k, bytes)) != cudaSuccess ||
      (e = cudaMalloc(&r->v, bytes)) != cudaSuccess ||
      (e = cudaMalloc(&r->st, sizeof(RingState) * nseq)) != cudaSuccess ||
      (e = cudaMemsetAsync(r->k, 0, bytes, st)) != cudaSuccess ||
      (e = cudaMemsetAsync(r->v, 0, bytes, st)) != cudaSuccess) {
    cudaFree(r->k); cudaFree(r->v); cudaFree(r->st);
    delete r;
    return cuda_fail(err, e, "ring allocation");
  }
  for (int q = 0; q < nseq && e == cudaSuccess; ++q) e = launch_ring_reset(r->st + q, 0, st);
  if (e != cudaSuccess || (e = cudaStreamSynchronize(st)) != cudaSuccess) {
    cudaFree(r->k); cudaFree(r->v); cudaFree(r->st);
    delete r;
    return cuda_fail(err, e, "ring allocation");
  }
  *out = r;
  return DFLASH_OK;
}

void ring_free(ring_cache* r) {
  if (!r) return;
  if (r->view) { delete r; return; }
  cudaFree(r->k);
  cudaFree(r->v);
  cudaFree(r->st);
  delete r;
}

// Exact device offset (syncs); used only when an append-only bound is close.
int ring_sync_offset(ring_cache* r, long long* off) {
  RingState s;
  CK(r->err, cudaStreamSynchronize(r->stream));
  CK(r->err, cudaMemcpy(&s, r->st, sizeof s, cudaMemcpyDeviceToHost));
  *off = s.offset;
  return DFLASH_OK;
}

LinearArgs lin_args(const void* x, int ldx, void* y, int ldy, int M, int N, int K) {
  LinearArgs a{};
  a.x = x; a.ldx = ldx; a.y = y; a.ldy = ldy; a.M = M; a.N = N; a.K = K;
  a.nseg = 1; a.seg_end[0] = N; a.epi = kEpiStore;
  return a;
}

const void* LW(const dflash_ctx* c, int l, int which) {
  return c->layers[(size_t)l * DFLASH_LAYER_TENSORS + which];
}

// Ring elements of one sequence (all layers) and sequence s's K / V base.
size_t seq_kv_elems(const dflash_ctx* c) { return (size_t)c->cfg.n_layers * c->nkv * c->ring->cap * c->hd; }
char* ring_k_of(const dflash_ctx* c, int s) { return static_cast<char*>(c->ring->k) + s * seq_kv_elems(c) * c->esz; }
char* ring_v_of(const dflash_ctx* c, int s) { return static_cast<char*>(c->ring->v) + s * seq_kv_elems(c) * c->esz; }

int bn_index(int M) { return M <= 16 ? 0 : 1; }
int bn_of(int M) { return M <= 16 ? 16 : 32; }

TcGemmArgs tc_args(dflash_ctx* c, int M, int N, int K, int epi) {
  TcGemmArgs a{};
  a.M = M; a.N = N; a.K = K; a.epi = epi;
  a.tiles = (N + 127) / 128;
  a.kchunks = K / 64;
  a.partials = c->tc_part;
  a.tile_ctr = c->tc_tiles;
  a.err = c->tc_err;
  return a;
}

// Next slot(s) of the per-launch kernel trace, or none when tracing is off.
KTrace ktrace_slot(dflash_ctx* c, const std::string& name, int nslots = 1) {
  if (!c->ktr_on || !c->ktr || c->ktr_n + nslots > kKTraceSlots) return KTrace{nullptr, 0};
  const KTrace t{c->ktr, c->ktr_n};
  for (int i = 0; i < nslots; ++i) c->ktr_names.push_back(i ? name + "." + std::to_string(i) : name);
  c->ktr_n += nslots;
  return t;
}

void tc_segments(TcGemmArgs& a, std::initializer_list<std::pair<const CUtensorMap*, int>> segs) {
  int i = 0, tiles = 0;
  for (auto& sg : segs) {
    a.a_map[i] = *sg.first;
    tiles += (sg.second + 127) / 128;
    a.seg_tiles[i] = tiles;
    ++i;
  }
  a.nseg = i;
}

// More than 32 rows (wide verify blocks, batches): the finish-free GEMMs
// (kEpiRed, kEpiRedPair) run once per group of up to 160 rows and the lm_head
// argmax once per group of up to 128 (64, 128 or 160 block rows a launch),
// each launch streaming the weights again; b_map must then have been encoded
// with 32-row boxes (bn_of of the whole row count), which a last group of 32
// rows or fewer also uses.
cudaError_t tc_run(dflash_ctx* c, const TcGemmArgs& a) {
  if (a.M <= 32) return launch_tc_gemm(a, bn_of(a.M), c->num_sms, true, c->stream);
  if (a.epi != kEpiRed && a.epi != kEpiRedPair && a.epi != kEpiArgmax) return cudaErrorInvalidValue;
  // (fp32 sums: up to 160 rows in one launch)
  const int group = a.epi == kEpiArgmax ? 128 : 160;
  for (int r0 = 0; r0 < a.M; r0 += group) {
    TcGemmArgs g = a;
    g.M = a.M - r0 < group ? a.M - r0 : group;
    g.b_row0 = a.b_row0 + r0;
    if (g.acc) g.acc += (size_t)r0 * a.ldacc;
    if (g.ids) g.ids += r0;
    if (g.ids2) g.ids2 += r0;
    if (g.maxv) g.maxv += r0;
    if (a.epi == kEpiArgmax) g.whole_tiles = g.M > 8;
    const int bn = g.M <= 32 ? 32 : g.M <= 64 ? 64 : g.M <= 128 ? 128 : 160;
    const cudaError_t e = launch_tc_gemm(g, bn, c->num_sms, true, c->stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// The tensor-core path for `rows` block rows: up to 32 rows every GEMM of
// the round; more in groups of up to 160 (128 for the argmax), which needs
// the finish-free QKV of the head_dim-128 attention.
bool tc_rows(const dflash_ctx* c, int rows) {
  return c->use_tc && (rows <= 32 || attention_mma_ok(c->dt, c->hd));
}

// Context rows -> ring: fc -> hidden_norm -> per layer [Wk | Wv] -> k-norm +
// RoPE / copy into ring slots. use_dev: positions from the device offset
// (block append), else pos_host (ingest).
int context_rows_to_ring(dflash_ctx* c, const void* resid, int rows, void* f, void* cn, void* kv,
                         float2* rope, int use_dev, long long pos_host) {
  const int dt = c->dt;
  cudaStream_t st = c->stream;
  // an append (use_dev) writes every sequence of the batch, rows / nseq rows
  // each; an ingest writes sequence seq_cur
  const int ns = use_dev ? c->nseq : 1;
  const int rps = rows / ns;
  const int sq = use_dev ? 0 : c->seq_cur;
  RingState* rst = c->ring->st + sq;
  CK(c->err, launch_rope_table(c->inv_freq, c->half, use_dev ? rst : nullptr, pos_host, rps, rope, st, ns));
  const bool tc = tc_rows(c, rows) && cn == c->app_c;
  if (tc) {
    // encoder.fc adds its fp32 sums into c->acc; hidden_norm rounds them
    // (f = rnd(acc)) and normalises
    TcGemmArgs t = tc_args(c, rows, c->H, c->kin, kEpiRed);
    tc_segments(t, {{&c->fc_map, c->H}});
    if (!tc_encode_map(&t.b_map, resid, c->kin, rows, (uint64_t)c->kin * 2, 64, bn_of(rows)))
      return fail(c->err, DFLASH_ECUDA, "cuTensorMapEncodeTiled failed for the residual rows");
    t.acc = c->acc; t.ldacc = c->H;
    if (use_dev) t.trace = ktrace_slot(c, "append.fc", 4);
    CK(c->err, tc_run(c, t));
    CK(c->err, launch_resid_rmsnorm(nullptr, 0, c->acc, c->H, c->hidden_norm, cn, c->H, rows, c->H,
                                    c->cfg.rms_eps, st,
                                    use_dev ? ktrace_slot(c, "append.hidden_norm") : KTrace{nullptr, 0}));
  } else {
    LinearArgs a = lin_args(resid, c->kin, f, c->H, rows, c->H, c->kin);
    a.w[0] = c->fc;
    CK(c->err, rows > 32 ? launch_linear_tiled(dt, a, st) : launch_linear_rows(dt, a, st));
    CK(c->err, launch_rmsnorm(dt, f, c->H, c->hidden_norm, cn, c->H, rows, c->H, c->cfg.rms_eps, st,
                              use_dev ? ktrace_slot(c, "append.hidden_norm") : KTrace{nullptr, 0}));
  }
  if (tc && c->hd == 128) {
    // One GEMM per group of up to five layers over [Wk_l | Wv_l ...] adds its
    // fp32 sums into c->kv_acc; one finishing kernel then norms, rotates and
    // writes K and V of every layer into the ring.
    const int L = c->cfg.n_layers;
    for (int l0 = 0; l0 < L; l0 += kTcMaxSeg / 2) {
      const int nl = L - l0 < kTcMaxSeg / 2 ? L - l0 : kTcMaxSeg / 2;
      TcGemmArgs t = tc_args(c, rows, nl * 2 * c->kvdim, c->H, kEpiRed);
      t.acc = c->kv_acc + (size_t)l0 * 2 * c->kvdim;
      t.ldacc = L * 2 * c->kvdim;
      t.nseg = 2 * nl;
      int tiles = 0;
      for (int j = 0; j < nl; ++j) {
        t.a_map[2 * j] = c->lmaps[l0 + j].wk;
        t.a_map[2 * j + 1] = c->lmaps[l0 + j].wv;
        tiles += c->kvdim / 128;
        t.seg_tiles[2 * j] = tiles;
        tiles += c->kvdim / 128;
        t.seg_tiles[2 * j + 1] = tiles;
      }
      t.b_map = c->appc_map[bn_index(rows)];
      const size_t lay = (size_t)l0 * c->nkv * c->ring->cap * c->hd * c->esz;
      t.ring_k = static_cast<char*>(c->ring->k) + lay;
      t.ring_v = static_cast<char*>(c->ring->v) + lay;
      t.cap = c->ring->cap;
      t.ring = c->ring->st;
      t.rope = rope;
      t.kgain = c->kgain_dev + l0;
      t.nkv = c->nkv;
      t.neox = c->cfg.rope_neox;
      t.append_only = c->ring->append_only;
      t.eps = c->cfg.rms_eps;
      if (use_dev) t.trace = ktrace_slot(c, "append.kv", 4);
      CK(c->err, tc_run(c, t));
    }
    CK(c->err, launch_kv_acc_to_ring(c->kv_acc, L * 2 * c->kvdim, rows, L, c->nkv, c->kgain_dev,
                                     c->cfg.rms_eps, rope, c->cfg.rope_neox, ring_k_of(c, sq), ring_v_of(c, sq),
                                     c->ring->cap, c->ring->append_only, rst, st,
                                     use_dev ? ktrace_slot(c, "append.kv_ring") : KTrace{nullptr, 0}, rps,
                                     (long long)seq_kv_elems(c)));
    return DFLASH_OK;
  }
  for (int l = 0; l < c->cfg.n_layers; ++l) {
    if (tc) {
      TcGemmArgs t = tc_args(c, rows, 2 * c->kvdim, c->H, kEpiStore);
      tc_segments(t, {{&c->lmaps[l].wk, c->kvdim}, {&c->lmaps[l].wv, c->kvdim}});
      t.b_map = c->appc_map[bn_index(rows)];
      t.y = kv; t.ldy = 2 * c->kvdim;
      CK(c->err, tc_run(c, t));
    } else {
      LinearArgs b = lin_args(cn, c->H, kv, 2 * c->kvdim, rows, 2 * c->kvdim, c->H);
      b.nseg = 2;
      b.w[0] = LW(c, l, kWk); b.seg_end[0] = c->kvdim;
      b.w[1] = LW(c, l, kWv); b.seg_end[1] = 2 * c->kvdim;
      CK(c->err, rows > 32 ? launch_linear_tiled(dt, b, st) : launch_linear_rows(dt, b, st));
    }
    const size_t lay = (size_t)l * c->nkv * c->ring->cap * c->hd * c->esz;
    CK(c->err, launch_kv_to_ring(dt, kv, 2 * c->kvdim, rows, c->nkv, c->hd, LW(c, l, kKNorm),
                                 c->cfg.rms_eps, rope, c->cfg.rope_neox, ring_k_of(c, sq) + lay,
                                 ring_v_of(c, sq) + lay, c->ring->cap, c->ring->append_only, rst, use_dev,
                                 pos_host, st, rps, (long long)seq_kv_elems(c)));
  }
  return DFLASH_OK;
}

// Context rows on the tensor cores (many rows): fc -> hidden_norm -> all
// layers' [Wk | Wv] in launches of up to five layers -> ring writes.
int context_rows_wide(dflash_ctx* c, const void* resid, int rows, void* f, void* cn, void* kv,
                      float2* rope, long long pos_host) {
  const int dt = c->dt;
  cudaStream_t st = c->stream;
  CK(c->err, launch_rope_table(c->inv_freq, c->half, nullptr, pos_host, rows, rope, st));
  TcWideArgs a{};
  a.M = rows; a.K = c->kin; a.N = c->H; a.nseg = 1; a.seg_rows[0] = c->H;
  a.w_map[0] = c->fcw_map;
  a.y = f; a.ldy = c->H; a.err = c->tc_err;
  if (!tc_encode_map(&a.x_map, resid, c->kin, rows, (uint64_t)c->kin * 2, 64, 128))
    return fail(c->err, DFLASH_ECUDA, "cuTensorMapEncodeTiled failed for the context rows");
  const unsigned evf = c->capturing ? cudaEventRecordExternal : 0;
  if (c->ing_timing) CK(c->err, cudaEventRecordWithFlags(c->ing_ev[0], st, evf));
  CK(c->err, launch_tc_wide(a, c->num_sms, st));
  if (c->ing_timing) CK(c->err, cudaEventRecordWithFlags(c->ing_ev[1], st, evf));
  CK(c->err, launch_rmsnorm(dt, f, c->H, c->hidden_norm, cn, c->H, rows, c->H, c->cfg.rms_eps, st));
  if (c->ing_timing) CK(c->err, cudaEventRecordWithFlags(c->ing_ev[2], st, evf));
  const int L = c->cfg.n_layers;
  const int ldkv = L * 2 * c->kvdim;
  // head_dim 128 with whole 256-column tiles per K or V: the wide GEMM's
  // epilogue does the k-norm + RoPE and the ring stores itself.
  const bool to_ring = c->hd == 128 && c->kvdim % 256 == 0;
  for (int l0 = 0; l0 < L; l0 += kTcMaxSeg / 2) {
    const int nl = L - l0 < kTcMaxSeg / 2 ? L - l0 : kTcMaxSeg / 2;
    TcWideArgs b{};
    b.M = rows; b.K = c->H; b.N = nl * 2 * c->kvdim; b.nseg = 2 * nl;
    for (int j = 0; j < nl; ++j) {
      b.w_map[2 * j] = c->lmaps_wide[l0 + j].wk;
      b.w_map[2 * j + 1] = c->lmaps_wide[l0 + j].wv;
      b.seg_rows[2 * j] = (2 * j + 1) * c->kvdim;
      b.seg_rows[2 * j + 1] = (2 * j + 2) * c->kvdim;
    }
    b.y = static_cast<char*>(kv) + (size_t)l0 * 2 * c->kvdim * c->esz;
    b.ldy = ldkv;
    b.err = c->tc_err;
    if (to_ring) {
      b.ring_k = ring_k_of(c, c->seq_cur); b.ring_v = ring_v_of(c, c->seq_cur); b.cap = c->ring->cap;
      b.pos0 = pos_host; b.ring = c->ring->st + c->seq_cur; b.rope = rope; b.kgain = c->kgain_dev;
      b.nkv = c->nkv; b.kvdim = c->kvdim; b.l0 = l0; b.append_only = c->ring->append_only;
      b.neox = c->cfg.rope_neox; b.eps = c->cfg.rms_eps;
    }
    if (!tc_encode_map(&b.x_map, cn, c->H, rows, (uint64_t)c->H * 2, 64, 128))
      return fail(c->err, DFLASH_ECUDA, "cuTensorMapEncodeTiled failed for the normed context rows");
    CK(c->err, launch_tc_wide(b, c->num_sms, st));
  }
  if (c->ing_timing) {
    CK(c->err, cudaEventRecordWithFlags(c->ing_ev[3], st, evf));
    c->ing_recorded = true;
  }
  for (int l = 0; l < L && !to_ring; ++l) {
    const size_t lay = (size_t)l * c->nkv * c->ring->cap * c->hd * c->esz;
    CK(c->err, launch_kv_to_ring(dt, static_cast<char*>(kv) + (size_t)l * 2 * c->kvdim * c->esz, ldkv,
                                 rows, c->nkv, c->hd, LW(c, l, kKNorm), c->cfg.rms_eps, rope,
                                 c->cfg.rope_neox, ring_k_of(c, c->seq_cur) + lay,
                                 ring_v_of(c, c->seq_cur) + lay, c->ring->cap, c->ring->append_only,
                                 c->ring->st + c->seq_cur, 0, pos_host, st, rows, 0));
  }
  return DFLASH_OK;
}

// A target forward's residual capture: the stream after `layer` (now in
// c->x) into every capture slot that names it.
int capture_stream(dflash_ctx* c, int layer, int rows) {
  if (!c->is_target || !c->cap_out) return DFLASH_OK;
  const size_t row = (size_t)c->H * c->esz, pitch = c->capture.size() * row;
  for (size_t j = 0; j < c->capture.size(); ++j)
    if (c->capture[j] == layer)
      CK(c->err, cudaMemcpy2DAsync(static_cast<char*>(c->cap_out) + j * row, pitch, c->x, row, row, rows,
                                   cudaMemcpyDeviceToDevice, c->stream));
  return DFLASH_OK;
}

int layer_forward(dflash_ctx* c, int l, int rows) {
  const int dt = c->dt;
  cudaStream_t st = c->stream;
  const float eps = c->cfg.rms_eps;
  const std::string ln = "L" + std::to_string(l) + ".";
  const bool tc = tc_rows(c, rows);
  // The residual GEMMs (O, down) of the tensor-core path add their fp32 sums
  // into c->acc and leave the residual add to the RMSNorm that follows them:
  // x = rnd(x + rnd(acc)), then the norm of x.
  if (tc && l > 0) {
    CK(c->err, launch_resid_rmsnorm(c->x, c->H, c->acc, c->H, LW(c, l, kInNorm), c->xn, c->H, rows, c->H,
                                    eps, st, ktrace_slot(c, ln + "in_norm")));
    int rc = capture_stream(c, l - 1, rows);   // x now holds layer l - 1's output
    if (rc) return rc;
  } else
    CK(c->err, launch_rmsnorm(dt, c->x, c->H, LW(c, l, kInNorm), c->xn, c->H, rows, c->H, eps, st,
                              ktrace_slot(c, ln + "in_norm")));
  const int bi = bn_index(rows);
  // With the tensor-core attention the QKV GEMM adds its fp32 sums into
  // c->qkv_acc and one finishing kernel rounds them and applies the q/k head
  // norm + RoPE (before it lets the attention launch: see launch_qkv_finish);
  // otherwise the GEMM stores and two head-norm kernels follow.
  const bool qkv_red = tc && attention_mma_ok(dt, c->hd);
  if (tc) {
    TcGemmArgs t = tc_args(c, rows, c->qkv_n, c->H, qkv_red ? kEpiRed : kEpiStore);
    tc_segments(t, {{&c->lmaps[l].wq, c->qdim}, {&c->lmaps[l].wk, c->kvdim}, {&c->lmaps[l].wv, c->kvdim}});
    t.b_map = c->xn_map[bi];
    t.y = c->qkv; t.ldy = c->qkv_n;
    t.acc = c->qkv_acc; t.ldacc = c->qkv_n;
    t.trace = ktrace_slot(c, ln + "qkv", 4);
    CK(c->err, tc_run(c, t));
  } else {
    LinearArgs q = lin_args(c->xn, c->H, c->qkv, c->qkv_n, rows, c->qkv_n, c->H);
    q.nseg = 3;
    q.w[0] = LW(c, l, kWq); q.seg_end[0] = c->qdim;
    q.w[1] = LW(c, l, kWk); q.seg_end[1] = c->qdim + c->kvdim;
    q.w[2] = LW(c, l, kWv); q.seg_end[2] = c->qkv_n;
    CK(c->err, launch_linear_rows(dt, q, st));
  }
  if (qkv_red) {
    CK(c->err, launch_qkv_finish(c->qkv_acc, c->qkv_n, c->qkv, c->qkv_n, rows, c->nq, c->nkv, LW(c, l, kQNorm),
                                 LW(c, l, kKNorm), eps, c->rope, c->cfg.rope_neox, st,
                                 ktrace_slot(c, ln + "qkv_finish")));
  } else {
    CK(c->err, launch_head_norm_rope(dt, c->qkv, c->qkv_n, rows, c->nq, c->hd, LW(c, l, kQNorm), eps,
                                     c->rope, c->cfg.rope_neox, st));
    CK(c->err, launch_head_norm_rope(dt, static_cast<char*>(c->qkv) + (size_t)c->qdim * c->esz,
                                     c->qkv_n, rows, c->nkv, c->hd, LW(c, l, kKNorm), eps, c->rope,
                                     c->cfg.rope_neox, st));
  }
  AttnArgs at{};
  at.q = c->qkv; at.ldq = c->qkv_n;
  at.kb = static_cast<char*>(c->qkv) + (size_t)c->qdim * c->esz;
  at.vb = static_cast<char*>(c->qkv) + (size_t)(c->qdim + c->kvdim) * c->esz;
  at.ldkv = c->qkv_n;
  // a target's full layer attends over its append-only cache, causally
  const bool full = c->is_target && c->full_idx[l] >= 0;
  ring_cache* rg = full ? c->ring_full : c->ring;
  const size_t lay = (size_t)(full ? c->full_idx[l] : l) * c->nkv * rg->cap * c->hd * c->esz;
  at.ring_k = static_cast<char*>(rg->k) + lay;
  at.ring_v = static_cast<char*>(rg->v) + lay;
  at.cap = rg->cap;
  at.ring = rg->st;
  at.window = full ? 0 : c->cfg.window;
  at.causal = c->is_target ? 1 : 0;
  at.rows = rows / c->nseq; at.nq = c->nq; at.nkv = c->nkv; at.hd = c->hd;
  at.nseq = c->nseq; at.seq_kv = (long long)seq_kv_elems(c);
  at.max_ctx = full ? static_cast<int>(rg->cap) : c->cfg.window > 0 ? c->cfg.window : c->max_ctx;
  at.partial = c->attn_part;
  at.out = c->attn; at.ldo = c->qdim;
  at.err = c->tc_err;
  at.trace = ktrace_slot(c, ln + "attn", 5);
  at.early_ctx = qkv_red ? 1 : 0;                // launch_qkv_finish precedes it
  if (tc && !c->is_target) {
    // (measured at the Muse shape: rounds 2.2% faster at width 4, 1.5% at 16)
    at.l2_next[0] = LW(c, l, kWg);
    at.l2_next[1] = LW(c, l, kWu);
    at.l2_next_bytes = (long long)c->I * c->H * c->esz;
  }
  CK(c->err, launch_attention(dt, at, st));
  // a target's block rows join its cache (positions offset .., advanced once
  // the whole forward is enqueued)
  if (c->is_target)
    CK(c->err, launch_kv_rows_to_ring(dt, c->qkv, c->qkv_n, c->qdim, c->qdim + c->kvdim, rows, c->nkv, c->hd,
                                      static_cast<char*>(rg->k) + lay, static_cast<char*>(rg->v) + lay, rg->cap,
                                      rg->append_only, rg->st, st));
  if (tc) {
    TcGemmArgs t = tc_args(c, rows, c->H, c->qdim, kEpiRed);
    tc_segments(t, {{&c->lmaps[l].wo, c->H}});
    t.b_map = c->attn_map[bi];
    t.acc = c->acc; t.ldacc = c->H;
    t.trace = ktrace_slot(c, ln + "o", 4);
    CK(c->err, tc_run(c, t));
    CK(c->err, launch_resid_rmsnorm(c->x, c->H, c->acc, c->H, LW(c, l, kPostNorm), c->xn, c->H, rows, c->H,
                                    eps, st, ktrace_slot(c, ln + "post_norm")));
  } else {
    LinearArgs o = lin_args(c->attn, c->qdim, c->x, c->H, rows, c->H, c->qdim);
    o.w[0] = LW(c, l, kWo); o.epi = kEpiResid; o.r = c->x; o.ldr = c->H;
    CK(c->err, launch_linear_rows(dt, o, st));
    CK(c->err, launch_rmsnorm(dt, c->x, c->H, LW(c, l, kPostNorm), c->xn, c->H, rows, c->H, eps, st,
                              ktrace_slot(c, ln + "post_norm")));
  }
  if (tc) {
    // gate and up add their fp32 sums into c->gu_acc; the SwiGLU finish
    // rounds them and writes the down GEMM's operand
    TcGemmArgs t = tc_args(c, rows, c->I, c->H, kEpiRedPair);
    tc_segments(t, {{&c->lmaps[l].wg, c->I}});
    t.a2_map = c->lmaps[l].wu;
    t.b_map = c->xn_map[bi];
    t.acc = c->gu_acc; t.ldacc = 2 * c->I;
    t.trace = ktrace_slot(c, ln + "gate_up", 4);
    CK(c->err, tc_run(c, t));
    CK(c->err, launch_swiglu_finish(c->gu_acc, 2 * c->I, c->sbuf, c->I, rows, c->I, st,
                                    ktrace_slot(c, ln + "swiglu")));
    TcGemmArgs d = tc_args(c, rows, c->H, c->I, kEpiRed);
    tc_segments(d, {{&c->lmaps[l].wd, c->H}});
    d.b_map = c->sbuf_map[bi];
    d.acc = c->acc; d.ldacc = c->H;
    d.trace = ktrace_slot(c, ln + "down", 4);
    CK(c->err, tc_run(c, d));
  } else {
    LinearArgs g = lin_args(c->xn, c->H, c->sbuf, c->I, rows, c->I, c->H);
    g.w[0] = LW(c, l, kWg); g.w2 = LW(c, l, kWu); g.epi = kEpiSwiglu;
    CK(c->err, launch_linear_rows(dt, g, st));
    LinearArgs d = lin_args(c->sbuf, c->I, c->x, c->H, rows, c->H, c->I);
    d.w[0] = LW(c, l, kWd); d.epi = kEpiResid; d.r = c->x; d.ldr = c->H;
    CK(c->err, launch_linear_rows(dt, d, st));
    int rc = capture_stream(c, l, rows);
    if (rc) return rc;
  }
  return DFLASH_OK;
}

// Append-only rings: make sure `rows` more rows fit (syncs only when the
// conservative host bound says they might not, and never while capturing).
int ensure_room(dflash_ctx* c, int rows, ring_cache* r = nullptr) {
  if (!r) r = c->ring;
  if (!r->append_only) return DFLASH_OK;
  if (r->pos_hi + rows - r->host_base <= r->cap) return DFLASH_OK;
  if (c->capturing)
    return fail(c->err, DFLASH_EFULL, "append-only cache may be full; cannot check while capturing");
  long long off;
  int rc = ring_sync_offset(r, &off);
  if (rc) { c->err = r->err; return rc; }
  r->pos_hi = off;
  if (off + rows - r->host_base > r->cap)
    return fail(c->err, DFLASH_EFULL, "append-only cache full: %lld + %d rows > %lld",
                off - r->host_base, rows, r->cap);
  return DFLASH_OK;
}

// Tensor maps of every weight and activation operand of the tensor-core path
// (bf16 configs whose output dimensions are whole 128-row tiles).
int setup_tensor_core_path(dflash_ctx* c) {
  const dflash_config& g = c->cfg;
  c->use_tc = false;
  if (g.dtype != DFLASH_BF16) return DFLASH_OK;
  if (c->H % 128 || c->qdim % 128 || c->kvdim % 128 || c->I % 128 || c->kin % 64) return DFLASH_OK;
  int dev = 0, sms = 0;
  CK(c->err, cudaGetDevice(&dev));
  CK(c->err, cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  c->num_sms = sms < kTcGrid ? sms : kTcGrid;
  const uint64_t H = c->H;
  auto wmap = [&](CUtensorMap* m, const void* w, uint64_t rows, uint64_t inner) {
    return tc_encode_map(m, w, inner, rows, inner * 2, 64, 128);
  };
  bool ok = wmap(&c->fc_map, c->fc, H, c->kin) && wmap(&c->lm_map, c->lm_head, c->V, H);
  c->lmaps.resize(g.n_layers);
  for (int l = 0; l < g.n_layers && ok; ++l) {
    auto& m = c->lmaps[l];
    ok = wmap(&m.wq, LW(c, l, kWq), c->qdim, H) && wmap(&m.wk, LW(c, l, kWk), c->kvdim, H) &&
         wmap(&m.wv, LW(c, l, kWv), c->kvdim, H) && wmap(&m.wo, LW(c, l, kWo), H, c->qdim) &&
         wmap(&m.wg, LW(c, l, kWg), c->I, H) && wmap(&m.wu, LW(c, l, kWu), c->I, H) &&
         wmap(&m.wd, LW(c, l, kWd), H, c->I);
  }
  auto wide = [&](CUtensorMap* m, const void* w, uint64_t rows, uint64_t inner) {
    return tc_encode_map(m, w, inner, rows, inner * 2, 64, 256);
  };
  ok = ok && wide(&c->fcw_map, c->fc, H, c->kin);
  c->lmaps_wide.resize(g.n_layers);
  for (int l = 0; l < g.n_layers && ok; ++l)
    ok = wide(&c->lmaps_wide[l].wk, LW(c, l, kWk), c->kvdim, H) &&
         wide(&c->lmaps_wide[l].wv, LW(c, l, kWv), c->kvdim, H);
  for (int b = 0; b < 2 && ok; ++b) {
    const uint32_t bn = b ? 32 : 16;
    const uint64_t R = c->R;
    ok = tc_encode_map(&c->xn_map[b], c->xn, H, R, H * 2, 64, bn) &&
         tc_encode_map(&c->attn_map[b], c->attn, c->qdim, R, (uint64_t)c->qdim * 2, 64, bn) &&
         tc_encode_map(&c->sbuf_map[b], c->sbuf, c->I, R, (uint64_t)c->I * 2, 64, bn) &&
         tc_encode_map(&c->appc_map[b], c->app_c, H, R, H * 2, 64, bn) &&
         tc_encode_map(&c->xf_map[0][b], c->xf, H, R, H * 2, 64, bn) &&
         tc_encode_map(&c->xf_map[1][b], static_cast<char*>(c->xf) + H * 2, H, R - 1, H * 2, 64, bn);
  }
  if (!ok) return DFLASH_OK;   // no tensor-map encoder: the CUDA-core path serves
  CK(c->err, init_tc_attrs());
  c->use_tc = true;
  return DFLASH_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
extern "C" {

int32_t dflash_speculative_slack(int32_t block) { return block < 1 ? -1 : slack_rule(block, true); }

int dflash_stats_ratios(const dflash_stats* s, double* apr, double* epr, double* acc) {
  if (!s || s->rounds <= 0 || s->draft_n <= 0) return DFLASH_EINVAL;
  const double a = static_cast<double>(s->accepted) / static_cast<double>(s->rounds);
  if (apr) *apr = a;
  if (epr) *epr = a + 1.0;
  if (acc) *acc = static_cast<double>(s->accepted) / static_cast<double>(s->draft_n);
  return DFLASH_OK;
}

int dflash_config_check(const dflash_config* cfg) { return check_config(cfg, g_create_err); }

const char* dflash_last_error(const dflash_ctx* ctx) {
  return ctx ? ctx->err.c_str() : g_create_err.c_str();
}

void dflash_ctx_destroy(dflash_ctx* ctx) {
  if (!ctx) return;
  if (ctx->capturing) {
    cudaGraph_t g = nullptr;
    cudaStreamEndCapture(ctx->stream, &g);
    if (g) cudaGraphDestroy(g);
  }
  cudaStreamSynchronize(ctx->stream);
  for (auto& g : ctx->graphs)
    if (g) cudaGraphExecDestroy(g);
  for (ring_cache* v : ctx->views) ring_free(v);
  ring_free(ctx->ring);
  ring_free(ctx->ring_full);
  cudaFree(ctx->tok);
  cudaFree(ctx->fc_unused);
  cudaFree(ctx->arena);
  cudaFree(ctx->ktr);
  for (auto& ev : ctx->ing_ev)
    if (ev) cudaEventDestroy(ev);
  for (auto& ev : ctx->lm_ev)
    if (ev) cudaEventDestroy(ev);
  delete ctx;
}

int ctx_create_impl(const dflash_config* cfg, const dflash_weights* w, int32_t n_seq, void* stream,
                    dflash_ctx** out, int max_ctx_floor);

int dflash_ctx_create_batched(const dflash_config* cfg, const dflash_weights* w, int32_t n_seq,
                              void* stream, dflash_ctx** out) {
  return ctx_create_impl(cfg, w, n_seq, stream, out, 0);
}

// max_ctx_floor: context rows the attention scratch must cover at least (the
// target's full layers see more than its window).
int ctx_create_impl(const dflash_config* cfg, const dflash_weights* w, int32_t n_seq, void* stream,
                    dflash_ctx** out, int max_ctx_floor) {
  std::string& err = g_create_err;
  if (!out) return fail(err, DFLASH_EINVAL, "out is NULL");
  *out = nullptr;
  int rc = check_config(cfg, err);
  if (rc) return rc;
  if (n_seq < 1 || n_seq > 64) return fail(err, DFLASH_ERANGE, "n_seq %d outside [1, 64]", n_seq);
  if (n_seq > 1 && (cfg->window <= 0 || cfg->markov_rank > 0))
    return fail(err, DFLASH_EINVAL, "a batch needs a sliding window and no Markov head");
  if ((int64_t)n_seq * cfg->max_block > kMaxBlock)
    return fail(err, DFLASH_ERANGE, "n_seq * max_block = %lld exceeds %d rows",
                (long long)n_seq * cfg->max_block, kMaxBlock);
  {
    dflash_config wide = *cfg;
    wide.max_block = n_seq * cfg->max_block;     // the products the batch's row count reaches
    rc = check_config(&wide, err);
    if (rc) return rc;
  }
  if (!w || !w->embed || !w->fc || !w->hidden_norm || !w->final_norm || !w->lm_head || !w->layers)
    return fail(err, DFLASH_EINVAL, "a weight pointer is NULL");
  const void* tops[] = {w->embed, w->fc, w->hidden_norm, w->final_norm, w->lm_head};
  for (const void* p : tops)
    if (!aligned16(p)) return fail(err, DFLASH_EINVAL, "weight pointers must be 16-byte aligned");
  for (int i = 0; i < cfg->n_layers * DFLASH_LAYER_TENSORS; ++i) {
    if (!w->layers[i]) return fail(err, DFLASH_EINVAL, "layer weight %d is NULL", i);
    if (!aligned16(w->layers[i])) return fail(err, DFLASH_EINVAL, "layer weight %d is not 16-byte aligned", i);
  }
  if (cfg->markov_rank > 0 && (!w->markov_w1 || !w->markov_w2 || !aligned16(w->markov_w1) ||
                               !aligned16(w->markov_w2)))
    return fail(err, DFLASH_ERANGE, "markov_rank > 0 needs aligned markov_w1 [V, r] and markov_w2 [r, V]");

  dflash_ctx* c = new (std::nothrow) dflash_ctx();
  if (!c) return fail(err, DFLASH_ECUDA, "out of host memory");
  c->cfg = *cfg;
  c->embed = w->embed; c->fc = w->fc; c->hidden_norm = w->hidden_norm;
  c->final_norm = w->final_norm; c->lm_head = w->lm_head;
  c->w1 = cfg->markov_rank > 0 ? w->markov_w1 : nullptr;
  c->w2 = cfg->markov_rank > 0 ? w->markov_w2 : nullptr;
  c->layers.assign(w->layers, w->layers + (size_t)cfg->n_layers * DFLASH_LAYER_TENSORS);
  c->stream = static_cast<cudaStream_t>(stream);
  c->dt = cfg->dtype;
  c->esz = cfg->dtype == DFLASH_BF16 ? 2 : 4;
  c->H = cfg->hidden; c->nq = cfg->n_q_heads; c->nkv = cfg->n_kv_heads; c->hd = cfg->head_dim;
  c->half = c->hd / 2; c->I = cfg->intermediate; c->V = cfg->vocab;
  c->kin = cfg->k_target_layers * cfg->target_hidden;
  c->qdim = c->nq * c->hd; c->kvdim = c->nkv * c->hd; c->qkv_n = c->qdim + 2 * c->kvdim;
  c->nseq = n_seq;
  c->rows_max = n_seq * cfg->max_block;
  c->max_ctx = cfg->window > 0 ? cfg->window : cfg->max_context;
  if (c->max_ctx < max_ctx_floor) c->max_ctx = max_ctx_floor;

  rc = ring_create_impl(cfg->n_layers, c->nkv, c->hd, cfg->window, cfg->max_block, cfg->dtype,
                        cfg->max_context, 0, c->stream, &c->ring, err, n_seq);
  if (rc) { delete c; return rc; }
  c->ring->owned_by_ctx = true;
  c->seq_ctx.assign(n_seq, 0);
  for (int q = 0; q < n_seq; ++q) {
    ring_cache* v = new (std::nothrow) ring_cache(*c->ring);
    if (!v) { ring_free(c->ring); delete c; return fail(err, DFLASH_ECUDA, "out of host memory"); }
    v->view = true;
    v->nseq = 1;
    v->k = static_cast<char*>(c->ring->k) + (size_t)q * c->ring->L * c->nkv * c->ring->cap * c->hd * c->esz;
    v->v = static_cast<char*>(c->ring->v) + (size_t)q * c->ring->L * c->nkv * c->ring->cap * c->hd * c->esz;
    v->st = c->ring->st + q;
    c->views.push_back(v);
  }

  c->R = c->rows_max + 1 > 33 ? c->rows_max + 1 : 33;
  const size_t E = c->esz, R = c->R;
  c->ing_rows = c->max_ctx < kIngestChunk ? c->max_ctx : kIngestChunk;
  c->lm_grid = lmhead_grid(c->V);
  c->vf_chunks = verify_chunks(c->V);
  c->mk_grid = markov_grid(c->V);
  if (cfg->markov_rank > 0) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0 &&
        markov_coop_ok(cfg->dtype, c->V, cfg->markov_rank, sms)) {
      c->mk_coop = true;
      c->mk_coop_grid = sms;
    }
  }
  size_t attn_floats = attention_scratch_floats(c->rows_max, c->nq, c->nkv, c->hd, c->max_ctx);
  const size_t attn_mma_floats = attention_mma_scratch_floats(c->rows_max, c->nq, c->nkv, c->max_ctx);
  if (attn_mma_floats > attn_floats) attn_floats = attn_mma_floats;
  const size_t sizes[] = {
      sizeof(RoundState) * n_seq, sizeof(double) * c->half,
      R * c->H * E, R * c->H * E, R * c->qkv_n * E, R * c->qdim * E, R * c->I * E, R * c->H * E,
      R * c->half * sizeof(float2), attn_floats * sizeof(float),
      R * c->H * E, R * c->H * E, R * 2 * c->kvdim * E, R * c->half * sizeof(float2),
      (size_t)c->ing_rows * c->H * E, (size_t)c->ing_rows * c->H * E,
      (size_t)c->ing_rows * 2 * c->kvdim * E * cfg->n_layers, (size_t)c->ing_rows * c->half * sizeof(float2),
      (size_t)c->lm_grid * R * 4, (size_t)c->lm_grid * R * 4, R * c->vf_chunks * 4,
      R * c->vf_chunks * 4, R * 8, (size_t)c->mk_grid * 4, 8 * sizeof(unsigned),
      R * 4, R * 4, cfg->markov_add && cfg->markov_rank > 0 ? R * (size_t)c->V * 4 : 0,
      (size_t)kTcGrid * 2 * 2 * 32 * 128 * 4, (size_t)kTcTiles * 4, 64,
      (size_t)kTcGrid * 32 * 4, (size_t)kTcGrid * 32 * 4, 64,
      (size_t)cfg->n_layers * sizeof(void*), R * 4, R * 4, R * 4, 64, R * c->H * 4, R * c->qkv_n * 4, R * 2 * c->I * 4,
      R * (size_t)cfg->n_layers * 2 * c->kvdim * 4, R * 4, R * 4, sizeof(unsigned) * n_seq};
  size_t total = 0;
  for (size_t s : sizes) total += (s + 255) & ~size_t(255);
  cudaError_t e = cudaMalloc(&c->arena, total);
  if (e != cudaSuccess) { ring_free(c->ring); delete c; return cuda_fail(err, e, "scratch allocation"); }
  c->arena_bytes = total;
  char* cur = c->arena;
  int si = 0;
  c->rs = carve<RoundState>(cur, sizes[si++]);
  c->inv_freq = carve<double>(cur, sizes[si++]);
  c->x = carve<char>(cur, sizes[si++]);
  c->xn = carve<char>(cur, sizes[si++]);
  c->qkv = carve<char>(cur, sizes[si++]);
  c->attn = carve<char>(cur, sizes[si++]);
  c->sbuf = carve<char>(cur, sizes[si++]);
  c->xf = carve<char>(cur, sizes[si++]);
  c->rope = carve<float2>(cur, sizes[si++]);
  c->attn_part_floats = attn_floats;
  c->attn_part = carve<float>(cur, sizes[si++]);
  c->app_f = carve<char>(cur, sizes[si++]);
  c->app_c = carve<char>(cur, sizes[si++]);
  c->app_kv = carve<char>(cur, sizes[si++]);
  c->app_rope = carve<float2>(cur, sizes[si++]);
  c->ing_f = carve<char>(cur, sizes[si++]);
  c->ing_c = carve<char>(cur, sizes[si++]);
  c->ing_kv = carve<char>(cur, sizes[si++]);
  c->ing_rope = carve<float2>(cur, sizes[si++]);
  c->lm_pv = carve<float>(cur, sizes[si++]);
  c->lm_pi = carve<int>(cur, sizes[si++]);
  c->vf_pv = carve<float>(cur, sizes[si++]);
  c->vf_pi = carve<int>(cur, sizes[si++]);
  c->mk_pv = carve<float>(cur, sizes[si++]);
  c->mk_pi = carve<int>(cur, sizes[si++]);
  c->counters = carve<unsigned>(cur, sizes[si++]);
  c->maxv = carve<float>(cur, sizes[si++]);
  c->backbone_ids = carve<int>(cur, sizes[si++]);
  c->zlog = sizes[si] ? carve<float>(cur, sizes[si]) : nullptr;
  ++si;
  c->tc_part = carve<float>(cur, sizes[si++]);
  c->tc_tiles = carve<unsigned>(cur, sizes[si++]);
  c->tc_err = carve<int>(cur, sizes[si++]);
  c->tc_best = carve<unsigned long long>(cur, sizes[si++]);
  c->tc_lm_pi = carve<int>(cur, sizes[si++]);
  c->tc_done = carve<unsigned>(cur, sizes[si++]);
  c->kgain_dev = carve<const void*>(cur, sizes[si++]);
  c->samp_acc = carve<int>(cur, sizes[si++]);
  c->samp_cand = carve<int>(cur, sizes[si++]);
  c->samp_pd = carve<float>(cur, sizes[si++]);
  c->samp_ctr = carve<unsigned>(cur, sizes[si++]);
  c->acc = carve<float>(cur, sizes[si++]);
  c->qkv_acc = carve<float>(cur, sizes[si++]);
  c->gu_acc = carve<float>(cur, sizes[si++]);
  c->kv_acc = carve<float>(cur, sizes[si++]);
  c->ids_all = carve<int>(cur, sizes[si++]);
  c->maxv_all = carve<float>(cur, sizes[si++]);
  c->vf_ctr = carve<unsigned>(cur, sizes[si++]);

  std::vector<const void*> kg(cfg->n_layers);
  for (int l = 0; l < cfg->n_layers; ++l) kg[l] = c->layers[(size_t)l * DFLASH_LAYER_TENSORS + 5];
  std::vector<double> inv(c->half);
  for (int i = 0; i < c->half; ++i)
    inv[i] = std::pow(static_cast<double>(cfg->rope_theta), -2.0 * i / static_cast<double>(c->hd));
  if ((e = cudaMemsetAsync(c->arena, 0, total, c->stream)) != cudaSuccess ||
      (e = cudaMemcpyAsync(c->inv_freq, inv.data(), sizeof(double) * c->half,
                           cudaMemcpyHostToDevice, c->stream)) != cudaSuccess ||
      (e = cudaMemcpyAsync(c->kgain_dev, kg.data(), sizeof(void*) * kg.size(),
                           cudaMemcpyHostToDevice, c->stream)) != cudaSuccess ||
      (e = init_lmhead_attrs(c->H)) != cudaSuccess ||
      (e = init_attention_attrs(c->hd)) != cudaSuccess ||
      (e = cudaEventCreate(&c->lm_ev[0])) != cudaSuccess ||
      (e = cudaEventCreate(&c->lm_ev[1])) != cudaSuccess ||
      (e = cudaEventCreate(&c->ing_ev[0])) != cudaSuccess ||
      (e = cudaEventCreate(&c->ing_ev[1])) != cudaSuccess ||
      (e = cudaEventCreate(&c->ing_ev[2])) != cudaSuccess ||
      (e = cudaEventCreate(&c->ing_ev[3])) != cudaSuccess ||
      (e = cudaStreamSynchronize(c->stream)) != cudaSuccess) {
    dflash_ctx_destroy(c);
    return cuda_fail(err, e, "context initialisation");
  }
  rc = setup_tensor_core_path(c);
  if (rc) { std::string m = c->err; dflash_ctx_destroy(c); return fail(err, rc, "%s", m.c_str()); }
  *out = c;
  return DFLASH_OK;
}

int dflash_ctx_create(const dflash_config* cfg, const dflash_weights* w, void* stream,
                      dflash_ctx** out) {
  return dflash_ctx_create_batched(cfg, w, 1, stream, out);
}

int dflash_ingest_context(dflash_ctx* c, const void* resid, int64_t rows, int64_t first_pos,
                          int32_t anchor) {
  return dflash_ingest_context_seq(c, 0, resid, rows, first_pos, anchor);
}

int dflash_ingest_context_seq(dflash_ctx* c, int32_t seq, const void* resid, int64_t rows, int64_t first_pos,
                              int32_t anchor) {
  if (!c) return DFLASH_EINVAL;
  if (c->is_target) return fail(c->err, DFLASH_EINVAL, "a target context takes the dflash_target_* calls");
  if (seq < 0 || seq >= c->nseq) return fail(c->err, DFLASH_ERANGE, "seq %d outside [0, %d)", seq, c->nseq);
  c->seq_cur = seq;
  if (rows <= 0) return fail(c->err, DFLASH_EEMPTY, "empty context (rows = %lld)", (long long)rows);
  if (!resid || !aligned16(resid)) return fail(c->err, DFLASH_EINVAL, "resid is NULL or misaligned");
  if (first_pos < 0) return fail(c->err, DFLASH_EINVAL, "first_pos must be >= 0");
  if (anchor < 0 || anchor >= c->V)
    return fail(c->err, DFLASH_ERANGE, "anchor %d outside [0, vocab=%d)", anchor, c->V);
  const long long next = first_pos + rows;
  long long kept_first = first_pos;
  if (c->cfg.window > 0 && next - c->cfg.window > kept_first) kept_first = next - c->cfg.window;
  const long long kept = next - kept_first;
  if (c->ring->append_only && kept > c->ring->cap)
    return fail(c->err, DFLASH_EFULL, "%lld context rows exceed max_context %lld", kept, c->ring->cap);
  CK(c->err, launch_ring_reset(c->ring->st + seq, kept_first, c->stream));
  const char* src = static_cast<const char*>(resid) + (size_t)(kept_first - first_pos) * c->kin * c->esz;
  const bool wide = c->use_tc && c->H % 256 == 0 && c->kvdim % 256 == 0;
  for (long long s = 0; s < kept; s += c->ing_rows) {
    const int n = static_cast<int>(kept - s < c->ing_rows ? kept - s : c->ing_rows);
    const void* rows_ptr = src + (size_t)s * c->kin * c->esz;
    int rc = (wide && n > 32)
                 ? context_rows_wide(c, rows_ptr, n, c->ing_f, c->ing_c, c->ing_kv, c->ing_rope, kept_first + s)
                 : context_rows_to_ring(c, rows_ptr, n, c->ing_f, c->ing_c, c->ing_kv, c->ing_rope, 0,
                                        kept_first + s);
    if (rc) return rc;
  }
  CK(c->err, launch_ring_advance(c->ring->st + seq, static_cast<int>(kept), 2, c->stream));
  CK(c->err, launch_set_anchor(c->rs + seq, anchor, c->stream));
  c->ring->host_base = kept_first;
  c->ring->pos_hi = next;
  c->ring->host_appended = 0;
  c->seq_ctx[seq] = 1;
  c->has_context = true;
  for (char h : c->seq_ctx) c->has_context = c->has_context && h;
  c->appended_block = 0;
  return DFLASH_OK;
}

int dflash_set_anchor(dflash_ctx* c, int32_t anchor) {
  if (!c) return DFLASH_EINVAL;
  if (anchor < 0 || anchor >= c->V)
    return fail(c->err, DFLASH_ERANGE, "anchor %d outside [0, vocab=%d)", anchor, c->V);
  CK(c->err, launch_set_anchor(c->rs, anchor, c->stream));
  return DFLASH_OK;
}

// DSpark: the rank-r Markov chain proposes the draft from the anchor, adding
// the backbone's logits when configured.
cudaError_t draft_markov(dflash_ctx* c, int R, int32_t* draft_ids) {
  MarkovArgs mk{};
  mk.w1 = c->w1; mk.w2 = c->w2; mk.V = c->V; mk.r = c->cfg.markov_rank;
  mk.rs = c->rs; mk.anchor_host = -1;
  mk.z = c->cfg.markov_add ? c->zlog : nullptr; mk.ldz = c->V;
  mk.gamma = R; mk.out = draft_ids; mk.out2 = nullptr;
  mk.key = reinterpret_cast<unsigned long long*>(c->mk_pv); mk.counter = c->counters + 2;
  mk.grid = c->mk_grid;
  mk.bar = c->counters + 4; mk.err = c->tc_err;
  if (c->mk_coop && !c->mk_stepwise) {
    mk.trace = ktrace_slot(c, "markov", 1);
    return launch_markov_chain_coop(c->dt, mk, c->mk_coop_grid, c->stream);
  }
  mk.trace = ktrace_slot(c, "markov", mk.gamma);
  return launch_markov_chain(c->dt, mk, c->stream);
}

int dflash_draft_block(dflash_ctx* c, int32_t anchor, int64_t anchor_pos, int32_t block,
                       int32_t* draft_ids) {
  if (!c) return DFLASH_EINVAL;
  if (c->is_target) return fail(c->err, DFLASH_EINVAL, "a target context takes the dflash_target_* calls");
  if (!draft_ids) return fail(c->err, DFLASH_EINVAL, "draft_ids is NULL");
  if (block < 2 || block > c->cfg.max_block)
    return fail(c->err, DFLASH_ERANGE, "block %d outside [2, max_block=%d]", block, c->cfg.max_block);
  if (anchor >= c->V)
    return fail(c->err, DFLASH_ERANGE, "anchor %d outside [0, vocab=%d)", anchor, c->V);
  if (c->nseq > 1 && (anchor >= 0 || anchor_pos >= 0))
    return fail(c->err, DFLASH_EINVAL, "a batch drafts from its device-resident anchors (pass -1, -1)");
  if (!c->has_context) return fail(c->err, DFLASH_EEMPTY, "no context ingested");
  const int dspark = c->cfg.kind == DFLASH_KIND_DSPARK;
  const int rps = dspark ? block - 1 : block;      // block rows of one sequence
  const int rows = rps * c->nseq;                  // rows of the whole batch
  const int read0 = dspark ? 0 : 1;
  const int R = block - 1;
  const int dt = c->dt;
  cudaStream_t st = c->stream;
  const bool markov = c->cfg.markov_rank > 0;
  if (c->ktr_on && c->ktr) {
    c->ktr_n = 0;
    c->ktr_names.clear();
    CK(c->err, cudaMemsetAsync(c->ktr, 0xFF, sizeof(unsigned long long) * kKTraceSlots, st));
    CK(c->err, cudaMemsetAsync(c->ktr + kKTraceSlots, 0, 2 * sizeof(unsigned long long) * kKTraceSlots, st));
  }
  CK(c->err, launch_embed_block(dt, c->embed, c->H, c->V, c->rs, c->cfg.mask_token_id, rps, c->x,
                                c->ring->st, c->inv_freq, c->half, rps, c->rope,
                                anchor < 0 ? -1 : anchor, anchor_pos < 0 ? -1 : anchor_pos, st, c->nseq));
  for (int l = 0; l < c->cfg.n_layers; ++l) {
    int rc = layer_forward(c, l, rows);
    if (rc) return rc;
  }
  if (tc_rows(c, rows))   // the last down GEMM's sums are still in c->acc
    CK(c->err, launch_resid_rmsnorm(c->x, c->H, c->acc, c->H, c->final_norm, c->xf, c->H, rows, c->H,
                                    c->cfg.rms_eps, st, ktrace_slot(c, "final_norm")));
  else
    CK(c->err, launch_rmsnorm(dt, c->x, c->H, c->final_norm, c->xf, c->H, rows, c->H,
                              c->cfg.rms_eps, st, ktrace_slot(c, "final_norm")));
  // One sequence: the read-out rows read0 .. are contiguous and the argmax
  // writes the proposals directly. A batch: the argmax runs over every block
  // row and the read-out rows of each sequence are picked out afterwards.
  const bool batch = c->nseq > 1;
  const int lm_rows = batch ? rows : R;
  LmHeadArgs lm{};
  lm.x = static_cast<char*>(c->xf) + (size_t)(batch ? 0 : read0) * c->H * c->esz;
  lm.ldx = c->H;
  lm.w = c->lm_head;
  lm.R = lm_rows; lm.H = c->H; lm.V = c->V;
  lm.softcap = c->cfg.softcap;
  lm.ids = batch ? c->ids_all : (markov ? c->backbone_ids : draft_ids);
  lm.ids2 = (batch || markov) ? nullptr : c->backbone_ids;
  lm.maxv = batch ? c->maxv_all : c->maxv;
  lm.logits = (markov && c->cfg.markov_add) ? c->zlog : nullptr;
  lm.part_v = c->lm_pv; lm.part_i = c->lm_pi;
  lm.counter = c->counters + 0;
  lm.grid = c->lm_grid;
  if (c->lm_timing) CK(c->err, cudaEventRecordWithFlags(c->lm_ev[0], st, c->capturing ? cudaEventRecordExternal : 0));
  if (tc_rows(c, lm_rows) && lm.logits == nullptr) {
    TcGemmArgs t = tc_args(c, lm_rows, c->V, c->H, kEpiArgmax);
    tc_segments(t, {{&c->lm_map, c->V}});
    t.b_map = c->xf_map[batch ? 0 : read0][bn_index(lm_rows)];
    t.softcap = c->cfg.softcap;
    t.ids = lm.ids; t.ids2 = lm.ids2; t.maxv = lm.maxv;
    t.best_key = c->tc_best; t.done_ctr = c->tc_done; t.whole_tiles = t.M > 8;
    t.trace = ktrace_slot(c, "lm_head", 4);
    CK(c->err, tc_run(c, t));
  } else {
    CK(c->err, launch_lmhead_argmax(dt, lm, st));
  }
  if (c->lm_timing) {
    CK(c->err, cudaEventRecordWithFlags(c->lm_ev[1], st, c->capturing ? cudaEventRecordExternal : 0));
    c->lm_recorded = true;
  }
  if (batch)
    CK(c->err, launch_split_ids(c->ids_all, c->maxv_all, rps, read0, c->nseq, draft_ids, c->backbone_ids,
                                c->maxv, st));
  if (markov) CK(c->err, draft_markov(c, R, draft_ids));
  c->last_draft_block = block;
  return DFLASH_OK;
}

int dflash_verify_accept(dflash_ctx* c, const void* target_logits, int32_t block,
                         const int32_t* draft_ids, int32_t* tokens, int32_t* n) {
  if (!c) return DFLASH_EINVAL;
  if (!target_logits || !draft_ids || !tokens || !n)
    return fail(c->err, DFLASH_EINVAL, "a verify pointer is NULL");
  if (block < 2 || block > c->cfg.max_block)
    return fail(c->err, DFLASH_ERANGE, "block %d outside [2, max_block=%d]", block, c->cfg.max_block);
  VerifyArgs v{};
  v.L = target_logits; v.B = block; v.V = c->V; v.d = draft_ids; v.tokens = tokens; v.n = n;
  v.rs = c->rs; v.part_v = c->vf_pv; v.part_i = c->vf_pi; v.counter = c->vf_ctr;
  v.nseq = c->nseq;
  v.chunks = c->vf_chunks;
  v.trace = ktrace_slot(c, "verify");
  CK(c->err, launch_verify(c->dt, v, c->stream));
  c->last_verify_block = block;
  c->last_tokens = tokens;
  c->last_n = n;
  c->last_tokens_block = block;
  return DFLASH_OK;
}

int dflash_verify_sampled(dflash_ctx* c, const void* target_logits, int32_t block,
                          const int32_t* draft_ids, const float* uniforms, float temperature,
                          float softcap, int32_t* tokens, int32_t* n, float* p_draft) {
  if (!c) return DFLASH_EINVAL;
  if (!target_logits || !draft_ids || !uniforms || !tokens || !n)
    return fail(c->err, DFLASH_EINVAL, "a sampled-verify pointer is NULL");
  if (block < 2 || block > c->cfg.max_block)
    return fail(c->err, DFLASH_ERANGE, "block %d outside [2, max_block=%d]", block, c->cfg.max_block);
  if (!(temperature > 0.f) || !std::isfinite(temperature) || !(softcap >= 0.f) || !std::isfinite(softcap))
    return fail(c->err, DFLASH_EINVAL, "temperature must be > 0 and softcap >= 0, both finite");
  if (c->nseq > 1) return fail(c->err, DFLASH_EINVAL, "the sampled verify takes one sequence");
  SampledVerifyArgs a{};
  a.L = target_logits; a.B = block; a.V = c->V; a.d = draft_ids; a.u = uniforms;
  a.temperature = temperature; a.softcap = softcap; a.tokens = tokens; a.n = n; a.rs = c->rs;
  a.acc = c->samp_acc; a.cand = c->samp_cand; a.pd = p_draft ? p_draft : c->samp_pd;
  a.counter = c->samp_ctr;
  CK(c->err, launch_verify_sampled(c->dt, a, c->stream));
  c->last_verify_block = block;
  c->last_tokens = tokens;
  c->last_n = n;
  c->last_tokens_block = block;
  return DFLASH_OK;
}

int dflash_sync_round(dflash_ctx* c, int32_t* tokens_host, int32_t* n_host) {
  if (!c) return DFLASH_EINVAL;
  if (!tokens_host || !n_host) return fail(c->err, DFLASH_EINVAL, "tokens_host or n_host is NULL");
  if (c->capturing) return fail(c->err, DFLASH_ESTATE, "dflash_sync_round while capturing");
  if (!c->last_tokens || !c->last_n) return fail(c->err, DFLASH_ESTATE, "no verify yet");
  CK(c->err, cudaMemcpyAsync(n_host, c->last_n, sizeof(int32_t) * c->nseq, cudaMemcpyDeviceToHost, c->stream));
  CK(c->err, cudaMemcpyAsync(tokens_host, c->last_tokens, sizeof(int32_t) * c->last_tokens_block * c->nseq,
                             cudaMemcpyDeviceToHost, c->stream));
  CK(c->err, cudaStreamSynchronize(c->stream));
  return DFLASH_OK;
}

int dflash_append_block(dflash_ctx* c, const void* resid, int32_t block) {
  if (!c) return DFLASH_EINVAL;
  if (c->is_target) return fail(c->err, DFLASH_EINVAL, "a target context takes the dflash_target_* calls");
  if (!resid || !aligned16(resid)) return fail(c->err, DFLASH_EINVAL, "resid is NULL or misaligned");
  if (block < 1 || block > c->cfg.max_block)
    return fail(c->err, DFLASH_ERANGE, "block %d outside [1, max_block=%d]", block, c->cfg.max_block);
  if (!c->has_context) return fail(c->err, DFLASH_EEMPTY, "no context ingested");
  if (c->appended_block) return fail(c->err, DFLASH_ESTATE, "append without a commit of the previous append");
  int rc = ensure_room(c, block);
  if (rc) return rc;
  rc = context_rows_to_ring(c, resid, block * c->nseq, c->app_f, c->app_c, c->app_kv, c->app_rope, 1, 0);
  if (rc) return rc;
  CK(c->err, launch_ring_advance(c->ring->st, block, 0, c->stream, c->nseq));
  c->appended_block = block;
  c->ring->host_appended = block;
  c->ring->pos_hi += block;
  return DFLASH_OK;
}

int dflash_commit(dflash_ctx* c, int32_t keep) {
  if (!c) return DFLASH_EINVAL;
  if (!c->appended_block) return fail(c->err, DFLASH_ESTATE, "commit without an append");
  if (keep > c->appended_block)
    return fail(c->err, DFLASH_EINVAL, "keep %d exceeds the appended block %d", keep, c->appended_block);
  if (keep < 0 && c->last_verify_block != c->appended_block)
    return fail(c->err, DFLASH_ESTATE, "commit(-1) needs a verify at the appended width %d", c->appended_block);
  CK(c->err, launch_commit(c->rs, c->ring->st, c->appended_block, keep, c->stream, c->nseq));
  if (keep >= 0) c->ring->pos_hi -= c->appended_block - keep;
  c->appended_block = 0;
  c->last_verify_block = 0;
  c->ring->host_appended = 0;
  return DFLASH_OK;
}

int dflash_round(dflash_ctx* c, const void* target_logits, const void* resid, int32_t block,
                 int32_t* draft_ids, int32_t* tokens, int32_t* n) {
  int rc = dflash_draft_block(c, -1, -1, block, draft_ids);
  if (!rc) rc = dflash_verify_accept(c, target_logits, block, draft_ids, tokens, n);
  if (!rc) rc = dflash_append_block(c, resid, block);
  if (!rc) rc = dflash_commit(c, -1);
  return rc;
}

int dflash_linear(dflash_ctx* c, const void* x, int32_t M, int32_t K, const void* w, const void* w2,
                  int32_t N, const void* r, void* y, int32_t epi) {
  if (!c) return DFLASH_EINVAL;
  if (!x || !w || !y || (epi == kEpiSwiglu && !w2) || (epi == kEpiResid && !r))
    return fail(c->err, DFLASH_EINVAL, "a linear operand is NULL");
  if (epi < 0 || epi > 2) return fail(c->err, DFLASH_EINVAL, "epi must be 0, 1 or 2");
  if (M < 1 || K < 8 || N < 1 || K % 8) return fail(c->err, DFLASH_EINVAL, "bad linear shape");
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (w2 && !aligned16(w2)) || (r && !aligned16(r)))
    return fail(c->err, DFLASH_EINVAL, "linear operands must be 16-byte aligned");
  if (c->use_tc && M > 32 && K % 64 == 0 && N % 256 == 0 && epi == kEpiStore) {
    TcWideArgs a{};
    a.M = M; a.N = N; a.K = K; a.nseg = 1; a.seg_rows[0] = N;
    a.y = y; a.ldy = N; a.err = c->tc_err;
    if (!tc_encode_map(&a.x_map, x, K, M, (uint64_t)K * 2, 64, 128) ||
        !tc_encode_map(&a.w_map[0], w, K, N, (uint64_t)K * 2, 64, 256))
      return fail(c->err, DFLASH_ECUDA, "cuTensorMapEncodeTiled failed");
    CK(c->err, launch_tc_wide(a, c->num_sms, c->stream));
  } else if (c->use_tc && M <= 32 && K % 64 == 0) {
    TcGemmArgs t = tc_args(c, M, N, K, epi);
    CUtensorMap wa, wb;
    bool ok = tc_encode_map(&wa, w, K, N, (uint64_t)K * 2, 64, 128) &&
              tc_encode_map(&t.b_map, x, K, M, (uint64_t)K * 2, 64, bn_of(M));
    if (ok && epi == kEpiSwiglu) ok = tc_encode_map(&wb, w2, K, N, (uint64_t)K * 2, 64, 128);
    if (!ok) return fail(c->err, DFLASH_ECUDA, "cuTensorMapEncodeTiled failed");
    tc_segments(t, {{&wa, N}});
    if (epi == kEpiSwiglu) t.a2_map = wb;
    t.y = y; t.ldy = N; t.r = r; t.ldr = N;
    CK(c->err, tc_run(c, t));
  } else {
    LinearArgs a = lin_args(x, K, y, N, M, N, K);
    a.w[0] = w; a.w2 = w2; a.r = r; a.ldr = N; a.epi = epi;
    CK(c->err, (M > 32 && epi == kEpiStore) ? launch_linear_tiled(c->dt, a, c->stream)
                                            : launch_linear_rows(c->dt, a, c->stream));
  }
  return DFLASH_OK;
}

int dflash_lm_head_argmax(dflash_ctx* c, const void* x, int32_t rows, int32_t* ids, float* maxv) {
  if (!c) return DFLASH_EINVAL;
  if (!x || !ids || !maxv) return fail(c->err, DFLASH_EINVAL, "an lm_head operand is NULL");
  if (rows < 1 || rows > c->cfg.max_block) return fail(c->err, DFLASH_ERANGE, "rows outside [1, max_block]");
  if (!aligned16(x)) return fail(c->err, DFLASH_EINVAL, "x must be 16-byte aligned");
  if (c->use_tc) {
    TcGemmArgs t = tc_args(c, rows, c->V, c->H, kEpiArgmax);
    tc_segments(t, {{&c->lm_map, c->V}});
    if (!tc_encode_map(&t.b_map, x, c->H, rows, (uint64_t)c->H * 2, 64, bn_of(rows)))
      return fail(c->err, DFLASH_ECUDA, "cuTensorMapEncodeTiled failed");
    t.softcap = c->cfg.softcap;
    t.ids = ids; t.ids2 = nullptr; t.maxv = maxv;
    t.best_key = c->tc_best; t.done_ctr = c->tc_done; t.whole_tiles = t.M > 8;
    CK(c->err, tc_run(c, t));
  } else {
    LmHeadArgs lm{};
    lm.x = x; lm.ldx = c->H; lm.w = c->lm_head; lm.R = rows; lm.H = c->H; lm.V = c->V;
    lm.softcap = c->cfg.softcap; lm.ids = ids; lm.maxv = maxv;
    lm.part_v = c->lm_pv; lm.part_i = c->lm_pi; lm.counter = c->counters + 0; lm.grid = c->lm_grid;
    CK(c->err, launch_lmhead_argmax(c->dt, lm, c->stream));
  }
  return DFLASH_OK;
}

int dflash_markov_chain(dflash_ctx* c, int32_t anchor, int32_t gamma, const float* z, int32_t* out) {
  if (!c) return DFLASH_EINVAL;
  if (!out) return fail(c->err, DFLASH_EINVAL, "out is NULL");
  if (c->cfg.markov_rank <= 0) return fail(c->err, DFLASH_ERANGE, "the config has no Markov head");
  if (c->nseq > 1) return fail(c->err, DFLASH_EINVAL, "the Markov chain takes one sequence");
  if (anchor < 0 || anchor >= c->V)
    return fail(c->err, DFLASH_ERANGE, "anchor %d outside [0, vocab=%d)", anchor, c->V);
  if (gamma < 1 || gamma > c->cfg.max_block)
    return fail(c->err, DFLASH_ERANGE, "gamma %d outside [1, max_block]", gamma);
  MarkovArgs mk{};
  mk.w1 = c->w1; mk.w2 = c->w2; mk.V = c->V; mk.r = c->cfg.markov_rank;
  mk.rs = c->rs; mk.anchor_host = anchor; mk.z = z; mk.ldz = c->V; mk.gamma = gamma;
  mk.out = out; mk.out2 = nullptr;
  mk.key = reinterpret_cast<unsigned long long*>(c->mk_pv); mk.counter = c->counters + 2; mk.grid = c->mk_grid;
  mk.bar = c->counters + 4; mk.err = c->tc_err;
  if (c->mk_coop && !c->mk_stepwise)
    CK(c->err, launch_markov_chain_coop(c->dt, mk, c->mk_coop_grid, c->stream));
  else CK(c->err, launch_markov_chain(c->dt, mk, c->stream));
  return DFLASH_OK;
}

int dflash_get_hidden(dflash_ctx* c, void* out) {
  if (!c || !out) return DFLASH_EINVAL;
  if (!c->last_draft_block) return fail(c->err, DFLASH_ESTATE, "no draft yet");
  const int rows = (c->cfg.kind == DFLASH_KIND_DSPARK ? c->last_draft_block - 1 : c->last_draft_block) * c->nseq;
  CK(c->err, cudaMemcpyAsync(out, c->xf, (size_t)rows * c->H * c->esz, cudaMemcpyDeviceToDevice, c->stream));
  CK(c->err, cudaStreamSynchronize(c->stream));
  return DFLASH_OK;
}

int dflash_get_draft_max_logit(dflash_ctx* c, float* out) {
  if (!c || !out) return DFLASH_EINVAL;
  if (!c->last_draft_block) return fail(c->err, DFLASH_ESTATE, "no draft yet");
  CK(c->err, cudaMemcpyAsync(out, c->maxv, sizeof(float) * (c->last_draft_block - 1) * c->nseq,
                             cudaMemcpyDeviceToDevice, c->stream));
  CK(c->err, cudaStreamSynchronize(c->stream));
  return DFLASH_OK;
}

int dflash_get_backbone_ids(dflash_ctx* c, int32_t* out) {
  if (!c || !out) return DFLASH_EINVAL;
  if (!c->last_draft_block) return fail(c->err, DFLASH_ESTATE, "no draft yet");
  CK(c->err, cudaMemcpyAsync(out, c->backbone_ids, sizeof(int) * (c->last_draft_block - 1) * c->nseq,
                             cudaMemcpyDeviceToDevice, c->stream));
  CK(c->err, cudaStreamSynchronize(c->stream));
  return DFLASH_OK;
}

int dflash_get_state(dflash_ctx* c, dflash_round_state* out) { return dflash_get_state_seq(c, 0, out); }

int dflash_get_state_seq(dflash_ctx* c, int32_t seq, dflash_round_state* out) {
  if (!c || !out) return DFLASH_EINVAL;
  if (seq < 0 || seq >= c->nseq) return fail(c->err, DFLASH_ERANGE, "seq %d outside [0, %d)", seq, c->nseq);
  RoundState rs;
  RingState ring;
  CK(c->err, cudaStreamSynchronize(c->stream));
  CK(c->err, cudaMemcpy(&rs, c->rs + seq, sizeof rs, cudaMemcpyDeviceToHost));
  CK(c->err, cudaMemcpy(&ring, c->ring->st + seq, sizeof ring, cudaMemcpyDeviceToHost));
  out->position = ring.offset;
  out->anchor = rs.anchor;
  out->last_n = rs.n;
  out->last_accepted = rs.a;
  int tcerr = 0;
  if (c->tc_err) CK(c->err, cudaMemcpy(&tcerr, c->tc_err, sizeof tcerr, cudaMemcpyDeviceToHost));
  out->error = rs.error | ring.error | (tcerr ? 4 : 0);
  return DFLASH_OK;
}

int dflash_get_stats(dflash_ctx* c, dflash_stats* out) { return dflash_get_stats_seq(c, 0, out); }

int dflash_get_stats_seq(dflash_ctx* c, int32_t seq, dflash_stats* out) {
  if (!c || !out) return DFLASH_EINVAL;
  if (seq < 0 || seq >= c->nseq) return fail(c->err, DFLASH_ERANGE, "seq %d outside [0, %d)", seq, c->nseq);
  RoundState rs;
  CK(c->err, cudaStreamSynchronize(c->stream));
  CK(c->err, cudaMemcpy(&rs, c->rs + seq, sizeof rs, cudaMemcpyDeviceToHost));
  out->rounds = rs.rounds;
  out->draft_n = rs.proposed;
  out->accepted = rs.accepted;
  out->emitted = rs.emitted;
  return DFLASH_OK;
}

int dflash_reset_stats(dflash_ctx* c) {
  if (!c) return DFLASH_EINVAL;
  for (int q = 0; q < c->nseq; ++q)
    CK(c->err, cudaMemsetAsync(&c->rs[q].rounds, 0, 4 * sizeof(long long), c->stream));
  return DFLASH_OK;
}

int dflash_ring(dflash_ctx* c, ring_cache** out) { return dflash_ring_seq(c, 0, out); }

int dflash_ring_seq(dflash_ctx* c, int32_t seq, ring_cache** out) {
  if (!c || !out) return DFLASH_EINVAL;
  if (seq < 0 || seq >= c->nseq) return fail(c->err, DFLASH_ERANGE, "seq %d outside [0, %d)", seq, c->nseq);
  *out = c->nseq == 1 ? c->ring : c->views[seq];
  return DFLASH_OK;
}

int dflash_batch_size(const dflash_ctx* c) { return c ? c->nseq : 0; }

int dflash_capture_begin(dflash_ctx* c) {
  if (!c) return DFLASH_EINVAL;
  if (c->capturing) return fail(c->err, DFLASH_ESTATE, "already capturing");
  if (!c->stream) return fail(c->err, DFLASH_ESTATE, "the legacy default stream cannot be captured");
  CK(c->err, cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal));
  c->capturing = true;
  c->saved_flags[0] = c->last_draft_block;
  c->saved_flags[1] = c->last_verify_block;
  c->saved_flags[2] = c->appended_block;
  c->saved_flags[3] = static_cast<int>(c->ring->pos_hi - c->ring->host_base);
  return DFLASH_OK;
}

int dflash_capture_end(dflash_ctx* c, int32_t slot) {
  if (!c) return DFLASH_EINVAL;
  if (!c->capturing) return fail(c->err, DFLASH_ESTATE, "not capturing");
  cudaGraph_t g = nullptr;
  cudaError_t e = cudaStreamEndCapture(c->stream, &g);
  c->capturing = false;
  c->last_draft_block = c->saved_flags[0];
  c->last_verify_block = c->saved_flags[1];
  c->appended_block = c->saved_flags[2];
  c->ring->pos_hi = c->ring->host_base + c->saved_flags[3];
  if (e != cudaSuccess) { if (g) cudaGraphDestroy(g); return cuda_fail(c->err, e, "cudaStreamEndCapture"); }
  if (slot < 0 || slot >= 64) { cudaGraphDestroy(g); return fail(c->err, DFLASH_ERANGE, "slot %d outside [0, 64)", slot); }
  size_t nn = 0;
  long long kernels = 0;
  if (cudaGraphGetNodes(g, nullptr, &nn) == cudaSuccess && nn) {
    std::vector<cudaGraphNode_t> nodes(nn);
    if (cudaGraphGetNodes(g, nodes.data(), &nn) == cudaSuccess)
      for (size_t i = 0; i < nn; ++i) {
        cudaGraphNodeType t;
        if (cudaGraphNodeGetType(nodes[i], &t) == cudaSuccess && t == cudaGraphNodeTypeKernel) ++kernels;
      }
  }
  cudaGraphExec_t ex = nullptr;
  e = cudaGraphInstantiate(&ex, g, 0);
  cudaGraphDestroy(g);
  if (e != cudaSuccess) return cuda_fail(c->err, e, "cudaGraphInstantiate");
  if (c->graphs[slot]) cudaGraphExecDestroy(c->graphs[slot]);
  c->graphs[slot] = ex;
  c->graph_kernels[slot] = kernels;
  return DFLASH_OK;
}

int dflash_graph_launch(dflash_ctx* c, int32_t slot) {
  if (!c) return DFLASH_EINVAL;
  if (slot < 0 || slot >= 64 || !c->graphs[slot]) return fail(c->err, DFLASH_ESTATE, "graph slot %d is empty", slot);
  CK(c->err, cudaGraphLaunch(c->graphs[slot], c->stream));
  return DFLASH_OK;
}

int dflash_graph_kernel_count(dflash_ctx* c, int32_t slot, int64_t* out) {
  if (!c || !out) return DFLASH_EINVAL;
  if (slot < 0 || slot >= 64 || !c->graphs[slot]) return fail(c->err, DFLASH_ESTATE, "graph slot %d is empty", slot);
  *out = c->graph_kernels[slot];
  return DFLASH_OK;
}

int dflash_set_option(dflash_ctx* c, int32_t option, int64_t value) {
  if (!c) return DFLASH_EINVAL;
  if (option == DFLASH_OPT_KERNEL_TRACE) {
    if (value != 0 && value != 1) return fail(c->err, DFLASH_EINVAL, "option value %lld", (long long)value);
    if (value && !c->ktr) CK(c->err, cudaMalloc(&c->ktr, 3 * sizeof(unsigned long long) * kKTraceSlots));
    c->ktr_on = value != 0;
    return DFLASH_OK;
  }
  if (option == DFLASH_OPT_MARKOV_STEPWISE) {
    if (value != 0 && value != 1) return fail(c->err, DFLASH_EINVAL, "option value %lld", (long long)value);
    c->mk_stepwise = value != 0;
    return DFLASH_OK;
  }
  return fail(c->err, DFLASH_EINVAL, "unknown option %d", option);
}

int dflash_kernel_trace(dflash_ctx* c, uint64_t* out, int64_t capacity, int32_t* count, char* names,
                        int64_t names_cap) {
  if (!c) return DFLASH_EINVAL;
  if (!count) return fail(c->err, DFLASH_EINVAL, "count is NULL");
  if (!c->ktr) return fail(c->err, DFLASH_ESTATE, "kernel tracing was never enabled");
  *count = c->ktr_n;
  std::string joined;
  for (const auto& nm : c->ktr_names) joined += nm + "\n";
  if (!out || capacity < 3LL * c->ktr_n || !names || names_cap < (int64_t)joined.size() + 1)
    return fail(c->err, DFLASH_ERANGE, "need %d stamps and %zu name bytes", 3 * c->ktr_n, joined.size() + 1);
  std::vector<unsigned long long> h(3 * kKTraceSlots);
  CK(c->err, cudaMemcpyAsync(h.data(), c->ktr, h.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost,
                             c->stream));
  CK(c->err, cudaStreamSynchronize(c->stream));
  for (int i = 0; i < c->ktr_n; ++i)
    for (int k = 0; k < 3; ++k) out[3 * i + k] = h[(size_t)k * kKTraceSlots + i];
  std::memcpy(names, joined.c_str(), joined.size() + 1);
  return DFLASH_OK;
}

int dflash_get_option(dflash_ctx* c, int32_t option, int64_t* value) {
  if (!c) return DFLASH_EINVAL;
  if (!value) return fail(c->err, DFLASH_EINVAL, "value is NULL");
  if (option == DFLASH_OPT_KERNEL_TRACE) { *value = c->ktr_on ? 1 : 0; return DFLASH_OK; }
  if (option == DFLASH_OPT_MARKOV_STEPWISE) { *value = c->mk_stepwise ? 1 : 0; return DFLASH_OK; }
  return fail(c->err, DFLASH_EINVAL, "unknown option %d", option);
}

int dflash_lm_head_timing(dflash_ctx* c, int32_t enable) {
  if (!c) return DFLASH_EINVAL;
  c->lm_timing = enable != 0;
  return DFLASH_OK;
}

int dflash_lm_head_elapsed_ms(dflash_ctx* c, float* ms) {
  if (!c || !ms) return DFLASH_EINVAL;
  if (!c->lm_recorded) return fail(c->err, DFLASH_ESTATE, "lm_head timing events never recorded");
  CK(c->err, cudaEventSynchronize(c->lm_ev[1]));
  CK(c->err, cudaEventElapsedTime(ms, c->lm_ev[0], c->lm_ev[1]));
  return DFLASH_OK;
}

int dflash_ingest_gemm_timing(dflash_ctx* c, int32_t enable) {
  if (!c) return DFLASH_EINVAL;
  c->ing_timing = enable != 0;
  return DFLASH_OK;
}

int dflash_ingest_gemm_ms(dflash_ctx* c, float* fc_ms, float* kv_ms) {
  if (!c || !fc_ms || !kv_ms) return DFLASH_EINVAL;
  if (!c->ing_recorded) return fail(c->err, DFLASH_ESTATE, "ingest GEMM timing events never recorded");
  CK(c->err, cudaEventSynchronize(c->ing_ev[3]));
  CK(c->err, cudaEventElapsedTime(fc_ms, c->ing_ev[0], c->ing_ev[1]));
  CK(c->err, cudaEventElapsedTime(kv_ms, c->ing_ev[2], c->ing_ev[3]));
  return DFLASH_OK;
}

int dflash_sync(dflash_ctx* c) {
  if (!c) return DFLASH_EINVAL;
  CK(c->err, cudaStreamSynchronize(c->stream));
  return DFLASH_OK;
}

int dflash_synth_target(dflash_ctx* c, const void* logit_pool, const void* plant,
                        const uint8_t* coins, const void* resid_pool, int32_t n_logit_pool,
                        int32_t n_coin_rows, int32_t n_resid_pool, int32_t block_max, int32_t block,
                        const int32_t* draft_ids, void* logits_out, void* resid_out) {
  if (!c) return DFLASH_EINVAL;
  if (!logit_pool || !plant || !coins || !resid_pool || !draft_ids || !logits_out || !resid_out)
    return fail(c->err, DFLASH_EINVAL, "a stand-in target pointer is NULL");
  if (n_logit_pool < 1 || n_coin_rows < 1 || n_resid_pool < 1)
    return fail(c->err, DFLASH_EINVAL, "pool sizes must be positive");
  if (block < 2 || block > block_max || block > c->cfg.max_block)
    return fail(c->err, DFLASH_ERANGE, "block %d outside [2, min(block_max, max_block)]", block);
  SynthArgs a{};
  a.logit_pool = logit_pool; a.plant = plant; a.coins = coins; a.resid_pool = resid_pool;
  a.n_logit = n_logit_pool; a.n_coin = n_coin_rows; a.n_resid = n_resid_pool;
  a.block_max = block_max; a.block = block; a.V = c->V; a.kin = c->kin;
  a.d = draft_ids; a.logits_out = logits_out; a.resid_out = resid_out; a.rs = c->rs;
  a.nseq = c->nseq;
  a.trace = ktrace_slot(c, "synth_target");
  CK(c->err, launch_synth_target(c->dt, a, c->stream));
  return DFLASH_OK;
}

// ---- LFM2 short convolution ----------------------------------------------------------
namespace {
int short_conv_check(int32_t layers, int32_t lcache, int32_t channels, int32_t block, int32_t dtype) {
  if (layers < 1 || channels < 1 || block < 1 || dtype < 0 || dtype > 1) {
    g_create_err = "short conv: dimensions must be positive and dtype DFLASH_F32 or DFLASH_BF16";
    return DFLASH_EINVAL;
  }
  if (lcache < 2 || lcache > kShortConvMaxL) {
    g_create_err = "short conv: lcache outside [2, 16]";
    return DFLASH_ERANGE;
  }
  if ((int64_t)layers * channels * (block > lcache ? block : lcache) > kI32Max) {
    g_create_err = "short conv: a dimension product would wrap an int32";
    return DFLASH_EINVAL;
  }
  return DFLASH_OK;
}
}  // namespace

int dflash_short_conv_block(const void* state, const void* bx, const void* w, int32_t layers,
                            int32_t lcache, int32_t channels, int32_t block, int32_t dtype, void* y,
                            void* state_after, void* stream) {
  int rc = short_conv_check(layers, lcache, channels, block, dtype);
  if (rc) return rc;
  if (!bx || !w || !y) {
    g_create_err = "short conv: bx, w and y must not be NULL";
    return DFLASH_EINVAL;
  }
  cudaError_t e = launch_short_conv(dtype, state, bx, w, layers, lcache, channels, block, y, state_after,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(g_create_err, e, "short conv");
  return DFLASH_OK;
}

int dflash_short_conv_rollback(const void* prev_state, const void* bx, const int32_t* n_dev,
                               int32_t layers, int32_t lcache, int32_t channels, int32_t block,
                               int32_t dtype, void* state_out, void* stream) {
  int rc = short_conv_check(layers, lcache, channels, block, dtype);
  if (rc) return rc;
  if (!bx || !n_dev || !state_out) {
    g_create_err = "short conv rollback: bx, n_dev and state_out must not be NULL";
    return DFLASH_EINVAL;
  }
  cudaError_t e = launch_short_conv_rollback(dtype, prev_state, bx, n_dev, layers, lcache, channels, block,
                                             state_out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(g_create_err, e, "short conv rollback");
  return DFLASH_OK;
}

// ---- standalone ring ----------------------------------------------------------------
int ring_cache_create_ex(int32_t n_layers, int32_t kv_heads, int32_t head_dim, int32_t window,
                         int32_t max_block, int32_t dtype, int32_t max_context, int32_t flags,
                         void* stream, ring_cache** out) {
  return ring_create_impl(n_layers, kv_heads, head_dim, window, max_block, dtype, max_context,
                          flags, static_cast<cudaStream_t>(stream), out, g_create_err);
}

int ring_cache_create(int32_t n_layers, int32_t kv_heads, int32_t head_dim, int32_t window,
                      int32_t max_block, int32_t dtype, int32_t max_context, void* stream,
                      ring_cache** out) {
  return ring_cache_create_ex(n_layers, kv_heads, head_dim, window, max_block, dtype, max_context,
                              0, stream, out);
}

void ring_cache_destroy(ring_cache* r) {
  if (!r || r->owned_by_ctx) return;
  cudaStreamSynchronize(r->stream);
  ring_free(r);
}

int ring_cache_append(ring_cache* r, const void* k, const void* v, int32_t n) {
  if (!r) return DFLASH_EINVAL;
  if (n < 0 || n > r->cap) return fail(r->err, DFLASH_EINVAL, "n = %d outside [0, capacity=%lld]", n, r->cap);
  if (n == 0) return DFLASH_OK;
  if (!k || !v) return fail(r->err, DFLASH_EINVAL, "k or v is NULL");
  if (r->append_only && r->pos_hi + n - r->host_base > r->cap) {
    long long off;
    int rc = ring_sync_offset(r, &off);
    if (rc) return rc;
    r->pos_hi = off;
    if (off + n - r->host_base > r->cap)
      return fail(r->err, DFLASH_EFULL, "append-only ring full (%lld + %d > %lld)", off - r->host_base, n, r->cap);
  }
  CK(r->err, launch_ring_append(r->dtype, k, v, r->L, n, r->nkv, r->hd, r->k, r->v, r->cap, r->st,
                                r->stream));
  r->host_appended += n;
  r->pos_hi += n;
  return DFLASH_OK;
}

int ring_cache_trim(ring_cache* r, int32_t m) {
  if (!r) return DFLASH_EINVAL;
  if (m < 0) return fail(r->err, DFLASH_EINVAL, "trim of %d rows", m);
  if (m > r->host_appended)
    return fail(r->err, DFLASH_EREWIND, "short rewind: trim %d > %d rows appended since the last trim",
                m, r->host_appended);
  // A sliding ring keeps the rows behind the offset only for `slack` slots
  // past the window: rows appended beyond that have already overwritten
  // window rows that a rewind would make visible again.
  if (!r->append_only && m > r->cap - r->window)
    return fail(r->err, DFLASH_EREWIND,
                "trim %d > slack %lld: the window rows it would expose were overwritten", m,
                r->cap - r->window);
  CK(r->err, launch_ring_advance(r->st, m, 1, r->stream));
  r->host_appended = 0;
  r->pos_hi -= m;
  return DFLASH_OK;
}

int ring_cache_offset(ring_cache* r, int64_t* off) {
  if (!r || !off) return DFLASH_EINVAL;
  long long o;
  int rc = ring_sync_offset(r, &o);
  if (rc) return rc;
  *off = o;
  return DFLASH_OK;
}

int ring_cache_capacity(const ring_cache* r, int64_t* cap) {
  if (!r || !cap) return DFLASH_EINVAL;
  *cap = r->cap;
  return DFLASH_OK;
}

int ring_cache_gather(ring_cache* r, int64_t pos0, int32_t count, void* k_out, void* v_out) {
  if (!r) return DFLASH_EINVAL;
  if (!k_out || !v_out || count < 0 || pos0 < 0)
    return fail(r->err, DFLASH_EINVAL, "bad gather arguments");
  CK(r->err, launch_ring_gather(r->dtype, r->k, r->v, r->L, r->cap, r->nkv, r->hd, pos0, count,
                                k_out, v_out, r->stream));
  return DFLASH_OK;
}

const char* ring_cache_last_error(const ring_cache* r) { return r ? r->err.c_str() : g_create_err.c_str(); }

// ---- the synthetic target ------------------------------------------------------

int dflash_target_create(const dflash_target_config* tc, const dflash_target_weights* tw, void* stream,
                         dflash_ctx** out) {
  std::string& err = g_create_err;
  if (!out) return fail(err, DFLASH_EINVAL, "out is NULL");
  *out = nullptr;
  if (!tc || !tw || !tw->embed || !tw->final_norm || !tw->lm_head || !tw->layers)
    return fail(err, DFLASH_EINVAL, "a target config or weight pointer is NULL");
  if (tc->n_layers < 1 || tc->n_layers > 64) return fail(err, DFLASH_ERANGE, "n_layers outside [1, 64]");
  if (tc->window <= 0) return fail(err, DFLASH_EINVAL, "the sliding layers need a window > 0");
  if (tc->max_block < 2 || tc->max_block > 32) return fail(err, DFLASH_ERANGE, "max_block outside [2, 32]");
  if (tc->n_capture < 1 || tc->n_capture > 8) return fail(err, DFLASH_ERANGE, "n_capture outside [1, 8]");
  for (int j = 0; j < tc->n_capture; ++j)
    if (tc->capture[j] < 0 || tc->capture[j] >= tc->n_layers)
      return fail(err, DFLASH_ERANGE, "capture layer %d outside [0, %d)", tc->capture[j], tc->n_layers);
  if (tc->n_layers < 64 && (tc->full_layers >> tc->n_layers))
    return fail(err, DFLASH_ERANGE, "full_layers names a layer past n_layers");
  const int n_full = __builtin_popcountll(tc->full_layers);
  if (n_full && tc->max_context < tc->max_block)
    return fail(err, DFLASH_ERANGE, "max_context must hold at least max_block rows");
  // the drafter's context machinery with a zeroed stand-in for its encoder.fc
  // (a target never ingests residual rows)
  dflash_config cfg{};
  cfg.n_layers = tc->n_layers; cfg.hidden = tc->hidden; cfg.n_q_heads = tc->n_q_heads;
  cfg.n_kv_heads = tc->n_kv_heads; cfg.head_dim = tc->head_dim; cfg.intermediate = tc->intermediate;
  cfg.vocab = tc->vocab; cfg.window = tc->window; cfg.k_target_layers = 1; cfg.target_hidden = 64;
  cfg.mask_token_id = 0; cfg.rope_neox = tc->rope_neox; cfg.max_block = tc->max_block;
  cfg.kind = DFLASH_KIND_DFLASH; cfg.dtype = tc->dtype; cfg.max_context = tc->max_context;
  cfg.rope_theta = tc->rope_theta; cfg.rms_eps = tc->rms_eps;
  const size_t esz = tc->dtype == DFLASH_BF16 ? 2 : 4;
  void* fc = nullptr;
  cudaError_t e = cudaMalloc(&fc, (size_t)tc->hidden * 64 * esz);
  if (e != cudaSuccess) return cuda_fail(err, e, "target allocation");
  if ((e = cudaMemset(fc, 0, (size_t)tc->hidden * 64 * esz)) != cudaSuccess) {
    cudaFree(fc);
    return cuda_fail(err, e, "target allocation");
  }
  dflash_weights w{};
  w.embed = tw->embed; w.fc = fc; w.hidden_norm = tw->final_norm; w.final_norm = tw->final_norm;
  w.lm_head = tw->lm_head; w.layers = tw->layers;
  dflash_ctx* c = nullptr;
  int rc = ctx_create_impl(&cfg, &w, 1, stream, &c, n_full ? tc->max_context : 0);
  if (rc) { cudaFree(fc); return rc; }
  c->fc_unused = fc;
  c->is_target = true;
  c->full_idx.assign(tc->n_layers, -1);
  for (int l = 0, k = 0; l < tc->n_layers; ++l)
    if ((tc->full_layers >> l) & 1) c->full_idx[l] = k++;
  c->capture.assign(tc->capture, tc->capture + tc->n_capture);
  if (n_full) {
    rc = ring_create_impl(n_full, c->nkv, c->hd, 0, tc->max_block, tc->dtype, tc->max_context, 0, c->stream,
                          &c->ring_full, err);
    if (rc) { dflash_ctx_destroy(c); return rc; }
  }
  if ((e = cudaMalloc(&c->tok, sizeof(int) * tc->max_block)) != cudaSuccess) {
    dflash_ctx_destroy(c);
    return cuda_fail(err, e, "target allocation");
  }
  c->has_context = true;
  *out = c;
  return DFLASH_OK;
}

int dflash_target_forward(dflash_ctx* c, const int32_t* tokens, int32_t rows, int32_t logit_rows, void* logits,
                          void* captured) {
  if (!c) return DFLASH_EINVAL;
  if (!c->is_target) return fail(c->err, DFLASH_EINVAL, "not a target context (dflash_target_create)");
  if (!tokens) return fail(c->err, DFLASH_EINVAL, "tokens is NULL");
  if (rows < 1 || rows > c->cfg.max_block)
    return fail(c->err, DFLASH_ERANGE, "rows %d outside [1, max_block=%d]", rows, c->cfg.max_block);
  if (logit_rows < 0 || logit_rows > rows)
    return fail(c->err, DFLASH_ERANGE, "logit_rows %d outside [0, rows=%d]", logit_rows, rows);
  if ((logit_rows > 0) != (logits != nullptr))
    return fail(c->err, DFLASH_EINVAL, "logits must be given exactly when logit_rows > 0");
  if ((logits && !aligned16(logits)) || (captured && !aligned16(captured)))
    return fail(c->err, DFLASH_EINVAL, "logits and captured must be 16-byte aligned");
  if (c->ring_full) {
    int rc = ensure_room(c, rows, c->ring_full);
    if (rc) return rc;
  }
  const int dt = c->dt;
  cudaStream_t st = c->stream;
  CK(c->err, launch_rope_table(c->inv_freq, c->half, c->ring->st, 0, rows, c->rope, st));
  CK(c->err, launch_embed_tokens(dt, c->embed, c->H, c->V, tokens, rows, c->x, c->rs, st));
  c->cap_out = captured;
  for (int l = 0; l < c->cfg.n_layers; ++l) {
    int rc = layer_forward(c, l, rows);
    if (rc) { c->cap_out = nullptr; return rc; }
  }
  const bool tc = tc_rows(c, rows);
  if (tc) {
    CK(c->err, launch_resid_rmsnorm(c->x, c->H, c->acc, c->H, c->final_norm, c->xf, c->H, rows, c->H,
                                    c->cfg.rms_eps, st, ktrace_slot(c, "final_norm")));
    int rc = capture_stream(c, c->cfg.n_layers - 1, rows);
    if (rc) { c->cap_out = nullptr; return rc; }
  } else {
    CK(c->err, launch_rmsnorm(dt, c->x, c->H, c->final_norm, c->xf, c->H, rows, c->H, c->cfg.rms_eps, st,
                              ktrace_slot(c, "final_norm")));
  }
  c->cap_out = nullptr;
  if (logit_rows > 0) {
    const void* xf = static_cast<const char*>(c->xf) + (size_t)(rows - logit_rows) * c->H * c->esz;
    if (tc) {
      TcGemmArgs t = tc_args(c, logit_rows, c->V, c->H, kEpiStore);
      tc_segments(t, {{&c->lm_map, c->V}});
      if (!tc_encode_map(&t.b_map, xf, c->H, logit_rows, (uint64_t)c->H * 2, 64, bn_of(logit_rows)))
        return fail(c->err, DFLASH_ECUDA, "cuTensorMapEncodeTiled failed for the final-normed rows");
      t.y = logits; t.ldy = c->V;
      t.trace = ktrace_slot(c, "target_logits", 4);
      CK(c->err, tc_run(c, t));
    } else {
      LinearArgs a = lin_args(xf, c->H, logits, c->V, logit_rows, c->V, c->H);
      a.w[0] = c->lm_head;
      CK(c->err, launch_linear_rows(dt, a, st));
    }
  }
  CK(c->err, launch_ring_advance(c->ring->st, rows, 0, st));
  if (c->ring_full) {
    CK(c->err, launch_ring_advance(c->ring_full->st, rows, 0, st));
    c->ring_full->pos_hi += rows;
  }
  return DFLASH_OK;
}

int dflash_target_verify(dflash_ctx* c, const dflash_ctx* drafter, int32_t block, const int32_t* draft_ids,
                         void* logits, void* captured) {
  if (!c || !drafter) return DFLASH_EINVAL;
  if (!c->is_target || drafter->is_target)
    return fail(c->err, DFLASH_EINVAL, "needs a target context and a drafter context");
  if (drafter->nseq != 1) return fail(c->err, DFLASH_EINVAL, "the drafter must run one sequence");
  if (drafter->stream != c->stream) return fail(c->err, DFLASH_EINVAL, "the drafter and the target must share a stream");
  if (!draft_ids || !logits) return fail(c->err, DFLASH_EINVAL, "draft_ids or logits is NULL");
  if (block < 2 || block > c->cfg.max_block)
    return fail(c->err, DFLASH_ERANGE, "block %d outside [2, max_block=%d]", block, c->cfg.max_block);
  CK(c->err, launch_verify_tokens(drafter->rs, drafter->ring->st, draft_ids, block, c->tok, c->ring->st, c->rs,
                                  c->stream));
  return dflash_target_forward(c, c->tok, block, block, logits, captured);
}

int dflash_target_commit(dflash_ctx* c, const int32_t* n_dev, int32_t block) {
  if (!c) return DFLASH_EINVAL;
  if (!c->is_target) return fail(c->err, DFLASH_EINVAL, "not a target context (dflash_target_create)");
  if (!n_dev) return fail(c->err, DFLASH_EINVAL, "n_dev is NULL");
  if (block < 1 || block > c->cfg.max_block)
    return fail(c->err, DFLASH_ERANGE, "block %d outside [1, max_block=%d]", block, c->cfg.max_block);
  CK(c->err, launch_target_trim(c->ring->st, c->ring_full ? c->ring_full->st : nullptr, n_dev, block, c->rs,
                                c->stream));
  return DFLASH_OK;
}

int dflash_target_full_ring(dflash_ctx* c, ring_cache** out) {
  if (!c || !out) return DFLASH_EINVAL;
  if (!c->is_target) return fail(c->err, DFLASH_EINVAL, "not a target context (dflash_target_create)");
  *out = c->ring_full;
  return DFLASH_OK;
}

}  // extern "C"
