/*
 * dflash.h -- C ABI of libdflash: one DFlash speculative round at batch 1 on
 * a single GB300 (sm_103a).
 *
 * Sources, cited by page title and section:
 *   [Muse]   "Muse Glimmer DFlash assistant drafter on the round loop"
 *            (mlxcel pull request 1762)
 *   [Head]   "Load Meta's Muse-Glimmer-30B-assistant DFlash head via a
 *            draft-adapter registry" (z-lab/dflash pull request 168)
 *   [DSpark] "LFM2 / LFM2.5 DSpark drafter on the DFlash loop"
 *            (mlxcel pull request 1751)
 *
 * Conventions for every call:
 *   - All tensor arguments are DEVICE pointers unless the name ends in _host.
 *     They are borrowed: the caller owns them and keeps them alive while the
 *     enqueued work runs. Tensors are dense row-major; linear weights are
 *     [out_features, in_features]. Element type is the config's dtype
 *     (fp32 or bf16) unless stated. Every tensor pointer must be 16-byte
 *     aligned.
 *   - Every call that takes a context enqueues its GPU work on the context's
 *     stream and returns without waiting, except the calls marked "syncs".
 *     The round calls allocate nothing and never synchronize, so a caller may
 *     capture whole rounds into a CUDA graph (dflash_capture_begin / _end /
 *     dflash_graph_launch).
 *   - Every call returns a status (DFLASH_OK == 0) and never aborts or throws
 *     [Muse "Pre-merge review round", third finding; DSpark "Security fixes":
 *     a bad checkpoint value must be a request error, not a process abort].
 *     The context keeps the message of its last error (dflash_last_error).
 *     Arguments are checked on the host before any GPU work is enqueued.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
enum {
  DFLASH_OK = 0,
  DFLASH_EINVAL = 1,  /* null pointer, bad dtype/kind, dimension <= 0, a
                         dimension product that would wrap an int32, bad
                         alignment [Muse "Pre-merge review round", third
                         finding: config dimensions bounded as i32] */
  DFLASH_ERANGE = 2,  /* token id outside [0, vocab), mask_token_id >= vocab,
                         block < 2 or block > max_block, Markov shape mismatch
                         [DSpark "Review fixes": mask id and width bounds,
                         Markov factor shapes] */
  DFLASH_EREWIND = 3, /* trim longer than the rows appended since the last
                         trim: the "short rewind" [Muse "Pre-merge review
                         round", second finding] */
  DFLASH_EEMPTY = 4,  /* empty context where a draft needs one, or zero rows
                         [DSpark "Security fixes": empty prompt / window] */
  DFLASH_ECUDA = 5,   /* a CUDA call failed; dflash_last_error has its text */
  DFLASH_ESTATE = 6,  /* call out of order (commit before append, capture
                         misuse, unknown graph slot) */
  DFLASH_EFULL = 7    /* an unbounded-window (append-only) cache is out of
                         rows (config.max_context) */
};

enum { DFLASH_F32 = 0, DFLASH_BF16 = 1 };
enum { DFLASH_KIND_DFLASH = 0, DFLASH_KIND_DSPARK = 1 };

/* Number of weight pointers per drafter layer in dflash_weights.layers, in
 * this order: in_norm[H], wq[nq*hd, H], wk[nkv*hd, H], wv[nkv*hd, H],
 * q_norm[hd], k_norm[hd], wo[H, nq*hd], post_norm[H], wg[I, H], wu[I, H],
 * wd[H, I]. */
#define DFLASH_LAYER_TENSORS 11

typedef struct dflash_config {
  int32_t n_layers;        /* drafter layers (5 on every page) */
  int32_t hidden;          /* H, a multiple of 8 */
  int32_t n_q_heads;       /* nq */
  int32_t n_kv_heads;      /* nkv; nq % nkv == 0 (grouped-query attention) */
  int32_t head_dim;        /* hd, a multiple of 8, at most 256 */
  int32_t intermediate;    /* I (SwiGLU), a multiple of 8 */
  int32_t vocab;           /* V */
  int32_t window;          /* W of the bidirectional sliding mask |q-k| <= W
                              [Muse "What changed"]; <= 0: no mask and an
                              append-only cache [DSpark "Verified against the
                              issue": mask None, append-only] */
  int32_t k_target_layers; /* captured target residual streams (5) */
  int32_t target_hidden;   /* width of each captured stream; k * width is a
                              multiple of 8 */
  int32_t mask_token_id;   /* < vocab [DSpark "Review fixes"] */
  int32_t rope_neox;       /* 1: neox pairs (i, i+hd/2); 0: traditional
                              pairs (2i, 2i+1) [DSpark "Verified against
                              the issue": rope_is_neox_style false] */
  int32_t max_block;       /* largest verify width B any round will use
                              (2..1024); sizes the ring slack and scratch */
  int32_t kind;            /* DFLASH_KIND_DFLASH: block of B rows, rows
                              1..B-1 read out; DFLASH_KIND_DSPARK: block of
                              B-1 rows, every row read out [DSpark
                              "Verified against the issue"] */
  int32_t markov_rank;     /* r of the DSpark Markov head, 0 = none */
  int32_t markov_add;      /* 0: proposals are argmax(W1[prev].W2); 1:
                              argmax(z_j + W1[prev].W2) over the lm_head
                              logits z_j */
  int32_t dtype;           /* DFLASH_F32 or DFLASH_BF16, for weights, inputs,
                              activations and the ring; accumulation is fp32 */
  int32_t max_context;     /* window <= 0 only: rows the append-only cache
                              holds; ignored for a sliding window */
  float rope_theta;        /* RoPE base (1e6 on the pages' drafters) */
  float rms_eps;           /* RMSNorm epsilon */
  float softcap;           /* c of c*tanh(z/c) on the drafter logits, 0 = off
                              [Head "How": inherited final_logit_softcapping] */
} dflash_config;

typedef struct dflash_weights {
  const void* embed;        /* [V, H] the target's raw embedding table
                               [Muse "What changed"; "Real-checkpoint
                               validation" item 5: not the embed_norm lookup] */
  const void* fc;           /* [H, k*target_hidden] encoder.fc */
  const void* hidden_norm;  /* [H] encoder.output_norm_enc */
  const void* final_norm;   /* [H] RMSNorm gain before the lm_head */
  const void* lm_head;      /* [V, H]; may equal embed (tied, as DSpark) */
  const void* markov_w1;    /* [V, r] or NULL when markov_rank == 0 */
  const void* markov_w2;    /* [r, V] or NULL when markov_rank == 0 */
  const void* const* layers;/* HOST array of n_layers * DFLASH_LAYER_TENSORS
                               device pointers; copied at create */
} dflash_weights;

typedef struct dflash_stats {
  int64_t rounds;     /* draft_rounds */
  int64_t draft_n;    /* proposals made (block - 1 per round) */
  int64_t accepted;   /* draft_n_accepted: sum of a */
  int64_t emitted;    /* tokens emitted by verifies: sum of n = a + 1 */
} dflash_stats;

typedef struct dflash_round_state {
  int64_t position;   /* absolute position of the current anchor; equals the
                         committed context length */
  int32_t anchor;     /* the current anchor token */
  int32_t last_n;     /* n of the last verify (accepted + 1) */
  int32_t last_accepted; /* a of the last verify */
  int32_t error;      /* device-side error bits: 1 = append-only cache full
                         (rows skipped), 2 = a token id outside the vocabulary
                         reached the embedding gather (row 0 used), 4 = a
                         bounded wait in a tensor-core kernel gave up, 8 = a
                         draft's anchor_pos was not the committed length */
} dflash_round_state;

typedef struct dflash_ctx dflash_ctx;
typedef struct ring_cache ring_cache;

/* ---- pure host helpers -------------------------------------------------- */

/* Speculative slack rows for a verify block: max(clamp(8*block, 32, 128),
 * block) [Muse "Pre-merge review round", second finding]. Returns -1 for
 * block < 1. */
int32_t dflash_speculative_slack(int32_t block);

/* Derived round counters. accepted_per_round = accepted / rounds (the Muse
 * page's "mean accepted"); emitted_per_round = accepted / rounds + 1 (the
 * DSpark page's "mean accepted length"); acceptance = accepted / draft_n.
 * Any output pointer may be NULL. EINVAL if stats is NULL or a denominator
 * is zero. */
int dflash_stats_ratios(const dflash_stats* stats, double* accepted_per_round,
                        double* emitted_per_round, double* acceptance);

/* Validates a config without touching the GPU (the same checks as create). */
int dflash_config_check(const dflash_config* cfg);

/* ---- context lifecycle --------------------------------------------------- */

/* Creates a drafter context on the current CUDA device: validates cfg and the
 * weight pointers, copies the layer pointer table, allocates the ring
 * (window + slack(max_block) rows per layer, or max_context rows for an
 * unbounded window) and all scratch in device memory owned by the context.
 * stream is a cudaStream_t (NULL: the legacy default stream). On failure *out
 * is NULL and the status says why (text: dflash_last_error(NULL)). */
int dflash_ctx_create(const dflash_config* cfg, const dflash_weights* w,
                      void* stream, dflash_ctx** out);
void dflash_ctx_destroy(dflash_ctx* ctx);

/* ---- batched rounds ------------------------------------------------------------ */

/* A context for n_seq sequences drafted, verified and committed together,
 * the batched mode the Muse page leaves out ["Muse Glimmer DFlash assistant
 * drafter on the round loop", "Not in this PR": batched (B > 1) windows
 * decline through supports_batched()]. The sequences share the drafter's
 * forward: every linear layer streams its weights once for the n_seq * block
 * rows of a round. Each sequence has its own ring (window + slack rows),
 * anchor, position and counters. The round calls keep their meaning with
 * sequence-major tensors: dflash_draft_block writes draft_ids [n_seq][block-1]
 * (anchor and anchor_pos must be -1: each sequence drafts from its device
 * anchor), dflash_verify_accept takes target_logits [n_seq][block][V] and
 * draft_ids [n_seq][block-1] and writes tokens [n_seq][block] and n
 * [n_seq], dflash_append_block takes resid [n_seq][block][k*target_hidden],
 * dflash_commit(ctx, -1) keeps each sequence's own n (a keep >= 0 applies to
 * all), dflash_sync_round and dflash_synth_target are per sequence in the same
 * layout (the stand-in target draws pool entry round * n_seq + s for sequence
 * s). Sequences are ingested one by one (dflash_ingest_context_seq); a draft
 * needs all of them. Needs 1 <= n_seq <= 64, n_seq * max_block <= 1024, a
 * sliding window (window > 0) and no Markov head (EINVAL / ERANGE
 * otherwise); the sampled verify and the Markov chain take one sequence.
 * dflash_ctx_create is dflash_ctx_create_batched with n_seq = 1. */
int dflash_ctx_create_batched(const dflash_config* cfg, const dflash_weights* w, int32_t n_seq,
                              void* stream, dflash_ctx** out);
/* Sequences per round of the context (1 for dflash_ctx_create). */
int dflash_batch_size(const dflash_ctx* ctx);
/* dflash_ingest_context for sequence seq (0 <= seq < n_seq; ERANGE
 * otherwise); dflash_ingest_context is seq 0. */
int dflash_ingest_context_seq(dflash_ctx* ctx, int32_t seq, const void* resid, int64_t rows,
                              int64_t first_pos, int32_t anchor);

/* Text of the last error on this context (or of the last failed create when
 * ctx is NULL). Never NULL. */
const char* dflash_last_error(const dflash_ctx* ctx);

/* ---- the round ------------------------------------------------------------ */

/* Ingests captured residual rows resid [rows, k*target_hidden] at absolute
 * positions first_pos .. first_pos+rows-1 and sets the next anchor to
 * `anchor` at position first_pos + rows. Rows older than the window (position
 * < first_pos + rows - W) are dropped before encoder.fc [Muse "Pre-merge
 * review round", third finding]; the kept rows go through fc ->
 * hidden_norm -> per-layer Wk/Wv -> k-norm + RoPE into the ring. Replaces any
 * earlier context. EEMPTY if rows == 0; ERANGE if anchor is out of range;
 * EFULL if an append-only cache cannot hold the kept rows. */
int dflash_ingest_context(dflash_ctx* ctx, const void* resid, int64_t rows,
                          int64_t first_pos, int32_t anchor);

/* Replaces the device-resident anchor token (the position is unchanged). */
int dflash_set_anchor(dflash_ctx* ctx, int32_t anchor);

/* Drafts one block of verify width `block` from the anchor token at absolute
 * position anchor_pos [Muse "What changed"; DSpark "Verified against the
 * issue"]: embeds [anchor, mask x (rows-1)] from the raw embedding table,
 * runs the drafter layers (per-head q/k RMSNorm, RoPE at absolute positions,
 * bidirectional sliding attention over the ring plus the block), the final
 * norm, the lm_head with softcap and the per-row argmax (no [rows, V] logit
 * tensor is written), and for a config with a Markov head the chain.
 * Writes block-1 proposals d_1..d_{block-1} to draft_ids [block-1] (int32).
 *
 * anchor < 0 takes the device-resident anchor (set by dflash_ingest_context,
 * dflash_set_anchor or the last dflash_commit: the bonus token t_a), which
 * is what lets whole rounds run from a CUDA graph with nothing passed from
 * the host; anchor >= 0 replaces it. The position is always the committed
 * context length held on the device (the ring offset): every row of the
 * ring is addressed by it, so it cannot be set per call. anchor_pos < 0
 * skips the check; anchor_pos >= 0 is compared with it on the device and a
 * mismatch sets error bit 8 of dflash_round_state (the draft still runs at
 * the committed position).
 * ERANGE unless 2 <= block <= max_block and anchor < vocab; EEMPTY if no
 * context was ingested. */
int dflash_draft_block(dflash_ctx* ctx, int32_t anchor, int64_t anchor_pos, int32_t block,
                       int32_t* draft_ids);

/* Greedy exact-match verify [DSpark intro; "Short-conv rollback"]: t_i =
 * argmax target_logits[i, :] (lowest index on ties) for i < block; a = the
 * longest prefix with draft_ids[i] == t_i; writes tokens [block] (int32)
 * = d_1..d_a, t_a, followed by -1 padding, and n [1] (int32) = a + 1.
 * target_logits is [block, V] in the config dtype. Keeps n, a and the bonus
 * token t_a on the device for dflash_commit. */
int dflash_verify_accept(dflash_ctx* ctx, const void* target_logits,
                         int32_t block, const int32_t* draft_ids,
                         int32_t* tokens, int32_t* n);

/* Appends the verify block's captured residual rows resid [block,
 * k*target_hidden] at positions p .. p+block-1 (p = device position) into the
 * ring through fc -> hidden_norm -> Wk/Wv -> k-norm + RoPE; like
 * ring_cache_append, the offset advances by block until dflash_commit trims
 * it. ERANGE unless 1 <= block <= max_block. */
int dflash_append_block(dflash_ctx* ctx, const void* resid, int32_t block);

/* Partial-accept rollback: keeps the first `keep` appended rows and trims
 * the other block - keep (KVCache::trim(block - n) [DSpark "Short-conv
 * rollback"]); keep < 0 takes n from the last verify. The anchor becomes the
 * verify's bonus token and the counters advance. EINVAL if keep > block;
 * ESTATE without an append since the last commit. */
int dflash_commit(dflash_ctx* ctx, int32_t keep);

/* The one host synchronization of a round: waits for the context's stream
 * and copies what the last dflash_verify_accept wrote (to its tokens and n
 * device buffers) into host memory: n_host [1] = a + 1 and tokens_host
 * [block] = d_1..d_a, t_a, then -1 padding (block = that verify's width)
 * [DSpark "Implementation Review Summary": one materialisation of the
 * argmax per round]. Syncs. ESTATE before any verify or while capturing. */
int dflash_sync_round(dflash_ctx* ctx, int32_t* tokens_host, int32_t* n_host);

/* Speculative-sampling verify at temperature T > 0, the counterpart of
 * dflash_verify_accept for sampled decoding ["Load Meta's
 * Muse-Glimmer-30B-assistant DFlash head", "Measured": the sampled-acceptance
 * run at T = 1]. The drafter proposes its argmaxes, so its proposal
 * distribution is a point mass on d_{i+1} and the speculative-sampling rule
 * min(1, p/q) accepts d_{i+1} iff uniforms[i] < p_i(d_{i+1}), with p_i =
 * softmax(c * tanh(target_logits[i] / c) / temperature) (c = softcap, 0 =
 * no cap). a = the accepted prefix; the bonus token is drawn by inverse CDF
 * in vocabulary order with uniforms[block - 1], from p_a without d_{a+1}
 * after a rejection (the residual max(p - q, 0)), from p_{block-1} after a
 * full accept. The emitted tokens then follow the target distribution
 * exactly. Writes tokens [block] = d_1..d_a, bonus, then -1 padding, n [1] =
 * a + 1 and, when p_draft is not NULL, p_draft [block] = p_i(d_{i+1}) (0 for
 * the last row). uniforms [block] fp32 in [0, 1) are caller-drawn (device).
 * Keeps n, a and the bonus on the device for dflash_commit like the greedy
 * verify. Top-k / top-p filtering is not applied. ERANGE unless 2 <= block
 * <= max_block; EINVAL for a NULL pointer, temperature <= 0 or softcap < 0. */
int dflash_verify_sampled(dflash_ctx* ctx, const void* target_logits, int32_t block,
                          const int32_t* draft_ids, const float* uniforms, float temperature,
                          float softcap, int32_t* tokens, int32_t* n, float* p_draft);

/* One whole round: draft_block (device anchor), verify_accept, append_block,
 * commit(-1). */
int dflash_round(dflash_ctx* ctx, const void* target_logits, const void* resid,
                 int32_t block, int32_t* draft_ids, int32_t* tokens,
                 int32_t* n);

/* DSpark Markov chain alone [DSpark "Verified against the issue": seeded
 * with the anchor, each step's argmax feeds the next step's W1 gather]:
 * out[j] = argmax_v (z[j, v] + W1[prev] . W2[:, v]) with prev = anchor for
 * j = 0 and out[j-1] after; z is [gamma, V] fp32 or NULL (then 0).
 * ERANGE if the context has no Markov head, anchor is out of range or gamma
 * is outside 1..max_block. */
int dflash_markov_chain(dflash_ctx* ctx, int32_t anchor, int32_t gamma,
                        const float* z, int32_t* out);

/* ---- single ops of the round (same kernels, same stream) --------------------- */

/* One linear layer of the drafter on the context's stream and scratch:
 * y[m, n] = rnd(sum_k x[m, k] w[n, k]) (epi 0), rnd(r[m, n] + rnd(...))
 * (epi 1, r may alias y), or rnd(silu(rnd(x.w^T)) * rnd(x.w2^T)) (epi 2,
 * the SwiGLU of Qwen-shaped MLPs [Head "Why"]); x [M, K], w and w2 [N, K],
 * r and y [M, N], all dense in the config dtype, accumulation fp32. bf16
 * with K % 64 == 0 runs on the tensor cores: M <= 32 as a weight-streaming
 * GEMM, M > 32 (epi 0, N % 256 == 0) as the many-row GEMM of the context
 * ingest. */
int dflash_linear(dflash_ctx* ctx, const void* x, int32_t M, int32_t K,
                  const void* w, const void* w2, int32_t N, const void* r,
                  void* y, int32_t epi);
/* The fused lm_head of dflash_draft_block on given rows: for x [rows, H]
 * (normed hidden rows), ids[m] = argmax_v c*tanh((x[m].lm_head[v])/c) (c =
 * softcap, 0 = no cap; lowest index on ties) and maxv[m] the selected value
 * (fp32). No [rows, V] logit tensor is written. 1 <= rows <= max_block. */
int dflash_lm_head_argmax(dflash_ctx* ctx, const void* x, int32_t rows,
                          int32_t* ids, float* maxv);

/* ---- inspection (these sync) ------------------------------------------------- */

/* Copies the final-normed hidden rows of the last draft [rows, H] (rows =
 * block for DFlash, block - 1 for DSpark) into out (device). */
int dflash_get_hidden(dflash_ctx* ctx, void* out);
/* Copies the softcapped maximum logit of each read-out row of the last draft
 * [block - 1] (fp32, device): the value the argmax selected. */
int dflash_get_draft_max_logit(dflash_ctx* ctx, float* out);
/* Copies the lm_head argmax ids of the last draft's read-out rows (before
 * any Markov chain) [block - 1] (int32, device). */
int dflash_get_backbone_ids(dflash_ctx* ctx, int32_t* out);
/* State and counters of sequence 0 (syncs); the _seq forms take any
 * sequence of a batch (ERANGE outside [0, n_seq)). dflash_reset_stats clears
 * the counters of every sequence. */
int dflash_get_state(dflash_ctx* ctx, dflash_round_state* out_host);
int dflash_get_stats(dflash_ctx* ctx, dflash_stats* out_host);
int dflash_get_state_seq(dflash_ctx* ctx, int32_t seq, dflash_round_state* out_host);
int dflash_get_stats_seq(dflash_ctx* ctx, int32_t seq, dflash_stats* out_host);
int dflash_reset_stats(dflash_ctx* ctx);
/* The context's ring, or sequence seq's ring of a batch (borrowed; owned and
 * destroyed by the context). */
int dflash_ring(dflash_ctx* ctx, ring_cache** out);
int dflash_ring_seq(dflash_ctx* ctx, int32_t seq, ring_cache** out);

/* ---- CUDA graphs of whole rounds -------------------------------------------- */

/* Begins stream capture on the context's stream. Calls made until
 * dflash_capture_end are recorded, not run. */
int dflash_capture_begin(dflash_ctx* ctx);
/* Ends the capture and instantiates it into graph slot `slot` (0..63),
 * replacing what the slot held. */
int dflash_capture_end(dflash_ctx* ctx, int32_t slot);
/* Launches graph slot `slot` on the context's stream. */
int dflash_graph_launch(dflash_ctx* ctx, int32_t slot);
/* Waits for the context's stream (syncs). */
int dflash_sync(dflash_ctx* ctx);
/* Number of kernel launches graph slot `slot` holds (its kernel nodes). */
int dflash_graph_kernel_count(dflash_ctx* ctx, int32_t slot, int64_t* out_host);

/* ---- options ------------------------------------------------------------------ */

/* DFLASH_OPT_KERNEL_TRACE: 1 makes dflash_draft_block on the one-kernel-per-
 * operation path (and the dflash_append_block that follows it) stamp the
 * GPU's global timer (ns) for each traced launch:
 * earliest CTA entry, latest return from the wait on the preceding kernel,
 * latest CTA exit (allocates 6 KB on first use; 0 stops it). Read with
 * dflash_kernel_trace. */
#define DFLASH_OPT_KERNEL_TRACE 4
/* DFLASH_OPT_MARKOV_STEPWISE: 1 runs the DSpark Markov chain one launch per
 * step instead of the one cooperative launch that holds W2 in shared memory
 * (the fallback where W2 does not fit; same results); 0 (default) takes the
 * cooperative launch where it fits. */
#define DFLASH_OPT_MARKOV_STEPWISE 8
/* EINVAL for an unknown option or value. Takes effect from the next call. */
int dflash_set_option(dflash_ctx* ctx, int32_t option, int64_t value);
int dflash_get_option(dflash_ctx* ctx, int32_t option, int64_t* value_host);
/* The kernel trace of the last traced dflash_draft_block: count entries,
 * out_host [count][3] stamps (entry, wait return, exit) and names_host their
 * newline-separated names (e.g. "L0.qkv"). A weight-streaming GEMM "X" adds
 * entries for phases of its latest CTA: "X.1" [1] last MMA issued, [2] own
 * tiles published; "X.2" [1] split-tile contributors present, [2] finished;
 * "X.3" [1] split groups reduced. An attention "L<l>.attn" adds "L<l>.attn.1",
 * its split-merge kernel (entry, wait return, exit). Unused stamps read as
 * their reset value (all ones for [0], zero otherwise). Syncs the context's
 * stream.
 * ERANGE if out_host / names_host are NULL or too small (count is still
 * set); ESTATE if tracing was never enabled. */
int dflash_kernel_trace(dflash_ctx* ctx, uint64_t* out_host, int64_t capacity, int32_t* count,
                        char* names_host, int64_t names_capacity);

/* ---- measurement ------------------------------------------------------------- */

/* When enabled, dflash_draft_block brackets its lm_head kernel with two CUDA
 * events owned by the context, recorded on the context's stream (as event nodes when the
 * draft is being captured into a graph). */
int dflash_lm_head_timing(dflash_ctx* ctx, int32_t enable);
/* Milliseconds between the two events as last recorded (syncs on the end
 * event). ESTATE if they were never recorded. */
int dflash_lm_head_elapsed_ms(dflash_ctx* ctx, float* ms_host);

/* When enabled, dflash_ingest_context brackets the tensor-core context GEMMs
 * of each ingest chunk (encoder.fc over the chunk's rows; the K|V projections
 * of every layer) with context-owned CUDA events (event nodes when captured).
 * Applies to the 128 x 256 tensor-core ingest path only. */
int dflash_ingest_gemm_timing(dflash_ctx* ctx, int32_t enable);
/* Milliseconds of the fc GEMM and of the K|V GEMM(s) of the last recorded
 * chunk (syncs on the last event). ESTATE if never recorded. */
int dflash_ingest_gemm_ms(dflash_ctx* ctx, float* fc_ms_host, float* kv_ms_host);

/* ---- verify without allocation ------------------------------------------------ */

/* The greedy verify of dflash_verify_accept for callers that cannot allocate
 * device memory: no context (creating one allocates), no cudaMalloc, no
 * cudaFree, no allocating library call. Meant for code whose device memory
 * all comes from a host framework's own pool, or for a latency-critical loop
 * that must never pay cudaMalloc's implicit device-wide synchronization. The
 * pages have no counterpart of this call.
 *
 * Same result as dflash_verify_accept: tokens [block] = d_1..d_a, t_a, then
 * -1 padding, and n [1] = a + 1, for target_logits [block, vocab] of `dtype`
 * and draft_ids [block - 1], enqueued on `stream` (a cudaStream_t; NULL is
 * the legacy default stream). Its scratch is one static device array of
 * about 64 KB that every GPU loading the library holds until the process
 * exits, so it accepts only 2 <= block <= 64 and 2 <= vocab <= 1048576
 * (ERANGE beyond, with the reason in dflash_last_error(NULL)). Each call
 * made outside a stream capture looks up the array's device address with the
 * current device (so a device reset, which reloads the library's device code,
 * is followed); a call on a capturing stream reuses the address its device's
 * last call found, so make the first call on a device before any stream
 * capture. All calls share the array:
 * calls that overlap on the GPU (other streams, other host threads) race.
 * Returns EINVAL for a NULL pointer or a bad dtype, ECUDA if a CUDA call
 * fails. */
int dflash_verify_accept_static(const void* target_logits, int32_t dtype,
                                int32_t vocab, int32_t block,
                                const int32_t* draft_ids, int32_t* tokens,
                                int32_t* n, void* stream);

/* ---- stand-in target (benchmark and test harness) ---------------------------- */

/* Fills the round's target inputs the way a target model would, from pools
 * of synthetic data. r = the context's committed-round counter (device);
 * logits_out [block, V] = logit_pool[r % n_logit_pool][:block] with
 * logits_out[i, draft_ids[i]] = plant[r % n_logit_pool][i] wherever
 * coins[r % n_coin_rows][i] != 0 (i < block - 1); resid_out
 * [block, k*target_hidden] = resid_pool[r % n_resid_pool][:block].
 * logit_pool is [n, block_max, V], plant [n, block_max], resid_pool
 * [n, block_max, k*target_hidden], coins uint8 [n_coin_rows, block_max].
 * This is not a step of the round: it stands in for the target model. */
int dflash_synth_target(dflash_ctx* ctx, const void* logit_pool,
                        const void* plant, const uint8_t* coins,
                        const void* resid_pool, int32_t n_logit_pool,
                        int32_t n_coin_rows, int32_t n_resid_pool,
                        int32_t block_max, int32_t block,
                        const int32_t* draft_ids, void* logits_out,
                        void* resid_out);

/* ---- LFM2 short convolution and its rollback ---------------------------------- */

/* The causal depthwise short convolution of an LFM2 conv layer over a verify
 * block ["LFM2 / LFM2.5 DSpark drafter on the DFlash loop", "Short-conv
 * rollback"], for `layers` layers at once: with x = concat(state [lcache-1,
 * C] (NULL: zeros), bx [block, C]) per layer, y[t, c] = sum_k w[c, k] *
 * x[t + k, c] for t < block (fp32 accumulation, stored in dtype), and
 * state_after (may be NULL, may alias state) = the last lcache - 1 rows of x.
 * Layouts: state/state_after [layers, lcache-1, C], bx and y [layers, block,
 * C], w [layers, C, lcache]; all device memory, dense. Enqueued on `stream`
 * (a cudaStream_t; NULL: the legacy default stream); no context, no
 * allocation. EINVAL for NULL bx/w/y or a bad size or dtype, ERANGE for
 * lcache outside [2, 16]; the reason is in dflash_last_error(NULL). */
int dflash_short_conv_block(const void* state, const void* bx, const void* w, int32_t layers,
                            int32_t lcache, int32_t channels, int32_t block, int32_t dtype, void* y,
                            void* state_after, void* stream);

/* Partial-accept rollback of short-conv states (same page and section): a
 * conv state cannot be trimmed like a KV cache, so the committed state is
 * recomputed as the last lcache - 1 rows of concat(prev_state (NULL: zeros),
 * bx[:n]), n = *n_dev read on the device (the verify's n = a + 1, clamped to
 * [0, block]), so a captured round needs no host read. prev_state is the
 * state before the block, bx the block's gated conv input; state_out [layers,
 * lcache-1, C] may alias prev_state. Bit-exact copies. Same conventions and
 * errors as dflash_short_conv_block. */
int dflash_short_conv_rollback(const void* prev_state, const void* bx, const int32_t* n_dev,
                               int32_t layers, int32_t lcache, int32_t channels, int32_t block,
                               int32_t dtype, void* state_out, void* stream);

/* ---- the synthetic target: a real verify forward ------------------------------ */

/* A Qwen3-shaped causal decoder standing in for the target model [Muse "What
 * changed", the Muse target: residual-stream capture before the final norm,
 * trim rollback over the mixed sliding / full caches]. Layers have the
 * drafter's layout (in_norm, Wq/Wk/Wv, per-head q/k norms + RoPE, Wo,
 * post_norm, SwiGLU), with a causal mask: a sliding layer sees key j from
 * query i iff 0 <= pos_i - pos_j <= window, a full layer iff pos_j <= pos_i.
 * The sliding layers keep a ring of window + slack(max_block) rows, the full
 * layers an append-only cache of max_context rows. */
typedef struct dflash_target_config {
  int32_t n_layers;        /* 1..64 */
  int32_t hidden;          /* the drafter's target_hidden */
  int32_t n_q_heads, n_kv_heads, head_dim, intermediate, vocab;
  int32_t window;          /* > 0: the sliding layers' window */
  uint64_t full_layers;    /* bit l set: layer l is a full-attention layer */
  int32_t n_capture;       /* 1..8: residual streams captured per row */
  int32_t capture[8];      /* layer l: the residual stream after layer l, in
                              this order (the drafter's k_target_layers
                              streams) */
  int32_t rope_neox;
  int32_t max_block;       /* largest forward (2..32 rows) */
  int32_t dtype;           /* DFLASH_F32 or DFLASH_BF16 */
  int32_t max_context;     /* rows the full layers' caches hold */
  float rope_theta;
  float rms_eps;
} dflash_target_config;

typedef struct dflash_target_weights {
  const void* embed;        /* [V, H] the raw embedding table (the drafter binds the same) */
  const void* final_norm;   /* [H] */
  const void* lm_head;      /* [V, H] untied (the drafter binds the same) */
  const void* const* layers;/* HOST array of n_layers * DFLASH_LAYER_TENSORS device pointers */
} dflash_target_weights;

/* Creates a target (a dflash_ctx on which only the dflash_target_* calls,
 * dflash_get_state, dflash_ctx_destroy, dflash_last_error and the ring
 * accessors apply; drafting calls return EINVAL). Same conventions as
 * dflash_ctx_create. EINVAL / ERANGE for a bad config (capture layers
 * outside [0, n_layers), window <= 0, max_block outside [2, 32]). */
int dflash_target_create(const dflash_target_config* cfg, const dflash_target_weights* w, void* stream,
                         dflash_ctx** out);

/* Forward of `rows` tokens (DEVICE int32 [rows]) at the positions after the
 * target's committed length: appends their K/V to every layer's cache,
 * writes the logits of the LAST logit_rows rows (DEVICE [logit_rows, V],
 * storage dtype, no softcap; NULL when logit_rows == 0) and, when captured is
 * not NULL, the captured residual rows (DEVICE [rows, n_capture * hidden],
 * the streams in capture order). Used for the prompt prefill (chunks of up to
 * max_block rows) and by dflash_target_verify. Enqueued only. EINVAL / ERANGE
 * for bad arguments, EFULL when the full layers' caches may overflow. */
int dflash_target_forward(dflash_ctx* target, const int32_t* tokens, int32_t rows, int32_t logit_rows,
                          void* logits, void* captured);

/* The verify forward of a round: the block [anchor, d_1 .. d_{block-1}] with
 * the anchor read from the drafter's device state and draft_ids (DEVICE
 * [block-1]); logits of every block row (DEVICE [block, V]) and the captured
 * rows (DEVICE [block, n_capture * hidden]) that dflash_verify_accept and
 * dflash_append_block then take. The drafter's committed length must equal
 * the target's (device check: error bit 8 of the target's state). */
int dflash_target_verify(dflash_ctx* target, const dflash_ctx* drafter, int32_t block,
                         const int32_t* draft_ids, void* logits, void* captured);

/* The trim after a verify of `block` rows: every layer's cache drops its
 * last block - n rows, n = *n_dev (DEVICE int32: the verify's n = a + 1)
 * [DSpark "Short-conv rollback": attention layers trim their KV cache]. A
 * trim longer than the rows appended since the last one is refused on the
 * device (error bit 16 of the target's state). Enqueued only. */
int dflash_target_commit(dflash_ctx* target, const int32_t* n_dev, int32_t block);

/* The full layers' cache (NULL when every layer slides); the sliding layers'
 * ring is dflash_ring(target). */
int dflash_target_full_ring(dflash_ctx* target, ring_cache** out);

/* ---- ring KV cache (usable standalone) ---------------------------------------- */

#define DFLASH_RING_UNFLOORED 1 /* test-only: size the slack by the unfloored
                                   clamp(8*block, 32, 128), to show the window
                                   corruption the floor prevents */

/* A per-layer ring of K and V rows [kv_heads, head_dim] addressed by absolute
 * position: position q lives in slot q mod capacity, capacity = window +
 * slack(max_block) [Muse "What changed": the mask needs absolute key
 * positions; "Pre-merge review round": the slack past the window]. window
 * <= 0 makes an append-only cache of max_context rows. stream as in
 * dflash_ctx_create. */
int ring_cache_create(int32_t n_layers, int32_t kv_heads, int32_t head_dim,
                      int32_t window, int32_t max_block, int32_t dtype,
                      int32_t max_context, void* stream, ring_cache** out);
int ring_cache_create_ex(int32_t n_layers, int32_t kv_heads, int32_t head_dim,
                         int32_t window, int32_t max_block, int32_t dtype,
                         int32_t max_context, int32_t flags, void* stream,
                         ring_cache** out);
/* Destroys a standalone ring; a context's ring is destroyed with it. */
void ring_cache_destroy(ring_cache* rc);
/* Appends n rows at positions offset .. offset+n-1; k and v are
 * [n_layers, n, kv_heads, head_dim]. EINVAL if n < 0 or n > capacity; EFULL
 * if an append-only cache would overflow. */
int ring_cache_append(ring_cache* rc, const void* k, const void* v, int32_t n);
/* Rewinds the offset by n_rows without restoring any slot; EREWIND if n_rows
 * exceeds the rows appended since the last trim or commit, or (sliding ring)
 * exceeds the slack, capacity - window: rows appended past the slack have
 * overwritten window rows that the rewind would make visible again [Muse
 * "Pre-merge review round", second finding: trim must restore exactly the
 * window seen before the append]. */
int ring_cache_trim(ring_cache* rc, int32_t n_rows);
/* Offset (syncs): the next absolute position to be written. */
int ring_cache_offset(ring_cache* rc, int64_t* offset_host);
int ring_cache_capacity(const ring_cache* rc, int64_t* capacity_host);
/* Copies the raw slot contents for positions pos0 .. pos0+count-1 into k_out
 * and v_out [n_layers, count, kv_heads, head_dim] (device). No validity
 * check: a slot overwritten since returns what it now holds. */
int ring_cache_gather(ring_cache* rc, int64_t pos0, int32_t count,
                      void* k_out, void* v_out);
const char* ring_cache_last_error(const ring_cache* rc);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */
