"""Plain fp64 CPU oracle of one DFlash speculative round at batch 1.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or call
anything here. The CUDA library never does, and nothing here is shared with it:
the GPU side and this file are two independent statements of the same round.

Everything is numpy in float64. Matrix products use ``numpy.matmul`` as a library
step; there is no blocking, fusion or reordering beyond the definitions below.
Where the GPU stores an activation in its storage type (fp32 or bf16) this file
rounds the fp64 value to that type at the same point (``rounder``), so both sides
describe the same rounded quantities; logits are never rounded to bf16.

Sources, cited by page title and section:

* "Muse Glimmer DFlash assistant drafter on the round loop" (mlxcel pull
  request 1762) -- the drafter layout, the sliding mask, the ring slack rule,
  the window drop before ``encoder.fc``.
* "Load Meta's Muse-Glimmer-30B-assistant DFlash head via a draft-adapter
  registry" (z-lab/dflash pull request 168) -- ``fc`` / ``hidden_norm`` naming,
  Qwen3 shape, bidirectional (non-causal) block attention, softcap inheritance.
* "LFM2 / LFM2.5 DSpark drafter on the DFlash loop" (mlxcel pull request 1751)
  -- the greedy exact-match verify rule, n = accepted + 1 and trim(block - n),
  the DSpark block input and read-out rows, the Markov chain, traditional RoPE.

Readings of points the pages leave open:

 R1  RMSNorm is x / sqrt(mean(x^2) + eps) * g with a plain gain (Qwen shape).
 R2  q/k norm is an RMSNorm over head_dim with one gain vector shared by all
     heads, applied before RoPE.
 R3  RoPE inverse frequency theta^(-2i/hd); neox pairs (i, i + hd/2),
     traditional pairs (2i, 2i + 1); positions are absolute.
 R4  The context path is C = hidden_norm(fc(X)) fed straight into each layer's
     Wk / Wv (+ k-norm + RoPE); it has no input norm and no query.
 R5  Key j is visible to query i iff |pos_i - pos_j| <= W (W <= 0: no mask);
     block rows see every block row (bidirectional).
 R6  A final RMSNorm precedes the lm_head.
 R7  DFlash reads out block rows 1..B-1 (mask positions); DSpark drafts a
     gamma = B - 1 row block and reads out every row.
 R8  Target row i predicts position p + i + 1, so d_{i+1} is checked against
     t_i; the bonus token is t_a and n = a + 1.
 R9  argmax ties go to the lowest index; the decision is taken in fp32.
 R10 Softcap is c * tanh(z / c) on the fp32 logit, c = 0 meaning off.
 R11 The Markov chain proposes argmax(W1[prev] . W2) by default, or
     argmax(z_j + W1[prev] . W2) when ``markov_add`` is set.
 R12 Rounding points (storage type): GEMM outputs, norm outputs, the fused
     q/k-norm + RoPE output, attention output, residual sums, the SwiGLU
     product; logits stay fp32.
 R13 Sampled verify (T > 0): the drafter proposes its argmaxes, so its
     proposal distribution is a point mass and the standard speculative-
     sampling rule accepts d with probability p(d); the bonus after a
     rejection comes from p with d removed; uniforms are inputs and the
     inverse CDF runs in vocabulary order.
 R14 The synthetic target is a Qwen3-shaped causal decoder with the drafter's
     layer layout (R1, R2, R3, R12). Its sliding layers see key j from query
     i iff 0 <= pos_i - pos_j <= W; its full layers iff pos_j <= pos_i. It
     shares the raw embedding table and the untied lm_head with the drafter.
 R15 The captured residual rows are the residual stream after each capture
     layer, concatenated in capture order; the last capture layer may be the
     last layer, whose output is the final norm's input.
 R16 The target's logits are fp32 lm_head outputs of the final-normed rows,
     without softcap (the greedy verify is unchanged by it; the sampled
     verify applies it), rounded to the storage type as the GEMM stores them.
 R17 A verify forward appends the block's K/V to every layer's cache; the
     trim after the verify drops the last B - n rows of every layer (the
     sliding layers' rings with the drafter's slack rule, the full layers'
     caches append-only).

Parity status: every function here has a named pin. The slack rule, the ring
restore, accept = prefix + 1, the mask, attention, RoPE, RMSNorm, linear,
window drop, softcap, argmax ties, bf16 rounding, verify and the Markov
feedback are pinned by ``tests/test_oracle_pins.py`` (page values, torch
fp64 routines, closed forms, brute force). The composition is pinned by
``tests/test_oracle_composition.py`` with closed forms on constructed
weights: the drafter layer (uniform attention gives x + Wo . mean of the
visible values; a gate/up fixture gives the MLP's output by hand; the MLP's
input depends on Wo), the context path (one-hot fc / Wk / Wv give each K and
V row by hand, RoPE at the absolute position, no input norm), the draft's
read-out rows through the final norm, lm_head and softcap, and the session's
history against the ring model. The pages print no numbers for the layer
layout itself (readings R1, R2, R4, R6, R12): those pins fix the reading
taken, not a value from the pages. The synthetic target (R14-R17) is pinned
by ``tests/test_oracle_target.py``: the causal mask against triangle / band
constructions and brute force, the masked attention against torch's
scaled-dot-product attention, identity layers (raw-embedding streams, plain
logits), the capture order, uniform attention (the causal mean of the
visible values), one pass against prefill-then-verify, and a trim against
never having appended the dropped rows.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "speculative_slack", "ring_capacity", "round_bf16", "round_f32", "rounder",
    "bf16_bits_to_f64", "as_f64", "rmsnorm", "head_rmsnorm", "rope",
    "visible_mask", "attention", "linear", "silu", "softcap", "argmax_lowest",
    "window_drop", "context_kv", "block_tokens", "drafter_layer",
    "lm_head_argmax", "draft_block", "markov_chain",
    "verify_accept", "sampled_probs", "verify_sampled", "short_conv_block",
    "short_conv_rollback", "RingModel", "OracleSession", "stats_ratios",
    "causal_mask", "causal_attention", "target_layer", "layer_window",
    "target_forward", "TargetSession",
]


# ---------------------------------------------------------------------------
# Speculative slack and the ring
# ---------------------------------------------------------------------------

def speculative_slack(block: int, floor: bool = True) -> int:
    """Rows of speculative buffer past the window for a verify block.

    Muse Glimmer DFlash assistant drafter on the round loop, "Pre-merge review
    round", second finding: the buffer is clamp(block * 8, 32, 128) and is
    floored at the block size. ``floor=False`` gives the earlier, unfloored
    rule (only used to show the corruption the floor prevents).
    """
    if block < 1:
        raise ValueError("block must be positive")
    s = min(max(8 * block, 32), 128)
    return max(s, block) if floor else s


def ring_capacity(window: int, block: int, floor: bool = True) -> int:
    """Slots of a sliding ring: the window plus the speculative slack
    (same page and finding: the slack sits past max_size)."""
    return window + speculative_slack(block, floor)


class RingModel:
    """A slot array of ``capacity`` rows addressed by absolute position, next to
    the dense history it is meant to reproduce.

    Muse Glimmer DFlash assistant drafter on the round loop, "Pre-merge review
    round", second finding: append writes rows past the window into the slack;
    trim rewinds the offset without restoring any overwritten slot. The model
    keeps both views so a test can see when the slot view of the visible window
    stops matching the history (the corruption the block-size floor prevents).
    """

    def __init__(self, window: int, capacity: int, row_shape=(1,)):
        self.window = window
        self.capacity = capacity
        self.slots = np.full((capacity,) + tuple(row_shape), np.nan)
        self.slot_pos = np.full(capacity, -1, dtype=np.int64)
        self.history: dict[int, np.ndarray] = {}
        self.offset = 0
        self.appended_since_trim = 0

    def append(self, rows: np.ndarray) -> None:
        for j in range(rows.shape[0]):
            pos = self.offset + j
            self.slots[pos % self.capacity] = rows[j]
            self.slot_pos[pos % self.capacity] = pos
            self.history[pos] = np.array(rows[j], copy=True)
        self.offset += rows.shape[0]
        self.appended_since_trim += rows.shape[0]

    def trim(self, m: int) -> None:
        """KVCache::trim(m): rewind the offset by m rows (DSpark page, "Short-conv
        rollback"). m larger than the rows appended since the last trim is the
        'short rewind' the Muse page makes an error."""
        if m < 0 or m > self.appended_since_trim:
            raise ValueError("short rewind")
        for pos in range(self.offset - m, self.offset):
            del self.history[pos]
        self.offset -= m
        self.appended_since_trim = 0

    def window_positions(self, next_pos: int | None = None) -> np.ndarray:
        """Positions a query at ``next_pos`` (default: the offset) can see."""
        p = self.offset if next_pos is None else next_pos
        lo = max(0, p - self.window) if self.window > 0 else 0
        return np.arange(lo, p, dtype=np.int64)

    def slot_view(self, positions) -> np.ndarray:
        return np.stack([self.slots[q % self.capacity] for q in positions])

    def history_view(self, positions) -> np.ndarray:
        return np.stack([self.history[q] for q in positions])


# ---------------------------------------------------------------------------
# Storage rounding
# ---------------------------------------------------------------------------

def round_bf16(x) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits with the fp32 exponent range, so the
    quantum of a value in [2^(e-1), 2^e) is 2^(e-8), never finer than the
    subnormal quantum 2^-133. Dividing by a power of two is exact, and
    ``numpy.rint`` rounds half to even.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    q = np.ldexp(1.0, np.maximum(e - 8, -133))
    return np.rint(x / q) * q


def round_f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def rounder(dtype: str):
    """The storage rounding of reading R12 for a config's dtype."""
    if dtype == "bf16":
        return round_bf16
    if dtype == "f32":
        return round_f32
    raise ValueError(f"unknown dtype {dtype!r}")


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bfloat16 bit patterns (uint16)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def as_f64(a, dtype: str) -> np.ndarray:
    """Exact fp64 value of a stored tensor (uint16 bf16 bits or float32)."""
    if dtype == "bf16":
        return bf16_bits_to_f64(a)
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------
# Per-op definitions
# ---------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    """Reading R1 (Qwen shape per the Muse head page, "Why"): RMSNorm over the
    last axis with a plain gain."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * gain


def head_rmsnorm(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    """Per-head q/k RMSNorm (Muse page, "What changed": per-head q/k norms);
    x is [..., heads, head_dim] and one gain [head_dim] serves every head (R2)."""
    return rmsnorm(x, gain, eps)


def rope(x: np.ndarray, pos, theta: float, neox: bool) -> np.ndarray:
    """Rotary embedding of x [rows, heads, hd] at absolute positions ``pos``.

    Reading R3. DSpark page, "Verified against the issue, line by line":
    rope_is_neox_style false means the traditional pairing. Neox rotates the
    pair (i, i + hd/2); traditional rotates (2i, 2i + 1); both by angle
    pos * theta^(-2i/hd).
    """
    hd = x.shape[-1]
    half = hd // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / hd)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    if neox:
        x1, x2 = x[..., :half], x[..., half:]
    else:
        x1, x2 = x[..., 0::2], x[..., 1::2]
    y1 = x1 * c - x2 * s
    y2 = x1 * s + x2 * c
    out = np.empty_like(x, dtype=np.float64)
    if neox:
        out[..., :half], out[..., half:] = y1, y2
    else:
        out[..., 0::2], out[..., 1::2] = y1, y2
    return out


def visible_mask(q_pos, k_pos, window: int) -> np.ndarray:
    """Muse page, "What changed": bidirectional sliding mask over absolute
    positions, key visible iff |q - k| <= W (reading R5; W <= 0: no mask)."""
    q_pos = np.asarray(q_pos, dtype=np.int64)
    k_pos = np.asarray(k_pos, dtype=np.int64)
    if window <= 0:
        return np.ones((q_pos.size, k_pos.size), dtype=bool)
    return np.abs(q_pos[:, None] - k_pos[None, :]) <= window


def attention(q, k, v, q_pos, k_pos, window: int) -> np.ndarray:
    """Grouped-query attention with the sliding mask, scale 1/sqrt(hd).

    q [Bq, nq, hd], k and v [Nk, nkv, hd]. Query head h reads kv head
    h // (nq / nkv). The whole [Bq, Nk] score matrix is formed and masked
    explicitly; the softmax runs in fp64.
    """
    bq, nq, hd = q.shape
    nkv = k.shape[1]
    group = nq // nkv
    mask = visible_mask(q_pos, k_pos, window)
    out = np.zeros((bq, nq, hd), dtype=np.float64)
    for h in range(nq):
        g = h // group
        s = (q[:, h, :] @ k[:, g, :].T) / math.sqrt(hd)
        s = np.where(mask, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, g, :]
    return out


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = x . W^T with W stored [out_features, in_features]."""
    return x @ w.T


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def softcap(z32: np.ndarray, cap: float) -> np.ndarray:
    """Reading R10: c * tanh(z / c) on fp32 logits, returned as fp32 values
    (Muse head page, "How": the head inherits final_logit_softcapping)."""
    z32 = np.asarray(z32, dtype=np.float32)
    if cap <= 0.0:
        return z32
    return (cap * np.tanh(z32.astype(np.float64) / cap)).astype(np.float32)


def argmax_lowest(z: np.ndarray) -> np.ndarray:
    """Row-wise argmax, ties to the lowest index (reading R9).

    ``numpy.argmax`` returns the first maximal index, which is the lowest."""
    return np.argmax(np.asarray(z), axis=-1).astype(np.int64)


# ---------------------------------------------------------------------------
# Context side: window drop, encoder.fc, hidden_norm, context K/V
# ---------------------------------------------------------------------------

def window_drop(resid: np.ndarray, first_pos: int, next_pos: int, window: int):
    """Rows of a residual slab a query at ``next_pos`` can still see.

    Muse page, "Pre-merge review round", third finding: rows past the sliding
    window are dropped before encoder.fc runs; fc and output_norm_enc are per
    row, so the kept rows' results are unchanged. Row r has position
    first_pos + r and is kept iff position >= next_pos - W (reading of the
    same |q - k| <= W bound for the nearest query).
    """
    pos = first_pos + np.arange(resid.shape[0], dtype=np.int64)
    if window > 0:
        keep = pos >= next_pos - window
        return resid[keep], pos[keep]
    return resid, pos


def context_kv(cfg: dict, w: dict, resid: np.ndarray, pos: np.ndarray):
    """Context K/V rows for every drafter layer from captured residual rows.

    Muse page, "What changed": encoder.fc plus encoder.output_norm_enc (the
    head page's fc / hidden_norm) over the concatenated residual streams; the
    DSpark page ("Verified against the issue") keeps only context K/V in the
    drafter cache. Reading R4: C goes straight into each layer's Wk / Wv, then
    k-norm and RoPE at each row's absolute position.

    Returns (K, V, C): K and V are lists over layers of [R, nkv, hd]; C is the
    normed fc output [R, H]. All are rounded to the storage type.
    """
    rnd = rounder(cfg["dtype"])
    nkv, hd = cfg["n_kv_heads"], cfg["head_dim"]
    f = rnd(linear(resid, w["fc"]))
    c = rnd(rmsnorm(f, w["hidden_norm"], cfg["rms_eps"]))
    ks, vs = [], []
    for lw in w["layers"]:
        k = rnd(linear(c, lw["wk"])).reshape(-1, nkv, hd)
        v = rnd(linear(c, lw["wv"])).reshape(-1, nkv, hd)
        k = rnd(rope(head_rmsnorm(k, lw["k_norm"], cfg["rms_eps"]), pos,
                     cfg["rope_theta"], cfg["rope_neox"]))
        ks.append(k)
        vs.append(v)
    return ks, vs, c


# ---------------------------------------------------------------------------
# Drafter block forward, lm_head + softcap + argmax, Markov chain
# ---------------------------------------------------------------------------

def block_tokens(cfg: dict, anchor: int, block: int):
    """The drafter's block input and the rows read out (reading R7).

    DFlash (Muse page, "What changed"): ``block`` rows [anchor, mask x (B-1)]
    at positions p..p+B-1; rows 1..B-1 propose the tokens at their own
    positions. DSpark (DSpark page, "Verified against the issue"): gamma =
    block - 1 rows [anchor, mask x (gamma-1)], every row read out, row j
    proposing position p + j + 1. Both give block - 1 proposals.
    """
    if cfg.get("kind", "dflash") == "dspark":
        rows = block - 1
        read = np.arange(rows)
    else:
        rows = block
        read = np.arange(1, rows)
    toks = np.array([anchor] + [cfg["mask_token_id"]] * (rows - 1), dtype=np.int64)
    return toks, read


def drafter_layer(cfg, lw, x, pos, ctx_k, ctx_v, ctx_pos):
    """One sliding-attention drafter layer on the block (reading R12 rounding).

    Muse page, "What changed": per-head q/k norms, bidirectional sliding mask
    over absolute positions; head page, "Why": Qwen3 layout, is_causal False.
    The block's own K/V join the context K/V for this forward only.
    """
    rnd = rounder(cfg["dtype"])
    eps = cfg["rms_eps"]
    nq, nkv, hd = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    rows = x.shape[0]
    xn = rnd(rmsnorm(x, lw["in_norm"], eps))
    q = rnd(linear(xn, lw["wq"])).reshape(rows, nq, hd)
    k = rnd(linear(xn, lw["wk"])).reshape(rows, nkv, hd)
    v = rnd(linear(xn, lw["wv"])).reshape(rows, nkv, hd)
    q = rnd(rope(head_rmsnorm(q, lw["q_norm"], eps), pos, cfg["rope_theta"], cfg["rope_neox"]))
    k = rnd(rope(head_rmsnorm(k, lw["k_norm"], eps), pos, cfg["rope_theta"], cfg["rope_neox"]))
    keys = np.concatenate([ctx_k, k], axis=0)
    vals = np.concatenate([ctx_v, v], axis=0)
    kpos = np.concatenate([ctx_pos, pos])
    a = rnd(attention(q, keys, vals, pos, kpos, cfg["window"]))
    o = rnd(linear(a.reshape(rows, nq * hd), lw["wo"]))
    h = rnd(x + o)
    hn = rnd(rmsnorm(h, lw["post_norm"], eps))
    g = rnd(linear(hn, lw["wg"]))
    u = rnd(linear(hn, lw["wu"]))
    s = rnd(silu(g) * u)
    d = rnd(linear(s, lw["wd"]))
    return rnd(h + d)


def lm_head_argmax(cfg: dict, w: dict, xf_rows: np.ndarray):
    """Logits of the read-out rows, softcap, argmax (readings R9, R10).

    Muse page, "What changed": the drafter binds the target's untied lm_head;
    head page, "How": it inherits final_logit_softcapping. Logits are formed
    in fp64, taken to fp32 (the decision precision), capped in fp32.
    Returns (capped fp32 logits [rows, V], ids [rows]).
    """
    z = linear(xf_rows, w["lm_head"]).astype(np.float32)
    zc = softcap(z, cfg.get("softcap", 0.0))
    return zc, argmax_lowest(zc)


def markov_chain(w1: np.ndarray, w2: np.ndarray, anchor: int, gamma: int,
                 z: np.ndarray | None = None) -> np.ndarray:
    """DSpark Markov token-transition chain (reading R11).

    DSpark page, "Verified against the issue": seeded with the anchor, each
    step's argmax feeds the next step's W1 gather. Step j scores
    m = W1[prev] . W2 (W1 [V, r], W2 [r, V]); with ``z`` given (the fp32 capped
    backbone logits of row j) the score is z_j + m, added in fp32.
    """
    prev = int(anchor)
    out = np.empty(gamma, dtype=np.int64)
    for j in range(gamma):
        m = (w1[prev] @ w2).astype(np.float32)
        score = m if z is None else (z[j].astype(np.float32) + m)
        prev = int(argmax_lowest(score))
        out[j] = prev
    return out


def draft_block(cfg: dict, w: dict, ctx_k, ctx_v, ctx_pos, anchor: int,
                anchor_pos: int, block: int) -> dict:
    """The drafter's full block forward and its proposals.

    ``ctx_k`` / ``ctx_v`` are lists over layers of [N, nkv, hd] with absolute
    positions ``ctx_pos``. Returns the final normed hidden of every block row
    ('hidden'), the capped fp32 logits and backbone argmax of the read-out rows,
    the Markov chain (if the config has one) and the proposals 'draft_ids'
    (block - 1 of them).
    """
    rnd = rounder(cfg["dtype"])
    toks, read = block_tokens(cfg, anchor, block)
    pos = anchor_pos + np.arange(toks.size, dtype=np.int64)
    x = rnd(w["embed"][toks])
    for li, lw in enumerate(w["layers"]):
        x = drafter_layer(cfg, lw, x, pos, ctx_k[li], ctx_v[li], ctx_pos)
    xf = rnd(rmsnorm(x, w["final_norm"], cfg["rms_eps"]))
    zc, ids = lm_head_argmax(cfg, w, xf[read])
    out = {"hidden": xf, "logits": zc, "backbone_ids": ids, "positions": pos}
    if cfg.get("markov_rank", 0) > 0:
        chain = markov_chain(w["markov_w1"], w["markov_w2"], anchor, read.size,
                             zc if cfg.get("markov_add", 0) else None)
        out["chain_ids"] = chain
        out["draft_ids"] = chain
    else:
        out["draft_ids"] = ids
    return out


# ---------------------------------------------------------------------------
# Verify and accept
# ---------------------------------------------------------------------------

def verify_accept(target_logits: np.ndarray, draft_ids: np.ndarray):
    """Greedy exact-match verification (reading R8).

    DSpark page, intro and "Short-conv rollback": the target's block argmax
    t_i = argmax L[i] (lowest index on ties) checks d_{i+1}; a is the longest
    matching prefix, the emitted tokens are d_1..d_a then the bonus t_a, and
    n = a + 1. ``draft_ids[i]`` holds d_{i+1}.
    """
    t = argmax_lowest(target_logits)
    b = t.size
    a = 0
    while a < b - 1 and int(draft_ids[a]) == int(t[a]):
        a += 1
    tokens = np.concatenate([np.asarray(draft_ids[:a], dtype=np.int64), t[a:a + 1]])
    return tokens, a + 1, t


def sampled_probs(logits: np.ndarray, temperature: float, cap: float) -> np.ndarray:
    """Target token probabilities of one verify row at temperature T > 0 on
    softcapped logits: softmax(c * tanh(L / c) / T) (reading R10 for the cap,
    c = 0 meaning none), formed in fp64 from the fp32 capped logits.

    "Load Meta's Muse-Glimmer-30B-assistant DFlash head", "Measured": the
    sampled-acceptance run at T = 1; "How": the head inherits the tanh cap.
    """
    z = softcap(np.asarray(logits, dtype=np.float32), cap).astype(np.float64) / temperature
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def verify_sampled(target_logits: np.ndarray, draft_ids: np.ndarray, u: np.ndarray,
                   temperature: float, cap: float):
    """Speculative-sampling verify for a drafter whose proposals are its
    argmaxes, i.e. whose proposal distribution q is a point mass on d_{i+1}
    (reading R13). Row i accepts d_{i+1} with probability min(1, p_i(d)/q(d))
    = p_i(d_{i+1}): accepted iff u[i] < p_i(d_{i+1}). a is the accepted
    prefix. The bonus token is drawn by inverse CDF with u[block - 1] in
    vocabulary order: after a rejection at row a from the residual
    max(p_a - q, 0) renormalised (p_a with d_{a+1} removed), after a full
    accept from p_{block-1}. Returns (tokens d_1..d_a + bonus, n = a + 1, a).
    ``u`` holds block values in [0, 1): the random numbers are inputs.
    """
    b = target_logits.shape[0]
    a = 0
    while a < b - 1:
        p = sampled_probs(target_logits[a], temperature, cap)
        if u[a] < p[int(draft_ids[a])]:
            a += 1
        else:
            break
    p = sampled_probs(target_logits[a], temperature, cap)
    if a < b - 1:
        p = p.copy()
        p[int(draft_ids[a])] = 0.0
    c = np.cumsum(p)
    t = u[b - 1] * c[-1]
    bonus = int(np.searchsorted(c, t, side="right"))
    bonus = min(bonus, int(np.nonzero(p > 0)[0][-1]))
    tokens = np.concatenate([np.asarray(draft_ids[:a], dtype=np.int64), [bonus]])
    return tokens, a + 1, a


def short_conv_block(state, bx, w):
    """LFM2 short convolution over a block (DSpark page, "Short-conv
    rollback"): a causal depthwise convolution of kernel length L over the
    gated input Bx. With the L - 1 rows of state before the block (zeros when
    there are none), y[t, c] = sum_k w[c, k] * x[t + k, c] over x = concat(
    state, bx), t < block; the state after the block is the last L - 1 rows of
    x. state [L-1, C] or None, bx [block, C], w [C, L]."""
    lc = w.shape[1]
    if state is None:
        state = np.zeros((lc - 1, bx.shape[1]))
    x = np.concatenate([state, bx], axis=0)
    y = np.stack([np.sum(w * x[t:t + lc].T, axis=1) for t in range(bx.shape[0])])
    return y, x[x.shape[0] - (lc - 1):]


def short_conv_rollback(prev_state, bx, n, lcache):
    """Partial-accept rollback of a short-conv state (DSpark page, "Short-conv
    rollback"): a conv state cannot be trimmed, so the committed state is
    recomputed as the last L - 1 rows of concat(prev_state or zeros, bx[:n])."""
    if prev_state is None:
        prev_state = np.zeros((lcache - 1, bx.shape[1]))
    x = np.concatenate([prev_state, bx[:n]], axis=0)
    return x[x.shape[0] - (lcache - 1):]


def stats_ratios(rounds: int, proposed: int, accepted: int) -> dict:
    """Round counters and the two 'mean accepted' definitions on the pages.

    Muse page, "Real-checkpoint validation": mean accepted = accepted / rounds.
    DSpark page, "Real-checkpoint validation": mean accepted length =
    accepted / rounds + 1 (emitted per verify) and acceptance = accepted /
    proposed.
    """
    return {
        "accepted_per_round": accepted / rounds,
        "emitted_per_round": accepted / rounds + 1.0,
        "acceptance": accepted / proposed,
        "emitted": accepted + rounds,
    }


# ---------------------------------------------------------------------------
# The synthetic target: causal verify forward, residual capture, cache trim
# ---------------------------------------------------------------------------

def causal_mask(q_pos, k_pos, window: int) -> np.ndarray:
    """Reading R14 (Muse page, "What changed", Muse target: sliding and full
    caches): key j visible to query i iff pos_j <= pos_i, and for a sliding
    layer (window > 0) also pos_i - pos_j <= window."""
    q_pos = np.asarray(q_pos, dtype=np.int64)
    k_pos = np.asarray(k_pos, dtype=np.int64)
    d = q_pos[:, None] - k_pos[None, :]
    vis = d >= 0
    if window > 0:
        vis &= d <= window
    return vis


def causal_attention(q, k, v, q_pos, k_pos, window: int) -> np.ndarray:
    """Grouped-query attention under the causal (sliding or full) mask; the
    same explicit score matrix and fp64 softmax as ``attention``."""
    bq, nq, hd = q.shape
    group = nq // k.shape[1]
    mask = causal_mask(q_pos, k_pos, window)
    out = np.zeros((bq, nq, hd), dtype=np.float64)
    for h in range(nq):
        g = h // group
        sc = (q[:, h, :] @ k[:, g, :].T) / math.sqrt(hd)
        sc = np.where(mask, sc, -np.inf)
        sc = sc - sc.max(axis=1, keepdims=True)
        pr = np.exp(sc)
        pr = pr / pr.sum(axis=1, keepdims=True)
        out[:, h, :] = pr @ v[:, g, :]
    return out


def target_layer(tcfg, lw, x, pos, hist_k, hist_v, hist_pos, window):
    """One target decoder layer over rows x at positions pos (reading R14):
    the drafter's layer with a causal mask, attending to the layer's cache
    (hist_*) followed by the rows themselves. Returns the layer output and the
    rows' K and V (normed + rotated K, rounded V), which join the cache."""
    rnd = rounder(tcfg["dtype"])
    eps = tcfg["rms_eps"]
    nq, nkv, hd = tcfg["n_q_heads"], tcfg["n_kv_heads"], tcfg["head_dim"]
    rows = x.shape[0]
    xn = rnd(rmsnorm(x, lw["in_norm"], eps))
    q = rnd(linear(xn, lw["wq"])).reshape(rows, nq, hd)
    k = rnd(linear(xn, lw["wk"])).reshape(rows, nkv, hd)
    v = rnd(linear(xn, lw["wv"])).reshape(rows, nkv, hd)
    q = rnd(rope(head_rmsnorm(q, lw["q_norm"], eps), pos, tcfg["rope_theta"], tcfg["rope_neox"]))
    k = rnd(rope(head_rmsnorm(k, lw["k_norm"], eps), pos, tcfg["rope_theta"], tcfg["rope_neox"]))
    keys = np.concatenate([hist_k, k], axis=0)
    vals = np.concatenate([hist_v, v], axis=0)
    kpos = np.concatenate([hist_pos, pos])
    a = rnd(causal_attention(q, keys, vals, pos, kpos, window))
    o = rnd(linear(a.reshape(rows, nq * hd), lw["wo"]))
    h = rnd(x + o)
    hn = rnd(rmsnorm(h, lw["post_norm"], eps))
    g = rnd(linear(hn, lw["wg"]))
    u = rnd(linear(hn, lw["wu"]))
    sw = rnd(silu(g) * u)
    d = rnd(linear(sw, lw["wd"]))
    return rnd(h + d), k, v


def layer_window(tcfg, layer: int) -> int:
    """A full layer attends to its whole history (window 0), a sliding one
    through the target's window."""
    return 0 if layer in tuple(tcfg["full_layers"]) else tcfg["window"]


def target_forward(tcfg, tw, tokens, pos0, hist, logit_rows=None):
    """The target's forward over ``tokens`` at positions pos0.. (readings
    R14-R16). ``hist`` holds per layer (K, V, positions) of the rows already
    in its cache. Returns the logits of the last ``logit_rows`` rows (all by
    default) [.., V] (storage-rounded fp32, no softcap), the captured residual
    rows [rows, len(capture) * H] and the rows' per-layer K and V."""
    rnd = rounder(tcfg["dtype"])
    toks = np.asarray(tokens, dtype=np.int64)
    pos = pos0 + np.arange(toks.size, dtype=np.int64)
    x = rnd(tw["embed"][toks])
    streams, new_k, new_v = {}, [], []
    for li, lw in enumerate(tw["layers"]):
        hk, hv, hp = hist[li]
        x, k, v = target_layer(tcfg, lw, x, pos, hk, hv, hp, layer_window(tcfg, li))
        streams[li] = x
        new_k.append(k)
        new_v.append(v)
    captured = np.concatenate([streams[l] for l in tcfg["capture"]], axis=1)
    xf = rnd(rmsnorm(x, tw["final_norm"], tcfg["rms_eps"]))
    if logit_rows is not None:
        xf = xf[xf.shape[0] - logit_rows:]
    logits = rnd(linear(xf, tw["lm_head"]).astype(np.float32).astype(np.float64))
    return {"logits": logits, "captured": captured, "k": new_k, "v": new_v, "positions": pos}


@dataclass
class TargetSession:
    """The target's caches as dense per-layer histories keyed by absolute
    position (reading R17): a forward appends its rows, ``commit`` keeps the
    first n rows of the last forward and drops the rest."""

    tcfg: dict
    tw: dict
    pos: int = 0
    hist: list = field(default_factory=list)
    last_rows: int = 0

    def __post_init__(self):
        nkv, hd = self.tcfg["n_kv_heads"], self.tcfg["head_dim"]
        if not self.hist:
            self.hist = [(np.zeros((0, nkv, hd)), np.zeros((0, nkv, hd)), np.zeros(0, dtype=np.int64))
                         for _ in self.tw["layers"]]

    def forward(self, tokens, logit_rows=None) -> dict:
        out = target_forward(self.tcfg, self.tw, tokens, self.pos, self.hist, logit_rows)
        for li in range(len(self.hist)):
            hk, hv, hp = self.hist[li]
            self.hist[li] = (np.concatenate([hk, out["k"][li]]), np.concatenate([hv, out["v"][li]]),
                             np.concatenate([hp, out["positions"]]))
        self.last_rows = len(tokens)
        self.pos += len(tokens)
        return out

    def commit(self, n: int) -> None:
        """Trim the last forward's rows past the first n (trim(rows - n))."""
        drop = self.last_rows - n
        if not 0 <= drop <= self.last_rows:
            raise ValueError("short rewind")
        if drop:
            self.hist = [(k[:-drop], v[:-drop], p[:-drop]) for k, v, p in self.hist]
            self.pos -= drop
        self.last_rows = 0

    def cache(self, layer: int):
        return self.hist[layer]


# ---------------------------------------------------------------------------
# Multi-round session: dense context history keyed by absolute position
# ---------------------------------------------------------------------------

@dataclass
class OracleSession:
    """The round loop over a dense context history.

    The history holds, per layer, the K/V rows of every committed context
    position (no ring, no capacity): the definition the GPU ring must reproduce
    for the visible window. One round is draft -> verify -> append(B) ->
    trim(B - n) (DSpark page, "Short-conv rollback"; Muse page, "What changed").
    """

    cfg: dict
    w: dict
    ctx_pos: np.ndarray = field(default_factory=lambda: np.zeros(0, dtype=np.int64))
    ctx_k: list = field(default_factory=list)
    ctx_v: list = field(default_factory=list)
    anchor: int = -1
    pos: int = 0
    rounds: int = 0
    proposed: int = 0
    accepted: int = 0

    def __post_init__(self):
        nkv, hd = self.cfg["n_kv_heads"], self.cfg["head_dim"]
        if not self.ctx_k:
            self.ctx_k = [np.zeros((0, nkv, hd)) for _ in self.w["layers"]]
            self.ctx_v = [np.zeros((0, nkv, hd)) for _ in self.w["layers"]]

    def ingest(self, resid: np.ndarray, first_pos: int, anchor: int) -> None:
        """Initial context: window drop, then context K/V; the next anchor sits
        at first_pos + R."""
        nxt = first_pos + resid.shape[0]
        kept, pos = window_drop(resid, first_pos, nxt, self.cfg["window"])
        self._append(kept, pos)
        self.pos = nxt
        self.anchor = int(anchor)

    def _append(self, resid, pos):
        if resid.shape[0] == 0:
            return
        ks, vs, _ = context_kv(self.cfg, self.w, resid, pos)
        self.ctx_pos = np.concatenate([self.ctx_pos, pos])
        for li in range(len(self.ctx_k)):
            self.ctx_k[li] = np.concatenate([self.ctx_k[li], ks[li]])
            self.ctx_v[li] = np.concatenate([self.ctx_v[li], vs[li]])
        self._forget_old()

    def _forget_old(self):
        """Drop history rows no future query can see (only to bound memory)."""
        win = self.cfg["window"]
        if win <= 0:
            return
        keep = self.ctx_pos >= self.pos - win - 1
        if keep.all():
            return
        self.ctx_pos = self.ctx_pos[keep]
        self.ctx_k = [k[keep] for k in self.ctx_k]
        self.ctx_v = [v[keep] for v in self.ctx_v]

    def visible_context(self):
        """Context rows any block query at self.pos can see."""
        win = self.cfg["window"]
        sel = self.ctx_pos < self.pos
        if win > 0:
            sel &= self.ctx_pos >= self.pos - win
        return ([k[sel] for k in self.ctx_k], [v[sel] for v in self.ctx_v],
                self.ctx_pos[sel])

    def draft(self, block: int) -> dict:
        k, v, p = self.visible_context()
        return draft_block(self.cfg, self.w, k, v, p, self.anchor, self.pos, block)

    def verify(self, target_logits, draft_ids):
        return verify_accept(target_logits, draft_ids)

    def append_and_trim(self, resid_rows: np.ndarray, keep: int) -> None:
        """Append the block's B captured rows at p..p+B-1, then trim(B - keep):
        only the first ``keep`` rows stay committed."""
        b = resid_rows.shape[0]
        if not 0 <= keep <= b:
            raise ValueError("short rewind")
        pos = self.pos + np.arange(b, dtype=np.int64)
        ks, vs, _ = context_kv(self.cfg, self.w, resid_rows, pos)
        self.ctx_pos = np.concatenate([self.ctx_pos, pos[:keep]])
        for li in range(len(self.ctx_k)):
            self.ctx_k[li] = np.concatenate([self.ctx_k[li], ks[li][:keep]])
            self.ctx_v[li] = np.concatenate([self.ctx_v[li], vs[li][:keep]])

    def commit(self, keep: int, next_anchor: int, block: int, accepted: int) -> None:
        """Advance past the ``keep`` committed rows; the next anchor is the
        verify's last emitted token. ``accepted`` is the verify's a (equal to
        keep - 1 in a normal round; a stress run may keep another count)."""
        self.rounds += 1
        self.proposed += block - 1
        self.accepted += accepted
        self.pos += keep
        self.anchor = int(next_anchor)
        self._forget_old()
