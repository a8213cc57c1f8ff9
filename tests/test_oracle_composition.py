"""Closed-form pins of how the oracle composes a drafter layer, the context
path and the draft read-out.

The per-op pins (tests/test_oracle_pins.py) fix RMSNorm, RoPE, attention,
silu, softcap and the ring. These tests fix the wiring between them, each on
weights built so that the result can be written down by hand, so that a
plausible slip fails one of them: the residual taken from the normed input,
the MLP reading x or the input norm instead of the post-attention norm, gate
and up swapped, the sliding window off by one, an input norm on the context
path, RoPE or the k-norm applied to V, the wrong read-out rows. Runs on CPU.

Sources: "Muse Glimmer DFlash assistant drafter on the round loop", "What
changed" (drafter layout, per-head q/k norms, sliding mask over absolute
positions); "Load Meta's Muse-Glimmer-30B-assistant DFlash head", "Why"
(Qwen3 layer shape, is_causal False) and "How" (fc / hidden_norm, softcap);
"LFM2 / LFM2.5 DSpark drafter on the DFlash loop", "Verified against the
issue" (context K/V only in the cache, DSpark read-out rows).
"""

import math
import struct

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O
from block_speculative_decoding_dflash_gb300 import synth

EPS = 1e-6


def _cfg(**over):
    return synth.config("tiny", n_layers=1, **over)


def _weights(cfg, seed=0):
    w = synth.make_weights(cfg, seed)
    out = {k: O.as_f64(v, "f32") for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: O.as_f64(v, "f32") for k, v in lw.items()} for lw in w["layers"]]
    return out


def _close(got, want, rtol):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    scale = np.maximum(np.abs(want).max(axis=-1, keepdims=True), 1e-30)
    assert np.all(np.abs(got - want) <= rtol * scale), np.abs(got - want).max()


def _context(cfg, w, rows=32, seed=4):
    resid = O.as_f64(synth.make_context(cfg, rows, seed=seed), "f32")
    pos = np.arange(rows, dtype=np.int64)
    k, v, _ = O.context_kv(cfg, w, resid, pos)
    return k, v, pos


# --- a drafter layer ---------------------------------------------------------------

def test_layer_with_zero_query_key_projections_averages_visible_values():
    """Wq = Wk = 0 makes every score 0, so each block query takes the plain
    mean of the values it may see: the context rows within W of its own
    absolute position and every block row. With Wg = 0 the MLP adds nothing,
    so the layer is x + Wo . mean(V). Pins the residual source (x, not the
    normed x), the key set of the mask (window edge inclusive, bidirectional
    block), the value path (Wv on the normed block rows) and Wo's
    orientation."""
    cfg = _cfg()
    w = _weights(cfg)
    lw = w["layers"][0]
    rng = np.random.default_rng(7)
    lw["wq"][:] = 0.0
    lw["wk"][:] = 0.0
    lw["wg"][:] = 0.0
    lw["in_norm"][:] = O.round_f32(0.5 + rng.random(cfg["hidden"]))    # makes xn != x
    ck, cv, cpos = _context(cfg, w)
    x = O.round_f32(rng.standard_normal((4, cfg["hidden"])))
    p = 32 + np.arange(4)
    got = O.drafter_layer(cfg, lw, x, p, ck[0], cv[0], cpos)

    W, nq, nkv, hd = cfg["window"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    xt = torch.from_numpy(x)
    xn = F.rms_norm(xt, (cfg["hidden"],), torch.from_numpy(lw["in_norm"]), eps=EPS)
    vb = F.linear(xn, torch.from_numpy(lw["wv"])).numpy().reshape(4, nkv, hd)
    want = np.empty_like(x)
    for m in range(4):
        keys = [cv[0][j] for j in range(cpos.size) if p[m] - W <= cpos[j]] + [vb[j] for j in range(4)]
        mean = np.mean(np.stack(keys), axis=0)                  # [nkv, hd]
        a = np.concatenate([mean[h // (nq // nkv)] for h in range(nq)])
        want[m] = x[m] + lw["wo"] @ a
    _close(got, want, 2e-6)
    # the context rows are really cut at distance W: row p - W - 1 is outside
    assert p[0] - W - 1 == 15 and (cpos < p[0] - W).sum() == 16


def _mlp_fixture():
    """Weights whose MLP output is known in closed form: block rows e_0
    (anchor) and e_1 (mask) of unit size, post-norm gain 1/8 (so the normed
    row is kappa * e_j), input-norm gain 3 (a different scale, used by
    nothing here), gate columns of 10 and up columns of known integers."""
    cfg = _cfg()
    H, I = cfg["hidden"], cfg["intermediate"]
    w = _weights(cfg)
    lw = w["layers"][0]
    lw["wo"][:] = 0.0
    lw["in_norm"][:] = 3.0
    lw["post_norm"][:] = 0.125
    lw["wg"][:] = 0.0
    lw["wu"][:] = 0.0
    lw["wd"][:] = 0.0
    up0 = (np.arange(H) % 3) + 1.0
    lw["wg"][:H, 0] = 10.0
    lw["wu"][:H, 0] = up0
    lw["wg"][H:, 1] = 10.0
    lw["wu"][H:, 1] = 2.0
    lw["wd"][np.arange(H), np.arange(H)] = 1.0          # row 0's gate rows -> outputs 0..H-1
    lw["wd"][np.arange(H), H + np.arange(H)] = 0.5      # row 1's gate rows -> every output
    x = np.zeros((4, H))
    x[0, 0] = 1.0
    x[1:, 1] = 1.0
    return cfg, lw, x, up0


def test_mlp_wiring_closed_form():
    """x' = h + Wd (silu(Wg hn) * (Wu hn)) with hn = post_norm(h), h = x here
    (Wo = 0). kappa = (1/8) / sqrt(1/64 + eps) and silu(z) = z / (1 + e^-z)
    at z = 10 kappa give the exact result; gate and up swapped, the input norm
    (gain 3) in place of the post-attention norm, no norm at all, or a
    residual taken from hn all change it."""
    cfg, lw, x, up0 = _mlp_fixture()
    H = cfg["hidden"]
    ck = np.zeros((0, cfg["n_kv_heads"], cfg["head_dim"]))
    got = O.drafter_layer(cfg, lw, x, 40 + np.arange(4), ck, ck, np.zeros(0, np.int64))
    kappa = 1.0 / math.sqrt(1.0 + H * EPS)
    z = 10.0 * kappa
    silu_z = z / (1.0 + math.exp(-z))
    want = x.copy()
    want[0] += silu_z * up0 * kappa
    want[1:] += silu_z * 2.0 * kappa * 0.5
    _close(got, want, 2e-6)
    swapped = x[0] + np.array([(u * kappa) / (1 + math.exp(-u * kappa)) * z for u in up0])
    assert np.abs(got[0] - swapped).max() > 1.0


def test_mlp_reads_the_post_attention_sum():
    """With uniform attention (Wq = Wk = 0), h = x + Wo . mean(V) is known
    (the first test). The MLP part of the layer, x' - h, must then change
    when Wo changes: an MLP reading x (or the input norm of x) would not see
    Wo at all."""
    cfg = _cfg()
    w = _weights(cfg)
    lw = w["layers"][0]
    lw["wq"][:] = 0.0
    lw["wk"][:] = 0.0
    ck, cv, cpos = _context(cfg, w)
    rng = np.random.default_rng(9)
    x = O.round_f32(rng.standard_normal((4, cfg["hidden"])))
    p = 32 + np.arange(4)
    diffs = []
    for scale in (1.0, 3.0):
        l2 = dict(lw, wo=lw["wo"] * scale)
        y = O.drafter_layer(cfg, l2, x, p, ck[0], cv[0], cpos)
        no_mlp = O.drafter_layer(cfg, dict(l2, wg=np.zeros_like(lw["wg"])), x, p, ck[0], cv[0], cpos)
        diffs.append(y - no_mlp)                       # the MLP's contribution
    assert np.abs(diffs[0] - diffs[1]).max() > 1e-3 * np.abs(diffs[0]).max()


# --- the context path ----------------------------------------------------------------

@pytest.mark.parametrize("neox", [True, False])
def test_context_kv_one_hot_rows(neox):
    """One-hot encoder.fc and Wk / Wv make every context row's K and V
    computable by hand: C = f / sqrt(mean(f^2) + eps) from two chosen
    residual entries, K = the per-head RMSNorm of the selected C entries,
    rotated at the row's absolute position, and V = the selected C entries
    unchanged (no norm, no RoPE). The layer's input-norm gain (7) must not
    enter: the context path has no input norm."""
    cfg = _cfg(rope_neox=neox)
    H, hd = cfg["hidden"], cfg["head_dim"]
    kin = cfg["k_target_layers"] * cfg["target_hidden"]
    w = _weights(cfg)
    lw = w["layers"][0]
    lw["in_norm"][:] = 7.0
    w["fc"][:] = 0.0
    w["fc"][np.arange(H), 5 * np.arange(H) + 3] = 1.0      # f_i = resid[5 i + 3]
    lw["wk"][:] = 0.0
    lw["wv"][:] = 0.0
    d1 = hd // 2 if neox else 1                             # partner of dim 0
    d3 = 3 if neox else 6                                   # a pair with frequency index 3
    lw["wk"][0, 0] = 1.0                                    # head 0, dim 0 <- C_0
    lw["wk"][d1, 1] = 1.0                                   # head 0, its partner <- C_1
    lw["wk"][hd + d3, 0] = 2.0                              # head 1, pair 3 <- 2 C_0
    lw["wv"][5, 1] = 1.0                                    # V head 0 dim 5 <- C_1
    lw["wv"][hd + 2, 0] = -1.0                              # V head 1 dim 2 <- -C_0
    pos = np.array([0, 7, 1000, 123457])
    a = np.array([1.0, -2.0, 0.5, 3.0])
    b = np.array([0.0, 1.0, -4.0, 0.25])
    resid = np.zeros((4, kin))
    resid[:, 3] = a
    resid[:, 8] = b
    K, V, C = O.context_kv(cfg, w, resid, pos)
    theta = cfg["rope_theta"]
    f3 = theta ** (-6.0 / hd)                               # inv freq of pair index 3
    for r in range(4):
        rms = math.sqrt((a[r] ** 2 + b[r] ** 2) / H + EPS)
        c0, c1 = a[r] / rms, b[r] / rms
        assert abs(C[r, 0] - c0) < 1e-5 * abs(c0) + 1e-6 and abs(C[r, 1] - c1) < 1e-5 * abs(c1) + 1e-6
        n0 = math.sqrt((c0 * c0 + c1 * c1) / hd + EPS)
        u, v = c0 / n0, c1 / n0
        ang = float(pos[r])
        k0 = np.zeros(hd)
        k0[0] = u * math.cos(ang) - v * math.sin(ang)
        k0[d1] = u * math.sin(ang) + v * math.cos(ang)
        n1 = math.sqrt((2 * c0) ** 2 / hd + EPS)
        u1 = 2 * c0 / n1
        k1 = np.zeros(hd)
        partner3 = d3 + hd // 2 if neox else d3 + 1
        k1[d3] = u1 * math.cos(ang * f3)
        k1[partner3] = u1 * math.sin(ang * f3)
        np.testing.assert_allclose(K[0][r, 0], k0, rtol=0, atol=2e-5 * abs(u1 if abs(u1) > 1 else 1) + 2e-5)
        np.testing.assert_allclose(K[0][r, 1], k1, rtol=0, atol=2e-5 * max(1.0, abs(u1)))
        v_want = np.zeros((2, hd))
        v_want[0, 5] = c1
        v_want[1, 2] = -c0
        np.testing.assert_allclose(V[0][r], v_want, rtol=0, atol=1e-5 * max(1.0, abs(c0), abs(c1)))


# --- the read-out ----------------------------------------------------------------------

@pytest.mark.parametrize("kind", ["dflash", "dspark"])
def test_draft_read_out_rows_and_lm_head(kind):
    """Identity layers (Wo = Wd = 0) leave the embedded rows; the final norm
    of a unit row e_j is kappa e_j * 8 * gain; an lm_head that copies hidden
    unit j into vocabulary entry 2 j makes the logits known. DFlash reads out
    block rows 1..B-1 (the mask rows), DSpark every row of its B-1 row block,
    so the ids and the capped maxima follow by hand; softcap c tanh(z / c)
    with c = 20."""
    cfg = _cfg(kind=kind, softcap=20.0)
    H, V = cfg["hidden"], cfg["vocab"]
    w = _weights(cfg)
    lw = w["layers"][0]
    lw["wo"][:] = 0.0
    lw["wd"][:] = 0.0
    anchor, mask = 5, cfg["mask_token_id"]
    w["embed"][anchor] = 0.0
    w["embed"][anchor, 3] = 1.0
    w["embed"][mask] = 0.0
    w["embed"][mask, 9] = -1.0
    w["final_norm"][:] = 0.5
    w["lm_head"][:] = 0.0
    w["lm_head"][2 * np.arange(H), np.arange(H)] = 1.0       # logit 2j = hidden j
    w["lm_head"][2 * np.arange(H) + 1, np.arange(H)] = -1.0  # logit 2j+1 = -hidden j
    ck = np.zeros((0, cfg["n_kv_heads"], cfg["head_dim"]))
    out = O.draft_block(cfg, w, [ck], [ck], np.zeros(0, np.int64), anchor, 100, 4)
    scale = 0.5 / math.sqrt(1.0 / H + EPS)                   # final-norm value of a unit entry
    if kind == "dflash":
        assert out["hidden"].shape[0] == 4
        want_ids = [2 * 9 + 1] * 3                           # mask rows: hidden 9 = -scale
    else:
        assert out["hidden"].shape[0] == 3
        want_ids = [2 * 3] + [2 * 9 + 1] * 2                 # anchor row: hidden 3 = +scale
    assert out["draft_ids"].tolist() == want_ids
    np.testing.assert_allclose(out["logits"].max(axis=1), 20.0 * math.tanh(scale / 20.0), rtol=1e-6)
    assert np.allclose(out["positions"], 100 + np.arange(out["hidden"].shape[0]))


# --- storage rounding and the session ------------------------------------------------------

def test_round_f32_is_ieee_single():
    vals = [1.0 / 3.0, 1e-40, -2.5e38, 0.1, 16777217.0, math.pi]
    want = [struct.unpack("f", struct.pack("f", v))[0] for v in vals]
    assert O.round_f32(np.array(vals)).tolist() == want


def test_session_history_is_the_ring_window():
    """The session's dense history (context rows by absolute position, the
    verify's kept rows appended) exposes exactly the rows a ring of capacity
    W + slack would hold for the window after the same appends and trims."""
    cfg = synth.config("tiny")
    w = _weights(synth.config("tiny"))
    stream = synth.make_target_stream(cfg, 12, 4, seed=2)
    s = O.OracleSession(cfg, w)
    s.ingest(O.as_f64(synth.make_context(cfg, 32, seed=2), "f32"), 0, anchor=5)
    ring = O.RingModel(cfg["window"], O.ring_capacity(cfg["window"], 4), row_shape=(1,))
    ring.append(np.arange(32, dtype=np.float64)[:, None])
    for r in range(12):
        d = s.draft(4)
        L = synth.planted_logits(stream, r, 4, d["draft_ids"])
        tokens, n, _ = s.verify(O.as_f64(L, "f32"), d["draft_ids"])
        s.append_and_trim(O.as_f64(synth.resid_rows(stream, r, 4), "f32"), n)
        ring.append((s.pos + np.arange(4, dtype=np.float64))[:, None])
        ring.trim(4 - n)
        s.commit(n, tokens[-1], 4, n - 1)
        _, _, vis = s.visible_context()
        assert s.pos == ring.offset
        assert vis.tolist() == ring.slot_view(ring.window_positions())[:, 0].astype(int).tolist()
