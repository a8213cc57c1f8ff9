"""The composition pins catch plausible slips: each test here plants one
mistake in the oracle (on the CPU, through monkeypatch, for this test only)
and checks that at least one closed-form pin of
tests/test_oracle_composition.py then fails, and that all of them pass on the
oracle as it is.

The mistakes are the ones a restatement of the pages' drafter could make: V
projected from the un-normed input, the sliding window one short, the
residual taken from the normed input, the MLP reading x or the input norm
instead of the post-attention norm, the MLP norm using the input norm's gain,
gate and up swapped, the layer's output residual taken from the MLP norm, an
input norm on the context path, RoPE or the k-norm applied to the context V,
context positions shifted by one, and the DFlash read-out taking the anchor
row instead of the mask rows.
"""

import inspect

import numpy as np
import pytest

import oracle as O
import test_oracle_composition as T
from oracle import dflash_oracle as D

_PARAMS = {
    "test_context_kv_one_hot_rows": [True, False],
    "test_draft_read_out_rows_and_lm_head": ["dflash", "dspark"],
}


def _failing_pins():
    """Names of the composition pins that fail on the oracle as patched."""
    fails = set()
    for name, fn in inspect.getmembers(T, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        for p in _PARAMS.get(name, [None]):
            try:
                fn() if p is None else fn(p)
            except Exception:   # an assertion, or a shape the slip broke
                fails.add(name)
    return sorted(fails)


def _mutant_layer(mut):
    """The oracle's drafter layer with one slip planted."""

    def layer(cfg, lw, x, pos, ctx_k, ctx_v, ctx_pos):
        rnd = D.rounder(cfg["dtype"])
        eps = cfg["rms_eps"]
        nq, nkv, hd = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
        rows = x.shape[0]
        xn = rnd(D.rmsnorm(x, lw["in_norm"], eps))
        q = rnd(D.linear(xn, lw["wq"])).reshape(rows, nq, hd)
        k = rnd(D.linear(xn, lw["wk"])).reshape(rows, nkv, hd)
        v = rnd(D.linear(x if mut == "v_from_x" else xn, lw["wv"])).reshape(rows, nkv, hd)
        q = rnd(D.rope(D.head_rmsnorm(q, lw["q_norm"], eps), pos, cfg["rope_theta"], cfg["rope_neox"]))
        k = rnd(D.rope(D.head_rmsnorm(k, lw["k_norm"], eps), pos, cfg["rope_theta"], cfg["rope_neox"]))
        keys = np.concatenate([ctx_k, k])
        vals = np.concatenate([ctx_v, v])
        kpos = np.concatenate([ctx_pos, pos])
        win = cfg["window"] - 1 if mut == "window_short" else cfg["window"]
        a = rnd(D.attention(q, keys, vals, pos, kpos, win))
        o = rnd(D.linear(a.reshape(rows, nq * hd), lw["wo"]))
        h = rnd((xn if mut == "resid_from_xn" else x) + o)
        gain = lw["in_norm"] if mut == "mlp_in_gain" else lw["post_norm"]
        if mut == "mlp_reads_xn":
            hn = xn
        else:
            hn = rnd(D.rmsnorm(x if mut == "mlp_reads_x" else h, gain, eps))
        g = rnd(D.linear(hn, lw["wg"]))
        u = rnd(D.linear(hn, lw["wu"]))
        if mut == "gate_up_swapped":
            g, u = u, g
        s = rnd(D.silu(g) * u)
        d = rnd(D.linear(s, lw["wd"]))
        return rnd((hn if mut == "out_resid_from_hn" else h) + d)

    return layer


def _mutant_context(mut):
    """The oracle's context K/V path with one slip planted."""

    def context_kv(cfg, w, resid, pos):
        rnd = D.rounder(cfg["dtype"])
        eps = cfg["rms_eps"]
        nkv, hd = cfg["n_kv_heads"], cfg["head_dim"]
        c = rnd(D.rmsnorm(rnd(D.linear(resid, w["fc"])), w["hidden_norm"], eps))
        ks, vs = [], []
        for lw in w["layers"]:
            cc = rnd(D.rmsnorm(c, lw["in_norm"], eps)) if mut == "ctx_input_norm" else c
            k = rnd(D.linear(cc, lw["wk"])).reshape(-1, nkv, hd)
            v = rnd(D.linear(cc, lw["wv"])).reshape(-1, nkv, hd)
            kp = pos + 1 if mut == "ctx_pos_shift" else pos
            k = rnd(D.rope(D.head_rmsnorm(k, lw["k_norm"], eps), kp, cfg["rope_theta"], cfg["rope_neox"]))
            if mut == "ctx_v_rope":
                v = rnd(D.rope(v, pos, cfg["rope_theta"], cfg["rope_neox"]))
            if mut == "ctx_v_norm":
                v = rnd(D.head_rmsnorm(v, lw["k_norm"], eps))
            ks.append(k)
            vs.append(v)
        return ks, vs, c

    return context_kv


def _anchor_read_out(orig):
    def block_tokens(cfg, anchor, block):
        toks, read = orig(cfg, anchor, block)
        if cfg.get("kind", "dflash") != "dspark":
            read = np.arange(0, block - 1)
        return toks, read

    return block_tokens


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(D, name, fn)
    monkeypatch.setattr(O, name, fn)


def test_pins_pass_on_the_oracle():
    assert _failing_pins() == []


@pytest.mark.parametrize("mut", ["v_from_x", "window_short", "resid_from_xn", "mlp_reads_x", "mlp_reads_xn",
                                 "mlp_in_gain", "gate_up_swapped", "out_resid_from_hn"])
def test_a_slip_in_the_layer_fails_a_pin(monkeypatch, mut):
    _patch(monkeypatch, "drafter_layer", _mutant_layer(mut))
    assert _failing_pins(), mut


@pytest.mark.parametrize("mut", ["ctx_input_norm", "ctx_v_rope", "ctx_v_norm", "ctx_pos_shift"])
def test_a_slip_in_the_context_path_fails_a_pin(monkeypatch, mut):
    _patch(monkeypatch, "context_kv", _mutant_context(mut))
    assert _failing_pins(), mut


def test_reading_out_the_anchor_row_fails_a_pin(monkeypatch):
    _patch(monkeypatch, "block_tokens", _anchor_read_out(D.block_tokens))
    assert _failing_pins()


def test_the_unpatched_layer_copy_agrees_with_the_oracle():
    """The mutant factory with no slip reproduces the oracle's layer exactly,
    so each mutant differs from the oracle by its one slip only."""
    cfg = T._cfg()
    w = T._weights(cfg)
    k, v, pos = T._context(cfg, w)
    x = np.random.default_rng(1).standard_normal((4, cfg["hidden"]))
    p = np.arange(32, 36)
    want = D.drafter_layer(cfg, w["layers"][0], x, p, k[0], v[0], pos)
    got = _mutant_layer(None)(cfg, w["layers"][0], x, p, k[0], v[0], pos)
    np.testing.assert_array_equal(got, want)
    resid = O.as_f64(T.synth.make_context(cfg, 8, seed=2), "f32")
    a, b = D.context_kv(cfg, w, resid, np.arange(8)), _mutant_context(None)(cfg, w, resid, np.arange(8))
    for x0, x1 in zip(a[0] + a[1] + [a[2]], b[0] + b[1] + [b[2]]):
        np.testing.assert_array_equal(x0, x1)
