"""Pins of the oracle's synthetic target (the verify forward, the residual
capture and the cache trim), each against something other than the oracle's
own formulas: explicit triangular/band constructions and brute force for the
causal mask, torch's scaled-dot-product attention for the masked attention,
closed forms on constructed weights (identity layers, uniform attention),
and invariants of the cache (one pass equals prefill then verify; a trim
equals never having appended the dropped rows). Runs on CPU.

Sources: "Muse Glimmer DFlash assistant drafter on the round loop", "What
changed" (the Muse target: residual-stream capture before the final norm,
trim rollback over the mixed sliding / full caches); "LFM2 / LFM2.5 DSpark
drafter on the DFlash loop", "Short-conv rollback" (attention layers trim
their KV cache after a partial accept).
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O
from block_speculative_decoding_dflash_gb300 import synth


def _f64(w):
    out = {k: O.as_f64(v, "f32") for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: O.as_f64(v, "f32") for k, v in lw.items()} for lw in w["layers"]]
    return out


@pytest.fixture(scope="module")
def tiny():
    cfg = synth.config("tiny")
    tc = synth.target_config("tiny")
    return tc, _f64(synth.make_target_weights(tc, synth.make_weights(cfg, 0)))


def test_causal_mask_against_triangles_and_brute_force():
    n = 12
    pos = np.arange(n)
    tri = np.tril(np.ones((n, n), dtype=bool))
    assert np.array_equal(O.causal_mask(pos, pos, 0), tri)
    for w in (1, 3, 11, 20):
        band = tri & np.triu(np.ones((n, n), dtype=bool), -w)
        assert np.array_equal(O.causal_mask(pos, pos, w), band)
    rng = np.random.default_rng(0)
    q, k = rng.integers(0, 40, 7), rng.integers(0, 40, 9)
    for w in (0, 5):
        brute = np.array([[kk <= qq and (w == 0 or qq - kk <= w) for kk in k] for qq in q])
        assert np.array_equal(O.causal_mask(q, k, w), brute)


@pytest.mark.parametrize("window", [0, 4])
def test_causal_attention_matches_torch_sdpa(window):
    rng = np.random.default_rng(1)
    nq, nkv, hd, hist, rows = 4, 2, 8, 10, 5
    q = rng.standard_normal((rows, nq, hd))
    k = rng.standard_normal((hist + rows, nkv, hd))
    v = rng.standard_normal((hist + rows, nkv, hd))
    qpos = np.arange(hist, hist + rows)
    kpos = np.arange(hist + rows)
    got = O.causal_attention(q, k, v, qpos, kpos, window)
    # torch: boolean mask from a shifted lower triangle (and band)
    full = torch.ones(rows, hist + rows, dtype=torch.bool).tril(hist)
    if window:
        full &= torch.ones(rows, hist + rows, dtype=torch.bool).triu(hist - window)
    qt = torch.from_numpy(q).permute(1, 0, 2)                      # [nq, rows, hd]
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(nq // nkv, 0)
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(nq // nkv, 0)
    want = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=full).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_identity_layers_give_raw_embedding_streams_and_plain_logits(tiny):
    """Wo = Wd = 0 makes every layer the identity, so every captured stream is
    the raw embedding row and the logits are lm_head(final_norm(embed)) in
    fp32, without softcap (readings R14-R16)."""
    tc, tw = tiny
    tw = dict(tw, layers=[dict(lw, wo=lw["wo"] * 0, wd=lw["wd"] * 0) for lw in tw["layers"]])
    toks = synth.make_prompt(tc, 9, seed=3)
    out = O.TargetSession(tc, tw).forward(toks)
    e = tw["embed"][toks]
    k = len(tc["capture"])
    np.testing.assert_array_equal(out["captured"], np.tile(e, (1, k)))
    ms = np.mean(e * e, axis=1, keepdims=True)
    xf = O.round_f32(e / np.sqrt(ms + tc["rms_eps"]))
    want = O.round_f32((xf @ tw["lm_head"].T).astype(np.float32))
    np.testing.assert_allclose(out["logits"], want, rtol=1e-6, atol=1e-7)


def test_capture_order_and_layer_indices(tiny):
    """Only layer 2 is not the identity: the streams after layers 0 and 1
    equal the embedding, those after 2.. equal layer 2's output, and the
    captured blocks follow the capture list's order."""
    tc, tw = tiny
    layers = [dict(lw, wo=lw["wo"] * 0, wd=lw["wd"] * 0) if i != 2 else lw for i, lw in enumerate(tw["layers"])]
    tc2 = dict(tc, capture=(4, 0, 1, 2))
    toks = synth.make_prompt(tc, 6, seed=4)
    out = O.TargetSession(tc2, dict(tw, layers=layers)).forward(toks)
    H = tc["hidden"]
    e = tw["embed"][toks]
    blocks = [out["captured"][:, i * H:(i + 1) * H] for i in range(4)]
    np.testing.assert_array_equal(blocks[1], e)
    np.testing.assert_array_equal(blocks[2], e)
    assert np.abs(blocks[3] - e).max() > 1e-3
    np.testing.assert_array_equal(blocks[0], blocks[3])


def test_uniform_attention_is_the_causal_mean_of_visible_values(tiny):
    """Wq = Wk = 0 makes every visible score 0: with Wg = 0 (no MLP) a layer
    is x + Wo . mean of the visible V rows, the keys in [pos - W, pos] for a
    sliding layer and [0, pos] for a full one (both pinned on one layer)."""
    tc, tw = tiny
    rng = np.random.default_rng(5)
    H, nq, nkv, hd = tc["hidden"], tc["n_q_heads"], tc["n_kv_heads"], tc["head_dim"]
    lw = dict(tw["layers"][0], wq=tw["layers"][0]["wq"] * 0, wk=tw["layers"][0]["wk"] * 0,
              wg=tw["layers"][0]["wg"] * 0)
    hist = 30
    hk = rng.standard_normal((hist, nkv, hd))
    hv = rng.standard_normal((hist, nkv, hd))
    hp = np.arange(hist)
    x = rng.standard_normal((3, H))
    pos = np.arange(hist, hist + 3)
    for window in (0, 7):
        y, _, v_rows = O.target_layer(tc, lw, x, pos, hk, hv, hp, window)
        allv = np.concatenate([hv, v_rows])
        allp = np.concatenate([hp, pos])
        for i in range(3):
            vis = (allp <= pos[i]) & ((window == 0) | (pos[i] - allp <= window))
            mean = allv[vis].mean(axis=0)                         # [nkv, hd]
            a = np.repeat(mean, nq // nkv, axis=0).reshape(-1)
            want = x[i] + O.round_f32(O.round_f32(a) @ lw["wo"].T)
            np.testing.assert_allclose(y[i], O.round_f32(want), rtol=1e-5, atol=1e-6)


def test_one_pass_equals_prefill_then_verify(tiny):
    tc, tw = tiny
    toks = synth.make_prompt(tc, 40, seed=6)
    one = O.TargetSession(tc, tw).forward(toks)
    s = O.TargetSession(tc, tw)
    s.forward(toks[:32])
    two = s.forward(toks[32:])
    np.testing.assert_allclose(two["logits"], one["logits"][32:], rtol=0, atol=1e-12)
    np.testing.assert_allclose(two["captured"], one["captured"][32:], rtol=0, atol=1e-12)


@pytest.mark.parametrize("n", [1, 3, 8])
def test_trim_equals_never_appending_the_dropped_rows(tiny, n):
    """verify(B) then commit(n) leaves the caches of a run that only ever saw
    the first n block tokens (reading R17): the next forward agrees."""
    tc, tw = tiny
    toks = synth.make_prompt(tc, 60, seed=7)
    prompt, block, nxt = toks[:40], toks[40:48], toks[48:52]
    a = O.TargetSession(tc, tw)
    a.forward(prompt)
    a.forward(block)
    a.commit(n)
    assert a.pos == 40 + n
    got = a.forward(nxt)
    b = O.TargetSession(tc, tw)
    b.forward(np.concatenate([prompt, block[:n]]))
    want = b.forward(nxt)
    np.testing.assert_allclose(got["logits"], want["logits"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["captured"], want["captured"], rtol=0, atol=1e-12)


def test_commit_refuses_a_short_rewind(tiny):
    tc, tw = tiny
    s = O.TargetSession(tc, tw)
    s.forward(synth.make_prompt(tc, 5))
    with pytest.raises(ValueError):
        s.commit(6)
