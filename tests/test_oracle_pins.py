"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties an oracle function to something other than itself: values the
pages print, closed forms, library routines (torch fp64), invariants, or brute
force on tiny inputs. Runs on CPU only.
"""

import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O
from block_speculative_decoding_dflash_gb300 import synth

RNG = np.random.default_rng(1234)


# --- slack rule and ring ---------------------------------------------------

def test_slack_rule_matches_page_table(golden):
    for b, floored, unfloored in golden("slack_rule.txt"):
        assert O.speculative_slack(int(b)) == int(floored)
        assert O.speculative_slack(int(b), floor=False) == int(unfloored)


def test_slack_never_below_block():
    for b in range(1, 600):
        assert O.speculative_slack(b) >= b


@pytest.mark.parametrize("block", [4, 5, 8, 16, 32, 129])
def test_ring_append_trim_restores_window(block):
    W = 2048
    ring = O.RingModel(W, O.ring_capacity(W, block), row_shape=(2,))
    ring.append(RNG.standard_normal((W + 300, 2)))
    pos = ring.window_positions()
    before = ring.slot_view(pos).copy()
    ring.append(RNG.standard_normal((block, 2)))
    ring.trim(block)
    after = ring.slot_view(ring.window_positions())
    assert np.array_equal(before, after)
    assert np.array_equal(after, ring.history_view(pos))


def test_unfloored_slack_corrupts_row_128_at_block_129():
    """Muse page, "Pre-merge review round": without the floor a 129-row
    append overwrites a still-visible window row that trim cannot restore."""
    W, B = 2048, 129
    ring = O.RingModel(W, O.ring_capacity(W, B, floor=False), row_shape=(1,))
    ring.append(np.arange(W + 300, dtype=np.float64)[:, None])
    pos = ring.window_positions()
    block_rows = -1.0 - np.arange(B, dtype=np.float64)[:, None]
    ring.append(block_rows)
    ring.trim(B)
    view = ring.slot_view(pos)
    truth = ring.history_view(pos)
    bad = np.nonzero(view[:, 0] != truth[:, 0])[0]
    assert bad.tolist() == [0]                     # the oldest visible row ...
    assert view[0, 0] == block_rows[128, 0]        # ... holds block row j = 128
    ring2 = O.RingModel(W, O.ring_capacity(W, B), row_shape=(1,))
    ring2.append(np.arange(W + 300, dtype=np.float64)[:, None])
    ring2.append(block_rows)
    ring2.trim(B)
    assert np.array_equal(ring2.slot_view(pos), ring2.history_view(pos))


def test_ring_wraparound_random_rounds():
    W, B = 64, 16
    ring = O.RingModel(W, O.ring_capacity(W, B), row_shape=(3,))
    ring.append(RNG.standard_normal((W, 3)))
    for _ in range(256):
        b = int(RNG.integers(1, B + 1))
        ring.append(RNG.standard_normal((b, 3)))
        ring.trim(int(RNG.integers(0, b + 1)))
        pos = ring.window_positions()
        assert np.array_equal(ring.slot_view(pos), ring.history_view(pos))


def test_short_rewind_is_an_error():
    ring = O.RingModel(8, O.ring_capacity(8, 4))
    ring.append(np.zeros((4, 1)))
    ring.trim(2)
    with pytest.raises(ValueError):
        ring.trim(1)          # nothing appended since the last trim
    ring.append(np.zeros((3, 1)))
    with pytest.raises(ValueError):
        ring.trim(4)


# --- verify / accept ---------------------------------------------------------

def _onehot_logits(t, V):
    L = np.zeros((len(t), V), dtype=np.float32)
    for i, ti in enumerate(t):
        L[i, ti] = 1.0
    return L


@pytest.mark.parametrize("B", [2, 3, 4, 5])
def test_accept_brute_force(B):
    V = 3
    for t in itertools.product(range(V), repeat=B):
        for d in itertools.product(range(V), repeat=B - 1):
            tokens, n, targ = O.verify_accept(_onehot_logits(t, V), np.array(d))
            assert targ.tolist() == list(t)
            cands = [a for a in range(B) if all(d[i] == t[i] for i in range(a))]
            a = max(cands)
            assert n == a + 1
            assert tokens.tolist() == list(d[:a]) + [t[a]]


def test_verify_ties_take_lowest_index():
    L = np.zeros((3, 10), dtype=np.float32)
    L[:, 3] = 2.0
    L[:, 7] = 2.0
    tokens, n, t = O.verify_accept(L, np.array([3, 3]))
    assert t.tolist() == [3, 3, 3] and n == 3
    tokens, n, t = O.verify_accept(L, np.array([7, 3]))
    assert n == 1 and tokens.tolist() == [3]


def test_round_counters_match_pages(golden):
    for name, rounds, proposed, accepted, tokens, ratio, printed in golden("round_counters.txt"):
        r = O.stats_ratios(int(rounds), int(proposed), int(accepted))
        digits = len(printed.split(".")[1])
        assert round(r[ratio], digits) == float(printed), name
        if tokens != "-":
            assert r["emitted"] == int(tokens), name


# --- mask and attention ------------------------------------------------------

def test_mask_symmetric_and_bounded():
    pos = np.arange(40)
    for W in (1, 5, 16):
        M = O.visible_mask(pos, pos, W)
        assert np.array_equal(M, M.T)
        d = np.abs(pos[:, None] - pos[None, :])
        assert np.array_equal(M, d <= W)
        assert M[0, W] and not M[0, W + 1]
    assert O.visible_mask(pos, pos, 0).all()


def _sdpa_reference(q, k, v, q_pos, k_pos, W):
    """torch fp64 scaled_dot_product_attention with a boolean mask; kv heads
    expanded with repeat_interleave (contiguous query groups)."""
    nq, nkv = q.shape[1], k.shape[1]
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(nq // nkv, dim=0)
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(nq // nkv, dim=0)
    qp = torch.from_numpy(np.asarray(q_pos))
    kp = torch.from_numpy(np.asarray(k_pos))
    mask = None
    if W > 0:
        mask = (qp[:, None] - kp[None, :]).abs() <= W
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("W", [0, 3, 7, 100])
def test_attention_matches_torch_sdpa(W):
    nq, nkv, hd, nk, bq = 8, 2, 16, 30, 5
    q = RNG.standard_normal((bq, nq, hd))
    k = RNG.standard_normal((nk, nkv, hd))
    v = RNG.standard_normal((nk, nkv, hd))
    k_pos = np.arange(nk) + 3
    q_pos = np.arange(bq) + 20
    got = O.attention(q, k, v, q_pos, k_pos, W)
    ref = _sdpa_reference(q, k, v, q_pos, k_pos, W)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_attention_unbounded_window_equals_full_bidirectional():
    nq, nkv, hd, nk, bq = 4, 4, 8, 12, 12
    q = RNG.standard_normal((bq, nq, hd))
    k = RNG.standard_normal((nk, nkv, hd))
    v = RNG.standard_normal((nk, nkv, hd))
    pos = np.arange(12)
    a = O.attention(q, k, v, pos, pos, 1000)
    b = O.attention(q, k, v, pos, pos, 0)
    ref = _sdpa_reference(q, k, v, pos, pos, 0)
    np.testing.assert_allclose(a, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(a, b)


# --- RoPE ----------------------------------------------------------------------

def test_rope_traditional_is_complex_rotation():
    hd, theta = 16, 1e6
    x = RNG.standard_normal((5, 3, hd))
    pos = np.array([0, 1, 17, 1000, 123456])
    got = O.rope(x, pos, theta, neox=False)
    z = x[..., 0::2] + 1j * x[..., 1::2]
    freqs = np.array([theta ** (-(2 * i) / hd) for i in range(hd // 2)])
    rot = np.exp(1j * pos[:, None, None] * freqs[None, None, :])
    w = z * rot
    ref = np.empty_like(x)
    ref[..., 0::2], ref[..., 1::2] = w.real, w.imag
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-10)


def test_rope_neox_is_traditional_on_permuted_pairs():
    hd, theta = 16, 1e6
    x = RNG.standard_normal((4, 2, hd))
    pos = np.array([3, 9, 40, 77])
    perm = np.empty(hd, dtype=int)          # neox pair (i, i + hd/2) -> (2i, 2i+1)
    perm[0::2] = np.arange(hd // 2)
    perm[1::2] = np.arange(hd // 2) + hd // 2
    trad = O.rope(x[..., perm], pos, theta, neox=False)
    back = np.empty_like(trad)
    back[..., perm] = trad
    np.testing.assert_allclose(O.rope(x, pos, theta, neox=True), back, rtol=1e-12, atol=1e-12)


def test_rope_norm_preserving_and_relative():
    hd, theta = 32, 1e4
    q = RNG.standard_normal((1, 1, hd))
    k = RNG.standard_normal((1, 1, hd))
    for neox in (True, False):
        r = O.rope(q, np.array([57]), theta, neox)
        assert abs(np.linalg.norm(r) - np.linalg.norm(q)) < 1e-12
        dots = []
        for m in (5, 50, 500):
            dots.append(float(np.sum(O.rope(q, np.array([m + 7]), theta, neox) *
                                     O.rope(k, np.array([m]), theta, neox))))
        assert max(dots) - min(dots) < 1e-9
    assert not np.allclose(O.rope(q, np.array([3]), theta, True),
                           O.rope(q, np.array([3]), theta, False))


# --- RMSNorm, linear, silu, softcap, argmax, bf16 ------------------------------

def test_rmsnorm_matches_torch():
    x = RNG.standard_normal((7, 64))
    g = RNG.standard_normal(64)
    ref = F.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(O.rmsnorm(x, g, 1e-6), ref, rtol=1e-12, atol=1e-12)
    y = O.rmsnorm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, atol=1e-12)
    np.testing.assert_allclose(O.rmsnorm(3.5 * x, g, 0.0), O.rmsnorm(x, g, 0.0), atol=1e-12)


def test_linear_orientation():
    out_f, in_f = 5, 7
    perm = RNG.permutation(in_f)[:out_f]
    W = np.zeros((out_f, in_f))
    W[np.arange(out_f), perm] = 1.0          # output o reads input perm[o]
    x = RNG.standard_normal((3, in_f))
    np.testing.assert_array_equal(O.linear(x, W), x[:, perm])
    a, b = RNG.standard_normal(out_f), RNG.standard_normal(in_f)
    np.testing.assert_allclose(O.linear(x, np.outer(a, b)), np.outer(x @ b, a), atol=1e-12)


def test_silu_against_torch():
    x = RNG.standard_normal(100) * 5
    np.testing.assert_allclose(O.silu(x), F.silu(torch.from_numpy(x)).numpy(), rtol=1e-14)


def test_softcap_properties():
    z = np.linspace(-80, 80, 2001).astype(np.float32)
    c = O.softcap(z, 20.0)
    assert np.all(np.diff(c) >= 0) and np.all(np.abs(c) <= 20.0)
    # tanh(1) = 0.76159415595576488812 (tabulated constant)
    assert abs(float(O.softcap(np.float32([20.0]), 20.0)[0]) - 20.0 * 0.7615941559557649) < 2e-6
    small = np.float32([1e-3, -2e-3])
    np.testing.assert_allclose(O.softcap(small, 20.0), small, rtol=1e-5)
    np.testing.assert_array_equal(O.softcap(z, 0.0), z)
    zz = RNG.standard_normal((4, 1000)).astype(np.float32) * 3
    assert np.array_equal(O.argmax_lowest(O.softcap(zz, 20.0)), O.argmax_lowest(zz))


def test_argmax_ties_lowest():
    z = np.array([[1, 5, 5, 2], [7, 7, 7, 7], [0, 0, 0, 1]], dtype=np.float32)
    assert O.argmax_lowest(z).tolist() == [1, 0, 3]


def test_bf16_rounding_matches_torch():
    a = RNG.standard_normal(100000).astype(np.float32) * np.float32(10.0) ** RNG.integers(-30, 30, 100000).astype(np.float32)
    # exact ties: fp32 values halfway between two bf16 values
    base = (RNG.integers(0, 2 ** 15, 1000).astype(np.uint32) << 16) | np.uint32(0x8000)
    a = np.concatenate([a, base.view(np.float32), np.float32([0.0, -0.0, 1.0, -3.0])])
    a = a[np.isfinite(a)]
    ref = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_bf16(a.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_bf16_bits_roundtrip():
    bits = RNG.integers(0, 2 ** 16, 5000).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]          # finite patterns only
    vals = O.bf16_bits_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(vals, ref)


# --- window drop ----------------------------------------------------------------

def _tiny_f64(cfg, seed=0):
    w = synth.make_weights(cfg, seed)
    conv = lambda a: O.as_f64(a, cfg["dtype"])
    out = {k: conv(v) for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: conv(v) for k, v in lw.items()} for lw in w["layers"]]
    return out


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_window_drop_equivalence(dtype):
    """Muse page, "Pre-merge review round", third finding: fc and the norm are
    per row, so dropping rows before them leaves the kept rows unchanged."""
    cfg = synth.config("tiny", dtype=dtype)
    w = _tiny_f64(cfg)
    resid = O.as_f64(synth.make_context(cfg, 48, seed=3), dtype)
    first = 10
    nxt = first + 48
    kept, kpos = O.window_drop(resid, first, nxt, cfg["window"])
    assert kpos.tolist() == list(range(nxt - cfg["window"], nxt))
    k_all, v_all, c_all = O.context_kv(cfg, w, resid, first + np.arange(48))
    k_kept, v_kept, c_kept = O.context_kv(cfg, w, kept, kpos)
    sl = slice(48 - cfg["window"], 48)
    np.testing.assert_array_equal(c_all[sl], c_kept)
    for l in range(cfg["n_layers"]):
        np.testing.assert_array_equal(k_all[l][sl], k_kept[l])
        np.testing.assert_array_equal(v_all[l][sl], v_kept[l])


# --- Markov chain -----------------------------------------------------------------

def test_markov_chain_follows_permutation():
    """DSpark page, "Verified against the issue": the chain feeds each step's
    argmax into the next gather; a chain ignoring its own output would fail."""
    V, r = 1024, 16
    ids = RNG.choice(V, size=r, replace=False)
    sigma = np.roll(np.arange(r), -1)               # id j -> id j+1 (cyclic)
    W1 = RNG.standard_normal((V, r)) * 1e-3
    W2 = RNG.standard_normal((r, V)) * 1e-3
    for j in range(r):
        W1[ids[j]] = 0.0
        W1[ids[j], j] = 1.0                          # row of id j selects rank j
    for j in range(r):
        W2[j, ids[sigma[j]]] = 10.0                  # rank j scores id sigma(j)
    chain = O.markov_chain(W1, W2, int(ids[0]), 9)
    assert chain.tolist() == [int(ids[(k + 1) % r]) for k in range(9)]
    brute = []
    prev = int(ids[0])
    for _ in range(9):
        scores = [float(np.dot(W1[prev], W2[:, v])) for v in range(V)]
        prev = int(np.argmax(np.float32(scores)))
        brute.append(prev)
    assert chain.tolist() == brute
    z = np.zeros((9, V), dtype=np.float32)
    z[:, 5] = 100.0
    assert O.markov_chain(W1, W2, int(ids[0]), 9, z).tolist() == [5] * 9


# --- drafter layer invariants -------------------------------------------------------

def _session(cfg, w, ctx_rows=32, seed=0):
    resid = O.as_f64(synth.make_context(cfg, ctx_rows, seed=seed), cfg["dtype"])
    s = O.OracleSession(cfg, w)
    s.ingest(resid, 0, anchor=5)
    return s


def test_identity_layers():
    cfg = synth.config("tiny")
    w = _tiny_f64(cfg)
    for lw in w["layers"]:
        lw["wo"] = np.zeros_like(lw["wo"])
        lw["wd"] = np.zeros_like(lw["wd"])
    s = _session(cfg, w)
    out = s.draft(4)
    x0 = w["embed"][[5, 1023, 1023, 1023]]
    np.testing.assert_allclose(out["hidden"], O.round_f32(O.rmsnorm(x0, w["final_norm"], 1e-6)), rtol=1e-7)


def test_translation_invariance_of_positions():
    """Mask and RoPE only see position differences (Muse page: the mask is
    over absolute positions, |q - k| <= W)."""
    cfg = synth.config("tiny")
    w = _tiny_f64(cfg)
    resid = O.as_f64(synth.make_context(cfg, 32), "f32")
    outs = []
    for shift in (0, 1000):
        s = O.OracleSession(cfg, w)
        s.ingest(resid, shift, anchor=7)
        outs.append(s.draft(4)["hidden"])
    np.testing.assert_allclose(outs[0], outs[1], rtol=2e-4, atol=1e-5)


def test_window_bound_and_bidirectional():
    cfg = synth.config("tiny")
    w = _tiny_f64(cfg)
    s = _session(cfg, w)
    k, v, p = s.visible_context()
    base = O.draft_block(cfg, w, k, v, p, 5, s.pos, 4)
    W = cfg["window"]
    assert p.min() == s.pos - W
    # an older context row (distance W + 1 from the anchor) changes nothing
    k2 = [np.concatenate([np.full((1,) + kk.shape[1:], 9.0), kk]) for kk in k]
    v2 = [np.concatenate([np.full((1,) + vv.shape[1:], 9.0), vv]) for vv in v]
    p2 = np.concatenate([[s.pos - W - 1], p])
    np.testing.assert_array_equal(O.draft_block(cfg, w, k2, v2, p2, 5, s.pos, 4)["hidden"][0], base["hidden"][0])
    # ... while the row at distance exactly W does matter for the anchor row
    k3 = [kk.copy() for kk in k]
    for kk in k3:
        kk[0] += 1.0
    assert not np.array_equal(O.draft_block(cfg, w, k3, v, p, 5, s.pos, 4)["hidden"][0], base["hidden"][0])
    # bidirectional: the anchor row (block row 0) sees later block rows
    cfg2 = dict(cfg, mask_token_id=17)
    other = O.draft_block(cfg2, w, k, v, p, 5, s.pos, 4)
    assert not np.array_equal(other["hidden"][0], base["hidden"][0])


def test_neox_and_traditional_change_attention_output():
    """DSpark page: the RoPE test asserts the output changes, not a field."""
    cfg = synth.config("tiny")
    w = _tiny_f64(cfg)
    s1 = _session(cfg, w)
    s2 = _session(dict(cfg, rope_neox=False), w)
    assert not np.allclose(s1.draft(4)["hidden"], s2.draft(4)["hidden"])


def test_dspark_block_reads_all_positions():
    """DSpark page: [anchor] ++ mask * (gamma - 1), every position read out."""
    toks, read = O.block_tokens(dict(kind="dspark", mask_token_id=99), 7, 10)
    assert toks.tolist() == [7] + [99] * 8 and read.tolist() == list(range(9))
    toks, read = O.block_tokens(dict(kind="dflash", mask_token_id=99), 7, 4)
    assert toks.tolist() == [7, 99, 99, 99] and read.tolist() == [1, 2, 3]


def test_tiny_session_runs_rounds():
    cfg = synth.config("tiny")
    w = _tiny_f64(cfg)
    stream = synth.make_target_stream(cfg, 8, 4)
    s = _session(cfg, w)
    for r in range(8):
        d = s.draft(4)
        L = synth.planted_logits(stream, r, 4, d["draft_ids"])
        tokens, n, _ = s.verify(O.as_f64(L, "f32"), d["draft_ids"])
        s.append_and_trim(O.as_f64(synth.resid_rows(stream, r, 4), "f32"), n)
        s.commit(n, tokens[-1], 4, n - 1)
        for i in range(n - 1):
            assert stream["coins"][r, i] == 1 or tokens[i] == d["draft_ids"][i]
    assert s.rounds == 8 and s.pos == 32 + (s.accepted + 8)
