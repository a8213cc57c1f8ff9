"""Pins of the oracle's sampled verify (T > 0) and LFM2 short-conv rollback.

Sampled verify: the defining property of speculative sampling (the emitted
token follows the target distribution whatever the proposal), its limits
(u = 0 always accepts, T -> 0 is the greedy rule), and the bonus draw.
Short conv: a brute-force causal convolution (numpy.convolve per channel),
causality, and the rollback state against a one-pass run over the committed
prefix (DSpark page, "Short-conv rollback": the test compares the state and
the next step's output against a genuine one-pass reference). CPU only.
"""

import numpy as np
import pytest

import oracle as O

RNG = np.random.default_rng(77)


def test_sampled_probs_is_a_capped_tempered_softmax():
    z = np.float32([1.0, 3.0, -2.0, 25.0])
    p = O.sampled_probs(z, 0.5, 20.0)
    capped = 20.0 * np.tanh(z.astype(np.float64) / 20.0)
    e = np.exp(capped / 0.5 - (capped / 0.5).max())
    np.testing.assert_allclose(p, e / e.sum(), rtol=1e-5)          # the cap is taken in fp32
    assert abs(p.sum() - 1.0) < 1e-12
    np.testing.assert_allclose(O.sampled_probs(z, 1.0, 0.0), np.exp(z - 25.0) / np.exp(z - 25.0).sum(), rtol=1e-6)


@pytest.mark.parametrize("draft", [0, 2, 5])
def test_first_emitted_token_follows_the_target_distribution(draft):
    """Speculative sampling emits tokens distributed exactly as the target's,
    whatever the drafter proposed: P(first = d) = p(d) (accepted) and
    P(first = v) = (1 - p(d)) p(v) / (1 - p(d)) = p(v) otherwise."""
    V, N = 6, 40000
    L = np.float32([[0.3, -1.0, 1.2, 0.0, 0.5, -0.4], [0.1, 0.2, 0.3, 0.4, 0.5, 0.6]])
    p0 = O.sampled_probs(L[0], 1.0, 20.0)
    u = RNG.random((N, 2))
    counts = np.zeros(V)
    for k in range(N):
        tokens, n, a = O.verify_sampled(L, np.array([draft]), u[k], 1.0, 20.0)
        counts[tokens[0]] += 1
    sd = np.sqrt(N * p0 * (1 - p0))
    assert np.all(np.abs(counts - N * p0) < 5 * sd), (counts / N, p0)


def test_sampled_verify_limits():
    V = 50
    L = RNG.standard_normal((4, V)).astype(np.float32)
    d = RNG.integers(0, V, 3)
    # u = 0 accepts every proposal with positive probability; the bonus with
    # u = 0 is the first token of positive probability of the last row
    tokens, n, a = O.verify_sampled(L, d, np.zeros(4), 1.0, 0.0)
    assert n == 4 and tokens[:3].tolist() == d.tolist() and tokens[3] == 0
    # u close to 1 rejects at row 0 unless p(d) is about 1; the bonus skips d
    tokens, n, a = O.verify_sampled(L, d, np.full(4, 1 - 1e-12), 1.0, 0.0)
    assert n == 1 and tokens[0] != d[0]
    # a near-zero temperature is the greedy exact-match rule
    t = np.argmax(L, axis=1)
    for dd in (t[:3].copy(), np.array([t[0], (t[1] + 1) % V, t[2]])):
        g_tok, g_n, _ = O.verify_accept(L, dd)
        s_tok, s_n, _ = O.verify_sampled(L, dd, RNG.random(4) * 0.9, 1e-4, 0.0)
        assert s_n == g_n and s_tok.tolist() == g_tok.tolist()


def test_bonus_after_rejection_never_repeats_the_rejected_draft():
    L = np.float32([[5.0, 0.0, 0.0], [0.0, 0.0, 0.0]])
    for uu in np.linspace(0.0, 0.999, 50):
        tokens, n, a = O.verify_sampled(L, np.array([0]), np.array([0.999999, uu]), 1.0, 0.0)
        assert n == 1 and tokens[0] in (1, 2)


# --- short conv ------------------------------------------------------------------------

def test_short_conv_matches_per_channel_convolution():
    C, B, Lc = 5, 7, 3
    state = RNG.standard_normal((Lc - 1, C))
    bx = RNG.standard_normal((B, C))
    w = RNG.standard_normal((C, Lc))
    y, st = O.short_conv_block(state, bx, w)
    x = np.concatenate([state, bx])
    for c in range(C):
        ref = np.convolve(x[:, c], w[c, ::-1], mode="valid")     # correlation with the taps
        np.testing.assert_allclose(y[:, c], ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(st, x[-(Lc - 1):])
    y0, st0 = O.short_conv_block(None, bx, w)
    np.testing.assert_array_equal(y0[0], w[:, -1] * bx[0])          # zero state: only the last tap


@pytest.mark.parametrize("n", [0, 1, 2, 5, 7])
def test_rollback_equals_one_pass_over_the_committed_prefix(n):
    C, B, Lc = 6, 7, 3
    state = RNG.standard_normal((Lc - 1, C))
    bx = RNG.standard_normal((B, C))
    nxt = RNG.standard_normal((1, C))
    w = RNG.standard_normal((C, Lc))
    rolled = O.short_conv_rollback(state, bx, n, Lc)
    y_prefix, st_prefix = O.short_conv_block(state, bx[:n], w) if n else (None, state)
    np.testing.assert_array_equal(rolled, st_prefix)
    # causality: the block's first n outputs do not depend on the rejected rows
    y_full, _ = O.short_conv_block(state, bx, w)
    if n:
        np.testing.assert_array_equal(y_full[:n], y_prefix)
    # the next decode step from the rolled-back state equals the one-pass run
    y_next, _ = O.short_conv_block(rolled, nxt, w)
    y_ref, _ = O.short_conv_block(state, np.concatenate([bx[:n], nxt]), w)
    np.testing.assert_allclose(y_next[0], y_ref[-1], rtol=1e-12, atol=1e-12)
    # no previous state: the zeros fallback
    np.testing.assert_array_equal(O.short_conv_rollback(None, bx, n, Lc),
                                  np.concatenate([np.zeros((Lc - 1, C)), bx[:n]])[-(Lc - 1):])
