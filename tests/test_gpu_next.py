"""GPU parity of the sampled verify (T > 0) and the LFM2 short-conv rollback
against the CPU oracle, through the C ABI.

Sampled verify: p_i(d_{i+1}) within fp32 rounding of the oracle's; the accept
decisions and the bonus token exact except where the oracle's own numbers put
a decision within rounding of its threshold (u against p, the bonus draw
against a CDF boundary); the first emitted token's frequencies match the
target distribution over many draws. Short conv: outputs within rounding,
states and rollbacks bit-exact, the next step after a rollback identical to a
one-pass run over the committed prefix."""

import numpy as np
import pytest
import torch

import oracle as O
from block_speculative_decoding_dflash_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from block_speculative_decoding_dflash_gb300 import build
    build.build()
    from block_speculative_decoding_dflash_gb300 import binding
    return binding


def _ctx(B, dtype, V, max_block):
    cfg = synth.config("tiny", dtype=dtype, vocab=V, mask_token_id=V - 1, n_layers=1, max_block=max_block)
    return B.DFlashContext(cfg, B.weights_to_device(synth.make_weights(cfg, 0), dtype)), cfg


@pytest.mark.parametrize("dtype,V,block,T,cap", [("bf16", 202048, 16, 1.0, 20.0), ("bf16", 202048, 4, 0.7, 0.0),
                                               ("f32", 1000, 8, 1.0, 0.0), ("f32", 4099, 5, 0.5, 20.0)])
def test_sampled_verify_matches_oracle(B, dtype, V, block, T, cap):
    ctx, cfg = _ctx(B, dtype, V, block)
    rng = np.random.default_rng(V + block)
    near = 0
    for r in range(12):
        L32 = (rng.standard_normal((block, V)) * 2.0).astype(np.float32)
        d = rng.integers(0, V, block - 1)
        # make the drafts likely for about half the rows so acceptance varies
        for i in range(block - 1):
            if rng.random() < 0.6:
                L32[i, d[i]] = L32[i].max() + rng.uniform(0.0, 3.0)
        L = synth.to_storage(L32, dtype)
        Lf = O.as_f64(L, dtype).astype(np.float32)
        u = rng.random(block).astype(np.float32)
        tok = torch.full((block,), -7, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        pd = torch.zeros(block, dtype=torch.float32, device="cuda")
        ids = torch.tensor(d, dtype=torch.int32, device="cuda")
        ctx.verify_sampled(B.to_device(L, dtype), block, ids, torch.from_numpy(u).cuda(), T, tok, n,
                           softcap=cap, p_draft=pd)
        ctx.sync()
        got_pd = pd.cpu().numpy()
        want_pd = np.array([O.sampled_probs(Lf[i], T, cap)[d[i]] for i in range(block - 1)])
        np.testing.assert_allclose(got_pd[:-1], want_pd, rtol=2e-4, atol=1e-7)
        assert got_pd[-1] == 0.0
        tokens, nn, a = O.verify_sampled(Lf, d, u.astype(np.float64), T, cap)
        close = [abs(float(u[i]) - want_pd[i]) < 1e-4 for i in range(block - 1)]
        if any(close[: min(a + 1, block - 1)]):
            near += 1
            continue
        got_n = int(n.item())
        assert got_n == nn, (r, got_n, nn)
        got_tok = tok.cpu().numpy()
        assert got_tok[: nn - 1].tolist() == tokens[:-1].tolist() and np.all(got_tok[nn:] == -1)
        if got_tok[nn - 1] != tokens[-1]:
            # allowed only where the draw sits within rounding of a CDF boundary
            p = O.sampled_probs(Lf[a], T, cap)
            if a < block - 1:
                p[d[a]] = 0.0
            c = np.cumsum(p)
            t = u[-1] * c[-1]
            edge = min(abs(t - c[max(int(tokens[-1]) - 1, 0)]), abs(c[int(tokens[-1])] - t))
            assert edge < 1e-5 * c[-1], (r, got_tok[nn - 1], tokens[-1], edge)
            near += 1
        st = ctx.state()
        assert st["last_n"] == got_n
    assert near <= 3
    ctx.close()


def test_sampled_verify_emits_the_target_distribution(B):
    """Whatever the draft, the first emitted token follows p_0: frequencies of
    2000 GPU verifies (fresh uniforms each) within 5 standard deviations."""
    V, block, N = 8, 2, 2000
    ctx, cfg = _ctx(B, "f32", V, 4)
    L = np.float32([[0.2, 1.0, -0.5, 0.0, 0.7, -1.0, 0.3, 0.1], [0.0] * 8])
    p0 = O.sampled_probs(L[0], 1.0, 0.0)
    Ld = B.to_device(L, "f32")
    ids = torch.tensor([1], dtype=torch.int32, device="cuda")
    U = torch.from_numpy(np.random.default_rng(3).random((N, 2)).astype(np.float32)).cuda()
    toks = torch.zeros(N, 2, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    for k in range(N):
        ctx.verify_sampled(Ld, block, ids, U[k], 1.0, toks[k], n, softcap=0.0)
    ctx.sync()
    first = toks[:, 0].cpu().numpy()
    counts = np.bincount(first, minlength=V)
    sd = np.sqrt(N * p0 * (1 - p0))
    assert np.all(np.abs(counts - N * p0) < 5 * sd), (counts / N, p0)
    ctx.close()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_short_conv_and_rollback_match_oracle(B, dtype):
    layers, lc, C, blk = 3, 3, 192, 8
    rng = np.random.default_rng(5)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    st_h = synth.to_storage(rng.standard_normal((layers, lc - 1, C)).astype(np.float32), dtype)
    bx_h = synth.to_storage(rng.standard_normal((layers, blk, C)).astype(np.float32), dtype)
    w_h = synth.to_storage((rng.standard_normal((layers, C, lc)) * 0.5).astype(np.float32), dtype)
    st64, bx64, w64 = (O.as_f64(a, dtype) for a in (st_h, bx_h, w_h))
    st_d, bx_d, w_d = (B.to_device(a, dtype) for a in (st_h, bx_h, w_h))
    y = torch.empty(layers, blk, C, dtype=tdt, device="cuda")
    after = torch.empty(layers, lc - 1, C, dtype=tdt, device="cuda")
    B.short_conv_block(st_d, bx_d, w_d, layers, lc, C, blk, dtype, y, after)
    torch.cuda.synchronize()
    rnd = O.rounder(dtype)
    tol = 1e-5 if dtype == "f32" else 1e-2
    for l in range(layers):
        yr, sr = O.short_conv_block(st64[l], bx64[l], w64[l])
        got = y[l].to(torch.float64).cpu().numpy()
        assert np.all(np.abs(got - rnd(yr)) <= tol * np.abs(yr).max())
        np.testing.assert_array_equal(after[l].to(torch.float64).cpu().numpy(), sr)
    nxt_h = synth.to_storage(rng.standard_normal((layers, 1, C)).astype(np.float32), dtype)
    nxt_d = B.to_device(nxt_h, dtype)
    for n in range(0, blk + 1):
        n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
        out = torch.empty(layers, lc - 1, C, dtype=tdt, device="cuda")
        B.short_conv_rollback(st_d, bx_d, n_dev, layers, lc, C, blk, dtype, out)
        zero = torch.empty_like(out)
        B.short_conv_rollback(None, bx_d, n_dev, layers, lc, C, blk, dtype, zero)
        # the next decode step from the rolled-back state ...
        y1 = torch.empty(layers, 1, C, dtype=tdt, device="cuda")
        B.short_conv_block(out, nxt_d, w_d, layers, lc, C, 1, dtype, y1)
        # ... equals the one-pass run over the committed prefix and that step
        pre = torch.cat([bx_d[:, :n], nxt_d], dim=1).contiguous()
        yp = torch.empty(layers, n + 1, C, dtype=tdt, device="cuda")
        B.short_conv_block(st_d, pre, w_d, layers, lc, C, n + 1, dtype, yp)
        torch.cuda.synchronize()
        for l in range(layers):
            np.testing.assert_array_equal(out[l].to(torch.float64).cpu().numpy(),
                                          O.short_conv_rollback(st64[l], bx64[l], n, lc))
            np.testing.assert_array_equal(zero[l].to(torch.float64).cpu().numpy(),
                                          O.short_conv_rollback(None, bx64[l], n, lc))
        assert torch.equal(y1[:, 0], yp[:, n])
    # in place: the output may alias the previous state
    n_dev = torch.tensor([3], dtype=torch.int32, device="cuda")
    inplace = st_d.clone()
    B.short_conv_rollback(inplace, bx_d, n_dev, layers, lc, C, blk, dtype, inplace)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(inplace[0].to(torch.float64).cpu().numpy(),
                                  O.short_conv_rollback(st64[0], bx64[0], 3, lc))


def test_next_step_errors(B):
    x = torch.zeros(64, device="cuda")
    with pytest.raises(B.DFlashError) as e:
        B.short_conv_block(x, x, x, 1, 1, 4, 2, "f32", x)
    assert e.value.code == B.ERANGE
    with pytest.raises(B.DFlashError) as e:
        B.short_conv_rollback(x, x, None, 1, 3, 4, 2, "f32", x)
    assert e.value.code == B.EINVAL
    ctx, cfg = _ctx(B, "f32", 1000, 4)
    ids = torch.zeros(3, dtype=torch.int32, device="cuda")
    with pytest.raises(B.DFlashError) as e:
        ctx.verify_sampled(torch.zeros(4, 1000, device="cuda"), 4, ids, torch.zeros(4, device="cuda"), 0.0,
                           ids, ids)
    assert e.value.code == B.EINVAL
    ctx.close()
