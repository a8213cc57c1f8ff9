"""The tensor-core (tcgen05 + TMA) weight-streaming GEMM and the fused
lm_head + softcap + argmax, against a plain PyTorch fp32 reference of the
same op: outputs equal the reference rounded to bf16 up to one bf16 step;
argmax ids exact except at near ties."""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

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


def _ctx(B, vocab, softcap=0.0, seed=0, max_block=32):
    cfg = synth.config("muse", n_layers=1, vocab=vocab, mask_token_id=vocab - 1, max_block=max_block,
                       softcap=softcap)
    w = synth.make_weights(cfg, seed)
    return B.DFlashContext(cfg, B.weights_to_device(w, "bf16")), w


def _close(y, ref, what):
    y, ref = y.float().cpu(), ref.float().cpu()
    tol = 1e-2 * ref.abs() + 1e-3 * ref.abs().max()      # one bf16 step of the element
    bad = ((y - ref).abs() > tol).nonzero()
    assert bad.numel() == 0, f"{what}: {bad.shape[0]} elements off, first {bad[:4].tolist()}"


@pytest.mark.parametrize("M,N,K,epi", [(1, 2048, 4096, 0), (4, 2048, 4096, 1), (16, 6144, 2048, 2),
                                       (32, 1000, 10240, 0), (13, 384, 64, 1), (7, 129, 128, 0),
                                       (16, 2048, 6144, 1), (24, 1024, 2048, 2)])
def test_linear_matches_torch(B, M, N, K, epi):
    ctx, _ = _ctx(B, 4096)
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N + K + epi)
    x = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    w2 = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    r = torch.randn(M, N, device="cuda", generator=g).to(torch.bfloat16)
    y = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    for rep in range(2):
        y.fill_(7.0)
        ctx.linear(x, M, K, w, N, y, epi=epi, w2=w2 if epi == 2 else None, r=r if epi == 1 else None)
        ctx.sync()
        acc = x.float() @ w.float().T
        if epi == 0:
            ref = acc.to(torch.bfloat16)
        elif epi == 1:
            ref = (r.float() + acc.to(torch.bfloat16).float()).to(torch.bfloat16)
        else:
            u = (x.float() @ w2.float().T).to(torch.bfloat16).float()
            ref = (F.silu(acc.to(torch.bfloat16).float()) * u).to(torch.bfloat16)
        _close(y, ref, f"linear M={M} N={N} K={K} epi={epi} rep={rep}")
    st = ctx.state()
    assert st["error"] == 0
    ctx.close()


@pytest.mark.parametrize("M,N,K", [(2048, 2048, 10240), (300, 2048, 2048), (128, 256, 64),
                                   (2048, 10240, 2048), (33, 512, 4096)])
def test_many_row_linear_matches_torch(B, M, N, K):
    """The context-ingest GEMM (128 x 256 x 16 tensor-core tiles)."""
    ctx, _ = _ctx(B, 4096)
    g = torch.Generator(device="cuda").manual_seed(M + N + K)
    x = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    y = torch.full((M, N), 7.0, device="cuda", dtype=torch.bfloat16)
    ctx.linear(x, M, K, w, N, y, epi=0)
    ctx.sync()
    ref = (x.float() @ w.float().T).to(torch.bfloat16)
    _close(y, ref, f"many-row linear M={M} N={N} K={K}")
    assert ctx.state()["error"] == 0
    ctx.close()


def test_linear_residual_in_place(B):
    ctx, _ = _ctx(B, 4096)
    M, N, K = 16, 2048, 4096
    g = torch.Generator(device="cuda").manual_seed(3)
    x = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    y = torch.randn(M, N, device="cuda", generator=g).to(torch.bfloat16)
    r0 = y.clone()
    ctx.linear(x, M, K, w, N, y, epi=1, r=y)
    ctx.sync()
    ref = (r0.float() + (x.float() @ w.float().T).to(torch.bfloat16).float()).to(torch.bfloat16)
    _close(y, ref, "in-place residual")
    ctx.close()


@pytest.mark.parametrize("vocab,rows,cap", [(202048, 3, 20.0), (202048, 15, 20.0), (65536, 9, 0.0),
                                            (4096, 32, 0.0), (1000, 5, 20.0), (202048, 100, 20.0),
                                            (65536, 64, 0.0), (4096, 129, 20.0), (65536, 300, 20.0)])
def test_lm_head_argmax_matches_torch(B, vocab, rows, cap):
    """Up to 32 rows one launch of 16 or 32; 33-128 one launch of 64 or 128
    rows (the accumulator read 32 columns at a time); 129 two launches; 300
    three (128, 128 and 44 rows, each writing its own rows' results)."""
    ctx, w = _ctx(B, vocab, softcap=cap, max_block=max(32, rows))
    lm = B.to_device(w["lm_head"], "bf16")
    g = torch.Generator(device="cuda").manual_seed(vocab + rows)
    x = torch.randn(rows, 2048, device="cuda", generator=g)
    x = (x / x.pow(2).mean(-1, keepdim=True).sqrt()).to(torch.bfloat16)
    ids = torch.empty(rows, dtype=torch.int32, device="cuda")
    mx = torch.empty(rows, dtype=torch.float32, device="cuda")
    for rep in range(2):
        ids.fill_(-1)
        ctx.lm_head_argmax(x, rows, ids, mx)
        ctx.sync()
        z = x.float() @ lm.float().T
        if cap > 0:
            z = cap * torch.tanh(z / cap)
        ref_ids = z.argmax(dim=1)
        top = z.max(dim=1).values
        for m in range(rows):
            i = int(ids[m])
            assert 0 <= i < vocab
            if i != int(ref_ids[m]):
                assert float(top[m] - z[m, i]) <= 1e-3 * float(z[m].abs().max()), (m, i, int(ref_ids[m]))
        assert torch.allclose(mx.cpu(), top.cpu(), rtol=1e-4, atol=1e-4)
    assert ctx.state()["error"] == 0
    ctx.close()


@pytest.mark.parametrize("rows", [4, 100])
def test_lm_head_argmax_exact_ties_take_lowest_index(B, rows):
    vocab = 202048
    cfg = synth.config("muse", n_layers=1, vocab=vocab, mask_token_id=vocab - 1, max_block=max(32, rows))
    w = synth.make_weights(cfg, 1)
    ctx0 = B.DFlashContext(cfg, B.weights_to_device(w, "bf16"))
    g = torch.Generator(device="cuda").manual_seed(9)
    x = torch.randn(rows, 2048, device="cuda", generator=g).to(torch.bfloat16)
    ids = torch.empty(rows, dtype=torch.int32, device="cuda")
    mx = torch.empty(rows, dtype=torch.float32, device="cuda")
    ctx0.lm_head_argmax(x, rows, ids, mx)
    ctx0.sync()
    first = ids.cpu().tolist()
    ctx0.close()
    lm = w["lm_head"].copy()
    lows, low_of, used = [], {}, set(first)
    for v in first:
        if v not in low_of:
            lo = v // 3
            while lo in used:         # a lower index no other row's winner or copy uses
                lo -= 1
            assert lo >= 0
            used.add(lo)
            low_of[v] = lo
            lm[lo] = lm[v]            # an identical row at a lower index, in another tile
        lows.append(low_of[v])
    w2 = dict(w, lm_head=lm)
    ctx = B.DFlashContext(cfg, B.weights_to_device(w2, "bf16"))
    ctx.lm_head_argmax(x, rows, ids, mx)
    ctx.sync()
    assert ids.cpu().tolist() == lows
    ctx.close()
