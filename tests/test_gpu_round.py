"""GPU parity of the DFlash round against the CPU oracle, through the C ABI.

Integer results (draft ids away from near ties, accepted counts, emitted
tokens, positions, anchors, counters) must match exactly; hidden states,
logits and ring K/V within 1e-4 (fp32) / 2e-2 (bf16) of the row's largest
magnitude.
"""

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


@pytest.fixture(scope="module")
def H(B):
    import gpu_harness
    return gpu_harness


# ---------------------------------------------------------------------------
# tiny fp32 configuration: every round compared
# ---------------------------------------------------------------------------

def test_tiny_64_rounds_match_oracle(B, H):
    cfg = synth.config("tiny")
    pair = H.Pair(cfg)
    resid = synth.make_context(cfg, cfg["context_rows"])
    pair.ingest(resid, 0, anchor=5)
    pair.check_ring()
    stream = synth.make_target_stream(cfg, cfg["rounds"], cfg["block"])
    ns = []
    for r in range(cfg["rounds"]):
        n, _ = pair.round(stream, r, cfg["block"])
        ns.append(n)
        pair.check_state()
        if r % 8 == 7:
            pair.check_ring()
    assert len(set(ns)) > 1, "planting should give varied accept lengths"
    assert pair.sess.pos > cfg["context_rows"] + cfg["window"]      # the ring has wrapped
    pair.close()


@pytest.mark.parametrize("block", [2, 3, 4])
def test_tiny_widths_and_neox_traditional(B, H, block):
    for neox in (True, False):
        cfg = synth.config("tiny", rope_neox=neox)
        pair = H.Pair(cfg, seed=3)
        pair.ingest(synth.make_context(cfg, 40, seed=3), 7, anchor=11)
        stream = synth.make_target_stream(cfg, 6, 4, seed=3)
        for r in range(6):
            pair.round(stream, r, block)
            pair.check_state()
        pair.check_ring()
        pair.close()


def test_tiny_bf16_matches_oracle(B, H):
    cfg = synth.config("tiny", dtype="bf16")
    pair = H.Pair(cfg, seed=1)
    pair.ingest(synth.make_context(cfg, 32, seed=1), 0, anchor=9)
    stream = synth.make_target_stream(cfg, 16, 4, seed=1)
    for r in range(16):
        pair.round(stream, r, 4)
        pair.check_state()
    pair.check_ring()
    pair.close()


def test_tiny_dspark_markov_both_modes(B, H):
    for add in (0, 1):
        cfg = synth.config("tiny", kind="dspark", window=0, max_context=32 + 8 * 5,
                           markov_rank=16, markov_add=add, rope_neox=False, tied_lm_head=True,
                           max_block=5, markov_std=0.05)
        pair = H.Pair(cfg, seed=2)
        pair.ingest(synth.make_context(cfg, 32, seed=2), 0, anchor=3)
        stream = synth.make_target_stream(cfg, 8, 5, seed=2)
        for r in range(8):
            pair.round(stream, r, 5)
            pair.check_state()
        pair.check_ring()
        pair.close()


def test_markov_chain_alone_follows_its_feedback(B, H):
    cfg = synth.config("tiny", kind="dspark", window=0, max_context=64, markov_rank=16,
                       tied_lm_head=True, max_block=10)
    w = synth.make_weights(cfg, 4)
    V, r = cfg["vocab"], 16
    rng = np.random.default_rng(5)
    ids = rng.choice(V, size=r, replace=False)
    W1 = (rng.standard_normal((V, r)) * 1e-3).astype(np.float32)
    W2 = (rng.standard_normal((r, V)) * 1e-3).astype(np.float32)
    for j in range(r):
        W1[ids[j]] = 0.0
        W1[ids[j], j] = 1.0
        W2[j, ids[(j + 1) % r]] = 10.0
    w["markov_w1"], w["markov_w2"] = W1, W2
    pair = H.Pair(cfg, weights=w)
    out = torch.empty(9, dtype=torch.int32, device="cuda")
    pair.ctx.markov_chain(int(ids[0]), 9, None, out)
    pair.ctx.sync()
    assert out.cpu().tolist() == [int(ids[(k + 1) % r]) for k in range(9)]
    assert out.cpu().tolist() == O.markov_chain(W1.astype(np.float64), W2.astype(np.float64),
                                                int(ids[0]), 9).tolist()
    pair.close()


# ---------------------------------------------------------------------------
# verify kernel: bit-exact, ties to the lowest index
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,V,block", [("f32", 1024, 4), ("bf16", 1000, 2), ("bf16", 202048, 16),
                                           ("f32", 8193, 129)])
def test_verify_bit_exact(B, H, dtype, V, block):
    cfg = synth.config("tiny", dtype=dtype, vocab=V, mask_token_id=V - 1, n_layers=1,
                       max_block=max(block, 4))
    pair = H.Pair(cfg)
    rng = np.random.default_rng(V + block)
    for trial in range(6):
        L = synth.to_storage(rng.standard_normal((block, V)).astype(np.float32), dtype)
        vals = O.as_f64(L, dtype)
        t = np.argmax(vals, axis=1)
        d = t[:block - 1].copy()
        cut = trial % block
        if cut < block - 1:
            d[cut] = (d[cut] + 1) % V
        if trial % 2:                        # an exact tie at a lower index
            L[0, 0] = L[0, t[0]]
        ids = torch.tensor(d, dtype=torch.int32, device="cuda")
        pair.verify(L, ids, d, block)
    pair.close()


# ---------------------------------------------------------------------------
# lm_head argmax: exact ties resolve to the lowest vocab index
# ---------------------------------------------------------------------------

def test_lm_head_ties_lowest_index(B, H):
    cfg = synth.config("tiny")
    w = synth.make_weights(cfg, 6)
    pair0 = H.Pair(cfg, weights=w)
    pair0.ingest(synth.make_context(cfg, 32, seed=6), 0, anchor=5)
    _, got, ref = pair0.draft(4)
    pair0.close()
    lm = w["lm_head"].copy()
    for m, v in enumerate(got):
        lo = int(v) // 2 if int(v) > 0 else 0
        if lo != int(v):
            lm[lo] = lm[int(v)]              # an identical row at a lower index
    w2 = dict(w, lm_head=lm)
    pair = H.Pair(cfg, weights=w2)
    pair.ingest(synth.make_context(cfg, 32, seed=6), 0, anchor=5)
    _, got2, ref2 = pair.draft(4)
    for v_old, v_new in zip(got, got2):
        assert int(v_new) == (int(v_old) // 2 if int(v_old) > 0 else 0)
    pair.close()


# ---------------------------------------------------------------------------
# graphs: a captured round is the same round
# ---------------------------------------------------------------------------

def test_graph_round_equals_eager_round(B, H):
    cfg = synth.config("tiny")
    w = synth.make_weights(cfg, 8)
    stream = synth.make_target_stream(cfg, 12, 4, seed=8)
    results = []
    for use_graph in (False, True):
        wd = B.weights_to_device(w, "f32")
        ctx = B.DFlashContext(cfg, wd)
        resid = synth.make_context(cfg, 32, seed=8)
        ctx.ingest_context(B.to_device(resid, "f32"), 32, 0, 5)
        pools = {k: torch.from_numpy(np.ascontiguousarray(stream[k])).cuda()
                 for k in ("logits", "plant", "coins", "resid")}
        ids = torch.zeros(3, dtype=torch.int32, device="cuda")
        tok = torch.zeros(4, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        Lb = torch.zeros(4, cfg["vocab"], dtype=torch.float32, device="cuda")
        Rb = torch.zeros(4, 320, dtype=torch.float32, device="cuda")

        def one_round():
            ctx.draft_block(4, ids)
            ctx.synth_target(pools["logits"], pools["plant"], pools["coins"], pools["resid"], 4, ids, Lb, Rb)
            ctx.verify_accept(Lb, 4, ids, tok, n)
            ctx.append_block(Rb, 4)
            ctx.commit(-1)

        if use_graph:
            one_round()                      # warm up outside capture
            ctx.capture_begin()
            one_round()
            ctx.capture_end(4)
            for _ in range(11):
                ctx.graph_launch(4)
        else:
            for _ in range(12):
                one_round()
        ctx.sync()
        results.append((ctx.state(), ctx.stats(), tok.cpu().tolist()))
        ctx.close()
    assert results[0] == results[1]


def test_host_driven_rounds_with_explicit_anchor_and_sync(B, H):
    """The round as the pages' loop drives it: the host passes the anchor and
    its position to the draft, and reads the verify's tokens and n back once
    per round (dflash_sync_round). The oracle runs the same rounds."""
    cfg = synth.config("tiny")
    pair = H.Pair(cfg, seed=3)
    pair.ingest(synth.make_context(cfg, 32, seed=3), 0, anchor=5)
    stream = synth.make_target_stream(cfg, 6, 4, seed=3)
    ids = torch.zeros(3, dtype=torch.int32, device="cuda")
    tok = torch.zeros(4, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    anchor, pos = 5, 32
    for r in range(6):
        if r == 3:
            anchor = 11                                 # the host may replace the anchor
            pair.sess.anchor = anchor
        pair.ctx.draft_block(4, ids, anchor=anchor, anchor_pos=pos)
        ref = pair.sess.draft(4)
        got = ids.cpu().numpy().astype(np.int64)
        H.check_ids(got, ref["backbone_ids"], ref["logits"], pair.tol, "draft ids")
        L = synth.planted_logits(stream, r, 4, got)
        pair.ctx.verify_accept(pair.to_dev(L), 4, ids, tok, n)
        pair.ctx.append_block(pair.to_dev(synth.resid_rows(stream, r, 4)), 4)
        pair.ctx.commit(-1)
        tokens_h, n_h = pair.ctx.sync_round(4)
        want, nn, _ = O.verify_accept(O.as_f64(L, "f32"), got)
        assert n_h == nn and tokens_h.tolist() == want.tolist()
        pair.sess.append_and_trim(O.as_f64(synth.resid_rows(stream, r, 4), "f32"), nn)
        pair.sess.commit(nn, int(want[-1]), 4, nn - 1)
        anchor, pos = int(tokens_h[-1]), pos + n_h
        pair.check_state()
    # a position that is not the committed length is flagged, not obeyed
    pair.ctx.draft_block(4, ids, anchor=anchor, anchor_pos=pos + 1)
    st = pair.ctx.state()
    assert st["error"] & 8 and st["position"] == pos
    with pytest.raises(B.DFlashError) as e:
        pair.ctx.draft_block(4, ids, anchor=cfg["vocab"])
    assert e.value.code == B.ERANGE
    pair.close()


def test_synth_target_kernel_matches_host(B, H):
    cfg = synth.config("tiny")
    pair = H.Pair(cfg)
    pair.ingest(synth.make_context(cfg, 32), 0, anchor=5)
    stream = synth.make_target_stream(cfg, 5, 4, seed=9)
    pools = {k: torch.from_numpy(np.ascontiguousarray(stream[k])).cuda()
             for k in ("logits", "plant", "coins", "resid")}
    d = np.array([3, stream["logits"].shape[2] - 1, 0])
    ids = torch.tensor(d, dtype=torch.int32, device="cuda")
    Lb = torch.zeros(4, cfg["vocab"], device="cuda")
    Rb = torch.zeros(4, 320, device="cuda")
    pair.ctx.synth_target(pools["logits"], pools["plant"], pools["coins"], pools["resid"], 4, ids, Lb, Rb)
    pair.ctx.sync()
    assert np.array_equal(Lb.cpu().numpy(), synth.planted_logits(stream, 0, 4, d))
    assert np.array_equal(Rb.cpu().numpy(), synth.resid_rows(stream, 0, 4))
    pair.close()


# ---------------------------------------------------------------------------
# errors never abort: they are status codes
# ---------------------------------------------------------------------------

def test_error_statuses(B, H):
    cfg = synth.config("tiny")
    pair = H.Pair(cfg)
    ctx = pair.ctx
    ids = torch.zeros(15, dtype=torch.int32, device="cuda")
    with pytest.raises(B.DFlashError) as e:
        ctx.draft_block(4, ids)
    assert e.value.code == B.EEMPTY
    resid = synth.make_context(cfg, 32)
    with pytest.raises(B.DFlashError) as e:
        ctx.ingest_context(B.to_device(resid, "f32"), 0, 0, 5)
    assert e.value.code == B.EEMPTY
    with pytest.raises(B.DFlashError) as e:
        ctx.ingest_context(B.to_device(resid, "f32"), 32, 0, 1024)
    assert e.value.code == B.ERANGE
    ctx.ingest_context(B.to_device(resid, "f32"), 32, 0, 5)
    for bad in (1, 5, 0):
        with pytest.raises(B.DFlashError) as e:
            ctx.draft_block(bad, ids)
        assert e.value.code == B.ERANGE
    with pytest.raises(B.DFlashError) as e:
        ctx.commit(-1)
    assert e.value.code == B.ESTATE
    with pytest.raises(B.DFlashError) as e:
        ctx.graph_launch(3)
    assert e.value.code == B.ESTATE
    with pytest.raises(B.DFlashError) as e:
        ctx.set_anchor(-3)
    assert e.value.code == B.ERANGE
    ring = ctx.ring()
    with pytest.raises(B.DFlashError) as e:
        ring.trim(1)
    assert e.value.code == B.EREWIND
    pair.close()


def test_append_only_cache_reports_full(B, H):
    cfg = synth.config("tiny", window=0, max_context=40, kind="dspark")
    pair = H.Pair(cfg)
    ctx = pair.ctx
    resid = synth.make_context(cfg, 41)
    with pytest.raises(B.DFlashError) as e:
        ctx.ingest_context(B.to_device(resid, "f32"), 41, 0, 5)
    assert e.value.code == B.EFULL
    ctx.ingest_context(B.to_device(resid[:38], "f32"), 38, 0, 5)
    rows = B.to_device(resid[:4], "f32")
    with pytest.raises(B.DFlashError) as e:
        ctx.append_block(rows, 4)
    assert e.value.code == B.EFULL
    ctx.append_block(rows[:2], 2)
    ctx.commit(2)
    assert ctx.state()["position"] == 40 and ctx.state()["error"] == 0
    pair.close()


# ---------------------------------------------------------------------------
# the standalone ring, bit-exact against the oracle's ring model
# ---------------------------------------------------------------------------

def _ring_rows(rng, L, n, nkv, hd):
    return rng.standard_normal((L, n, nkv, hd)).astype(np.float32)


def test_ring_wraparound_matches_history(B, H):
    L, nkv, hd, W, Bmax = 2, 2, 8, 24, 16
    ring = B.RingCache(L, nkv, hd, W, Bmax, "f32")
    cap = ring.capacity()
    assert cap == O.ring_capacity(W, Bmax)
    model = O.RingModel(W, cap, row_shape=(2, L, nkv, hd))
    rng = np.random.default_rng(11)

    def push(n):
        k, v = _ring_rows(rng, L, n, nkv, hd), _ring_rows(rng, L, n, nkv, hd)
        ring.append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), n)
        model.append(np.stack([k, v], axis=0).transpose(2, 0, 1, 3, 4))

    push(W)
    for _ in range(256):
        b = int(rng.integers(1, Bmax + 1))
        push(b)
        m = int(rng.integers(0, b + 1))
        ring.trim(m)
        model.trim(m)
        assert ring.offset() == model.offset
        pos = model.window_positions()
        ko = torch.empty(L, pos.size, nkv, hd, device="cuda")
        vo = torch.empty_like(ko)
        ring.gather(int(pos[0]), pos.size, ko, vo)
        truth = model.history_view(pos)            # [n, 2, L, nkv, hd]
        assert np.array_equal(ko.cpu().numpy(), truth[:, 0].transpose(1, 0, 2, 3))
        assert np.array_equal(vo.cpu().numpy(), truth[:, 1].transpose(1, 0, 2, 3))
    with pytest.raises(B.DFlashError) as e:
        ring.trim(1)
    assert e.value.code == B.EREWIND
    ring.close()


def test_ring_trim_past_slack_is_a_short_rewind(B, H):
    """Muse page, "Pre-merge review round", second finding: a trim must bring
    back exactly the window seen before the append. Appending more rows than
    the slack between trims overwrites window rows, so rewinding past the
    slack is refused (EREWIND) and the offset stays put."""
    L, nkv, hd, W, Bmax = 1, 1, 8, 24, 4
    ring = B.RingCache(L, nkv, hd, W, Bmax, "f32")
    slack = ring.capacity() - W
    assert slack == O.speculative_slack(Bmax) == 32
    rows = torch.zeros(L, slack + 1, nkv, hd, device="cuda")
    ring.append(rows[:, :W].contiguous(), rows[:, :W].contiguous(), W)
    ring.trim(0)
    ring.append(rows, rows, slack + 1)
    before = ring.offset()
    with pytest.raises(B.DFlashError) as e:
        ring.trim(slack + 1)
    assert e.value.code == B.EREWIND
    assert ring.offset() == before
    ring.trim(slack)                                # the slack itself may be rewound
    assert ring.offset() == before - slack
    ring.close()


@pytest.mark.parametrize("flags,corrupt", [(0, False), (1, True)])
def test_ring_floor_at_block_129(B, H, flags, corrupt):
    L, nkv, hd, W, Bk = 1, 1, 8, 2048, 129
    ring = B.RingCache(L, nkv, hd, W, Bk, "bf16", flags=flags)
    rng = np.random.default_rng(12)
    hist = rng.standard_normal((W + 300, hd)).astype(np.float32)
    histd = torch.from_numpy(hist).cuda().to(torch.bfloat16).view(L, -1, nkv, hd)
    half = (W + 300) // 2
    ring.append(histd[:, :half].contiguous(), histd[:, :half].contiguous(), half)
    ring.append(histd[:, half:].contiguous(), histd[:, half:].contiguous(), W + 300 - half)
    ring.trim(0)
    p = ring.offset()
    before_k = torch.empty(L, W, nkv, hd, dtype=torch.bfloat16, device="cuda")
    before_v = torch.empty_like(before_k)
    ring.gather(p - W, W, before_k, before_v)
    blk = torch.full((L, Bk, nkv, hd), -7.0, dtype=torch.bfloat16, device="cuda")
    ring.append(blk, blk, Bk)
    after_k = torch.empty_like(before_k)
    after_v = torch.empty_like(before_k)
    # the slots of the window seen before the append
    ring.gather(p - W, W, after_k, after_v)
    same = torch.equal(before_k, after_k)
    assert same != corrupt
    if corrupt:
        diff = (before_k != after_k).any(dim=-1).view(-1).nonzero().view(-1).tolist()
        assert diff == [0]                          # the oldest window row, overwritten by block row 128
        # a rewind would expose it: trim refuses to go past the slack
        with pytest.raises(B.DFlashError) as e:
            ring.trim(Bk)
        assert e.value.code == B.EREWIND
    else:
        ring.trim(Bk)
        assert ring.offset() == p
    ring.close()


# ---------------------------------------------------------------------------
# stand-in target: the block's logits with the planted draft tokens, and the
# captured residual rows, exactly as the host reference builds them
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,V,block", [("bf16", 1024, 4), ("bf16", 1001, 16), ("f32", 1024, 16),
                                           ("f32", 999, 4)])
def test_synth_target_matches_host(B, H, dtype, V, block):
    cfg = synth.config("tiny", dtype=dtype, vocab=V, mask_token_id=V - 1, n_layers=1, max_block=16)
    pair = H.Pair(cfg)
    stream = synth.make_target_stream(cfg, 4, 16, seed=V + block, logit_pool=2, resid_pool=2, p_plant=0.8)
    as_t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16
                                      else np.ascontiguousarray(a)).cuda()
    pools = {k: as_t(stream[k]) for k in ("logits", "plant", "coins", "resid")}
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    kin = cfg["k_target_layers"] * cfg["target_hidden"]
    d = np.random.default_rng(V).integers(0, V, block - 1).astype(np.int32)
    ids = torch.from_numpy(d).cuda()
    Lb = torch.zeros(block, V, dtype=tdt, device="cuda")
    Rb = torch.zeros(block, kin, dtype=tdt, device="cuda")
    pair.ctx.synth_target(pools["logits"].view(tdt) if dtype == "bf16" else pools["logits"],
                          pools["plant"].view(tdt) if dtype == "bf16" else pools["plant"],
                          pools["coins"], pools["resid"].view(tdt) if dtype == "bf16" else pools["resid"],
                          block, ids, Lb, Rb)
    pair.ctx.sync()
    r = pair.ctx.stats()["rounds"]
    want_l = synth.planted_logits(stream, r, block, d)
    want_r = stream["resid"][r % stream["resid_pool"], :block]
    got_l = Lb.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bf16" else Lb.cpu().numpy()
    got_r = Rb.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bf16" else Rb.cpu().numpy()
    assert np.array_equal(got_l, want_l)
    assert np.array_equal(got_r, want_r)
    pair.close()
