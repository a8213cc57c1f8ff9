"""Batched rounds: several sequences drafted, verified and committed together
through one context (dflash_ctx_create_batched), each compared round by
round with its own CPU oracle session -- draft ids exact away from near ties,
the verify's tokens and n, the committed position and anchor, the counters
and the ring's visible window exact, hidden rows within the parity rule."""

import numpy as np
import pytest
import torch

import oracle as O
from block_speculative_decoding_dflash_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def H():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from block_speculative_decoding_dflash_gb300 import build
    build.build()
    import gpu_harness
    return gpu_harness


class Batch:
    """A batched GPU context next to one oracle session per sequence."""

    def __init__(self, H, cfg, n_seq, w=None, w64=None, wd=None, ctx_rows=32):
        from block_speculative_decoding_dflash_gb300 import binding as B
        self.B, self.H, self.cfg, self.S = B, H, cfg, n_seq
        self.dt = cfg["dtype"]
        self.tol = H.TOL[self.dt]
        self.w = w if w is not None else synth.make_weights(cfg, 0)
        self.wd = wd if wd is not None else B.weights_to_device(self.w, self.dt)
        self.w64 = w64 if w64 is not None else H.f64_weights(self.w, self.dt)
        self.ctx = B.DFlashContext(cfg, self.wd, n_seq=n_seq)
        assert B.lib.dflash_batch_size(self.ctx.h) == n_seq
        self.sess = [O.OracleSession(cfg, self.w64) for _ in range(n_seq)]
        self.streams = []
        for s in range(n_seq):
            resid = synth.make_context(cfg, ctx_rows, seed=100 + s)
            self.ctx.ingest_context_seq(s, B.to_device(resid, self.dt), ctx_rows, 7 * s, 5 + 11 * s)
            self.sess[s].ingest(O.as_f64(resid, self.dt), 7 * s, 5 + 11 * s)
            self.streams.append(synth.make_target_stream(cfg, 64, cfg["max_block"], seed=200 + s,
                                                         logit_pool=2, resid_pool=4))

    def round(self, r, block, check_hidden=True):
        B, H, S, V = self.B, self.H, self.S, self.cfg["vocab"]
        ids = torch.zeros(S, block - 1, dtype=torch.int32, device="cuda")
        self.ctx.draft_block(block, ids)
        self.ctx.sync()
        got = ids.cpu().numpy().astype(np.int64)
        refs = [self.sess[s].draft(block) for s in range(S)]
        if check_hidden:
            rows = refs[0]["hidden"].shape[0]
            hid = torch.empty(S * rows, self.cfg["hidden"], dtype=H.torch_dtype(self.dt), device="cuda")
            self.ctx.get_hidden(hid)
            hid = H.dev_to_f64(hid)
            for s in range(S):
                H.assert_hidden_close(hid[s * rows:(s + 1) * rows], refs[s]["hidden"], self.tol, self.dt,
                                      f"hidden seq {s}")
        for s in range(S):
            H.check_ids(got[s], refs[s]["backbone_ids"], refs[s]["logits"], self.tol, f"seq {s} ids")
        L = np.stack([synth.planted_logits(self.streams[s], r, block, got[s]) for s in range(S)])
        tok = torch.full((S, block), -7, dtype=torch.int32, device="cuda")
        n = torch.zeros(S, dtype=torch.int32, device="cuda")
        self.ctx.verify_accept(B.to_device(L, self.dt), block, ids, tok, n)
        resid = np.stack([synth.resid_rows(self.streams[s], r, block) for s in range(S)])
        self.ctx.append_block(B.to_device(resid, self.dt), block)
        self.ctx.commit(-1)
        host = self.ctx.sync_round(block)
        for s in range(S):
            tokens, nn, _ = O.verify_accept(O.as_f64(L[s], self.dt), got[s])
            assert host[s][1] == nn and host[s][0].tolist() == tokens.tolist(), (r, s)
            self.sess[s].append_and_trim(O.as_f64(resid[s], self.dt), nn)
            self.sess[s].commit(nn, int(tokens[-1]), block, nn - 1)
            st, stats = self.ctx.state(s), self.ctx.stats(s)
            assert st["position"] == self.sess[s].pos and st["anchor"] == self.sess[s].anchor, (r, s)
            assert st["error"] == 0
            assert stats["rounds"] == self.sess[s].rounds and stats["accepted"] == self.sess[s].accepted

    def check_rings(self, max_rows=None):
        H, cfg = self.H, self.cfg
        for s in range(self.S):
            pair = H.Pair.__new__(H.Pair)
            pair.cfg, pair.dt, pair.tol, pair.dev = cfg, self.dt, self.tol, "cuda"
            pair.sess = self.sess[s]

            class _One:
                def __init__(self, ctx, s):
                    self.c, self.s = ctx, s

                def ring(self):
                    return self.c.ring(self.s)

                def sync(self):
                    self.c.sync()

            pair.ctx = _One(self.ctx, s)
            pair.check_ring(max_rows=max_rows)


@pytest.mark.parametrize("n_seq", [2, 3])
def test_tiny_batched_rounds_match_per_sequence_oracles(H, n_seq):
    cfg = synth.config("tiny", max_block=4)
    b = Batch(H, cfg, n_seq)
    for r in range(24):
        b.round(r, 4 if r % 3 else 3)
        if r % 6 == 5:
            b.check_rings()
    # the windows have wrapped the 48-slot rings
    assert all(s.pos > 32 + 48 for s in b.sess)
    b.ctx.close()


def test_tiny_batched_graph_replay_equals_eager(H):
    from block_speculative_decoding_dflash_gb300 import binding as B
    cfg = synth.config("tiny", max_block=4)
    S, blk = 3, 4
    results = []
    for use_graph in (False, True):
        b = Batch(H, cfg, S)
        st = synth.make_target_stream(cfg, 12, 4, seed=9, logit_pool=2, resid_pool=4)
        pools = [torch.from_numpy(np.ascontiguousarray(st[k])).cuda() for k in ("logits", "plant", "coins", "resid")]
        ids = torch.zeros(S, blk - 1, dtype=torch.int32, device="cuda")
        tok = torch.zeros(S, blk, dtype=torch.int32, device="cuda")
        n = torch.zeros(S, dtype=torch.int32, device="cuda")
        Lb = torch.zeros(S, blk, cfg["vocab"], device="cuda")
        Rb = torch.zeros(S, blk, 320, device="cuda")

        def one():
            b.ctx.draft_block(blk, ids)
            b.ctx.synth_target(*pools, blk, ids, Lb, Rb)
            b.ctx.verify_accept(Lb, blk, ids, tok, n)
            b.ctx.append_block(Rb, blk)
            b.ctx.commit(-1)

        if use_graph:
            one()
            b.ctx.capture_begin()
            one()
            b.ctx.capture_end(3)
            for _ in range(9):
                b.ctx.graph_launch(3)
        else:
            for _ in range(10):
                one()
        b.ctx.sync()
        results.append([(b.ctx.state(s), b.ctx.stats(s)) for s in range(S)] + [tok.cpu().tolist()])
        b.ctx.close()
    assert results[0] == results[1]


@pytest.fixture(scope="module")
def muse(H):
    from block_speculative_decoding_dflash_gb300 import binding as B
    cfg = synth.config("muse", max_block=16)
    w = synth.make_weights(cfg, 0)
    return cfg, w, B.weights_to_device(w, "bf16"), H.f64_weights(w, "bf16", lazy_embed=True)


@pytest.mark.parametrize("n_seq,block", [(4, 4), (2, 16), (4, 16)])
def test_muse_batched_rounds(H, muse, n_seq, block):
    """16 rows (four sequences of 4) and 32 rows (two of 16) on the tensor-core
    path: the weights stream once for the whole batch; 64 rows (four of 16):
    every GEMM in one launch of 64 block rows."""
    cfg, w, wd, w64 = muse
    b = Batch(H, dict(cfg, max_block=block), n_seq, w=w, w64=w64, wd=wd, ctx_rows=2048)
    for r in range(3):
        b.round(r, block)
    b.check_rings(max_rows=32)
    b.ctx.close()


def test_muse_batched_rounds_past_one_launch(H, muse):
    """176 rows (eleven sequences of 16): the fp32-sum GEMMs in groups of 160
    and 16 block rows, the lm_head argmax in groups of 128 and 48, the
    verify and the append over all 176 rows (a shorter context keeps the
    eleven oracle sessions quick)."""
    cfg, w, wd, w64 = muse
    b = Batch(H, dict(cfg, max_block=16), 11, w=w, w64=w64, wd=wd, ctx_rows=256)
    for r in range(2):
        b.round(r, 16)
    b.check_rings(max_rows=32)
    b.ctx.close()
