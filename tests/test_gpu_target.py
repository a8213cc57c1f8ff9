"""The synthetic target's verify forward through the C ABI against the CPU
oracle's TargetSession: the prompt prefill (captured residual rows of every
prompt row, the last row's logits), verify forwards with their cache trims
(logits of every block row, captured rows, committed positions), and whole
rounds drafter + target (draft ids, the verify's tokens and n, both
committed positions), eager and from a captured CUDA graph.

Parity rule: captured rows by the hidden-row rule; logits within the logit
tolerance of the row maximum; argmax decisions exact except at a near tie of
the oracle's logits, where the oracle follows the GPU's choice."""

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


class Setup:
    """A drafter and a target on one stream, beside their oracle sessions."""

    def __init__(self, H, name, prompt_rows, drafter=True):
        from block_speculative_decoding_dflash_gb300 import binding as B
        self.B, self.H = B, H
        cfg = synth.config(name, max_block=16)
        tc = synth.target_config(name)
        self.cfg, self.tc, self.dt = cfg, tc, cfg["dtype"]
        self.tol = H.TOL[self.dt]
        w = synth.make_weights(cfg, 0)
        tw = synth.make_target_weights(tc, w)
        self.w64 = H.f64_weights(w, self.dt, lazy_embed=name != "tiny")
        tw64 = {"embed": self.w64["embed"], "lm_head": self.w64["lm_head"],
                "final_norm": O.as_f64(tw["final_norm"], self.dt),
                "layers": [{k: O.as_f64(v, self.dt) for k, v in lw.items()} for lw in tw["layers"]]}
        wd = B.weights_to_device(w, self.dt)
        twd = {"embed": wd["embed"], "lm_head": wd["lm_head"],
               "final_norm": B.to_device(tw["final_norm"], self.dt),
               "layers": [{k: B.to_device(v, self.dt) for k, v in lw.items()} for lw in tw["layers"]]}
        self.stream = torch.cuda.Stream()
        self.target = B.TargetContext(tc, twd, stream=self.stream)
        self.drafter = B.DFlashContext(cfg, wd, stream=self.stream) if drafter else None
        self.tsess = O.TargetSession(tc, tw64)
        self.dsess = O.OracleSession(cfg, self.w64) if drafter else None
        self.kin = len(tc["capture"]) * tc["hidden"]
        self.V = tc["vocab"]
        self.prompt = synth.make_prompt(tc, prompt_rows, seed=11)
        self.tdt = H.torch_dtype(self.dt)

    def dev_tokens(self, toks):
        return torch.tensor(np.asarray(toks, dtype=np.int32), device="cuda")

    def prefill(self):
        """The prompt in chunks of max_block rows: captured rows of every
        row, the last row's logits."""
        P, mb = len(self.prompt), self.tc["max_block"]
        cap = torch.empty(P, self.kin, dtype=self.tdt, device="cuda")
        logits = torch.empty(1, self.V, dtype=self.tdt, device="cuda")
        toks = self.dev_tokens(self.prompt)
        for r0 in range(0, P, mb):
            rows = min(mb, P - r0)
            last = r0 + rows == P
            self.target.forward(toks[r0:], rows, 1 if last else 0, logits if last else None, cap[r0:])
        self.target.sync()
        ref = self.tsess.forward(self.prompt, logit_rows=1)
        self.H.assert_hidden_close(self.H.dev_to_f64(cap), ref["captured"], self.tol, self.dt, "prompt captured")
        self.check_logits(self.H.dev_to_f64(logits), ref["logits"], "prompt logits")
        return cap, ref

    def check_logits(self, got, ref, what):
        self.H.assert_rows_close(got, ref, self.tol, what)

    def argmax_follow(self, got_logits, ref_logits):
        """The GPU's argmax per row; it must be the oracle's except at a near tie."""
        g = got_logits.argmax(axis=1)
        self.H.check_ids(g, ref_logits.argmax(axis=1), ref_logits, self.tol, "target argmax")
        return g


@pytest.mark.parametrize("name,prompt", [("tiny", 40), ("muse", 96)])
def test_prefill_and_verify_forwards_with_trims(H, name, prompt):
    s = Setup(H, name, prompt, drafter=False)
    s.prefill()
    rng = np.random.default_rng(3)
    blk = min(8, s.tc["max_block"])
    logits = torch.empty(blk, s.V, dtype=s.tdt, device="cuda")
    cap = torch.empty(blk, s.kin, dtype=s.tdt, device="cuda")
    n_dev = torch.zeros(1, dtype=torch.int32, device="cuda")
    for r in range(30 if name == "tiny" else 3):
        toks = rng.integers(0, s.V, blk)
        s.target.forward(s.dev_tokens(toks), blk, blk, logits, cap)
        n = int(rng.integers(1, blk + 1))
        n_dev.fill_(n)
        s.target.commit(n_dev, blk)
        s.target.sync()
        ref = s.tsess.forward(toks)
        s.tsess.commit(n)
        s.check_logits(H.dev_to_f64(logits), ref["logits"], f"round {r} logits")
        H.assert_hidden_close(H.dev_to_f64(cap), ref["captured"], s.tol, s.dt, f"round {r} captured")
        st = s.target.state()
        assert st["position"] == s.tsess.pos and st["error"] == 0, (r, st, s.tsess.pos)
    # the sliding ring has wrapped (tiny): capacity 16 + 128 < the position
    if name == "tiny":
        assert s.tsess.pos > s.target.ring().capacity()
    s.target.close()


def _round(s, block, ids, logits, cap, tok, n):
    s.target._capturing = s.drafter._capturing       # one stream, one capture
    s.drafter.draft_block(block, ids)
    s.target.verify(s.drafter, block, ids, logits, cap)
    s.drafter.verify_accept(logits, block, ids, tok, n)
    s.drafter.append_block(cap, block)
    s.drafter.commit(-1)
    s.target.commit(n, block)


def _oracle_round(s, block, got_ids, got_logits, got_cap):
    ref = s.dsess.draft(block)
    s.H.check_ids(got_ids, ref["backbone_ids"], ref["logits"], s.tol, "draft ids")
    toks = np.concatenate([[s.dsess.anchor], got_ids]).astype(np.int64)
    tref = s.tsess.forward(toks)
    s.check_logits(got_logits, tref["logits"], "verify logits")
    # the verify on the GPU's logits decides (near ties of the oracle's own
    # logits may go either way); the oracle's argmax must agree elsewhere
    s.argmax_follow(got_logits, tref["logits"])
    tokens, nn, _ = O.verify_accept(got_logits, got_ids)
    s.H.assert_hidden_close(got_cap, tref["captured"], s.tol, s.dt, "verify captured")
    s.dsess.append_and_trim(got_cap, nn)           # the drafter's input: the GPU's captured rows
    s.dsess.commit(nn, int(tokens[-1]), block, nn - 1)
    s.tsess.commit(nn)
    return tokens, nn


@pytest.mark.parametrize("name,prompt,widths", [("tiny", 40, [4, 8, 3, 16] * 6), ("muse", 64, [4, 16, 4])])
def test_rounds_with_the_target_match_oracle(H, name, prompt, widths):
    s = Setup(H, name, prompt)
    cap, ref = s.prefill()
    anchor = int(ref["logits"][0].argmax())
    s.drafter.ingest_context(cap, prompt, 0, anchor)
    s.dsess.ingest(H.dev_to_f64(cap), 0, anchor)
    mb = max(widths)
    ids = torch.zeros(mb, dtype=torch.int32, device="cuda")
    tok = torch.zeros(mb, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.empty(mb, s.V, dtype=s.tdt, device="cuda")
    capb = torch.empty(mb, s.kin, dtype=s.tdt, device="cuda")
    for r, w in enumerate(widths):
        _round(s, w, ids, logits, capb, tok, n)
        s.drafter.sync()
        got_ids = ids[: w - 1].cpu().numpy().astype(np.int64)
        got_logits = H.dev_to_f64(logits[:w])
        tokens, nn = _oracle_round(s, w, got_ids, got_logits, H.dev_to_f64(capb[:w]))
        assert int(n.item()) == nn and tok[:nn].cpu().tolist() == tokens.tolist(), r
        dst, tst = s.drafter.state(), s.target.state()
        assert dst["position"] == s.dsess.pos == tst["position"] == s.tsess.pos, (r, dst, tst)
        assert dst["anchor"] == s.dsess.anchor and dst["error"] == 0 and tst["error"] == 0, (r, dst, tst)
    s.drafter.close()
    s.target.close()


def test_target_rounds_from_a_captured_graph_equal_eager(H):
    """The whole round (draft, target verify, accept, append, both commits)
    captured once and replayed gives the eager run's states and tokens."""
    results = []
    for use_graph in (False, True):
        s = Setup(H, "tiny", 40, drafter=True)
        cap, ref = s.prefill()
        s.drafter.ingest_context(cap, 40, 0, int(ref["logits"][0].argmax()))
        blk = 8
        ids = torch.zeros(blk, dtype=torch.int32, device="cuda")
        tok = torch.zeros(blk, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        logits = torch.empty(blk, s.V, dtype=s.tdt, device="cuda")
        capb = torch.empty(blk, s.kin, dtype=s.tdt, device="cuda")
        if use_graph:
            _round(s, blk, ids, logits, capb, tok, n)
            s.drafter.capture_begin()
            _round(s, blk, ids, logits, capb, tok, n)
            s.drafter.capture_end(5)
            for _ in range(10):
                s.drafter.graph_launch(5)
        else:
            for _ in range(11):                       # as many as 1 eager + 10 replays
                _round(s, blk, ids, logits, capb, tok, n)
        s.drafter.sync()
        results.append((s.drafter.state(), s.drafter.stats(), s.target.state(), tok.cpu().tolist()))
        s.drafter.close()
        s.target.close()
    assert results[0] == results[1]


def test_target_argument_errors(H):
    from block_speculative_decoding_dflash_gb300 import binding as B
    s = Setup(H, "tiny", 8)
    t = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(B.DFlashError) as e:
        s.target.forward(t, s.tc["max_block"] + 1)
    assert e.value.code == B.ERANGE
    with pytest.raises(B.DFlashError) as e:
        s.target.forward(t, 2, 1, None)
    assert e.value.code == B.EINVAL
    with pytest.raises(B.DFlashError) as e:
        s.target.draft_block(4, t)
    assert e.value.code == B.EINVAL
    # a drafter context is no target
    assert B.lib.dflash_target_forward(s.drafter.h, t.data_ptr(), 2, 0, None, None) == B.EINVAL
    s.drafter.close()
    s.target.close()
