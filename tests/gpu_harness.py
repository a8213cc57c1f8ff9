"""Lock-step runner of the GPU library next to the CPU oracle on the same
seeded inputs, with the comparison rules of the parity tests.

Rules: integer outputs (accepted counts, emitted tokens, positions, anchors)
are compared exactly; floating outputs within ``TOL[dtype]`` times the row's
largest magnitude; a draft id may differ from the oracle's only where the
oracle's own logits put the GPU's choice within that tolerance of the top
(a near tie). After such a tie the oracle continues with the GPU's id
(teacher forcing), so the following rounds stay comparable.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle as O
from block_speculative_decoding_dflash_gb300 import binding as B
from block_speculative_decoding_dflash_gb300 import synth

from tolerances import BF16_HIDDEN_L2, BF16_HIDDEN_MAXABS_RATIO, TOL


class LazyRows:
    """Rows of a stored table converted to fp64 only when indexed (the
    embedding gather reads a handful of rows of a [V, H] table)."""

    def __init__(self, a, dtype):
        self.a, self.dtype = a, dtype

    def __getitem__(self, idx):
        return O.as_f64(self.a[idx], self.dtype)


def f64_weights(w: dict, dtype: str, lazy_embed: bool = False) -> dict:
    out = {k: O.as_f64(v, dtype) for k, v in w.items()
           if k != "layers" and not (lazy_embed and k == "embed")}
    if lazy_embed:
        out["embed"] = LazyRows(w["embed"], dtype)
    out["layers"] = [{k: O.as_f64(v, dtype) for k, v in lw.items()} for lw in w["layers"]]
    return out


def torch_dtype(dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def dev_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def assert_rows_close(got, ref, tol, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    scale = np.maximum(np.abs(ref).reshape(ref.shape[0], -1).max(axis=1), 1e-30)
    err = np.abs(got - ref).reshape(ref.shape[0], -1).max(axis=1)
    bad = np.nonzero(err > tol * scale)[0]
    assert bad.size == 0, f"{what}: rows {bad[:8].tolist()} rel err {(err / scale)[bad[:8]].tolist()}"


def assert_hidden_close(got, ref, tol, dtype, what):
    """Final hidden rows. fp32: max-abs <= tol * row max. bf16: relative L2
    error <= BF16_HIDDEN_L2 and max-abs <= BF16_HIDDEN_MAXABS_RATIO *
    BF16_HIDDEN_L2 of the row's largest magnitude, the rule derived in
    test_bf16_tolerance.py (an fp32 implementation with the oracle's rounding
    points already sits at about 1.5% relative L2 after five bf16 layers)."""
    if dtype == "f32":
        return assert_rows_close(got, ref, tol, what)
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    l2 = np.linalg.norm(got - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    mx = np.abs(got - ref).max(axis=1) / np.maximum(np.abs(ref).max(axis=1), 1e-30)
    bad = np.nonzero((l2 > BF16_HIDDEN_L2) | (mx > BF16_HIDDEN_MAXABS_RATIO * BF16_HIDDEN_L2))[0]
    assert bad.size == 0, f"{what}: rows {bad[:8].tolist()} l2 {l2[bad[:8]].tolist()} maxabs {mx[bad[:8]].tolist()}"


def check_ids(got, ref_ids, ref_logits, tol, what):
    """Exact, except at a near tie of the oracle's logits."""
    ties = 0
    for m in range(len(got)):
        if int(got[m]) == int(ref_ids[m]):
            continue
        z = ref_logits[m].astype(np.float64)
        margin = z[int(ref_ids[m])] - z[int(got[m])]
        assert margin <= tol * np.abs(z).max(), f"{what}[{m}]: gpu {got[m]} oracle {ref_ids[m]} margin {margin}"
        ties += 1
    return ties


class Pair:
    """A GPU context and an oracle session fed the same inputs."""

    def __init__(self, cfg: dict, seed: int = 0, weights=None, w64=None, wd=None):
        self.cfg = cfg
        self.dt = cfg["dtype"]
        self.tol = TOL[self.dt]
        self.w = weights if weights is not None else synth.make_weights(cfg, seed)
        self.wd = wd if wd is not None else B.weights_to_device(self.w, self.dt)
        self.w64 = w64 if w64 is not None else f64_weights(self.w, self.dt)
        self.ctx = B.DFlashContext(cfg, self.wd)
        self.sess = O.OracleSession(cfg, self.w64)
        self.ties = 0
        self.dev = "cuda"

    def to_dev(self, a):
        return B.to_device(a, self.dt, self.dev)

    def ingest(self, resid: np.ndarray, first_pos: int, anchor: int):
        self.ctx.ingest_context(self.to_dev(resid), resid.shape[0], first_pos, anchor)
        self.sess.ingest(O.as_f64(resid, self.dt), first_pos, anchor)

    def draft(self, block: int, check_hidden: bool = True):
        """GPU draft; compared with the oracle; returns the GPU's ids."""
        ids = torch.empty(block - 1, dtype=torch.int32, device=self.dev)
        self.ctx.draft_block(block, ids)
        self.ctx.sync()
        ref = self.sess.draft(block)
        got = ids.cpu().numpy().astype(np.int64)
        if check_hidden:
            rows = ref["hidden"].shape[0]
            hid = torch.empty(rows, self.cfg["hidden"], dtype=torch_dtype(self.dt), device=self.dev)
            self.ctx.get_hidden(hid)
            assert_hidden_close(dev_to_f64(hid), ref["hidden"], self.tol, self.dt, "final hidden")
            mx = torch.empty(block - 1, dtype=torch.float32, device=self.dev)
            self.ctx.get_draft_max_logit(mx)
            zmax = ref["logits"].max(axis=1).astype(np.float64)
            scale = np.abs(ref["logits"]).max(axis=1)
            assert np.all(np.abs(mx.cpu().numpy() - zmax) <= self.tol * scale), "max logit"
        bb = torch.empty(block - 1, dtype=torch.int32, device=self.dev)
        self.ctx.get_backbone_ids(bb)
        self.ties += check_ids(bb.cpu().numpy(), ref["backbone_ids"], ref["logits"], self.tol, "backbone ids")
        if "chain_ids" in ref:
            self.check_chain(got, ref, block - 1)
        else:
            assert np.array_equal(got, bb.cpu().numpy()), "draft ids != backbone ids without a Markov head"
        return ids, got, ref

    def check_chain(self, got, ref, gamma):
        """Each chain step, seeded with the GPU's previous id, must pick a
        near-maximal oracle score."""
        w1, w2 = self.w64["markov_w1"], self.w64["markov_w2"]
        prev = self.sess.anchor
        for j in range(gamma):
            m = (w1[prev] @ w2).astype(np.float32)
            score = m if not self.cfg.get("markov_add") else ref["logits"][j].astype(np.float32) + m
            best = int(np.argmax(score))
            if int(got[j]) != best:
                margin = float(score[best]) - float(score[int(got[j])])
                assert margin <= self.tol * float(np.abs(score).max()), f"chain step {j}"
                self.ties += 1
            prev = int(got[j])

    def verify(self, logits: np.ndarray, ids_dev, got_ids, block: int):
        tok = torch.empty(block, dtype=torch.int32, device=self.dev)
        n = torch.empty(1, dtype=torch.int32, device=self.dev)
        self.ctx.verify_accept(self.to_dev(logits), block, ids_dev, tok, n)
        self.ctx.sync()
        tokens, nn, _ = O.verify_accept(O.as_f64(logits, self.dt), got_ids)
        assert int(n.item()) == nn, (int(n.item()), nn)
        t = tok.cpu().numpy()
        assert t[:nn].tolist() == tokens.tolist() and np.all(t[nn:] == -1)
        return tokens, nn

    def append_commit(self, resid_rows: np.ndarray, block: int, gpu_keep: int, keep: int, tokens,
                      accepted: int):
        """GPU: append + commit(gpu_keep) (-1: the verify's n); oracle: the
        same rows, keeping ``keep``."""
        self.ctx.append_block(self.to_dev(resid_rows), block)
        self.ctx.commit(gpu_keep)
        self.sess.append_and_trim(O.as_f64(resid_rows, self.dt), keep)
        self.sess.commit(keep, int(tokens[-1]), block, accepted)

    def check_state(self):
        st = self.ctx.state()
        assert st["position"] == self.sess.pos, (st, self.sess.pos)
        assert st["anchor"] == self.sess.anchor, (st, self.sess.anchor)
        assert st["error"] == 0
        stats = self.ctx.stats()
        assert stats["rounds"] == self.sess.rounds and stats["accepted"] == self.sess.accepted
        assert stats["draft_n"] == self.sess.proposed

    def check_ring(self, layers=None, max_rows=None):
        """The ring's visible window against the oracle history."""
        k, v, pos = self.sess.visible_context()
        if pos.size == 0:
            return
        if max_rows is not None and pos.size > max_rows:
            sel = np.linspace(0, pos.size - 1, max_rows).astype(np.int64)
        else:
            sel = np.arange(pos.size)
        ring = self.ctx.ring()
        L, nkv, hd = self.cfg["n_layers"], self.cfg["n_kv_heads"], self.cfg["head_dim"]
        p0, cnt = int(pos[0]), int(pos[-1] - pos[0] + 1)
        assert cnt == pos.size
        ko = torch.empty(L, cnt, nkv, hd, dtype=torch_dtype(self.dt), device=self.dev)
        vo = torch.empty_like(ko)
        ring.gather(p0, cnt, ko, vo)
        self.ctx.sync()
        ko, vo = dev_to_f64(ko), dev_to_f64(vo)
        for l in (layers if layers is not None else range(L)):
            assert_rows_close(ko[l][sel].reshape(sel.size, -1), k[l][sel].reshape(sel.size, -1),
                              self.tol, f"ring K layer {l}")
            assert_rows_close(vo[l][sel].reshape(sel.size, -1), v[l][sel].reshape(sel.size, -1),
                              self.tol, f"ring V layer {l}")

    def round(self, stream: dict, r: int, block: int, keep=None, check_hidden=True):
        ids_dev, got, ref = self.draft(block, check_hidden)
        L = synth.planted_logits(stream, r, block, got)
        tokens, nn = self.verify(L, ids_dev, got, block)
        k = nn if keep is None else keep
        self.append_commit(synth.resid_rows(stream, r, block), block, -1 if keep is None else keep,
                           k, tokens, nn - 1)
        return nn, k

    def close(self):
        self.ctx.close()
