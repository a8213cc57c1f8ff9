"""The timed path against the oracle: Muse-shape rounds replayed from the CUDA
graphs that bench.py captures (one per verify width, tensor-core kernels,
programmatic dependent launch, stand-in target on the device), compared with
the CPU oracle round by round: draft ids (exact away from near ties), the
verify's emitted tokens and n, the committed position and anchor, the round
counters and the ring's visible window."""

import types

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


def test_muse_graph_rounds_match_oracle(H):
    import bench
    args = types.SimpleNamespace(rounds=32, window=8, challenge_every=4)
    job = bench.Job(args, "cuda")
    c, cfg = job.ctx, job.cfg
    # replay the captured ingest (drops the warm-up rounds' state), then
    # rounds from the plain width graphs
    c.graph_launch(job.SLOT_INGEST)
    c.reset_stats()
    c.sync()
    check = H.Pair.__new__(H.Pair)
    check.cfg, check.dt, check.tol, check.dev, check.ties = cfg, "bf16", H.TOL["bf16"], "cuda", 0
    check.ctx = c
    check.sess = O.OracleSession(cfg, H.f64_weights(job.w, "bf16", lazy_embed=True))
    check.sess.ingest(O.as_f64(job.resid_host, "bf16"), 0, 5)
    sess = check.sess
    widths = [4] * 6 + [16] * 6 + [4] * 2
    for r, w in enumerate(widths):
        assert c.stats()["rounds"] == r
        c.graph_launch(w)
        c.sync()
        got = job.ids[: w - 1].cpu().numpy().astype(np.int64)
        ref = sess.draft(w)
        check.ties += H.check_ids(got, ref["backbone_ids"], ref["logits"], check.tol, f"round {r} ids")
        L = synth.planted_logits(job.ts, r, w, got)
        tokens, nn, _ = O.verify_accept(O.as_f64(L, "bf16"), got)
        assert int(job.n.item()) == nn, (r, int(job.n.item()), nn)
        assert job.tok[:nn].cpu().tolist() == tokens.tolist()
        sess.append_and_trim(O.as_f64(synth.resid_rows(job.ts, r, w), "bf16"), nn)
        sess.commit(nn, int(tokens[-1]), w, nn - 1)
        check.check_state()
        if r % 5 == 4:
            check.check_ring(max_rows=32)
    c.close()
