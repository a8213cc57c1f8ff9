"""GPU parity at the pages' full shapes (bf16): the Muse-assistant-shaped
drafter (vocab 202048, window 2048, softcap 20), its long-context slab
stress and block-width sweep, and the DSpark-shaped drafter with its Markov
head. Sampled where the oracle would be slow; integer state exact at every
round."""

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


@pytest.fixture(scope="module")
def muse(H):
    """Muse weights on the host (storage), on the device, and in fp64."""
    cfg = synth.config("muse")
    w = synth.make_weights(cfg, 0)
    from block_speculative_decoding_dflash_gb300 import binding as B
    wd = B.weights_to_device(w, "bf16")
    w64 = H.f64_weights(w, "bf16", lazy_embed=True)
    return cfg, w, wd, w64


def _pair(H, muse, **over):
    cfg, w, wd, w64 = muse
    return H.Pair(dict(cfg, **over), weights=w, w64=w64, wd=wd)


def test_muse_ingest_and_rounds(H, muse):
    pair = _pair(H, muse)
    cfg = pair.cfg
    resid = synth.make_context(cfg, 2048)
    pair.ingest(resid, 0, anchor=1234)
    pair.check_ring(max_rows=48)
    stream = synth.make_target_stream(cfg, 8, 16, logit_pool=2, resid_pool=8)
    for r, blk in enumerate((4, 4, 4, 16, 16)):
        pair.round(stream, r, blk)
        pair.check_state()
    pair.check_ring(max_rows=48)
    pair.close()


def test_muse_block_sweep(H, muse):
    """Block in {4, 5, 8, 16, 32, 129}; 129 checks the slack floor."""
    pair = _pair(H, muse, max_block=129)
    cfg = pair.cfg
    assert pair.ctx.ring().capacity() == 2048 + 129
    pair.ingest(synth.make_context(cfg, 2048, seed=2), 0, anchor=77)
    for i, (blk, p) in enumerate([(4, 0.3), (5, 0.7), (8, 0.95), (16, 0.7), (32, 0.95), (129, 0.95)]):
        stream = synth.make_target_stream(cfg, 1, blk, seed=10 + i, logit_pool=1, resid_pool=1, p_plant=p)
        pair.round(stream, 0, blk)
        pair.check_state()
    pair.check_ring(max_rows=64)
    pair.close()


def test_muse_slab_stress_wraparound(H, muse):
    """16384-row slab, rows older than W dropped before fc; block 16, slack
    128; 256 rounds keeping n ~ U{0..16} rows, so append and trim cross the
    ring boundary. The ring content does not depend on the drafts, so the
    oracle tracks every round's ring; the drafts are checked on the first
    rounds and then on one round in 32, long after the ring has wrapped
    (the oracle takes the GPU's anchor there: teacher forcing)."""
    from block_speculative_decoding_dflash_gb300 import binding as B
    pair = _pair(H, muse)
    cfg = pair.cfg
    assert pair.ctx.ring().capacity() == 2048 + 128
    slab = synth.make_context(cfg, 16384, seed=3, name="slab")
    pair.ingest(slab, 0, anchor=4321)
    pair.check_ring(max_rows=64)
    rounds = 256
    stream = synth.make_target_stream(cfg, rounds, 16, seed=3, logit_pool=4, resid_pool=32)
    keeps = np.random.default_rng(33).integers(0, 17, rounds)
    for r in range(3):
        pair.round(stream, r, 16, keep=int(keeps[r]))
        pair.check_state()
    # the remaining rounds: stand-in target on the device, oracle tracks the ring
    pools = {k: torch.from_numpy(np.ascontiguousarray(stream[k])).cuda()
             for k in ("logits", "plant", "coins", "resid")}
    ctx = pair.ctx
    ids = torch.zeros(15, dtype=torch.int32, device="cuda")
    tok = torch.zeros(16, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    Lb = torch.zeros(16, cfg["vocab"], dtype=torch.bfloat16, device="cuda")
    Rb = torch.zeros(16, 10240, dtype=torch.bfloat16, device="cuda")
    checked = 0
    for r in range(3, rounds):
        d = ids
        if r % 32 == 0:
            st = ctx.state()
            assert st["position"] == pair.sess.pos and st["error"] == 0
            pair.sess.anchor = st["anchor"]
            d, _, _ = pair.draft(16)               # compared with the oracle's draft
            checked += 1
        else:
            ctx.draft_block(16, d)
        ctx.synth_target(pools["logits"], pools["plant"], pools["coins"], pools["resid"], 16, d, Lb, Rb)
        ctx.verify_accept(Lb, 16, d, tok, n)
        ctx.append_block(Rb, 16)
        ctx.commit(int(keeps[r]))
        rows = stream["resid"][r % stream["resid_pool"], :16]
        pair.sess.append_and_trim(O.as_f64(rows, "bf16"), int(keeps[r]))
        pair.sess.pos += int(keeps[r])
        pair.sess._forget_old()
        if r % 64 == 63:
            st = ctx.state()
            assert st["position"] == pair.sess.pos and st["error"] == 0
            pair.check_ring(max_rows=32)
    assert pair.sess.pos == 16384 + int(keeps.sum())
    assert checked == 7
    pair.close()


@pytest.mark.parametrize("add", [0, 1])
@pytest.mark.parametrize("stepwise", [0, 1])
def test_dspark_rounds(H, add, stepwise):
    """stepwise 1: the Markov chain one launch per step (the fallback of the
    one cooperative launch)."""
    from block_speculative_decoding_dflash_gb300 import binding as B
    cfg = synth.config("dspark", markov_add=add, max_context=1024 + 4 * 10)
    w = synth.make_weights(cfg, 0)
    pair = H.Pair(cfg, weights=w, w64=H.f64_weights(w, "bf16"))
    pair.ctx.set_option(B.OPT_MARKOV_STEPWISE, stepwise)
    pair.ingest(synth.make_context(cfg, 1024, seed=4), 0, anchor=999)
    stream = synth.make_target_stream(cfg, 4, 10, seed=4, logit_pool=2, resid_pool=4)
    for r, blk in enumerate((8, 10, 8, 10)):
        pair.round(stream, r, blk)
        pair.check_state()
    pair.check_ring(max_rows=48)
    pair.close()
