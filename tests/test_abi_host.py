"""The C ABI library loads, exports every declared symbol, and its pure host
logic (slack rule, counter ratios, config checks) is right. No GPU needed:
none of these calls reaches CUDA."""

import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "dflash.h")


@pytest.fixture(scope="module")
def B():
    from block_speculative_decoding_dflash_gb300 import build
    build.build()
    from block_speculative_decoding_dflash_gb300 import binding
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?(?:int|void|int32_t|char)\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_round_calls():
    names = declared_functions()
    for must in ("dflash_ctx_create", "dflash_draft_block", "dflash_verify_accept",
                 "ring_cache_append", "ring_cache_trim", "dflash_markov_chain"):
        assert must in names


def test_library_exports_every_declared_symbol(B):
    lib = ctypes.CDLL(B.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_slack_rule_in_library(B, golden):
    for b, floored, _ in golden("slack_rule.txt"):
        assert B.speculative_slack(int(b)) == int(floored)
    assert B.speculative_slack(0) == -1


def test_stats_ratios_match_pages(B, golden):
    for name, rounds, proposed, accepted, tokens, ratio, printed in golden("round_counters.txt"):
        r = B.stats_ratios(int(rounds), int(proposed), int(accepted))
        digits = len(printed.split(".")[1])
        assert round(r[ratio], digits) == float(printed), name


def test_config_checks(B):
    from block_speculative_decoding_dflash_gb300 import synth
    for name in ("tiny", "muse", "dspark"):
        cfg = synth.config(name)
        if cfg["window"] <= 0:
            cfg["max_context"] = 6144
        assert B.config_check(cfg) == B.OK, (name, B.last_error())
    base = synth.config("tiny")
    bad = [
        (dict(mask_token_id=1024), B.ERANGE),
        (dict(mask_token_id=-1), B.ERANGE),
        (dict(max_block=1), B.ERANGE),
        (dict(max_block=2000), B.ERANGE),
        (dict(hidden=0), B.EINVAL),
        (dict(hidden=60), B.EINVAL),
        (dict(n_kv_heads=3), B.EINVAL),
        (dict(head_dim=512), B.EINVAL),
        (dict(window=0, max_context=0), B.EINVAL),
        (dict(vocab=2 ** 31 - 1, max_block=4), B.EINVAL),      # max_block * vocab wraps an int32
        (dict(markov_rank=16, vocab=1020, mask_token_id=5), B.EINVAL),
        (dict(rms_eps=float("nan")), B.EINVAL),
    ]
    for over, code in bad:
        cfg = dict(base, **over)
        assert B.config_check(cfg) == code, (over, B.last_error())
        assert B.last_error() != ""


def test_create_rejects_null_weights_before_cuda(B):
    from block_speculative_decoding_dflash_gb300 import synth
    c = B.make_config(synth.config("tiny"))
    w = B.Weights()
    h = ctypes.c_void_p()
    rc = B.lib.dflash_ctx_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h))
    assert rc == B.EINVAL and h.value is None
    c.mask_token_id = 5000
    assert B.lib.dflash_ctx_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h)) == B.ERANGE


def test_null_context_calls_return_einval(B):
    assert B.lib.dflash_draft_block(None, -1, -1, 4, None) == B.EINVAL
    assert B.lib.dflash_sync_round(None, None, None) == B.EINVAL
    assert B.lib.dflash_commit(None, -1) == B.EINVAL
    assert B.lib.ring_cache_trim(None, 1) == B.EINVAL
    B.lib.dflash_ctx_destroy(None)


def test_batched_create_checks_before_cuda(B):
    """n_seq outside [1, 64], a batch without a sliding window or with a Markov
    head, and n_seq * max_block > 1024 are refused before any GPU work."""
    from block_speculative_decoding_dflash_gb300 import synth
    w = B.Weights()
    h = ctypes.c_void_p()
    c = B.make_config(synth.config("tiny"))
    assert B.lib.dflash_ctx_create_batched(ctypes.byref(c), ctypes.byref(w), 0, None, ctypes.byref(h)) == B.ERANGE
    assert B.lib.dflash_ctx_create_batched(ctypes.byref(c), ctypes.byref(w), 65, None, ctypes.byref(h)) == B.ERANGE
    c2 = B.make_config(dict(synth.config("tiny"), window=0, max_context=64))
    assert B.lib.dflash_ctx_create_batched(ctypes.byref(c2), ctypes.byref(w), 2, None, ctypes.byref(h)) == B.EINVAL
    c3 = B.make_config(dict(synth.config("tiny"), max_block=600))
    assert B.lib.dflash_ctx_create_batched(ctypes.byref(c3), ctypes.byref(w), 2, None, ctypes.byref(h)) == B.ERANGE
    assert "1024" in B.last_error()
    assert h.value is None
    assert B.lib.dflash_batch_size(None) == 0
