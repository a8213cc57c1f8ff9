"""dflash_verify_accept_static: the verify entry point for callers that may
not allocate device memory (everything they use comes from a host framework's
pool, or their loop must never trigger cudaMalloc's device-wide sync). It must
give exactly what dflash_verify_accept on a context gives, call after call,
while its scratch lives in one static device array shared by all calls."""

import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from block_speculative_decoding_dflash_gb300 import build
    build.build()
    from block_speculative_decoding_dflash_gb300 import binding
    f = binding.lib.dflash_verify_accept_static
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return binding


@pytest.mark.parametrize("dtype,V,block", [("bf16", 202048, 16), ("f32", 1000, 4),
                                           ("bf16", 1 << 20, 64), ("bf16", 1 << 20, 2)])
def test_static_verify_matches_context_verify_twice(B, dtype, V, block):
    from block_speculative_decoding_dflash_gb300 import synth
    cfg = synth.config("tiny", dtype=dtype, vocab=V, mask_token_id=V - 1, n_layers=1,
                       max_block=max(block, 4))
    ctx = B.DFlashContext(cfg, B.weights_to_device(synth.make_weights(cfg, 0), dtype))
    rng = np.random.default_rng(V + block)
    cur = torch.cuda.current_stream()
    for call in range(2):                       # two calls in a row share the scratch
        L = synth.to_storage(rng.standard_normal((block, V)).astype(np.float32), dtype)
        vals = L.astype(np.uint32) << 16 if dtype == "bf16" else None
        t = np.argmax(vals.view(np.float32) if dtype == "bf16" else L, axis=1)
        d = t[:block - 1].copy()
        d[(call * 5 + 2) % (block - 1)] += 1       # a mismatch partway in: 1 <= n < block
        if block == 2 and call == 1:
            d[0] -= 1                              # and all accepted: n == block
        Ld = B.to_device(L, dtype)
        ids = torch.tensor(d % V, dtype=torch.int32, device="cuda")
        ref_tok = torch.full((block,), -7, dtype=torch.int32, device="cuda")
        ref_n = torch.zeros(1, dtype=torch.int32, device="cuda")
        ctx.verify_accept(Ld, block, ids, ref_tok, ref_n)
        ctx.sync()
        tok = torch.full((block,), -7, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = B.lib.dflash_verify_accept_static(Ld.data_ptr(), B.BF16 if dtype == "bf16" else B.F32,
                                               V, block, ids.data_ptr(), tok.data_ptr(),
                                               n.data_ptr(), cur.cuda_stream)
        assert rc == B.OK, B.last_error()
        cur.synchronize()
        assert int(n.item()) == int(ref_n.item())
        assert 1 <= int(n.item()) <= block
        assert tok.cpu().tolist() == ref_tok.cpu().tolist()
    ctx.close()


def test_static_verify_rejects_sizes_beyond_its_scratch(B):
    x = torch.zeros(4, dtype=torch.int32, device="cuda")
    rc = B.lib.dflash_verify_accept_static(x.data_ptr(), B.F32, 2000000, 4, x.data_ptr(),
                                           x.data_ptr(), x.data_ptr(), None)
    assert rc == B.ERANGE and "static scratch" in B.last_error()
    rc = B.lib.dflash_verify_accept_static(x.data_ptr(), B.F32, 1000, 65, x.data_ptr(),
                                           x.data_ptr(), x.data_ptr(), None)
    assert rc == B.ERANGE


def test_static_verify_allocates_no_device_memory(B):
    """The property this entry point exists for: after a first call on the
    device, further calls leave the device's free memory unchanged."""
    V, block = 202048, 16
    rng = np.random.default_rng(5)
    L = torch.from_numpy(rng.standard_normal((block, V)).astype(np.float32)).cuda()
    ids = torch.zeros(block - 1, dtype=torch.int32, device="cuda")
    tok = torch.zeros(block, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    cur = torch.cuda.current_stream()
    call = lambda: B.lib.dflash_verify_accept_static(L.data_ptr(), B.F32, V, block, ids.data_ptr(),
                                                      tok.data_ptr(), n.data_ptr(), cur.cuda_stream)
    assert call() == B.OK
    cur.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(20):
        assert call() == B.OK
    cur.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert int(n.item()) >= 1
