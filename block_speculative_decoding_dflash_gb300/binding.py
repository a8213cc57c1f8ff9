"""Python binding of libdflash (ctypes; argument marshalling only).

Every call below forwards to the C ABI in ``include/dflash.h`` with the same
name; tensors are passed as raw device pointers taken from ``torch`` tensors.
Importing this module loads ``libdflash.so`` and fails loudly if it has not
been built -- there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdflash.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() "
                      "or python -m block_speculative_decoding_dflash_gb300.build")
lib = ctypes.CDLL(LIB_PATH)

OK, EINVAL, ERANGE, EREWIND, EEMPTY, ECUDA, ESTATE, EFULL = range(8)
STATUS = {0: "OK", 1: "EINVAL", 2: "ERANGE", 3: "EREWIND", 4: "EEMPTY", 5: "ECUDA",
          6: "ESTATE", 7: "EFULL"}
F32, BF16 = 0, 1
KIND_DFLASH, KIND_DSPARK = 0, 1
RING_UNFLOORED = 1
LAYER_TENSORS = 11
LAYER_KEYS = ("in_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "post_norm",
              "wg", "wu", "wd")


class DFlashError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "intermediate", "vocab",
        "window", "k_target_layers", "target_hidden", "mask_token_id", "rope_neox",
        "max_block", "kind", "markov_rank", "markov_add", "dtype", "max_context")] + [
        ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float), ("softcap", ctypes.c_float)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "embed", "fc", "hidden_norm", "final_norm", "lm_head", "markov_w1", "markov_w2")] + [
        ("layers", ctypes.POINTER(ctypes.c_void_p))]


class TargetConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "intermediate", "vocab", "window")] + [
        ("full_layers", ctypes.c_uint64), ("n_capture", ctypes.c_int32), ("capture", ctypes.c_int32 * 8)] + [
        (n, ctypes.c_int32) for n in ("rope_neox", "max_block", "dtype", "max_context")] + [
        ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float)]


class TargetWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("embed", "final_norm", "lm_head")] + [
        ("layers", ctypes.POINTER(ctypes.c_void_p))]


class Stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("rounds", "draft_n", "accepted", "emitted")]


class RoundStateC(ctypes.Structure):
    _fields_ = [("position", ctypes.c_int64), ("anchor", ctypes.c_int32),
                ("last_n", ctypes.c_int32), ("last_accepted", ctypes.c_int32),
                ("error", ctypes.c_int32)]


_vp, _i32, _i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
OPT_KERNEL_TRACE = 4
OPT_MARKOV_STEPWISE = 8


def _sig(name, res, *args):
    f = getattr(lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_sig("dflash_speculative_slack", _i32, _i32)
_sig("dflash_stats_ratios", ctypes.c_int, ctypes.POINTER(Stats), ctypes.POINTER(ctypes.c_double),
     ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double))
_sig("dflash_config_check", ctypes.c_int, ctypes.POINTER(Config))
_sig("dflash_ctx_create", ctypes.c_int, ctypes.POINTER(Config), ctypes.POINTER(Weights), _vp,
     ctypes.POINTER(_vp))
_sig("dflash_ctx_destroy", None, _vp)
_sig("dflash_last_error", ctypes.c_char_p, _vp)
_sig("dflash_ingest_context", ctypes.c_int, _vp, _vp, _i64, _i64, _i32)
_sig("dflash_set_anchor", ctypes.c_int, _vp, _i32)
_sig("dflash_draft_block", ctypes.c_int, _vp, _i32, _i64, _i32, _vp)
_sig("dflash_sync_round", ctypes.c_int, _vp, _vp, _vp)
_sig("dflash_ctx_create_batched", ctypes.c_int, ctypes.POINTER(Config), ctypes.POINTER(Weights), _i32, _vp,
     ctypes.POINTER(_vp))
_sig("dflash_batch_size", ctypes.c_int, _vp)
_sig("dflash_ingest_context_seq", ctypes.c_int, _vp, _i32, _vp, _i64, _i64, _i32)
_sig("dflash_get_state_seq", ctypes.c_int, _vp, _i32, ctypes.POINTER(RoundStateC))
_sig("dflash_get_stats_seq", ctypes.c_int, _vp, _i32, ctypes.POINTER(Stats))
_sig("dflash_ring_seq", ctypes.c_int, _vp, _i32, ctypes.POINTER(_vp))
_sig("dflash_verify_sampled", ctypes.c_int, _vp, _vp, _i32, _vp, _vp, ctypes.c_float, ctypes.c_float,
     _vp, _vp, _vp)
_sig("dflash_short_conv_block", ctypes.c_int, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp)
_sig("dflash_short_conv_rollback", ctypes.c_int, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp)
_sig("dflash_verify_accept", ctypes.c_int, _vp, _vp, _i32, _vp, _vp, _vp)
_sig("dflash_append_block", ctypes.c_int, _vp, _vp, _i32)
_sig("dflash_commit", ctypes.c_int, _vp, _i32)
_sig("dflash_round", ctypes.c_int, _vp, _vp, _vp, _i32, _vp, _vp, _vp)
_sig("dflash_markov_chain", ctypes.c_int, _vp, _i32, _i32, _vp, _vp)
_sig("dflash_linear", ctypes.c_int, _vp, _vp, _i32, _i32, _vp, _vp, _i32, _vp, _vp, _i32)
_sig("dflash_lm_head_argmax", ctypes.c_int, _vp, _vp, _i32, _vp, _vp)
_sig("dflash_get_hidden", ctypes.c_int, _vp, _vp)
_sig("dflash_get_draft_max_logit", ctypes.c_int, _vp, _vp)
_sig("dflash_get_backbone_ids", ctypes.c_int, _vp, _vp)
_sig("dflash_get_state", ctypes.c_int, _vp, ctypes.POINTER(RoundStateC))
_sig("dflash_get_stats", ctypes.c_int, _vp, ctypes.POINTER(Stats))
_sig("dflash_reset_stats", ctypes.c_int, _vp)
_sig("dflash_ring", ctypes.c_int, _vp, ctypes.POINTER(_vp))
_sig("dflash_capture_begin", ctypes.c_int, _vp)
_sig("dflash_capture_end", ctypes.c_int, _vp, _i32)
_sig("dflash_graph_launch", ctypes.c_int, _vp, _i32)
_sig("dflash_sync", ctypes.c_int, _vp)
_sig("dflash_graph_kernel_count", ctypes.c_int, _vp, _i32, ctypes.POINTER(_i64))
_sig("dflash_set_option", ctypes.c_int, _vp, _i32, _i64)
_sig("dflash_get_option", ctypes.c_int, _vp, _i32, ctypes.POINTER(_i64))
_sig("dflash_kernel_trace", ctypes.c_int, _vp, _vp, _i64, ctypes.POINTER(_i32), ctypes.c_char_p, _i64)
_sig("dflash_lm_head_timing", ctypes.c_int, _vp, _i32)
_sig("dflash_ingest_gemm_timing", ctypes.c_int, _vp, _i32)
_sig("dflash_ingest_gemm_ms", ctypes.c_int, _vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float))
_sig("dflash_lm_head_elapsed_ms", ctypes.c_int, _vp, ctypes.POINTER(ctypes.c_float))
_sig("dflash_synth_target", ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
     _vp, _vp, _vp)
_sig("dflash_target_create", ctypes.c_int, ctypes.POINTER(TargetConfig), ctypes.POINTER(TargetWeights), _vp,
     ctypes.POINTER(_vp))
_sig("dflash_target_forward", ctypes.c_int, _vp, _vp, _i32, _i32, _vp, _vp)
_sig("dflash_target_verify", ctypes.c_int, _vp, _vp, _i32, _vp, _vp, _vp)
_sig("dflash_target_commit", ctypes.c_int, _vp, _vp, _i32)
_sig("dflash_target_full_ring", ctypes.c_int, _vp, ctypes.POINTER(_vp))
_sig("ring_cache_create", ctypes.c_int, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _vp,
     ctypes.POINTER(_vp))
_sig("ring_cache_create_ex", ctypes.c_int, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _vp,
     ctypes.POINTER(_vp))
_sig("ring_cache_destroy", None, _vp)
_sig("ring_cache_append", ctypes.c_int, _vp, _vp, _vp, _i32)
_sig("ring_cache_trim", ctypes.c_int, _vp, _i32)
_sig("ring_cache_offset", ctypes.c_int, _vp, ctypes.POINTER(_i64))
_sig("ring_cache_capacity", ctypes.c_int, _vp, ctypes.POINTER(_i64))
_sig("ring_cache_gather", ctypes.c_int, _vp, _i64, _i32, _vp, _vp)
_sig("ring_cache_last_error", ctypes.c_char_p, _vp)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def speculative_slack(block: int) -> int:
    return lib.dflash_speculative_slack(block)


def stats_ratios(rounds: int, draft_n: int, accepted: int, emitted: int = 0):
    s = Stats(rounds, draft_n, accepted, emitted)
    a, e, c = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    rc = lib.dflash_stats_ratios(ctypes.byref(s), ctypes.byref(a), ctypes.byref(e), ctypes.byref(c))
    if rc:
        raise DFlashError(rc, "stats_ratios")
    return {"accepted_per_round": a.value, "emitted_per_round": e.value, "acceptance": c.value}


def make_config(cfg: dict) -> Config:
    """C config from a config dict (the keys of ``synth.CONFIGS``)."""
    c = Config()
    for k in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "intermediate",
              "vocab", "window", "k_target_layers", "target_hidden", "mask_token_id",
              "max_block", "markov_rank", "markov_add"):
        setattr(c, k, int(cfg.get(k, 0)))
    c.rope_neox = 1 if cfg.get("rope_neox", True) else 0
    c.kind = KIND_DSPARK if cfg.get("kind", "dflash") == "dspark" else KIND_DFLASH
    c.dtype = BF16 if cfg["dtype"] == "bf16" else F32
    c.max_context = int(cfg.get("max_context", 0))
    c.rope_theta = float(cfg.get("rope_theta", 1e6))
    c.rms_eps = float(cfg.get("rms_eps", 1e-6))
    c.softcap = float(cfg.get("softcap", 0.0))
    return c


def config_check(cfg: dict) -> int:
    c = make_config(cfg)
    return lib.dflash_config_check(ctypes.byref(c))


def last_error(ctx=None) -> str:
    return lib.dflash_last_error(ctx).decode()


def to_device(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """Storage array (float32, or uint16 bf16 bits) -> device tensor."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    t = t.to(device)
    torch.cuda.current_stream().synchronize()
    return t


def weights_to_device(w: dict, dtype: str, device="cuda") -> dict:
    out = {}
    for k, v in w.items():
        if k == "layers":
            out["layers"] = [{kk: to_device(vv, dtype, device) for kk, vv in lw.items()} for lw in v]
        elif k == "lm_head" and v is w["embed"]:
            out[k] = None          # tied: filled below
        else:
            out[k] = to_device(v, dtype, device)
    if out.get("lm_head") is None:
        out["lm_head"] = out["embed"]
    return out


class RingCache:
    """A ring KV cache; standalone (owning) or borrowed from a context."""

    def __init__(self, n_layers=None, kv_heads=None, head_dim=None, window=None, max_block=None,
                 dtype="f32", max_context=0, flags=0, stream=None, handle=None, owner=None):
        self._owner = owner
        if handle is not None:
            self.h = handle
            self.borrowed = True
        else:
            self.stream = stream or torch.cuda.Stream()
            h = _vp()
            rc = lib.ring_cache_create_ex(n_layers, kv_heads, head_dim, window, max_block,
                                          BF16 if dtype == "bf16" else F32, max_context, flags,
                                          self.stream.cuda_stream, ctypes.byref(h))
            if rc:
                raise DFlashError(rc, last_error(None))
            self.h = h.value
            self.borrowed = False

    def _check(self, rc):
        if rc:
            raise DFlashError(rc, lib.ring_cache_last_error(self.h).decode())

    def append(self, k, v, n):
        self._check(lib.ring_cache_append(self.h, _ptr(k), _ptr(v), n))

    def trim(self, n):
        self._check(lib.ring_cache_trim(self.h, n))

    def offset(self) -> int:
        o = _i64()
        self._check(lib.ring_cache_offset(self.h, ctypes.byref(o)))
        return o.value

    def capacity(self) -> int:
        o = _i64()
        self._check(lib.ring_cache_capacity(self.h, ctypes.byref(o)))
        return o.value

    def gather(self, pos0, count, k_out, v_out):
        self._check(lib.ring_cache_gather(self.h, pos0, count, _ptr(k_out), _ptr(v_out)))

    def close(self):
        if not self.borrowed and self.h:
            lib.ring_cache_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DFlashContext:
    """One drafter context (C: dflash_ctx). Holds references to the weight
    tensors it borrows."""

    def __init__(self, cfg: dict, weights: dict, stream: torch.cuda.Stream | None = None, n_seq: int = 1):
        """n_seq > 1: a batch of sequences drafted, verified and committed
        together (dflash_ctx_create_batched)."""
        self.cfg = dict(cfg)
        self.n_seq = n_seq
        self.ccfg = make_config(cfg)
        self.weights = weights
        self.stream = stream or torch.cuda.Stream()
        layer_ptrs = []
        for lw in weights["layers"]:
            layer_ptrs += [lw[k].data_ptr() for k in LAYER_KEYS]
        self._layers = (ctypes.c_void_p * len(layer_ptrs))(*layer_ptrs)
        w = Weights()
        w.embed = weights["embed"].data_ptr()
        w.fc = weights["fc"].data_ptr()
        w.hidden_norm = weights["hidden_norm"].data_ptr()
        w.final_norm = weights["final_norm"].data_ptr()
        w.lm_head = weights["lm_head"].data_ptr()
        w.markov_w1 = weights["markov_w1"].data_ptr() if "markov_w1" in weights else None
        w.markov_w2 = weights["markov_w2"].data_ptr() if "markov_w2" in weights else None
        w.layers = ctypes.cast(self._layers, ctypes.POINTER(ctypes.c_void_p))
        h = _vp()
        rc = lib.dflash_ctx_create_batched(ctypes.byref(self.ccfg), ctypes.byref(w), n_seq,
                                           self.stream.cuda_stream, ctypes.byref(h))
        if rc:
            raise DFlashError(rc, last_error(None))
        self.h = h.value
        self._capturing = False

    def _check(self, rc):
        if rc:
            raise DFlashError(rc, lib.dflash_last_error(self.h).decode())

    def _prep(self):
        """Order the context's stream after the caller's current torch stream,
        so tensors torch just wrote are ready (skipped while capturing)."""
        if not self._capturing:
            self.stream.wait_stream(torch.cuda.current_stream())

    def ingest_context(self, resid, rows, first_pos, anchor):
        self._prep()
        self._check(lib.dflash_ingest_context(self.h, _ptr(resid), rows, first_pos, anchor))

    def set_anchor(self, anchor):
        self._prep()
        self._check(lib.dflash_set_anchor(self.h, anchor))

    def draft_block(self, block, draft_ids, anchor=-1, anchor_pos=-1):
        """anchor / anchor_pos < 0: the device-resident anchor and no
        position check (the CUDA-graph round path)."""
        self._prep()
        self._check(lib.dflash_draft_block(self.h, anchor, anchor_pos, block, _ptr(draft_ids)))

    def verify_sampled(self, logits, block, draft_ids, uniforms, temperature, tokens, n,
                       softcap=None, p_draft=None):
        self._prep()
        cap = self.cfg.get("softcap", 0.0) if softcap is None else softcap
        self._check(lib.dflash_verify_sampled(self.h, _ptr(logits), block, _ptr(draft_ids), _ptr(uniforms),
                                              float(temperature), float(cap), _ptr(tokens), _ptr(n),
                                              _ptr(p_draft) if p_draft is not None else None))

    def sync_round(self, block):
        """Waits for the stream; returns (tokens[:n], n) of the last verify
        (a list of them, one per sequence, for a batch)."""
        tok = np.zeros((self.n_seq, block), dtype=np.int32)
        n = np.zeros(self.n_seq, dtype=np.int32)
        self._check(lib.dflash_sync_round(self.h, tok.ctypes.data, n.ctypes.data))
        out = [(tok[s, : int(n[s])], int(n[s])) for s in range(self.n_seq)]
        return out[0] if self.n_seq == 1 else out

    def verify_accept(self, logits, block, draft_ids, tokens, n):
        self._prep()
        self._check(lib.dflash_verify_accept(self.h, _ptr(logits), block, _ptr(draft_ids),
                                             _ptr(tokens), _ptr(n)))

    def append_block(self, resid, block):
        self._prep()
        self._check(lib.dflash_append_block(self.h, _ptr(resid), block))

    def commit(self, keep=-1):
        self._prep()
        self._check(lib.dflash_commit(self.h, keep))

    def round(self, logits, resid, block, draft_ids, tokens, n):
        self._prep()
        self._check(lib.dflash_round(self.h, _ptr(logits), _ptr(resid), block, _ptr(draft_ids),
                                     _ptr(tokens), _ptr(n)))

    def markov_chain(self, anchor, gamma, z, out):
        self._prep()
        self._check(lib.dflash_markov_chain(self.h, anchor, gamma, _ptr(z), _ptr(out)))

    def linear(self, x, M, K, w, N, y, epi=0, w2=None, r=None):
        self._prep()
        self._check(lib.dflash_linear(self.h, _ptr(x), M, K, _ptr(w), _ptr(w2), N, _ptr(r), _ptr(y), epi))

    def lm_head_argmax(self, x, rows, ids, maxv):
        self._prep()
        self._check(lib.dflash_lm_head_argmax(self.h, _ptr(x), rows, _ptr(ids), _ptr(maxv)))

    def get_hidden(self, out):
        self._prep()
        self._check(lib.dflash_get_hidden(self.h, _ptr(out)))

    def get_draft_max_logit(self, out):
        self._prep()
        self._check(lib.dflash_get_draft_max_logit(self.h, _ptr(out)))

    def get_backbone_ids(self, out):
        self._prep()
        self._check(lib.dflash_get_backbone_ids(self.h, _ptr(out)))

    def ingest_context_seq(self, seq, resid, rows, first_pos, anchor):
        self._prep()
        self._check(lib.dflash_ingest_context_seq(self.h, seq, _ptr(resid), rows, first_pos, anchor))

    def state(self, seq: int = 0) -> dict:
        s = RoundStateC()
        self._check(lib.dflash_get_state_seq(self.h, seq, ctypes.byref(s)))
        return {"position": s.position, "anchor": s.anchor, "last_n": s.last_n,
                "last_accepted": s.last_accepted, "error": s.error}

    def stats(self, seq: int = 0) -> dict:
        s = Stats()
        self._check(lib.dflash_get_stats_seq(self.h, seq, ctypes.byref(s)))
        return {"rounds": s.rounds, "draft_n": s.draft_n, "accepted": s.accepted,
                "emitted": s.emitted}

    def reset_stats(self):
        self._check(lib.dflash_reset_stats(self.h))

    def ring(self, seq: int = 0) -> RingCache:
        h = _vp()
        self._check(lib.dflash_ring_seq(self.h, seq, ctypes.byref(h)))
        return RingCache(handle=h.value, owner=self)

    def capture_begin(self):
        self._prep()
        self._check(lib.dflash_capture_begin(self.h))
        self._capturing = True

    def capture_end(self, slot):
        self._capturing = False
        self._check(lib.dflash_capture_end(self.h, slot))

    def graph_launch(self, slot):
        self._check(lib.dflash_graph_launch(self.h, slot))

    def sync(self):
        self._check(lib.dflash_sync(self.h))

    def graph_kernel_count(self, slot) -> int:
        o = _i64()
        self._check(lib.dflash_graph_kernel_count(self.h, slot, ctypes.byref(o)))
        return o.value

    def set_option(self, option: int, value: int):
        self._check(lib.dflash_set_option(self.h, option, value))

    def kernel_trace(self, enable: bool):
        """Stamp each launch of the per-operation draft (see kernel_trace_read)."""
        self._check(lib.dflash_set_option(self.h, OPT_KERNEL_TRACE, 1 if enable else 0))

    def kernel_trace_read(self):
        """[(name, entry_ns, wait_return_ns, exit_ns)] of the last traced draft."""
        n = _i32()
        buf = np.zeros(3 * 256, dtype=np.uint64)
        names = ctypes.create_string_buffer(1 << 14)
        self._check(lib.dflash_kernel_trace(self.h, buf.ctypes.data, buf.size, ctypes.byref(n), names,
                                            len(names)))
        labels = names.value.decode().split("\n")
        return [(labels[i], int(buf[3 * i]), int(buf[3 * i + 1]), int(buf[3 * i + 2])) for i in range(n.value)]

    def lm_head_timing(self, enable: bool):
        self._check(lib.dflash_lm_head_timing(self.h, 1 if enable else 0))

    def ingest_gemm_timing(self, enable: bool):
        self._check(lib.dflash_ingest_gemm_timing(self.h, 1 if enable else 0))

    def ingest_gemm_ms(self):
        """(fc GEMM ms, K|V GEMM ms) of the last timed ingest chunk."""
        a, b = ctypes.c_float(), ctypes.c_float()
        self._check(lib.dflash_ingest_gemm_ms(self.h, ctypes.byref(a), ctypes.byref(b)))
        return a.value, b.value

    def lm_head_elapsed_ms(self) -> float:
        o = ctypes.c_float()
        self._check(lib.dflash_lm_head_elapsed_ms(self.h, ctypes.byref(o)))
        return o.value

    def synth_target(self, logit_pool, plant, coins, resid_pool, block, draft_ids, logits_out,
                     resid_out):
        self._prep()
        self._check(lib.dflash_synth_target(
            self.h, _ptr(logit_pool), _ptr(plant), _ptr(coins), _ptr(resid_pool),
            logit_pool.shape[0], coins.shape[0], resid_pool.shape[0], logit_pool.shape[1], block,
            _ptr(draft_ids), _ptr(logits_out), _ptr(resid_out)))

    def close(self):
        if getattr(self, "h", None):
            lib.dflash_ctx_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def short_conv_block(state, bx, w, layers, lcache, channels, block, dtype, y, state_after=None,
                     stream=None):
    """dflash_short_conv_block on the current torch stream (or `stream`)."""
    st = (stream or torch.cuda.current_stream()).cuda_stream
    rc = lib.dflash_short_conv_block(_ptr(state) if state is not None else None, _ptr(bx), _ptr(w), layers,
                                     lcache, channels, block, BF16 if dtype == "bf16" else F32, _ptr(y),
                                     _ptr(state_after) if state_after is not None else None, st)
    if rc:
        raise DFlashError(rc, last_error(None))


def short_conv_rollback(prev_state, bx, n_dev, layers, lcache, channels, block, dtype, state_out,
                        stream=None):
    """dflash_short_conv_rollback on the current torch stream (or `stream`)."""
    st = (stream or torch.cuda.current_stream()).cuda_stream
    rc = lib.dflash_short_conv_rollback(_ptr(prev_state) if prev_state is not None else None, _ptr(bx),
                                        _ptr(n_dev), layers, lcache, channels, block,
                                        BF16 if dtype == "bf16" else F32, _ptr(state_out), st)
    if rc:
        raise DFlashError(rc, last_error(None))


def make_target_config(tcfg: dict) -> TargetConfig:
    """C target config from a config dict (the keys of ``synth.TARGETS``)."""
    c = TargetConfig()
    for k in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "intermediate", "vocab", "window",
              "max_block", "max_context"):
        setattr(c, k, int(tcfg[k]))
    c.full_layers = sum(1 << int(l) for l in tcfg.get("full_layers", ()))
    cap = tuple(int(l) for l in tcfg["capture"])
    c.n_capture = len(cap)
    for i, l in enumerate(cap):
        c.capture[i] = l
    c.rope_neox = 1 if tcfg.get("rope_neox", True) else 0
    c.dtype = BF16 if tcfg["dtype"] == "bf16" else F32
    c.rope_theta = float(tcfg.get("rope_theta", 1e6))
    c.rms_eps = float(tcfg.get("rms_eps", 1e-6))
    return c


class TargetContext(DFlashContext):
    """The synthetic target (C: dflash_target_create): the verify forward,
    residual capture and cache trim. State, rings, graphs and close come from
    DFlashContext."""

    def __init__(self, tcfg: dict, weights: dict, stream: torch.cuda.Stream | None = None):
        self.cfg = dict(tcfg)
        self.n_seq = 1
        self.ccfg = make_target_config(tcfg)
        self.weights = weights
        self.stream = stream or torch.cuda.Stream()
        layer_ptrs = []
        for lw in weights["layers"]:
            layer_ptrs += [lw[k].data_ptr() for k in LAYER_KEYS]
        self._layers = (ctypes.c_void_p * len(layer_ptrs))(*layer_ptrs)
        w = TargetWeights()
        w.embed = weights["embed"].data_ptr()
        w.final_norm = weights["final_norm"].data_ptr()
        w.lm_head = weights["lm_head"].data_ptr()
        w.layers = ctypes.cast(self._layers, ctypes.POINTER(ctypes.c_void_p))
        h = _vp()
        rc = lib.dflash_target_create(ctypes.byref(self.ccfg), ctypes.byref(w), self.stream.cuda_stream,
                                      ctypes.byref(h))
        if rc:
            raise DFlashError(rc, last_error(None))
        self.h = h.value
        self._capturing = False

    def forward(self, tokens, rows, logit_rows=0, logits=None, captured=None):
        self._prep()
        self._check(lib.dflash_target_forward(self.h, _ptr(tokens), rows, logit_rows, _ptr(logits),
                                              _ptr(captured)))

    def verify(self, drafter, block, draft_ids, logits, captured=None):
        self._prep()
        self._check(lib.dflash_target_verify(self.h, drafter.h, block, _ptr(draft_ids), _ptr(logits),
                                             _ptr(captured)))

    def commit(self, n, block):
        """Trim block - n rows of every layer's cache; n is a DEVICE int32
        tensor (the verify's n)."""
        self._prep()
        self._check(lib.dflash_target_commit(self.h, _ptr(n), block))

    def full_ring(self) -> RingCache | None:
        h = _vp()
        self._check(lib.dflash_target_full_ring(self.h, ctypes.byref(h)))
        return RingCache(handle=h.value, owner=self) if h.value else None
