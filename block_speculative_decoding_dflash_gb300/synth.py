"""Seeded synthetic inputs for the DFlash round: configs, weights, context slabs,
and the stand-in target (block logits with planted draft matches, captured
residual rows).

This module holds no step of the round itself. It only draws inputs, so both
the CUDA library's tests and the CPU oracle can be fed the same arrays.
Every tensor is drawn from its own PCG64 stream keyed by (seed, name), so a
tensor's values do not depend on which other tensors were drawn first.

Storage format: fp32 tensors are ``float32`` arrays; bf16 tensors are
``uint16`` arrays holding the bfloat16 bit patterns (rounded to nearest even
from the fp32 draw by ``torch``'s conversion).
"""

from __future__ import annotations

import copy
import os
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

# Drafter shapes. "tiny" is the fp32 parity shape; "muse" is the Muse Glimmer
# assistant drafter shape; "dspark" is the DSpark backbone with its Markov head.
CONFIGS = {
    "tiny": dict(
        n_layers=5, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16,
        intermediate=128, vocab=1024, window=16, k_target_layers=5,
        target_hidden=64, mask_token_id=1023, rope_neox=True, rope_theta=1e6,
        rms_eps=1e-6, softcap=0.0, dtype="f32", kind="dflash",
        markov_rank=0, markov_add=0, tied_lm_head=False, max_block=4,
        context_rows=32, weight_std=0.02, logit_std=1.0, p_plant=0.6,
        block=4, rounds=64,
    ),
    "muse": dict(
        n_layers=5, hidden=2048, n_q_heads=32, n_kv_heads=8, head_dim=128,
        intermediate=6144, vocab=202048, window=2048, k_target_layers=5,
        target_hidden=2048, mask_token_id=202047, rope_neox=True,
        rope_theta=1e6, rms_eps=1e-6, softcap=20.0, dtype="bf16",
        kind="dflash", markov_rank=0, markov_add=0, tied_lm_head=False,
        max_block=16, context_rows=2048, weight_std=0.02, logit_std=3.0,
        p_plant=0.7, block=4, rounds=512,
    ),
    "dspark": dict(
        n_layers=5, hidden=2048, n_q_heads=16, n_kv_heads=8, head_dim=128,
        intermediate=8192, vocab=65536, window=0, k_target_layers=5,
        target_hidden=2048, mask_token_id=65535, rope_neox=False,
        rope_theta=1e6, rms_eps=1e-6, softcap=0.0, dtype="bf16",
        kind="dspark", markov_rank=256, markov_add=0, tied_lm_head=True,
        max_block=10, context_rows=1024, weight_std=0.02, markov_std=0.05,
        logit_std=1.0, p_plant=0.6, block=8, rounds=512,
    ),
}


def config(name: str, **overrides) -> dict:
    cfg = copy.deepcopy(CONFIGS[name])
    cfg.update(overrides)
    return cfg


def _stream(seed: int, name: str) -> np.random.Generator:
    return np.random.default_rng([int(seed), zlib.crc32(name.encode())])


def _f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bfloat16 bit patterns, nearest-even."""
    u = a.view(np.uint32)
    return ((u + (np.uint32(0x7FFF) + ((u >> 16) & np.uint32(1)))) >> 16).astype(np.uint16)


def to_storage(a: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 array -> storage array (float32, or uint16 bf16 bits)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a if dtype == "f32" else _f32_to_bf16_bits(a)


_CHUNK = 1 << 22


def normal(seed: int, name: str, shape, std: float, dtype: str) -> np.ndarray:
    """N(0, std) tensor in storage format. Element i belongs to chunk
    i // 2^22, and chunk c is drawn from its own PCG64 stream keyed by
    (seed, name, c), so large tensors are drawn on all cores with values
    independent of the thread count."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)
    key = zlib.crc32(name.encode())

    def fill(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = np.random.default_rng([int(seed), key, c])
        x = g.standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[lo:hi] = _f32_to_bf16_bits(x) if dtype == "bf16" else x

    chunks = (n + _CHUNK - 1) // _CHUNK
    if chunks > 1:
        with ThreadPoolExecutor(max_workers=min(chunks, os.cpu_count() or 4)) as ex:
            list(ex.map(fill, range(chunks)))
    else:
        fill(0)
    return out.reshape(shape)


def ones(shape, dtype: str) -> np.ndarray:
    return to_storage(np.ones(shape, dtype=np.float32), dtype)


def make_weights(cfg: dict, seed: int = 0) -> dict:
    """Drafter weights: linear layers and tables N(0, weight_std), norm gains
    1.0, Markov factors N(0, markov_std). Linear weights are [out, in]."""
    dt, std = cfg["dtype"], cfg["weight_std"]
    H, nq, nkv, hd = cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    I, V = cfg["intermediate"], cfg["vocab"]
    kin = cfg["k_target_layers"] * cfg["target_hidden"]
    w = {
        "embed": normal(seed, "embed", (V, H), std, dt),
        "fc": normal(seed, "fc", (H, kin), std, dt),
        "hidden_norm": ones((H,), dt),
        "final_norm": ones((H,), dt),
        "layers": [],
    }
    w["lm_head"] = w["embed"] if cfg.get("tied_lm_head") else normal(seed, "lm_head", (V, H), std, dt)
    for l in range(cfg["n_layers"]):
        p = f"layer{l}."
        w["layers"].append({
            "in_norm": ones((H,), dt),
            "wq": normal(seed, p + "wq", (nq * hd, H), std, dt),
            "wk": normal(seed, p + "wk", (nkv * hd, H), std, dt),
            "wv": normal(seed, p + "wv", (nkv * hd, H), std, dt),
            "q_norm": ones((hd,), dt),
            "k_norm": ones((hd,), dt),
            "wo": normal(seed, p + "wo", (H, nq * hd), std, dt),
            "post_norm": ones((H,), dt),
            "wg": normal(seed, p + "wg", (I, H), std, dt),
            "wu": normal(seed, p + "wu", (I, H), std, dt),
            "wd": normal(seed, p + "wd", (H, I), std, dt),
        })
    r = cfg.get("markov_rank", 0)
    if r > 0:
        ms = cfg.get("markov_std", 0.05)
        w["markov_w1"] = normal(seed, "markov_w1", (V, r), ms, dt)
        w["markov_w2"] = normal(seed, "markov_w2", (r, V), ms, dt)
    return w


LAYER_KEYS = ("in_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo",
              "post_norm", "wg", "wu", "wd")

# Synthetic targets for the verify forward: Qwen3-shaped causal decoders whose
# width is the drafter's target_hidden and whose captured layers feed its
# encoder.fc (k_target_layers of them); sliding layers with the drafter's
# window except the last, which sees its whole history.
TARGETS = {
    "tiny": dict(
        n_layers=6, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16,
        intermediate=128, vocab=1024, window=16, full_layers=(5,),
        capture=(1, 2, 3, 4, 5), rope_neox=True, rope_theta=1e6, rms_eps=1e-6,
        dtype="f32", max_block=16, max_context=512, weight_std=0.05,
    ),
    "muse": dict(
        n_layers=6, hidden=2048, n_q_heads=32, n_kv_heads=8, head_dim=128,
        intermediate=6144, vocab=202048, window=2048, full_layers=(5,),
        capture=(1, 2, 3, 4, 5), rope_neox=True, rope_theta=1e6, rms_eps=1e-6,
        dtype="bf16", max_block=32, max_context=8192, weight_std=0.02,
    ),
}


def target_config(name: str, **overrides) -> dict:
    cfg = copy.deepcopy(TARGETS[name])
    cfg.update(overrides)
    return cfg


def make_target_weights(tcfg: dict, drafter_weights: dict, seed: int = 1) -> dict:
    """Target weights: its own layers (N(0, weight_std), gains 1.0) and final
    norm; the raw embedding table and the untied lm_head are the drafter's
    (the drafter binds the target's)."""
    dt, std = tcfg["dtype"], tcfg["weight_std"]
    H, nq, nkv, hd, I = (tcfg[k] for k in ("hidden", "n_q_heads", "n_kv_heads", "head_dim", "intermediate"))
    w = {"embed": drafter_weights["embed"], "lm_head": drafter_weights["lm_head"],
         "final_norm": ones((H,), dt), "layers": []}
    for l in range(tcfg["n_layers"]):
        p = f"target{l}."
        w["layers"].append({
            "in_norm": ones((H,), dt),
            "wq": normal(seed, p + "wq", (nq * hd, H), std, dt),
            "wk": normal(seed, p + "wk", (nkv * hd, H), std, dt),
            "wv": normal(seed, p + "wv", (nkv * hd, H), std, dt),
            "q_norm": ones((hd,), dt),
            "k_norm": ones((hd,), dt),
            "wo": normal(seed, p + "wo", (H, nq * hd), std, dt),
            "post_norm": ones((H,), dt),
            "wg": normal(seed, p + "wg", (I, H), std, dt),
            "wu": normal(seed, p + "wu", (I, H), std, dt),
            "wd": normal(seed, p + "wd", (H, I), std, dt),
        })
    return w


def make_prompt(tcfg: dict, rows: int, seed: int = 0) -> np.ndarray:
    """Prompt token ids, uniform over the vocabulary."""
    return _stream(seed, "prompt").integers(0, tcfg["vocab"], rows).astype(np.int32)


def make_context(cfg: dict, rows: int, seed: int = 0, name: str = "context") -> np.ndarray:
    """Captured target residual rows [rows, k * target_hidden], N(0, 1)."""
    kin = cfg["k_target_layers"] * cfg["target_hidden"]
    return normal(seed, name, (rows, kin), 1.0, cfg["dtype"])


def make_target_stream(cfg: dict, rounds: int, block_max: int, seed: int = 0,
                       logit_pool: int = 8, resid_pool: int = 64,
                       p_plant: float | None = None) -> dict:
    """The stand-in target's per-round inputs.

    * ``logits``: a pool [logit_pool, block_max, V] of N(0, logit_std) rows;
      round r uses entry r % logit_pool.
    * ``plant``: [logit_pool, block_max] storage values max(row) + 1, the
      value a planted draft token gets so it becomes the row's unique argmax.
    * ``coins``: [rounds, block_max] uint8, 1 with probability p_plant: whether
      row i of round r plants the draft token d_{i+1}.
    * ``resid``: a pool [resid_pool, block_max, k * target_hidden] of N(0, 1)
      captured residual rows; round r uses entry r % resid_pool.
    """
    dt, V = cfg["dtype"], cfg["vocab"]
    p = cfg["p_plant"] if p_plant is None else p_plant
    g = _stream(seed, "logits")
    base = g.standard_normal(logit_pool * block_max * V, dtype=np.float32)
    base = base.reshape(logit_pool, block_max, V) * np.float32(cfg["logit_std"])
    logits = to_storage(base, dt)
    exact = _storage_values(logits, dt)
    plant = to_storage(exact.max(axis=-1) + np.float32(1.0), dt)
    coins = (_stream(seed, "coins").random((rounds, block_max)) < p).astype(np.uint8)
    kin = cfg["k_target_layers"] * cfg["target_hidden"]
    resid = normal(seed, "resid", (resid_pool, block_max, kin), 1.0, dt)
    return {"logits": logits, "plant": plant, "coins": coins, "resid": resid,
            "logit_pool": logit_pool, "resid_pool": resid_pool, "block_max": block_max}


def _storage_values(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32)
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def planted_logits(stream: dict, r: int, block: int, drafts) -> np.ndarray:
    """Round r's target block logits [block, V] in storage format: the pool
    entry with L[i, d_{i+1}] set to the row's plant value wherever coin[r, i]
    is set, for rows i < block - 1 (the last row is never planted, so it always
    supplies a free bonus token). ``drafts[i]`` holds d_{i+1}."""
    k = r % stream["logit_pool"]
    L = np.array(stream["logits"][k, :block], copy=True)
    for i in range(block - 1):
        if stream["coins"][r, i]:
            L[i, int(drafts[i])] = stream["plant"][k, i]
    return L


def resid_rows(stream: dict, r: int, block: int) -> np.ndarray:
    return stream["resid"][r % stream["resid_pool"], :block]
