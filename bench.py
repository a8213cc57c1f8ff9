#!/usr/bin/env python
"""Throughput of the DFlash speculative round at batch 1 on GB300.

One step = one whole Muse-assistant-shaped job: ingest 2048 captured context
rows (window 2048), then 512 rounds (draft, stand-in target, verify, ring
append, partial-accept trim) with the verify width starting at 4 and
widening to 16 when a measurement window pays for it. Metric: rounds/s
(whole job, all GPUs). Riding along: draft tokens/s; the HBM roofline
fraction of the lm_head kernel (the round's largest) and of the whole round
per width; a per-kernel-class breakdown from one traced round per width; the
end-to-end rate with host inputs; the CPU oracle on the host cores; and the
other shapes of the workload list (DSpark drafter, long-context slab stress,
block-width sweep), each through captured round graphs. Inputs are synthetic
(seeded), weights random-init bf16.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the CPU oracle (fp64 numpy) on the host cores on
a bounded sample of the same job.
"""

from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DFlash rounds/sec and draft tok/s at B=1; % HBM roofline on lm_head+decode GEMMs"
WORKLOAD = "muse_bf16_ctx2048_w2048_vocab202048_softcap20_512rounds_block4to16"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--rounds", type=int, default=512)
    ap.add_argument("--window", type=int, default=32, help="rounds per width measurement window")
    ap.add_argument("--challenge-every", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-rounds", type=int, default=3)
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the DSpark, slab-stress and width-sweep measurements")
    ap.add_argument("--no-breakdown", action="store_true", help="skip the per-kernel trace")
    ap.add_argument("--config-rounds", type=int, default=64,
                    help="timed rounds per point of the DSpark / width-sweep measurements")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local: int):
        import torch
        self.uuid = None
        try:
            self.uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
        except Exception:
            pass
        self.proc = None
        self.path = os.path.join("/tmp", f"dflash_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu=uuid,{self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = [[p.strip() for p in ln.split(",")] for ln in open(self.path)]
        lines = [p for p in lines if len(p) >= 10]
        mine = [p for p in lines if self.uuid and p[0] == self.uuid]
        for parts in (mine or lines):
            parts = parts[1:]
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
class Job:
    """Device-resident inputs, graphs and the round loop of one Muse job."""

    SLOT_INGEST, SLOT_TIMED, SLOT_E2E, SLOT_E2E_B = 1, 20, 40, 41   # graph slots (< 64) + width

    def __init__(self, args, device):
        import torch
        from block_speculative_decoding_dflash_gb300 import binding as B
        from block_speculative_decoding_dflash_gb300 import synth
        self.torch, self.B, self.synth = torch, B, synth
        self.args = args
        self.widths = (4, 16)
        cfg = synth.config("muse", max_block=max(self.widths))
        self.cfg = cfg
        t0 = time.time()
        self.w = synth.make_weights(cfg, 0)
        self.wd = B.weights_to_device(self.w, "bf16", device)
        self.ctx = B.DFlashContext(cfg, self.wd)
        self.stream = self.ctx.stream
        self.resid_host = synth.make_context(cfg, cfg["context_rows"])
        self.resid = B.to_device(self.resid_host, "bf16", device)
        self.ts = synth.make_target_stream(cfg, args.rounds, 16, logit_pool=8, resid_pool=64)
        i16 = lambda a: np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else np.ascontiguousarray(a)
        tt = lambda a: torch.from_numpy(i16(a)).to(device)
        self.pool_L = tt(self.ts["logits"]).view(torch.bfloat16)
        self.pool_P = tt(self.ts["plant"]).view(torch.bfloat16)
        self.pool_C = tt(self.ts["coins"])
        self.pool_R = tt(self.ts["resid"]).view(torch.bfloat16)
        V, kin = cfg["vocab"], cfg["k_target_layers"] * cfg["target_hidden"]
        self.ids = torch.zeros(16, dtype=torch.int32, device=device)
        self.tok = torch.zeros(16, dtype=torch.int32, device=device)
        self.n = torch.zeros(1, dtype=torch.int32, device=device)
        self.Lb = torch.zeros(16, V, dtype=torch.bfloat16, device=device)
        self.Rb = torch.zeros(16, kin, dtype=torch.bfloat16, device=device)
        # e2e staging: two pools of one entry each, refilled from pinned host
        # memory on a copy stream, round r into pool r % 2, so that round r + 1's
        # inputs cross while round r computes
        self.st = [(torch.zeros(1, 16, V, dtype=torch.bfloat16, device=device),
                    torch.zeros(1, 16, dtype=torch.bfloat16, device=device),
                    torch.zeros(1, 16, dtype=torch.uint8, device=device),
                    torch.zeros(1, 16, kin, dtype=torch.bfloat16, device=device)) for _ in range(2)]
        self.copy_stream = torch.cuda.Stream(device)
        self.copied = [torch.cuda.Event() for _ in range(2)]
        self.freed = [torch.cuda.Event() for _ in range(2)]
        pin = lambda a: torch.from_numpy(i16(a)).pin_memory()
        self.h_L = pin(self.ts["logits"]).view(torch.bfloat16)
        self.h_P = pin(self.ts["plant"]).view(torch.bfloat16)
        self.h_C = pin(self.ts["coins"])
        self.h_R = pin(self.ts["resid"]).view(torch.bfloat16)
        self.h_resid = pin(self.resid_host).view(torch.bfloat16)
        self.h_out = torch.zeros(args.rounds, 17, dtype=torch.int32).pin_memory()
        self.setup_s = time.time() - t0
        self._capture()

    def _round(self, pools):
        c = self.ctx
        L, P, C, R = pools
        c.draft_block(self.bw, self.ids)
        c.synth_target(L, P, C, R, self.bw, self.ids, self.Lb, self.Rb)
        c.verify_accept(self.Lb, self.bw, self.ids, self.tok, self.n)
        c.append_block(self.Rb, self.bw)
        c.commit(-1)

    def _capture(self):
        c = self.ctx
        c.ingest_context(self.resid, self.cfg["context_rows"], 0, 5)
        dev_pools = (self.pool_L, self.pool_P, self.pool_C, self.pool_R)
        for w in self.widths:
            self.bw = w
            self._round(dev_pools)                 # eager warm-up of this width
            for slot, timing, pools in ((w, False, dev_pools), (self.SLOT_TIMED + w, True, dev_pools),
                                        (self.SLOT_E2E + w, False, self.st[0]),
                                        (self.SLOT_E2E_B + w, False, self.st[1])):
                c.lm_head_timing(timing)
                c.capture_begin()
                self._round(pools)
                c.capture_end(slot)
            c.lm_head_timing(False)
        c.ingest_gemm_timing(True)
        c.capture_begin()
        c.ingest_context(self.resid, self.cfg["context_rows"], 0, 5)
        c.capture_end(self.SLOT_INGEST)
        c.ingest_gemm_timing(False)
        c.sync()
        self.kcount = {s: c.graph_kernel_count(s) for s in
                       [self.SLOT_INGEST] + [x + w for w in self.widths
                                             for x in (0, self.SLOT_TIMED, self.SLOT_E2E, self.SLOT_E2E_B)]}

    def run(self, e2e=False):
        """One job. Returns dict of counters; the caller brackets timing."""
        from block_speculative_decoding_dflash_gb300.policy import ThroughputController, resolve_widths
        torch, c, a = self.torch, self.ctx, self.args
        s = self.stream
        launches = 0
        if e2e:
            with torch.cuda.stream(s):
                self.resid.copy_(self.h_resid, non_blocking=True)
            for ev in self.freed:
                ev.record(s)
        c.reset_stats()
        i0, i1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        i0.record(s)
        c.graph_launch(self.SLOT_INGEST)
        i1.record(s)
        launches += self.kcount[self.SLOT_INGEST]
        gemm_ms = c.ingest_gemm_ms()
        # the Muse assistant declares a depth of 4 under the requested 16 rows
        depth, ceiling = resolve_widths(16, configured_depth=4)
        ctl = ThroughputController(depth, ceiling, window=a.window, challenge_every=a.challenge_every)
        done, lm_ms, emitted_prev, proposals = 0, [], 0, 0
        widths_used = []
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        while done < a.rounds:
            w = ctl.next_width()
            nr = min(a.window, a.rounds - done)
            e0.record(s)
            for i in range(nr):
                r = done + i
                if e2e:
                    k = r % 2
                    stL, stP, stC, stR = self.st[k]
                    cs = self.copy_stream
                    cs.wait_event(self.freed[k])   # the round that last read pool k is done
                    with torch.cuda.stream(cs):
                        stL[0, :w].copy_(self.h_L[r % 8, :w], non_blocking=True)
                        stP[0].copy_(self.h_P[r % 8], non_blocking=True)
                        stC[0].copy_(self.h_C[r], non_blocking=True)
                        stR[0, :w].copy_(self.h_R[r % 64, :w], non_blocking=True)
                        self.copied[k].record(cs)
                    s.wait_event(self.copied[k])
                    slot = (self.SLOT_E2E if k == 0 else self.SLOT_E2E_B) + w
                else:
                    slot = self.SLOT_TIMED + w if i == 0 else w
                c.graph_launch(slot)
                launches += self.kcount[slot]
                if e2e:
                    self.freed[r % 2].record(s)
                    with torch.cuda.stream(s):
                        self.h_out[r, :16].copy_(self.tok, non_blocking=True)
                        self.h_out[r, 16:].copy_(self.n, non_blocking=True)
            e1.record(s)
            e1.synchronize()
            st = c.stats()
            ctl.observe(w, st["emitted"] - emitted_prev, e0.elapsed_time(e1))
            emitted_prev = st["emitted"]
            if not e2e:
                lm_ms.append((w, c.lm_head_elapsed_ms()))
            widths_used += [w] * nr
            done += nr
        st = c.stats()
        return {"stats": st, "lm_ms": lm_ms, "launches": launches, "widths": widths_used,
                "controller": ctl.history, "ingest_ms": i0.elapsed_time(i1), "ingest_gemm_ms": gemm_ms}

    def e2e_bytes_per_step(self, widths):
        V, kin = self.cfg["vocab"], self.cfg["k_target_layers"] * self.cfg["target_hidden"]
        h2d = self.resid_host.nbytes + sum(w * V * 2 + 16 * 2 + 16 + w * kin * 2 for w in widths)
        d2h = len(widths) * 17 * 4
        return h2d, d2h


# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the lm_head
# kernel at width 4 (ncu capture of this kernel version on this workload,
# profiles/lmhead_argmax_muse_block4.md): 831.16 MB read + 3.23 MB written.
LMHEAD_TRAFFIC = 834_389_760


def lm_head_bytes(cfg, rows):
    return cfg["vocab"] * cfg["hidden"] * 2 + rows * cfg["hidden"] * 2 + rows * 8


def round_bytes(cfg, block, nctx, n_seq=1):
    """Algorithmic HBM bytes of one round at verify width `block` with `nctx`
    visible context rows: every drafter weight once (5 layers of Wq Wk Wv Wo
    Wg Wu Wd and their norm gains, the lm_head), the window's K and V of every
    layer, the block's embedding rows, the target's block logits, the captured
    residual rows and encoder.fc plus every layer's Wk and Wv for the append,
    and the ring rows it writes. A batch of n_seq sequences streams the
    weights once and everything else once per sequence."""
    H, I, hd, L = cfg["hidden"], cfg["intermediate"], cfg["head_dim"], cfg["n_layers"]
    V, kin = cfg["vocab"], cfg["k_target_layers"] * cfg["target_hidden"]
    qdim, kvdim = cfg["n_q_heads"] * hd, cfg["n_kv_heads"] * hd
    rows = block - 1 if cfg.get("kind") == "dspark" else block
    layer_w = (H * (qdim + 2 * kvdim) + qdim * H + 3 * H * I + 2 * H + 2 * hd) * 2
    shared = L * layer_w + 2 * H * 2 + V * H * 2 + H * kin * 2 + 2 * H * 2 + L * 2 * kvdim * H * 2
    per_seq = L * 2 * nctx * kvdim * 2 + (H * 2 if rows else 0) + block * V * 2 \
        + block * kin * 2 + L * 2 * block * kvdim * 2
    if cfg.get("markov_rank", 0):
        r = cfg["markov_rank"]
        shared += r * V * 2
        per_seq += (block - 1) * r * 2
    return shared + n_seq * per_seq


# bytes each traced kernel class must move per launch (Muse shape)
def _class_bytes(cfg, block):
    H, I, hd, L = cfg["hidden"], cfg["intermediate"], cfg["head_dim"], cfg["n_layers"]
    qdim, kvdim = cfg["n_q_heads"] * hd, cfg["n_kv_heads"] * hd
    kin = cfg["k_target_layers"] * cfg["target_hidden"]
    nctx = cfg["window"] if cfg["window"] > 0 else cfg["context_rows"]
    return {"qkv": H * (qdim + 2 * kvdim) * 2, "attn": 2 * nctx * kvdim * 2, "o": qdim * H * 2,
            "gate_up": 2 * H * I * 2, "down": I * H * 2, "lm_head": cfg["vocab"] * H * 2,
            "append.fc": H * kin * 2 + block * kin * 2, "append.kv": L * 2 * kvdim * H * 2}


def kernel_breakdown(job, peak):
    """One traced round per width (captured like the timed rounds): for every
    kernel of the round the time from the release of its programmatic
    dependency to its last CTA's exit (weights a kernel requested before the
    release stream during its predecessor), summed per class, with the class's
    algorithmic bytes over that time."""
    c, out = job.ctx, {}
    pools = (job.pool_L, job.pool_P, job.pool_C, job.pool_R)
    for w in job.widths:
        job.bw = w
        c.kernel_trace(True)
        c.capture_begin()
        job._round(pools)
        c.capture_end(60)
        c.kernel_trace(False)
        for _ in range(4):
            c.graph_launch(60)
        c.sync()
        tr = c.kernel_trace_read()
        # the attention's split merge is its own kernel (slot .1 of the attention)
        main = [(t[0].replace("attn.1", "attn_merge"),) + tuple(t[1:]) for t in tr
                if t[0].endswith("attn.1") or not re.search(r"\.\d+$", t[0])]
        t0 = min(t[1] for t in main)
        t1 = max(t[3] for t in main)
        by = {}
        for name, _entry, wait_ret, exit_ in main:
            cls = name.split(".", 1)[1] if name.startswith("L") else name
            by.setdefault(cls, []).append((exit_ - wait_ret) / 1e3)
        nb = _class_bytes(job.cfg, w)
        cl = {}
        for cls, us in sorted(by.items()):
            mean = statistics.mean(us)
            e = {"launches": len(us), "us_per_launch": round(mean, 2), "us_per_round": round(sum(us), 1)}
            if cls in nb:
                gbs = nb[cls] / (mean * 1e-6) / 1e9
                e.update({"bytes": nb[cls], "gbs": round(gbs, 1), "frac": round(gbs / peak, 3)})
            cl[cls] = e
        # the attention's phase marks (last CTA through each), after its
        # dependency resolves, averaged over the layers
        d = {name: (e, wr, x) for name, e, wr, x in tr}
        ph = {"loaded": [], "scored": [], "softmax": [], "o_back": [], "exit": [], "merge_exit": []}
        ok = lambda t: 0 < t < (1 << 63)
        for name, _e, wr, x in tr:
            if not name.endswith(".attn") or not ok(wr):
                continue
            s1, s2, s3 = d.get(name + ".1"), d.get(name + ".2"), d.get(name + ".3")
            for key, t in (("loaded", s2[1]), ("scored", s2[2]), ("softmax", s3[1]), ("o_back", s3[2]),
                           ("exit", x), ("merge_exit", s1[2])):
                if ok(t):
                    ph[key].append((t - wr) / 1e3)
        out[str(w)] = {"traced_span_us": round((t1 - t0) / 1e3, 1), "classes": cl,
                       "attn_phases_us": {k: round(statistics.mean(v), 2) for k, v in ph.items() if v}}
    return {"how": "kernel trace (globaltimer) of one captured round per width: per launch, "
                   "dependency release to last CTA exit; attn_phases_us: the attention's last CTA "
                   "through each phase, after its dependency resolves, mean over the layers",
            "by_width": out}


def _pools(B, ts, device):
    import torch
    i16 = lambda a: np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else np.ascontiguousarray(a)
    tt = lambda a: torch.from_numpy(i16(a)).to(device)
    bf = ts["logits"].dtype == np.uint16
    v = (lambda t: t.view(torch.bfloat16)) if bf else (lambda t: t)
    return (v(tt(ts["logits"])), v(tt(ts["plant"])), tt(ts["coins"]), v(tt(ts["resid"])))


class _Rounds:
    """Round buffers and graphs of one side measurement."""

    def __init__(self, ctx, cfg, bmax, device):
        import torch
        V, kin = cfg["vocab"], cfg["k_target_layers"] * cfg["target_hidden"]
        tdt = torch.bfloat16
        self.ctx, self.torch = ctx, torch
        self.ids = torch.zeros(bmax, dtype=torch.int32, device=device)
        self.tok = torch.zeros(bmax, dtype=torch.int32, device=device)
        self.n = torch.zeros(1, dtype=torch.int32, device=device)
        self.Lb = torch.zeros(bmax, V, dtype=tdt, device=device)
        self.Rb = torch.zeros(bmax, kin, dtype=tdt, device=device)

    def round(self, pools, w, keep=-1):
        c = self.ctx
        c.draft_block(w, self.ids)
        c.synth_target(*pools, w, self.ids, self.Lb, self.Rb)
        c.verify_accept(self.Lb, w, self.ids, self.tok, self.n)
        c.append_block(self.Rb, w)
        c.commit(keep)

    def capture(self, slot, pools, w, keep=-1):
        self.ctx.capture_begin()
        self.round(pools, w, keep)
        self.ctx.capture_end(slot)

    def timed(self, slots, s):
        """Launches the graph slots in order; returns elapsed ms."""
        torch = self.torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for sl in slots:
            self.ctx.graph_launch(sl)
        e1.record(s)
        e1.synchronize()
        return e0.elapsed_time(e1)


def side_configs(job, args, peak, device):
    """The other shapes the workload list names, each timed with CUDA events
    on the context's stream through captured round graphs: the DSpark drafter
    (widths 8 and 10, rank-256 Markov chain, append-only cache), the
    long-context slab stress (16384-row slab, window drop, width 16, keep ~
    U{0..16}), the Muse block-width sweep (widths 4..129 x planting
    probability 0.3 / 0.7 / 0.95), batched rounds (2 to 8 sequences at
    widths 4 and 16) and rounds with the synthetic target's verify forward."""
    import torch
    B, synth = job.B, job.synth
    R = args.config_rounds
    out = {}
    # -- DSpark ------------------------------------------------------------------------
    t0 = time.time()
    dcfg = synth.config("dspark", max_context=1024 + 3 * (R + 8) * 10)
    dw = B.weights_to_device(synth.make_weights(dcfg, 0), "bf16", device)
    ctx = B.DFlashContext(dcfg, dw)
    ctx.ingest_context(B.to_device(synth.make_context(dcfg, 1024, seed=4), "bf16", device), 1024, 0, 999)
    ts = synth.make_target_stream(dcfg, 2 * (R + 8) + 8, 10, seed=4, logit_pool=8, resid_pool=16)
    pools = _pools(B, ts, device)
    rb = _Rounds(ctx, dcfg, 10, device)
    res = {}
    for w in (8, 10):
        rb.round(pools, w)
        rb.capture(w, pools, w)
        for _ in range(4):
            ctx.graph_launch(w)
        st0 = ctx.stats()
        ms = rb.timed([w] * R, ctx.stream)
        st1 = ctx.stats()
        nctx = 1024 + (st1["emitted"])
        us = ms * 1e3 / R
        res[str(w)] = {"rounds_per_s": round(R / (ms / 1e3), 1),
                       "draft_tok_s": round(R * (w - 1) / (ms / 1e3), 1),
                       "accepted_per_round": round((st1["accepted"] - st0["accepted"]) / R, 3),
                       "round_us": round(us, 1),
                       "round_frac": round(round_bytes(dcfg, w, nctx) / (us * 1e-6) / 1e9 / peak, 3)}
    out["dspark"] = {"workload": "dspark_bf16_ctx1024_vocab65536_markov256_block8and10",
                     "rounds_timed_per_width": R, "by_width": res,
                     "note": "tied lm_head; proposals are the Markov chain argmax(W1[prev] W2)",
                     "setup_s": round(time.time() - t0, 1)}
    ctx.close()
    del dw
    # -- slab stress ----------------------------------------------------------------------
    t0 = time.time()
    cfg = job.cfg
    ctx = B.DFlashContext(cfg, job.wd)
    slab = B.to_device(synth.make_context(cfg, 16384, seed=3, name="slab"), "bf16", device)
    ctx.ingest_context(slab, 16384, 0, 4321)
    ctx.sync()
    i0, i1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    i0.record(ctx.stream)
    ctx.ingest_context(slab, 16384, 0, 4321)
    i1.record(ctx.stream)
    i1.synchronize()
    ingest_ms = i0.elapsed_time(i1)
    nr = 256
    ts = synth.make_target_stream(cfg, nr + 64, 16, seed=3, logit_pool=4, resid_pool=32)
    pools = _pools(B, ts, device)
    keeps = np.random.default_rng(33).integers(0, 17, nr)
    rb = _Rounds(ctx, cfg, 16, device)
    for k in range(17):
        rb.round(pools, 16, k)
        rb.capture(k, pools, 16, k)
    st0 = ctx.stats()
    ms = rb.timed([int(k) for k in keeps], ctx.stream)
    st1 = ctx.stats()
    us = ms * 1e3 / nr
    out["slab_stress"] = {"workload": "muse_bf16_slab16384_w2048_block16_keepU0to16_256rounds",
                          "ingest_ms": round(ingest_ms, 3),
                          "ingest_note": "16384-row slab: the 14336 rows older than the window are "
                                         "dropped before encoder.fc, 2048 kept",
                          "rounds_per_s": round(nr / (ms / 1e3), 1),
                          "draft_tok_s": round(nr * 15 / (ms / 1e3), 1), "round_us": round(us, 1),
                          "round_frac": round(round_bytes(cfg, 16, 2048) / (us * 1e-6) / 1e9 / peak, 3),
                          "rounds": st1["rounds"] - st0["rounds"],
                          "setup_s": round(time.time() - t0, 1)}
    ctx.close()
    del slab
    # -- block-width sweep ----------------------------------------------------------------
    t0 = time.time()
    scfg = dict(cfg, max_block=129)
    ctx = B.DFlashContext(scfg, job.wd)
    ctx.ingest_context(job.resid, 2048, 0, 77)
    rb = _Rounds(ctx, scfg, 129, device)
    sweep = {}
    for pi, p in enumerate((0.3, 0.7, 0.95)):
        ts = synth.make_target_stream(scfg, 8 * (R + 8), 129, seed=20 + pi, logit_pool=4, resid_pool=8,
                                      p_plant=p)
        pools = _pools(B, ts, device)
        for slot, w in enumerate((4, 5, 8, 16, 32, 129)):
            rb.round(pools, w)
            rb.capture(slot, pools, w)
            for _ in range(4):
                ctx.graph_launch(slot)
            st0 = ctx.stats()
            ms = rb.timed([slot] * R, ctx.stream)
            st1 = ctx.stats()
            us = ms * 1e3 / R
            sweep.setdefault(str(w), {})[str(p)] = {
                "rounds_per_s": round(R / (ms / 1e3), 1),
                "draft_tok_s": round(R * (w - 1) / (ms / 1e3), 1),
                "accepted_per_round": round((st1["accepted"] - st0["accepted"]) / R, 3),
                "round_us": round(us, 1),
                "round_frac": round(round_bytes(scfg, w, 2048) / (us * 1e-6) / 1e9 / peak, 3)}
        del pools
    out["width_sweep"] = {"workload": "muse_bf16_ctx2048_vocab202048_block4to129_p0.3_0.7_0.95",
                          "rounds_timed_per_point": R, "by_width_then_p": sweep,
                          "setup_s": round(time.time() - t0, 1)}
    ctx.close()
    # -- batched rounds --------------------------------------------------------------------
    t0 = time.time()
    kin = cfg["k_target_layers"] * cfg["target_hidden"]
    batched = {}
    for S, w in ((2, 4), (4, 4), (8, 4), (2, 16), (4, 16)):
        bcfg = dict(cfg, max_block=w)
        ctx = B.DFlashContext(bcfg, job.wd, n_seq=S)
        for sq in range(S):
            ctx.ingest_context_seq(sq, job.resid, 2048, 0, 77 + sq)
        ts = synth.make_target_stream(bcfg, S * (R + 8), w, seed=40 + S + w, logit_pool=4, resid_pool=8)
        pools = _pools(B, ts, device)
        ids = torch.zeros(S, w - 1, dtype=torch.int32, device=device)
        tok = torch.zeros(S, w, dtype=torch.int32, device=device)
        n = torch.zeros(S, dtype=torch.int32, device=device)
        Lb = torch.zeros(S, w, cfg["vocab"], dtype=torch.bfloat16, device=device)
        Rb = torch.zeros(S, w, kin, dtype=torch.bfloat16, device=device)

        def one():
            ctx.draft_block(w, ids)
            ctx.synth_target(*pools, w, ids, Lb, Rb)
            ctx.verify_accept(Lb, w, ids, tok, n)
            ctx.append_block(Rb, w)
            ctx.commit(-1)

        one()
        ctx.capture_begin()
        one()
        ctx.capture_end(1)
        for _ in range(4):
            ctx.graph_launch(1)
        st0 = [ctx.stats(sq) for sq in range(S)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(ctx.stream)
        for _ in range(R):
            ctx.graph_launch(1)
        e1.record(ctx.stream)
        e1.synchronize()
        ms = e0.elapsed_time(e1)
        st1 = [ctx.stats(sq) for sq in range(S)]
        acc = sum(st1[sq]["accepted"] - st0[sq]["accepted"] for sq in range(S)) / (R * S)
        us = ms * 1e3 / R
        batched[f"{S}x{w}"] = {
            "n_seq": S, "width": w, "rounds_per_s": round(R / (ms / 1e3), 1),
            "sequence_rounds_per_s": round(S * R / (ms / 1e3), 1),
            "draft_tok_s": round(S * R * (w - 1) / (ms / 1e3), 1),
            "accepted_per_sequence_round": round(acc, 3), "round_us": round(us, 1),
            "round_frac": round(round_bytes(bcfg, w, 2048, S) / (us * 1e-6) / 1e9 / peak, 3)}
        ctx.close()
        del pools, Lb, Rb
    out["batched"] = {"workload": "muse_bf16_ctx2048_w2048_vocab202048_batched_nseq2to8_block4and16",
                      "rounds_timed_per_point": R, "by_nseq_x_width": batched,
                      "note": "one round drafts, verifies and commits every sequence of the batch; "
                              "the weights stream once per round for all of them",
                      "setup_s": round(time.time() - t0, 1)}
    out["target_verify"] = target_rounds(job, R, peak, device)
    return out


def target_bytes(tcfg, block, pos):
    """Algorithmic HBM bytes of one verify forward of the synthetic target at
    committed length pos: its layer weights, the cache rows its layers read
    (window rows for a sliding layer, the whole history for a full one), the
    lm_head, the block's logits and captured rows written, its K/V rows."""
    H, I, hd, L = tcfg["hidden"], tcfg["intermediate"], tcfg["head_dim"], tcfg["n_layers"]
    qdim, kvdim, V = tcfg["n_q_heads"] * hd, tcfg["n_kv_heads"] * hd, tcfg["vocab"]
    layer_w = (H * (qdim + 2 * kvdim) + qdim * H + 3 * H * I + 2 * H + 2 * hd) * 2
    full = set(tcfg["full_layers"])
    kv = sum(2 * (pos if l in full else min(pos, tcfg["window"])) * kvdim * 2 for l in range(L))
    return (L * layer_w + kv + V * H * 2 + H * 2 + block * V * 2
            + block * len(tcfg["capture"]) * H * 2 + L * 2 * block * kvdim * 2)


def target_rounds(job, R, peak, device):
    """Rounds with the synthetic target's real verify forward in place of the
    stand-in logits: a 2048-token prompt prefilled through the target (its
    captured rows are the drafter's context), then rounds of draft -> target
    verify forward -> accept -> append the captured rows -> both commits, one
    CUDA graph per width, timed with CUDA events on the shared stream."""
    import torch
    B, synth = job.B, job.synth
    t0 = time.time()
    cfg = job.cfg
    tcfg = synth.target_config("muse")
    tw = synth.make_target_weights(tcfg, job.w)
    twd = {"embed": job.wd["embed"], "lm_head": job.wd["lm_head"],
           "final_norm": B.to_device(tw["final_norm"], "bf16", device),
           "layers": [{k: B.to_device(v, "bf16", device) for k, v in lw.items()} for lw in tw["layers"]]}
    stream = torch.cuda.Stream()
    target = B.TargetContext(tcfg, twd, stream=stream)
    drafter = B.DFlashContext(cfg, job.wd, stream=stream)
    P, mb, kin, V = 2048, tcfg["max_block"], len(tcfg["capture"]) * tcfg["hidden"], tcfg["vocab"]
    prompt = torch.tensor(synth.make_prompt(tcfg, P, seed=21), device=device)
    cap = torch.empty(P, kin, dtype=torch.bfloat16, device=device)
    last = torch.empty(1, V, dtype=torch.bfloat16, device=device)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for r0 in range(0, P, mb):
        rows = min(mb, P - r0)
        fin = r0 + rows == P
        target.forward(prompt[r0:], rows, 1 if fin else 0, last if fin else None, cap[r0:])
    p1.record(stream)
    p1.synchronize()
    prefill_ms = p0.elapsed_time(p1)
    drafter.ingest_context(cap, P, 0, int(last.float().argmax().item()))
    wmax = 16
    ids = torch.zeros(wmax, dtype=torch.int32, device=device)
    tok = torch.zeros(wmax, dtype=torch.int32, device=device)
    n = torch.zeros(1, dtype=torch.int32, device=device)
    logits = torch.empty(wmax, V, dtype=torch.bfloat16, device=device)
    capb = torch.empty(wmax, kin, dtype=torch.bfloat16, device=device)

    def one(w):
        target._capturing = drafter._capturing
        drafter.draft_block(w, ids)
        target.verify(drafter, w, ids, logits, capb)
        drafter.verify_accept(logits, w, ids, tok, n)
        drafter.append_block(capb, w)
        drafter.commit(-1)
        target.commit(n, w)

    res = {}
    for w in (4, 16):
        one(w)
        drafter.capture_begin()
        one(w)
        drafter.capture_end(w)
        target._capturing = False
        for _ in range(4):
            drafter.graph_launch(w)
        st0 = drafter.stats()
        pos0 = drafter.state()["position"]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(R):
            drafter.graph_launch(w)
        e1.record(stream)
        e1.synchronize()
        ms = e0.elapsed_time(e1)
        st1 = drafter.stats()
        us = ms * 1e3 / R
        nb = round_bytes(cfg, w, cfg["window"]) + target_bytes(tcfg, w, pos0)
        assert target.state()["error"] == 0 and drafter.state()["error"] == 0
        res[str(w)] = {"rounds_per_s": round(R / (ms / 1e3), 1),
                       "emitted_tok_s": round((st1["emitted"] - st0["emitted"]) / (ms / 1e3), 1),
                       "accepted_per_round": round((st1["accepted"] - st0["accepted"]) / R, 3),
                       "round_us": round(us, 1), "round_bytes": nb,
                       "round_frac": round(nb / (us * 1e-6) / 1e9 / peak, 3)}
    drafter.close()
    target.close()
    return {"workload": "muse_bf16_target6L_w2048_full1_prompt2048_block4and16",
            "prefill_ms": round(prefill_ms, 3), "rounds_timed_per_width": R, "by_width": res,
            "note": "random-weight target and drafter: acceptance is what two unrelated random models "
                    "give; the round time is the measurement",
            "setup_s": round(time.time() - t0, 1)}


def cpu_baseline(job, n_rounds, mix):
    """The oracle as it stands, on the host cores: ingest + n_rounds rounds at
    each verify width, weighted by the width mix of the GPU job (mix: width ->
    share of its rounds) and extrapolated to the 512-round job."""
    import oracle as O
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    cfg, w = job.cfg, job.w
    t0 = time.time()
    w64 = {k: O.as_f64(v, "bf16") for k, v in w.items() if k not in ("layers", "embed")}

    class Rows:
        def __getitem__(self, idx):
            return O.as_f64(w["embed"][idx], "bf16")

    w64["embed"] = Rows()
    w64["layers"] = [{k: O.as_f64(v, "bf16") for k, v in lw.items()} for lw in w["layers"]]
    setup = time.time() - t0
    sess = O.OracleSession(cfg, w64)
    t0 = time.time()
    sess.ingest(O.as_f64(job.resid_host, "bf16"), 0, 5)
    t_ingest = time.time() - t0
    ts = job.ts
    from block_speculative_decoding_dflash_gb300 import synth
    per_width, r = {}, 0
    for bw in sorted(mix):
        t0 = time.time()
        for _ in range(n_rounds):
            d = sess.draft(bw)
            L = synth.planted_logits(ts, r, bw, d["draft_ids"])
            tokens, n, _ = sess.verify(O.as_f64(L, "bf16"), d["draft_ids"])
            sess.append_and_trim(O.as_f64(synth.resid_rows(ts, r, bw), "bf16"), n)
            sess.commit(n, int(tokens[-1]), bw, n - 1)
            r += 1
        per_width[bw] = (time.time() - t0) / n_rounds
    t_round = sum(mix[bw] * per_width[bw] for bw in mix)
    job_s = t_ingest + job.args.rounds * t_round
    cores = len(os.sched_getaffinity(0))
    widths = ", ".join(f"width {bw}: {per_width[bw]:.2f} s/round x {mix[bw]:.2f} of the rounds"
                       for bw in sorted(mix))
    return {"value": job.args.rounds / job_s, "unit": "rounds/s", "cores": cores, "kind": "oracle",
            "sample": f"ingest of 2048 context rows ({t_ingest:.2f} s) + {n_rounds} rounds at each width "
                      f"({widths}), weighted by the GPU job's width mix and extrapolated to the "
                      f"{job.args.rounds}-round job; fp64 weight conversion ({setup:.1f} s) untimed"}


def run_ours(args, world, rank, local):
    import torch
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    job = Job(args, device)
    for _ in range(args.warmup):
        job.run()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(job.stream)
    results = [job.run() for _ in range(args.steps)]
    t_end.record(job.stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms = t_start.elapsed_time(t_end)
    ms_max = max_over_ranks(ms, world)
    rounds = args.rounds * args.steps * world
    value = rounds / (ms_max / 1e3)
    proposals = sum(r["stats"]["draft_n"] for r in results) * world
    accepted = sum(r["stats"]["accepted"] for r in results)
    nrounds = sum(r["stats"]["rounds"] for r in results)
    launches = sum(r["launches"] for r in results)
    lm = [x for r in results for x in r["lm_ms"]]
    peaks, which = measured_peaks()
    lm_bytes = [lm_head_bytes(job.cfg, w - 1) for w, _ in lm]
    kname = "tc_gemm_kernel<16, 3, 6, 2> (lm_head + softcap + argmax, tcgen05, paired K chunks)"
    unit_desc = "lm_head weights per launch"
    lm_t = [t for _, t in lm]
    achieved = sum(lm_bytes) / (sum(lm_t) / 1e3) / 1e9 if lm_t else None
    widths = [w for r in results for w in r["widths"]]
    per_width = {}
    for r in results:
        for (w, tokens, wms, _adopted) in r["controller"]:
            per_width.setdefault(w, []).append(wms / args.window)
    round_us = {str(w): round(1e3 * statistics.mean(v), 1) for w, v in sorted(per_width.items())}

    # context ingest: fc over the kept rows plus every layer's K|V projection
    cfg = job.cfg
    kin = cfg["k_target_layers"] * cfg["target_hidden"]
    rows = cfg["context_rows"]
    ingest_flop = 2 * rows * cfg["hidden"] * kin + \
        cfg["n_layers"] * 2 * rows * cfg["hidden"] * 2 * cfg["n_kv_heads"] * cfg["head_dim"]
    ingest_ms = statistics.median(r["ingest_ms"] for r in results)
    ingest_tf = ingest_flop / (ingest_ms / 1e3) / 1e12
    peak_tf = peaks.get("bf16_tflops", 1900.0)
    fc_flop = 2 * rows * cfg["hidden"] * kin
    kv_flop = ingest_flop - fc_flop
    fc_ms = statistics.median(r["ingest_gemm_ms"][0] for r in results)
    kv_ms = statistics.median(r["ingest_gemm_ms"][1] for r in results)
    gemm_tf = ingest_flop / ((fc_ms + kv_ms) / 1e3) / 1e12
    ingest = {"kernels": "tc_gemm_wide_kernel: encoder.fc, then every layer's K|V with k-norm + RoPE "
                         "into the ring in its epilogue; rmsnorm between",
              "gflop": round(ingest_flop / 1e9, 1), "ms": round(ingest_ms, 4), "tflops": round(ingest_tf, 1),
              "peak_tflops": peaks.get("bf16_tflops"), "frac": round(ingest_tf / peak_tf, 4),
              "gemms": {"fc_ms": round(fc_ms, 4), "fc_tflops": round(fc_flop / (fc_ms / 1e3) / 1e12, 1),
                        "kv_ms": round(kv_ms, 4), "kv_tflops": round(kv_flop / (kv_ms / 1e3) / 1e12, 1),
                        "tflops": round(gemm_tf, 1), "frac": round(gemm_tf / peak_tf, 4),
                        "timing": "CUDA events around the two GEMM launches inside the ingest graph"}}
    e2e = None
    if not args.no_e2e:
        for _ in range(1):
            job.run(e2e=True)
        torch.cuda.synchronize()
        barrier(world)
        e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        e_s.record(job.stream)
        eres = [job.run(e2e=True) for _ in range(args.steps)]
        e_e.record(job.stream)
        torch.cuda.synchronize()
        wall = time.time() - t0
        barrier(world)
        ems = max_over_ranks(e_s.elapsed_time(e_e), world)
        h2d, d2h = job.e2e_bytes_per_step(eres[0]["widths"])
        e2e = {"value": args.rounds * args.steps * world / (ems / 1e3), "unit": "rounds/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "host_wall_s": round(wall, 3)}

    # the round against its HBM roofline, per width: every byte a round must
    # move (round_bytes) over the mean round time the controller measured
    peak = peaks["hbm_gbs"]
    round_roof = {}
    for w, us in round_us.items():
        nb = round_bytes(cfg, int(w), cfg["window"])
        gbs = nb / (us * 1e-6) / 1e9
        round_roof[w] = {"bytes": nb, "us": us, "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)}
    nw = len(widths)
    mix = {w: widths.count(w) / nw for w in set(widths)}
    job_bytes = sum(round_bytes(cfg, w, cfg["window"]) for w in widths) / args.steps
    job_gbs = job_bytes / (ms_max / args.steps / 1e3) / 1e9 / world
    breakdown = None if args.no_breakdown else kernel_breakdown(job, peak)
    configs = None if args.no_configs else side_configs(job, args, peak, device)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(job, args.cpu_rounds, mix)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "rounds/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,0.02) bf16 weights, N(0,1) residual slabs, N(0,3) "
                    "target logits with planted draft matches p=0.7)",
            "config": {"workload": WORKLOAD, "rounds_per_step": args.rounds, "context_rows": 2048,
                       "widths": {"4": widths.count(4), "16": widths.count(16)},
                       "parallelism": f"replicas{world}",
                       "l2": "inputs larger than L2: ~1.5 GB of weights streamed per round"},
            "draft_tok_s": round(proposals / (ms_max / 1e3), 1),
            "round_us_by_width": round_us,
            "accepted_per_round": round(accepted / nrounds, 4),
            "emitted_per_round": round(accepted / nrounds + 1, 4),
            "roofline": {"kernel": kname, "bytes": unit_desc,
                         "bytes_per_launch": {str(w): lm_head_bytes(job.cfg, w - 1) for w in (4, 16)},
                         "bound": "hbm", "achieved": round(achieved, 1) if achieved else None,
                         "peak": peaks["hbm_gbs"], "peak_source": which, "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4) if achieved else None,
                         "traffic": LMHEAD_TRAFFIC, "launches_timed": len(lm_t),
                         "mean_ms": round(sum(lm_t) / len(lm_t), 4) if lm_t else None,
                         "round": {"by_width": round_roof,
                                   "job": {"gbs": round(job_gbs, 1), "frac": round(job_gbs / peak, 4)},
                                   "bytes": "every drafter weight once, the window's K and V of every "
                                            "layer, the block logits, residual rows, encoder.fc and "
                                            "every layer's Wk, Wv for the append, the ring rows "
                                            "written (round_bytes in bench.py)"}},
            "kernels": breakdown,
            "configs": configs,
            "context_ingest": ingest,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clk,
            "setup_s": round(job.setup_s, 1),
        }
        print(json.dumps(line), flush=True)
    job.ctx.close()


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle as O
    from block_speculative_decoding_dflash_gb300 import synth
    cfg = synth.config("muse")
    w = synth.make_weights(cfg, 0)
    w64 = {k: O.as_f64(v, "bf16") for k, v in w.items() if k not in ("layers", "embed")}

    class Rows:
        def __getitem__(self, idx):
            return O.as_f64(w["embed"][idx], "bf16")

    w64["embed"] = Rows()
    w64["layers"] = [{k: O.as_f64(v, "bf16") for k, v in lw.items()} for lw in w["layers"]]
    resid = synth.make_context(cfg, 2048)
    ts = synth.make_target_stream(cfg, args.warmup + args.steps, 16, logit_pool=8, resid_pool=64)
    sess = O.OracleSession(cfg, w64)
    t0 = time.time()
    sess.ingest(O.as_f64(resid, "bf16"), 0, 5)
    t_ingest = time.time() - t0

    def one(r):
        d = sess.draft(4)
        L = synth.planted_logits(ts, r, 4, d["draft_ids"])
        tokens, n, _ = sess.verify(O.as_f64(L, "bf16"), d["draft_ids"])
        sess.append_and_trim(O.as_f64(synth.resid_rows(ts, r, 4), "bf16"), n)
        sess.commit(n, int(tokens[-1]), 4, n - 1)

    for r in range(args.warmup):
        one(r)
    t0 = time.time()
    for r in range(args.steps):
        one(args.warmup + r)
    el = time.time() - t0
    # one step = one round of the job; the job's ingest is amortised over its rounds
    per_round = el / args.steps + t_ingest / args.rounds
    value = 1.0 / per_round
    cores = len(os.sched_getaffinity(0))
    sample = (f"{args.steps} timed oracle rounds at width 4 after {args.warmup} warm-up rounds, plus the "
              f"2048-row ingest ({t_ingest:.2f} s) amortised over {args.rounds} rounds")
    line = {"metric": METRIC, "value": round(value, 4), "unit": "rounds/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_round * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "rounds_per_step": 1, "context_rows": 2048,
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": round(value, 4), "unit": "rounds/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "rounds/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
