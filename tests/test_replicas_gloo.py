"""The multi-replica plumbing of bench.py on CPU: two gloo ranks.

`bench.py --gpus N` runs N independent replicas (batch-1 rounds have no
exchange step); what the ranks share is the rendezvous, the barrier around
the timed region and the max over ranks of its duration. The reference arm
runs on rank 0 only.
"""

import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

# bench.py picks NCCL when a GPU is visible, and two ranks must not share one
# GPU: this test is for the CPU runner only.
pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="CPU (gloo) test")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup(None)
    assert (w, r, local) == (world, rank, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    # each rank's duration differs; every rank must see the largest
    m = bench.max_over_ranks(10.0 + rank, w)
    # the reference arm does its (slow) work on rank 0 only; the others return at once
    other = bench.run_reference(None, w, r) if r != 0 else None
    bench.barrier(w)
    dist.destroy_process_group()
    out.put((rank, m, other))


def test_two_gloo_ranks_share_barrier_and_max():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    got = sorted(out.get(timeout=5) for _ in range(world))
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 10.0 + world - 1 for g in got)
    assert got[1][2] is None
