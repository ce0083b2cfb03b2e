"""Host logic of bench.py's multi-process mode, on CPU with gloo.

The layer has no exchange step, so N GPUs run N independent replicas; what
the ranks share is the timing protocol: a barrier on both sides of the timed
region and the maximum of the per-rank times.  These tests run that protocol
as two gloo ranks on 127.0.0.1 (no GPU), including a rank that arrives late.
"""
import os
import socket
import time

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_setup("gloo")
    assert (ws, r, local) == (world, rank, rank)
    # per-rank "step times": the job's time is the slowest rank's
    got = bench.max_over_ranks(1.5 + rank, ws)
    # a late rank: the barrier holds the others until it arrives
    if rank == 1:
        time.sleep(0.5)
    t0 = time.perf_counter()
    bench.barrier(ws)
    waited = time.perf_counter() - t0
    out.put((rank, got, waited))
    dist.destroy_process_group()


def test_two_gloo_ranks_share_max_time_and_barrier():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, got, waited = out.get(timeout=120)
        res[rank] = (got, waited)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank sees the maximum over ranks
    assert res[0][0] == pytest.approx(2.5)
    assert res[1][0] == pytest.approx(2.5)
    # rank 0 waited at the barrier for the late rank 1
    assert res[0][1] > 0.3


def test_single_process_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)  # no-op without a process group
