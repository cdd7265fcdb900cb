"""bench.py's whole-job aggregation over ranks, on two gloo processes (CPU):
timings take the max over ranks, work counts the sum; the reference arm runs
on rank 0 only; a rank that dies between steps makes the other's reduction
fail within the process-group timeout instead of waiting."""
import datetime
import os
import socket
import time

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        timings = [10.0 + rank, 20.0 - rank, 5.0 * (rank + 1)]
        counts = [1000.0 * (rank + 1), 128.0]
        t, c = bench.reduce_over_ranks(timings, counts, torch.device("cpu"))
        assert bench.dist_env() == (world, rank, rank)
        ref = bench.run_reference(_Args()) if rank != 0 else "skipped"
        out.put((rank, t, c, ref))
    finally:
        dist.destroy_process_group()


class _Args:
    workload = "tiny"
    steps = 3
    warmup = 3
    cpu_seconds = 1.0


def test_reduce_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = dict((r, (t, c, ref)) for r, t, c, ref in (q.get(timeout=5) for _ in procs))
    for r in (0, 1):
        t, c, _ = res[r]
        assert t == [11.0, 20.0, 10.0]          # max over ranks
        assert c == [3000.0, 256.0]             # sum over ranks
    assert res[1][2] is None                    # the reference arm does no work off rank 0


def test_reduce_without_process_group_is_identity():
    import bench
    assert not dist.is_initialized()
    assert bench.reduce_over_ranks([1, 2], [3], torch.device("cpu")) == ([1.0, 2.0], [3.0])


def _dying_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=20))
    if rank == 1:
        os._exit(3)                             # dies between steps, without a goodbye
    t0 = time.monotonic()
    try:
        bench.reduce_over_ranks([1.0], [1.0], torch.device("cpu"))
        out.put((rank, "no error", time.monotonic() - t0))
    except Exception as e:                      # the backend's error type varies by version
        out.put((rank, type(e).__name__, time.monotonic() - t0))


def test_dead_rank_fails_the_reduction_instead_of_hanging():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dying_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    rank, outcome, waited = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        if p.is_alive():
            p.kill()
    assert rank == 0
    assert outcome != "no error"                # the survivor learns of it on the host
    assert waited < 60.0                        # within the timeout, not a hang
    assert procs[1].exitcode == 3
