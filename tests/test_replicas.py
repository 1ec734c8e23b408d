"""The N > 1 path of bench.py (replicas only): two gloo ranks on the CPU check
that each rank gets its own batch and that the job's time is the slowest
rank's, reduced over the process group."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    from beam_decode_gb300 import workload as wl
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = bench.replica_workload(wl.make_workload("long"), rank)
        ms = bench.job_time_ms(10.0 * (rank + 1), world, "cpu")
        q.put((rank, w.seed, w.ctx_lens, ms, bench.job_value(ms / 4, world)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_reduce_time_and_seed_apart():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, c0, ms0, v0), (r1, s1, c1, ms1, v1) = res
    assert (r0, r1) == (0, 1)
    assert s0 != s1 and c0 == c1            # same shape, different draws
    assert ms0 == ms1 == 20.0                # the slowest rank's time on every rank
    assert v0 == v1 == pytest.approx(2 * 1000.0 / 5.0)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.job_time_ms(7.5, 1, "cpu") == 7.5
    assert bench.job_value(2.0, 1) == 500.0
