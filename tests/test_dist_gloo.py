"""The benchmark's multi-rank plumbing on CPU: two gloo ranks (no GPU) meet at
the barrier, agree on the slowest rank's time, and the reference arm runs on
rank 0 only."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        bench.barrier(ws)
        slowest = bench.max_over_ranks(10.0 * rank + 1.5, ws)
        bench.barrier(ws)
        out.put((rank, slowest, bench.run_reference(None, None, ws, rank) if rank > 0 else "skipped"))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ws = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, out)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(out.get(timeout=5) for _ in range(ws))
    assert [g[1] for g in got] == [11.5, 11.5]
    assert got[1][2] is None          # the reference arm does no work on rank 1


def test_job_value_counts_every_rank():
    import bench
    one = bench.job_value(1, 4096, 100, 33.0)
    assert bench.job_value(4, 4096, 100, 33.0) == pytest.approx(4 * one)
    assert one == pytest.approx(4096 * 100 / 0.033)
