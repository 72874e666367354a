"""Host logic of bench.py under several ranks, on CPU with the gloo backend (world size 2):
the job time is the slowest rank's, the rate counts every rank's units, and the baseline arm
runs on rank 0 only."""
import contextlib
import io
import os
import socket
import types

import pytest
import torch.distributed as dist
import torch.multiprocessing as tmp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]
        total = bench.max_over_ranks(local_ms, world)
        # the baseline arm prints its line on rank 0 only; other ranks return without work
        args = types.SimpleNamespace(workload="tiny_f32", warmup=0, steps=0, gpus=world)
        buf = io.StringIO()
        if rank != 0:
            with contextlib.redirect_stdout(buf):
                bench.run_reference(args, rank)
        dist.barrier()
        out.put((rank, total, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_both_replicas():
    world = 2
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    by_rank = {r: (t, s) for r, t, s in results}
    assert by_rank[0][0] == 5.0 and by_rank[1][0] == 5.0
    assert by_rank[1][1] == ""  # rank 1 printed nothing
    # 2 replicas x 1000 bytes x 10 steps over the slowest rank's 5 ms
    assert bench.job_rate(world, 1000, 10, 5.0) == pytest.approx(2 * 1000 * 10 / 5e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.job_rate(1, 10**9, 1, 1000.0) == pytest.approx(1.0)
