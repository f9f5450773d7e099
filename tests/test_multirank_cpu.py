"""The multi-rank (N > 1) host logic of bench.py on CPU: two gloo ranks, each
timing a different step, agree on the slowest rank's time and on the
whole-job throughput, and only rank 0 reports.  No GPU is used."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [12.5, 20.0][rank]
        ms_max = bench.max_over_ranks(local_ms, world, "cpu")
        value = bench.job_tflops(1.0e12, world, ms_max)
        bench.rank_barrier(world)
        out.put((rank, ms_max, value))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_rank_and_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms_max, value in res:
        assert ms_max == 20.0
        # 2 ranks x 1 TFLOP in 20 ms of the slowest rank: 100 TFLOP/s.
        assert value == pytest.approx(100.0)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_tflops(2.0e12, 1, 10.0) == pytest.approx(200.0)
