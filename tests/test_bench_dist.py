"""The multi-process side of bench.py without a GPU: two gloo ranks on the CPU
check that the timed region is taken as the maximum over ranks and that the
whole-job value counts every rank's steps (replicas, weak scaling)."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = [3.0, 5.0][rank]
        ms_max = bench.max_over_ranks(torch, ms, dist, torch.device("cpu"))
        value = bench.whole_job_gbs(world, 100, 9437184, ms_max)
        out.put((rank, ms_max, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_whole_job_value():
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
    for _, ms_max, value in res:
        assert ms_max == 5.0
        assert value == pytest.approx(2 * 100 * 9437184 / 5e-3 / 1e9)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(torch, 4.0, None, torch.device("cpu")) == 4.0
    assert bench.whole_job_gbs(1, 10, 1000, 1.0) == pytest.approx(10 * 1000 / 1e-3 / 1e9)
