"""The multi-process side of bench.py without a GPU: two gloo ranks on the CPU
check that the timed region is taken as the maximum over ranks and that the
whole-job value counts every rank's steps (replicas, weak scaling). Also the
reference arm (the CPU oracle), which needs no GPU either."""

import json
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


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


def test_reference_arm_prints_one_line():
    """`bench.py --impl reference` times the CPU oracle on the headline
    workload and prints one JSON line with the same metric, unit and config
    as the GPU arm, a cpu_baseline describing the run, and an e2e record
    (no host-device copies: it runs on the host)."""
    import subprocess
    import oracle
    oracle.build()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "1"], capture_output=True, text=True, timeout=600,
                       env={**os.environ, "RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    # at least three warm-up steps, whatever was asked
    assert d["steps"] == 2 and d["warmup"] == 3 and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"].startswith(bench.HEADLINE)
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_print_nothing():
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600,
                       env={**os.environ, "RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
