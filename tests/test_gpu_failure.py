"""Failure detection on the GPU without a fault: a bounded wait that runs out
raises QMV_STATUS_WAIT_TIMEOUT in the device status word and returns; the
context stays usable for ordinary calls afterwards."""

import time

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def test_wait_timeout_raises_status_and_returns():
    import __graft_entry__
    __graft_entry__.build()
    import ggml_format_dequant_gb300 as q

    q.qmv_device_status(clear=True)
    t0 = time.time()
    q.qmv_selftest_wait_timeout(10_000_000)   # 10 ms
    torch.cuda.synchronize()
    assert time.time() - t0 < 5.0
    st = q.qmv_device_status(clear=True)
    assert st & q.QMV_STATUS_WAIT_TIMEOUT
    assert q.qmv_device_status(clear=True) == 0

    # an ordinary call afterwards: correct result, no status raised
    st_ = synth.Stream(11)
    w = synth.gen_q4k_rows(st_, 64, 1024)
    x = synth.gen_normal(st_, 1024)
    y = torch.empty(64, dtype=torch.float32, device="cuda")
    q.qmv_q4k(torch.from_numpy(w).cuda(), torch.from_numpy(x).cuda(), y, 64, 1024)
    torch.cuda.synchronize()
    ref = oracle.qmv("q4k", w, x, 64, 1024)
    got = y.cpu().numpy().astype(np.float64)
    assert float(np.max(np.abs(ref - got)) / np.max(np.abs(ref))) <= 1e-4
    assert q.qmv_device_status(clear=True) == 0


@pytest.mark.parametrize("m", [1, 4])
def test_timeout_path_marks_outputs_nan(m):
    """The product kernel's own failure path, taken on purpose: every CTA
    behaves as if a staged weight copy had not landed in time. It raises the
    timeout bit, lets its copies land, writes NaN to all of its outputs (no
    stale y survives) and returns; ordinary calls afterwards are correct."""
    import __graft_entry__
    __graft_entry__.build()
    import ggml_format_dequant_gb300 as q

    st_ = synth.Stream(12 + m)
    rows, k = 300, 2048
    w = synth.gen_q4k_rows(st_, rows, k)
    x = synth.gen_normal(st_, m * k).reshape(m, k)
    wd, xd = torch.from_numpy(w).cuda(), torch.from_numpy(x).cuda()
    y = torch.zeros(m, rows, dtype=torch.float32, device="cuda")
    q.qmv_device_status(clear=True)
    q.qmv_selftest_timeout_path(wd, xd, y, rows, k, m)
    torch.cuda.synchronize()
    assert torch.isnan(y).all()
    assert q.qmv_device_status(clear=True) & q.QMV_STATUS_WAIT_TIMEOUT
    assert q.qmv_device_status(clear=True) == 0
    q.qmm_q4k(wd, xd, y, rows, k, m)
    torch.cuda.synchronize()
    ref = oracle.qmm("q4k", w, x, m, rows, k)
    got = y.cpu().numpy().astype(np.float64)
    for i in range(m):
        assert float(np.max(np.abs(ref[i] - got[i])) / np.max(np.abs(ref[i]))) <= 1e-4
    assert q.qmv_device_status(clear=True) == 0
