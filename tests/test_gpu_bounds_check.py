"""The checking build of the library (compiled with QMV_BOUNDS_CHECK): the
matvec kernel tests every shared- and global-memory access against the region
its plan gives it -- each bulk copy against its ring slot and the weights,
each unit a lane reads against the landed rows of its piece, each parked sum
and output against its buffer -- and raises QMV_STATUS_OUT_OF_BOUNDS instead
of making an access outside. A seeded sweep over every matvec family, the
dp4a, block-dot and fused entry points, MoE banks, the three launch modes and
forced plans must leave that bit clear and match the oracle. The sweep runs in
a process of its own, which loads the checking build instead of the product
library."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checking_build_sweep():
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ggml_format_dequant_gb300 import _build
    import ggml_format_dequant_gb300 as q
    _build.build(flavour="check")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "bounds_check_run.py")], capture_output=True,
                       text=True, timeout=1200)
    assert r.returncode == 0, r.stderr[-3000:]
    rec = json.loads(r.stdout.strip().splitlines()[-1])
    assert rec["n_failures"] == 0, rec["failures"]
    assert rec["calls"] >= 130, rec
    assert not rec["status"] & q.QMV_STATUS_OUT_OF_BOUNDS, rec


def test_checking_build_catches_a_planted_fault():
    """The same checks in a build whose planners make every ring slot half as
    long as its pieces need: the copies that would overrun their slot are
    skipped and QMV_STATUS_OUT_OF_BOUNDS is raised, by the matvec kernel and
    by the batch kernel."""
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ggml_format_dequant_gb300 import _build
    import ggml_format_dequant_gb300 as q
    _build.build(flavour="check_planted")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "bounds_check_run.py"), "planted"],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    rec = json.loads(r.stdout.strip().splitlines()[-1])
    assert rec["calls"] >= 4, rec
    assert rec["status"] & q.QMV_STATUS_OUT_OF_BOUNDS, rec         # the matvec kernel's checks
    assert rec["batch_status"] & q.QMV_STATUS_OUT_OF_BOUNDS, rec   # the batch kernel's checks
