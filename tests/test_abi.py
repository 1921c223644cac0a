"""The C ABI library without a GPU: it builds, loads, exports every function
include/qmv.h declares, and rejects bad arguments on the host before touching
CUDA (so these calls are safe on a machine with no device)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import ggml_format_dequant_gb300 as q
    return q


def declared_functions():
    src = open(os.path.join(ROOT, "include", "qmv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["qmv_q4k", "qmv_q6k", "qmv_q8_0", "quantize_act_q8", "qmv_q8_dp4a", "moe_qmv_q4k",
              "qmv_strerror"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    L = lib.load()
    for n in declared_functions():
        assert hasattr(L, n), n
    assert os.path.abspath(lib.library_path()).startswith(ROOT)


def test_checking_build_exports_every_declared_symbol(lib):
    """The bounds-checking flavour is the same boundary: every declared
    function, in a library file of its own inside the tree."""
    from ggml_format_dequant_gb300 import _build
    path = _build.lib_path("check")
    assert os.path.exists(path) and os.path.abspath(path).startswith(ROOT)
    assert path != lib.library_path()
    L = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(L, n), n


def test_strerror(lib):
    for code in [0, -1, -2, -3, -4, 12345]:
        assert isinstance(lib.strerror(code), str) and lib.strerror(code)
    assert lib.strerror(-2).startswith("misaligned")


def test_host_side_validation_without_gpu(lib):
    A = 0x10000   # a 16-byte aligned fake address; never dereferenced
    S = 0
    assert lib.qmv_q4k(A, A, A, 4, 300, stream=S, check=False) == lib.QMV_EINVAL
    assert lib.qmv_q4k(A, A, A, 0, 256, stream=S, check=False) == lib.QMV_EINVAL
    assert lib.qmv_q4k(A, A, A, -3, 256, stream=S, check=False) == lib.QMV_EINVAL
    assert lib.qmv_q4k(None, A, A, 4, 256, stream=S, check=False) == lib.QMV_EINVAL
    assert lib.qmv_q4k(A + 8, A, A, 4, 256, stream=S, check=False) == lib.QMV_EALIGN
    assert lib.qmv_q4k(A, A + 2, A, 4, 256, stream=S, check=False) == lib.QMV_EALIGN
    assert lib.qmv_q6k(A, A, A, 4, 32, stream=S, check=False) == lib.QMV_EINVAL
    assert lib.qmv_q8_0(A, A, A, 4, 33, stream=S, check=False) == lib.QMV_EINVAL
    assert lib.quantize_act_q8(A, A, A, None, 0, 32, stream=S, check=False) == lib.QMV_EINVAL
    assert lib.quantize_act_q8(A, A, None, None, 1, 32, stream=S, check=False) == lib.QMV_EINVAL
    assert lib.qmv_q8_dp4a(A, A + 4, A, A, 4, 32, stream=S, check=False) == lib.QMV_EALIGN
    assert lib.qmv_q8_dp4a(A, A, None, A, 4, 32, stream=S, check=False) == lib.QMV_EINVAL
    assert lib.moe_qmv_q4k(A, A, A, 4, 256, None, 2, 8, stream=S, check=False) == lib.QMV_EINVAL
    assert lib.moe_qmv_q4k(A, A, A, 4, 256, A, 70000, 8, stream=S, check=False) == lib.QMV_EINVAL
    assert lib.moe_qmv_q4k(A, A, A, 4, 256, A + 2, 2, 8, stream=S, check=False) == lib.QMV_EALIGN
    assert lib.qmv_dequant_q4k(A, A, 4, 100, stream=S, check=False) == lib.QMV_EINVAL
    assert lib.qmv_q8_dp4a_blockdots(A, A + 1, A, 4, 32, stream=S, check=False) == lib.QMV_EALIGN
    assert lib.qmv_selftest_wait_timeout(0, stream=S, check=False) == lib.QMV_EINVAL
    assert lib.qmv_selftest_wait_timeout(200_000_000, stream=S, check=False) == lib.QMV_EINVAL
    # the batched products: bad k, m, rows, pointers and alignment, for every format
    for fmt, qk in (("q4k", 256), ("q6k", 256), ("q8_0", 32), ("q5k", 256), ("q4_0", 32)):
        f = getattr(lib, f"qmm_{fmt}")
        assert f(A, A, A, 4, qk + 1, 2, stream=S, check=False) == lib.QMV_EINVAL
        assert f(A, A, A, 4, qk, 0, stream=S, check=False) == lib.QMV_EINVAL
        assert f(A, A, A, 0, qk, 2, stream=S, check=False) == lib.QMV_EINVAL
        assert f(None, A, A, 4, qk, 2, stream=S, check=False) == lib.QMV_EINVAL
        assert f(A, A + 4, A, 4, qk, 2, stream=S, check=False) == lib.QMV_EALIGN
        assert f(A, A, A + 2, 4, qk, 2, stream=S, check=False) == lib.QMV_EALIGN
    with pytest.raises(lib.QmvError):
        lib.qmv_q4k(A, A, A, 4, 300, stream=S)


def test_batch_launch_count():
    """The kernel launches a batched call makes (bench.py counts them): the
    matvec for one row of x, else one tensor-core launch per tile of up to 8
    rows, whatever the format and row length."""
    import ggml_format_dequant_gb300 as q
    for fmt in ("q4k", "q6k", "q8_0", "q5k", "q4_0"):
        for k in (256, 4096, 65536):
            assert q.qmm_launches(fmt, k, 1) == 1
            for m in (2, 3, 8):
                assert q.qmm_launches(fmt, k, m) == 1
            assert q.qmm_launches(fmt, k, 9) == 2
            assert q.qmm_launches(fmt, k, 17) == 3


def test_binding_fails_loudly_without_library(tmp_path):
    import ggml_format_dequant_gb300 as q
    saved = q._LIB
    try:
        q._LIB = None
        with pytest.raises(q.QmvLibraryMissing):
            q.load(str(tmp_path / "missing.so"))
    finally:
        q._LIB = saved


def test_launch_options_are_validated_per_call(lib):
    """The overlap mode is an argument of the call (qmv_opts), not process
    state: an unknown mode is refused on the host, and the planner's choice
    for one mode does not depend on any earlier call's mode."""
    A = 0x10000
    S = 0
    for bad in (-1, 3, 99):
        assert lib.qmv_q4k(A, A, A, 4, 256, stream=S, overlap=bad, check=False) == lib.QMV_EINVAL
        assert lib.qmm_q4k(A, A, A, 4, 256, 2, stream=S, overlap=bad, check=False) == lib.QMV_EINVAL
        assert lib.moe_qmv_q4k(A, A, A, 4, 256, A, 2, 8, stream=S, overlap=bad, check=False) == lib.QMV_EINVAL
        with pytest.raises(lib.QmvError):
            lib.qmv_plan_detail(lib.FMT_Q4K, 4096, 4096, overlap=bad)
    assert not hasattr(lib.load(), "qmv_set_weight_prefetch")
    plain = lib.qmv_plan_detail(lib.FMT_Q4K, 4096, 4096)
    indep = lib.qmv_plan_detail(lib.FMT_Q4K, 4096, 4096, overlap=lib.OVERLAP_INDEPENDENT)
    assert indep["ctas"] < plain["ctas"]   # independent calls take fewer CTAs so several are in flight
    assert lib.qmv_plan_detail(lib.FMT_Q4K, 4096, 4096) == plain
    assert lib.qmv_plan_detail(lib.FMT_Q4K, 4096, 4096, overlap=lib.OVERLAP_CHAIN) == plain
