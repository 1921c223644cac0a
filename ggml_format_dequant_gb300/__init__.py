"""Python binding of libqmv.so, the GB300 GGML-block quantized matvec library.

Argument marshalling only: every function forwards to the C entry point of the
same name (see ``include/qmv.h``), which enqueues the CUDA kernels on the
given stream. Arguments may be ``torch.Tensor`` objects on the GPU (their
``data_ptr()`` is passed) or raw device addresses as ``int``. The stream
defaults to torch's current stream on the current device.

There is no CPU fallback: if the compiled library is missing, loading raises
``QmvLibraryMissing``; build it with ``__graft_entry__.build()`` (or
``python -m ggml_format_dequant_gb300._build``).
"""

from __future__ import annotations

import ctypes
import os

from . import _build

QMV_OK = 0
QMV_EINVAL = -1
QMV_EALIGN = -2
QMV_ECUDA = -3
QMV_ETOOBIG = -4
QMV_STATUS_BAD_EXPERT_ID = 1
QMV_STATUS_WAIT_TIMEOUT = 2
QMV_STATUS_OUT_OF_BOUNDS = 4   # the checking build only (see _build.FLAVOURS)

# Plan ids of qmv_plan_info / qmv_plan_detail (13-15 are not plans).
(FMT_Q4K, FMT_Q6K, FMT_Q8_0, FMT_Q8_DP4A, FMT_MOE_Q4K, FMT_Q4K_DP4A, FMT_MOE_Q6K, FMT_MOE_Q4K_DP4A,
 FMT_Q5K, FMT_Q4_0, FMT_MOE_Q8_0, FMT_MOE_Q4_0, FMT_MOE_Q5K) = range(13)
FMT_Q6K_DP4A, FMT_MOE_Q6K_DP4A, FMT_Q8_DP4A_QUANT = 16, 17, 18


class QmvLibraryMissing(RuntimeError):
    pass


class QmvError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        msg = f"{fn} failed: {code} ({strerror(code)})"
        if code == QMV_ECUDA:
            msg += f": {load().qmv_last_cuda_error().decode()}"
        super().__init__(msg)


# Launch overlap of one call (qmv_opts.overlap, see qmv.h).
OVERLAP_NONE, OVERLAP_CHAIN, OVERLAP_INDEPENDENT = 0, 1, 2


class qmv_opts(ctypes.Structure):
    _fields_ = [("overlap", ctypes.c_int), ("ctas", ctypes.c_int), ("chunk_rows", ctypes.c_int),
                ("chunks", ctypes.c_int), ("unroll", ctypes.c_int), ("warps", ctypes.c_int),
                ("cluster", ctypes.c_int)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SIG = {
    "qmv_q4k": [_P, _P, _P, _I, _I, _P],
    "qmv_q6k": [_P, _P, _P, _I, _I, _P],
    "qmv_q8_0": [_P, _P, _P, _I, _I, _P],
    "quantize_act_q8": [_P, _P, _P, _P, _I, _I, _P],
    "qmv_q8_dp4a": [_P, _P, _P, _P, _I, _I, _P],
    "moe_qmv_q4k": [_P, _P, _P, _I, _I, _P, _I, _I, _P],
    "qmv_q4k_dp4a": [_P, _P, _P, _P, _I, _I, _P],
    "qmv_q8_dp4a_quant": [_P, _P, _P, _I, _I, _P],
    "qmv_q8_dp4a_quant_ex": [_P, _P, _P, _I, _I, _P, _P],
    "moe_qmv_q6k": [_P, _P, _P, _I, _I, _P, _I, _I, _P],
    "moe_qmv_q6k_ex": [_P, _P, _P, _I, _I, _P, _I, _I, _P, _P],
    "moe_qmv_q4k_dp4a": [_P, _P, _P, _P, _I, _I, _P, _I, _I, _P],
    "moe_qmv_q4k_dp4a_ex": [_P, _P, _P, _P, _I, _I, _P, _I, _I, _P, _P],
    "qmv_q4k_dp4a_ex": [_P, _P, _P, _P, _I, _I, _P, _P],
    "qmv_q4k_dp4a_blockdots": [_P, _P, _P, _I, _I, _P],
    "qmv_q6k_dp4a": [_P, _P, _P, _P, _I, _I, _P],
    "qmv_q6k_dp4a_ex": [_P, _P, _P, _P, _I, _I, _P, _P],
    "qmv_q6k_dp4a_blockdots": [_P, _P, _P, _I, _I, _P],
    "moe_qmv_q6k_dp4a": [_P, _P, _P, _P, _I, _I, _P, _I, _I, _P],
    "moe_qmv_q6k_dp4a_ex": [_P, _P, _P, _P, _I, _I, _P, _I, _I, _P, _P],
    "qmv_q4k_ex": [_P, _P, _P, _I, _I, _P, _P],
    "qmv_q6k_ex": [_P, _P, _P, _I, _I, _P, _P],
    "qmv_q8_0_ex": [_P, _P, _P, _I, _I, _P, _P],
    "qmv_q8_dp4a_ex": [_P, _P, _P, _P, _I, _I, _P, _P],
    "moe_qmv_q4k_ex": [_P, _P, _P, _I, _I, _P, _I, _I, _P, _P],
    "qmv_dequant_q4k": [_P, _P, _I, _I, _P],
    "qmv_dequant_q6k": [_P, _P, _I, _I, _P],
    "qmv_dequant_q8_0": [_P, _P, _I, _I, _P],
    "qmv_dequant_q5k": [_P, _P, _I, _I, _P],
    "qmv_dequant_q4_0": [_P, _P, _I, _I, _P],
    "qmm_q4k": [_P, _P, _P, _I, _I, _I, _P],
    "qmm_q4k_ex": [_P, _P, _P, _I, _I, _I, _P, _P],
    "qmm_q4k_tc5_ex": [_P, _P, _P, _I, _I, _I, _P, _P],
    "qmm_q4k_tc5_plan_detail": [_I, _I, _I, _P, _P, _P],
    "qmm_q6k": [_P, _P, _P, _I, _I, _I, _P],
    "qmm_q6k_ex": [_P, _P, _P, _I, _I, _I, _P, _P],
    "qmm_q8_0": [_P, _P, _P, _I, _I, _I, _P],
    "qmm_q8_0_ex": [_P, _P, _P, _I, _I, _I, _P, _P],
    "qmm_q5k": [_P, _P, _P, _I, _I, _I, _P],
    "qmm_q5k_ex": [_P, _P, _P, _I, _I, _I, _P, _P],
    "qmm_q4_0": [_P, _P, _P, _I, _I, _I, _P],
    "qmm_q4_0_ex": [_P, _P, _P, _I, _I, _I, _P, _P],
    "qmv_q5k": [_P, _P, _P, _I, _I, _P],
    "qmv_q5k_ex": [_P, _P, _P, _I, _I, _P, _P],
    "qmv_q4_0": [_P, _P, _P, _I, _I, _P],
    "qmv_q4_0_ex": [_P, _P, _P, _I, _I, _P, _P],
    "moe_qmv_q8_0": [_P, _P, _P, _I, _I, _P, _I, _I, _P],
    "moe_qmv_q8_0_ex": [_P, _P, _P, _I, _I, _P, _I, _I, _P, _P],
    "moe_qmv_q4_0": [_P, _P, _P, _I, _I, _P, _I, _I, _P],
    "moe_qmv_q4_0_ex": [_P, _P, _P, _I, _I, _P, _I, _I, _P, _P],
    "moe_qmv_q5k": [_P, _P, _P, _I, _I, _P, _I, _I, _P],
    "moe_qmv_q5k_ex": [_P, _P, _P, _I, _I, _P, _I, _I, _P, _P],
    "qmv_q8_dp4a_blockdots": [_P, _P, _P, _I, _I, _P],
    "qmv_device_status": [_P, _I],
    "qmv_selftest_wait_timeout": [ctypes.c_ulonglong, _P],
    "qmv_selftest_timeout_path": [_P, _P, _P, _I, _I, _I, _P],
    "qmm_q4k_tc5_selftest_timeout_path": [_P, _P, _P, _I, _I, _I, _P, _P],
    "qmv_plan_info": [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P],
    "qmv_plan_detail": [_I, _I, _I, _I, _P, _P, _P],
    "qmm_tc_plan_detail": [_I, _I, _I, _I, _P, _P, _P],
}

_LIB = None


def library_path() -> str:
    return _build.lib_path()


def load(path: str | None = None):
    """Load libqmv.so (once). Raises QmvLibraryMissing if it was not built."""
    global _LIB
    if _LIB is None:
        p = path or library_path()
        if not os.path.exists(p):
            raise QmvLibraryMissing(f"libqmv.so not built at {p}; run __graft_entry__.build()")
        lib = ctypes.CDLL(p)
        for name, args in _SIG.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        lib.qmv_strerror.argtypes = [ctypes.c_int]
        lib.qmv_strerror.restype = ctypes.c_char_p
        lib.qmv_last_cuda_error.argtypes = []
        lib.qmv_last_cuda_error.restype = ctypes.c_char_p
        _LIB = lib
    return _LIB


def strerror(code: int) -> str:
    return load().qmv_strerror(int(code)).decode()


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _opts(cfg, overlap=0):
    """The qmv_opts of one call: the overlap mode and an optional forced plan
    (a dict of the other qmv_opts fields); None for a plain call."""
    if cfg is None and not overlap:
        return None
    cfg = cfg or {}
    c = qmv_opts(int(overlap), int(cfg.get("ctas", 0)), int(cfg.get("chunk_rows", 0)), int(cfg.get("chunks", 0)),
                 int(cfg.get("unroll", 0)), int(cfg.get("warps", 0)), int(cfg.get("cluster", 0)))
    return ctypes.byref(c)


def _call(name, *args, check=True):
    rc = getattr(load(), name)(*args)
    if check and rc != QMV_OK:
        raise QmvError(name, rc)
    return rc


def qmv_q4k(w, x, y, rows, k, stream=None, cfg=None, overlap=0, check=True):
    if cfg is None and not overlap:
        return _call("qmv_q4k", _ptr(w), _ptr(x), _ptr(y), rows, k, _stream(stream), check=check)
    return _call("qmv_q4k_ex", _ptr(w), _ptr(x), _ptr(y), rows, k, _opts(cfg, overlap), _stream(stream), check=check)


def qmv_q6k(w, x, y, rows, k, stream=None, cfg=None, overlap=0, check=True):
    if cfg is None and not overlap:
        return _call("qmv_q6k", _ptr(w), _ptr(x), _ptr(y), rows, k, _stream(stream), check=check)
    return _call("qmv_q6k_ex", _ptr(w), _ptr(x), _ptr(y), rows, k, _opts(cfg, overlap), _stream(stream), check=check)


def qmv_q8_0(w, x, y, rows, k, stream=None, cfg=None, overlap=0, check=True):
    if cfg is None and not overlap:
        return _call("qmv_q8_0", _ptr(w), _ptr(x), _ptr(y), rows, k, _stream(stream), check=check)
    return _call("qmv_q8_0_ex", _ptr(w), _ptr(x), _ptr(y), rows, k, _opts(cfg, overlap), _stream(stream), check=check)


def _qmm(name, w, x, y, rows, k, m, stream, cfg, overlap, check):
    if cfg is None and not overlap:
        return _call(name, _ptr(w), _ptr(x), _ptr(y), rows, k, m, _stream(stream), check=check)
    return _call(name + "_ex", _ptr(w), _ptr(x), _ptr(y), rows, k, m, _opts(cfg, overlap), _stream(stream), check=check)


def qmm_q4k(w, x, y, rows, k, m, stream=None, cfg=None, overlap=0, check=True):
    return _qmm("qmm_q4k", w, x, y, rows, k, m, stream, cfg, overlap, check)


def qmm_q4k_tc5(w, x, y, rows, k, m, stream=None, cfg=None, overlap=0, check=True):
    return _call("qmm_q4k_tc5_ex", _ptr(w), _ptr(x), _ptr(y), rows, k, m, _opts(cfg, overlap), _stream(stream),
                 check=check)


def qmm_q6k(w, x, y, rows, k, m, stream=None, cfg=None, overlap=0, check=True):
    return _qmm("qmm_q6k", w, x, y, rows, k, m, stream, cfg, overlap, check)


def qmm_q8_0(w, x, y, rows, k, m, stream=None, cfg=None, overlap=0, check=True):
    return _qmm("qmm_q8_0", w, x, y, rows, k, m, stream, cfg, overlap, check)


def qmm_q5k(w, x, y, rows, k, m, stream=None, cfg=None, overlap=0, check=True):
    return _qmm("qmm_q5k", w, x, y, rows, k, m, stream, cfg, overlap, check)


def qmm_q4_0(w, x, y, rows, k, m, stream=None, cfg=None, overlap=0, check=True):
    return _qmm("qmm_q4_0", w, x, y, rows, k, m, stream, cfg, overlap, check)


def qmm_launches(fmt, k, m) -> int:
    """Kernel launches one qmm_<fmt> call makes: the matvec for m = 1, else the
    tensor-core kernel, one launch per tile of up to 8 rows of x (ceil(m / 8)),
    whatever k."""
    return 1 if m == 1 else -(-m // 8)


def qmv_q5k(w, x, y, rows, k, stream=None, cfg=None, overlap=0, check=True):
    if cfg is None and not overlap:
        return _call("qmv_q5k", _ptr(w), _ptr(x), _ptr(y), rows, k, _stream(stream), check=check)
    return _call("qmv_q5k_ex", _ptr(w), _ptr(x), _ptr(y), rows, k, _opts(cfg, overlap), _stream(stream), check=check)


def qmv_q4_0(w, x, y, rows, k, stream=None, cfg=None, overlap=0, check=True):
    if cfg is None and not overlap:
        return _call("qmv_q4_0", _ptr(w), _ptr(x), _ptr(y), rows, k, _stream(stream), check=check)
    return _call("qmv_q4_0_ex", _ptr(w), _ptr(x), _ptr(y), rows, k, _opts(cfg, overlap), _stream(stream), check=check)


def quantize_act_q8(x, xq, xs, xsum, m, k, stream=None, check=True):
    return _call("quantize_act_q8", _ptr(x), _ptr(xq), _ptr(xs), _ptr(xsum), m, k, _stream(stream), check=check)


def qmv_q8_dp4a(w, xq, xs, y, rows, k, stream=None, cfg=None, overlap=0, check=True):
    if cfg is None and not overlap:
        return _call("qmv_q8_dp4a", _ptr(w), _ptr(xq), _ptr(xs), _ptr(y), rows, k, _stream(stream), check=check)
    return _call("qmv_q8_dp4a_ex", _ptr(w), _ptr(xq), _ptr(xs), _ptr(y), rows, k, _opts(cfg, overlap), _stream(stream),
                 check=check)


def qmv_q8_dp4a_quant(w, x, y, rows, k, stream=None, cfg=None, overlap=0, check=True):
    if cfg is None and not overlap:
        return _call("qmv_q8_dp4a_quant", _ptr(w), _ptr(x), _ptr(y), rows, k, _stream(stream), check=check)
    return _call("qmv_q8_dp4a_quant_ex", _ptr(w), _ptr(x), _ptr(y), rows, k, _opts(cfg, overlap), _stream(stream),
                 check=check)


def qmv_q4k_dp4a(w, xq, xs, y, rows, k, stream=None, cfg=None, overlap=0, check=True):
    if cfg is None and not overlap:
        return _call("qmv_q4k_dp4a", _ptr(w), _ptr(xq), _ptr(xs), _ptr(y), rows, k, _stream(stream), check=check)
    return _call("qmv_q4k_dp4a_ex", _ptr(w), _ptr(xq), _ptr(xs), _ptr(y), rows, k, _opts(cfg, overlap), _stream(stream),
                 check=check)


def qmv_q6k_dp4a(w, xq, xs, y, rows, k, stream=None, cfg=None, overlap=0, check=True):
    if cfg is None and not overlap:
        return _call("qmv_q6k_dp4a", _ptr(w), _ptr(xq), _ptr(xs), _ptr(y), rows, k, _stream(stream), check=check)
    return _call("qmv_q6k_dp4a_ex", _ptr(w), _ptr(xq), _ptr(xs), _ptr(y), rows, k, _opts(cfg, overlap), _stream(stream),
                 check=check)


def qmv_q6k_dp4a_blockdots(w, xq, dots, rows, k, stream=None, check=True):
    return _call("qmv_q6k_dp4a_blockdots", _ptr(w), _ptr(xq), _ptr(dots), rows, k, _stream(stream), check=check)


def moe_qmv_q6k_dp4a(w_bank, xq, xs, y, rows, k, ids, slots, n_experts, stream=None, cfg=None, overlap=0, check=True):
    if cfg is None and not overlap:
        return _call("moe_qmv_q6k_dp4a", _ptr(w_bank), _ptr(xq), _ptr(xs), _ptr(y), rows, k, _ptr(ids), slots,
                     n_experts, _stream(stream), check=check)
    return _call("moe_qmv_q6k_dp4a_ex", _ptr(w_bank), _ptr(xq), _ptr(xs), _ptr(y), rows, k, _ptr(ids), slots,
                 n_experts, _opts(cfg, overlap), _stream(stream), check=check)


def qmv_q4k_dp4a_blockdots(w, xq, dots, rows, k, stream=None, check=True):
    return _call("qmv_q4k_dp4a_blockdots", _ptr(w), _ptr(xq), _ptr(dots), rows, k, _stream(stream), check=check)


def moe_qmv_q4k(w_bank, x, y, rows, k, ids, slots, n_experts, stream=None, cfg=None, overlap=0, check=True):
    if cfg is None and not overlap:
        return _call("moe_qmv_q4k", _ptr(w_bank), _ptr(x), _ptr(y), rows, k, _ptr(ids), slots, n_experts,
                     _stream(stream), check=check)
    return _call("moe_qmv_q4k_ex", _ptr(w_bank), _ptr(x), _ptr(y), rows, k, _ptr(ids), slots, n_experts,
                 _opts(cfg, overlap), _stream(stream), check=check)


def moe_qmv_q6k(w_bank, x, y, rows, k, ids, slots, n_experts, stream=None, cfg=None, overlap=0, check=True):
    if cfg is None and not overlap:
        return _call("moe_qmv_q6k", _ptr(w_bank), _ptr(x), _ptr(y), rows, k, _ptr(ids), slots, n_experts,
                     _stream(stream), check=check)
    return _call("moe_qmv_q6k_ex", _ptr(w_bank), _ptr(x), _ptr(y), rows, k, _ptr(ids), slots, n_experts,
                 _opts(cfg, overlap), _stream(stream), check=check)


def _moe_f32(name, w_bank, x, y, rows, k, ids, slots, n_experts, stream, cfg, overlap, check):
    if cfg is None and not overlap:
        return _call(name, _ptr(w_bank), _ptr(x), _ptr(y), rows, k, _ptr(ids), slots, n_experts,
                     _stream(stream), check=check)
    return _call(name + "_ex", _ptr(w_bank), _ptr(x), _ptr(y), rows, k, _ptr(ids), slots, n_experts,
                 _opts(cfg, overlap), _stream(stream), check=check)


def moe_qmv_q8_0(w_bank, x, y, rows, k, ids, slots, n_experts, stream=None, cfg=None, overlap=0, check=True):
    return _moe_f32("moe_qmv_q8_0", w_bank, x, y, rows, k, ids, slots, n_experts, stream, cfg, overlap, check)


def moe_qmv_q4_0(w_bank, x, y, rows, k, ids, slots, n_experts, stream=None, cfg=None, overlap=0, check=True):
    return _moe_f32("moe_qmv_q4_0", w_bank, x, y, rows, k, ids, slots, n_experts, stream, cfg, overlap, check)


def moe_qmv_q5k(w_bank, x, y, rows, k, ids, slots, n_experts, stream=None, cfg=None, overlap=0, check=True):
    return _moe_f32("moe_qmv_q5k", w_bank, x, y, rows, k, ids, slots, n_experts, stream, cfg, overlap, check)


def moe_qmv_q4k_dp4a(w_bank, xq, xs, y, rows, k, ids, slots, n_experts, stream=None, cfg=None, overlap=0, check=True):
    if cfg is None and not overlap:
        return _call("moe_qmv_q4k_dp4a", _ptr(w_bank), _ptr(xq), _ptr(xs), _ptr(y), rows, k, _ptr(ids), slots,
                     n_experts, _stream(stream), check=check)
    return _call("moe_qmv_q4k_dp4a_ex", _ptr(w_bank), _ptr(xq), _ptr(xs), _ptr(y), rows, k, _ptr(ids), slots,
                 n_experts, _opts(cfg, overlap), _stream(stream), check=check)


def qmv_dequant_q4k(w, out, rows, k, stream=None, check=True):
    return _call("qmv_dequant_q4k", _ptr(w), _ptr(out), rows, k, _stream(stream), check=check)


def qmv_dequant_q6k(w, out, rows, k, stream=None, check=True):
    return _call("qmv_dequant_q6k", _ptr(w), _ptr(out), rows, k, _stream(stream), check=check)


def qmv_dequant_q8_0(w, out, rows, k, stream=None, check=True):
    return _call("qmv_dequant_q8_0", _ptr(w), _ptr(out), rows, k, _stream(stream), check=check)


def qmv_dequant_q5k(w, out, rows, k, stream=None, check=True):
    return _call("qmv_dequant_q5k", _ptr(w), _ptr(out), rows, k, _stream(stream), check=check)


def qmv_dequant_q4_0(w, out, rows, k, stream=None, check=True):
    return _call("qmv_dequant_q4_0", _ptr(w), _ptr(out), rows, k, _stream(stream), check=check)


def qmv_q8_dp4a_blockdots(w, xq, dots, rows, k, stream=None, check=True):
    return _call("qmv_q8_dp4a_blockdots", _ptr(w), _ptr(xq), _ptr(dots), rows, k, _stream(stream), check=check)


def qmv_selftest_wait_timeout(limit_ns, stream=None, check=True):
    return _call("qmv_selftest_wait_timeout", int(limit_ns), _stream(stream), check=check)


def qmv_selftest_timeout_path(w, x, y, rows, k, m=1, stream=None, check=True):
    return _call("qmv_selftest_timeout_path", _ptr(w), _ptr(x), _ptr(y), rows, k, m, _stream(stream), check=check)


def qmm_q4k_tc5_selftest_timeout_path(w, x, y, rows, k, m=2, stream=None, overlap=0, check=True):
    return _call("qmm_q4k_tc5_selftest_timeout_path", _ptr(w), _ptr(x), _ptr(y), rows, k, m, _opts(None, overlap),
                 _stream(stream), check=check)


def qmv_device_status(clear=True) -> int:
    v = ctypes.c_uint(0)
    _call("qmv_device_status", ctypes.cast(ctypes.byref(v), ctypes.c_void_p), 1 if clear else 0)
    return v.value


def qmv_plan_info(fmt, rows, k, slots=1, cfg=None, overlap=0) -> dict:
    out = [ctypes.c_int(0) for _ in range(5)]
    _call("qmv_plan_info", fmt, rows, k, slots, _opts(cfg, overlap), *[ctypes.cast(ctypes.byref(o), ctypes.c_void_p)
                                                           for o in out])
    return dict(zip(["threads", "ctas", "chunk_rows", "chunks", "smem_bytes"], [o.value for o in out]))


PLAN_DETAIL_FIELDS = ("threads", "ctas", "unroll", "smem", "U", "KS", "GS", "NG", "CR", "S", "rowbytes", "W",
                      "slot_stride", "aligned8", "rq", "rrem", "gq0", "grem0", "gq1", "grem1", "off_la", "off_lb",
                      "off_lc", "off_xs", "off_xsum16", "off_red", "off_ring", "off_bars", "off_cnt", "CL")

# A GB300's numbers: 152 SMs, 227 KB opt-in shared memory per CTA, 228 KB per
# SM, 1 KB reserved per CTA.
GB300_DEVICE = (152, 232448, 233472, 1024)


def qmv_plan_detail(fmt, rows, k, slots=1, cfg=None, device=GB300_DEVICE, overlap=0) -> dict:
    """The planner's full choice for a described device, computed on the host
    (no GPU needed). Raises QmvError for shapes the planner rejects."""
    dev = (ctypes.c_int * 4)(*device)
    out = (ctypes.c_int * len(PLAN_DETAIL_FIELDS))()
    _call("qmv_plan_detail", fmt, rows, k, slots, _opts(cfg, overlap), ctypes.cast(dev, ctypes.c_void_p),
          ctypes.cast(out, ctypes.c_void_p))
    return dict(zip(PLAN_DETAIL_FIELDS, list(out)))


QMM_TC_PLAN_FIELDS = ("threads", "ctas", "smem", "KS", "CR", "S", "chunk_bytes", "stride", "slot_stride", "rq",
                      "rrem", "ngroups", "nchunks", "off_red", "off_sums", "off_ring", "off_bars", "off_cnt")


def qmm_tc_plan_detail(fmt, rows, k, m, cfg=None, device=GB300_DEVICE, overlap=0) -> dict:
    """The tensor-core batch planner's choice (fmt 0 = Q4_K, 1 = Q6_K, 2 = Q8_0)
    for a described device, computed on the host without a GPU."""
    out = (ctypes.c_int * len(QMM_TC_PLAN_FIELDS))()
    dev = (ctypes.c_int * 4)(*device)
    _call("qmm_tc_plan_detail", fmt, rows, k, m, _opts(cfg, overlap), dev, out)
    return dict(zip(QMM_TC_PLAN_FIELDS, list(out)))


TC5_PLAN_FIELDS = ("ctas", "threads", "smem", "CL", "S", "nsb", "off_b", "off_bm", "off_sc", "off_x", "off_in",
                   "off_bars", "streaming")


def qmm_q4k_tc5_plan_detail(rows, k, m, cfg=None, device=GB300_DEVICE, overlap=0) -> dict:
    """The plan of qmm_q4k_tc5 for one launch of m <= 8 rows of x on a
    described device, computed on the host without a GPU."""
    out = (ctypes.c_int * len(TC5_PLAN_FIELDS))()
    dev = (ctypes.c_int * 4)(*device)
    _call("qmm_q4k_tc5_plan_detail", rows, k, m, _opts(cfg, overlap), dev, out)
    return dict(zip(TC5_PLAN_FIELDS, list(out)))
