"""CPU oracle for the GGML-block quantized matvec -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this package. The product path (the CUDA library and
its Python binding) never imports, links or calls it, and shares no code with
it.

The arithmetic lives in ``qmv_oracle.c`` (plain C, f64 accumulation, IEEE f32
for the activation quantizer, compiled with ``-ffp-contract=off``). This module
only compiles it with gcc and marshals numpy arrays through ctypes.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms on hand-built blocks, an exhaustive f16 check against numpy,
brute-force dequantize-then-multiply, invariants of the matvec and
round-half-even tie cases for the quantizer); none is "parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = None
_LOCK = threading.Lock()

FMT = {"q4k": 0, "q6k": 1, "q8_0": 2, "q4_0": 3, "q5k": 4}
QK = {"q4k": 256, "q6k": 256, "q8_0": 32, "q4_0": 32, "q5k": 256}
BLOCK_BYTES = {"q4k": 144, "q6k": 210, "q8_0": 34, "q4_0": 18, "q5k": 176}


def lib_path() -> str:
    return os.path.join(_BUILD, f"liboracle_{platform.machine()}.so")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FP contraction)."""
    out = lib_path()
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lg = ctypes.c_long
            L.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
            L.orc_f16_to_f64.restype = ctypes.c_double
            for fmt in FMT:
                getattr(L, f"orc_{fmt}_block_decode").argtypes = [P, P]
                getattr(L, f"orc_{fmt}_block_decode").restype = None
            for f in (f"orc_{fmt}_elem" for fmt in FMT):
                getattr(L, f).argtypes = [P, ctypes.c_int]
                getattr(L, f).restype = ctypes.c_double
            L.orc_dequant.argtypes = [ctypes.c_int, P, lg, lg, P]
            L.orc_qmv.argtypes = [ctypes.c_int, P, P, lg, lg, P]
            L.orc_moe_qmv.argtypes = [ctypes.c_int, P, P, P, lg, lg, lg, lg, P]
            L.orc_qmm.argtypes = [ctypes.c_int, P, P, lg, lg, lg, P]
            L.orc_quantize_act_q8.argtypes = [P, lg, lg, P, P, P]
            L.orc_q8_blockdots.argtypes = [P, P, lg, lg, P]
            L.orc_qmv_q8_dp4a.argtypes = [P, P, P, lg, lg, P]
            L.orc_q4k_dp4a_blockdots.argtypes = [P, P, lg, lg, P]
            L.orc_qmv_q4k_dp4a.argtypes = [P, P, P, lg, lg, P]
            L.orc_moe_qmv_q4k_dp4a.argtypes = [P, P, P, P, lg, lg, lg, lg, P]
            L.orc_q6k_dp4a_groupdots.argtypes = [P, P, lg, lg, P]
            L.orc_qmv_q6k_dp4a.argtypes = [P, P, P, lg, lg, P]
            L.orc_moe_qmv_q6k_dp4a.argtypes = [P, P, P, P, lg, lg, lg, lg, P]
            _LIB = L
    return _LIB


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u8(w) -> np.ndarray:
    return np.ascontiguousarray(w, dtype=np.uint8)


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32)


def f16_to_f64(h: int) -> float:
    """Exact value of one IEEE binary16 bit pattern."""
    return _lib().orc_f16_to_f64(int(h) & 0xFFFF)


def decode_block(fmt: str, block) -> np.ndarray:
    """Loop-structured exact decode of one block (f64 array of QK[fmt])."""
    b = _u8(block)
    assert b.size == BLOCK_BYTES[fmt]
    out = np.empty(QK[fmt], dtype=np.float64)
    getattr(_lib(), f"orc_{fmt}_block_decode")(_p(b), _p(out))
    return out


def decode_elem(fmt: str, block, i: int) -> float:
    """Per-element closed-form decode of element ``i`` of one block."""
    b = _u8(block)
    assert b.size == BLOCK_BYTES[fmt]
    return getattr(_lib(), f"orc_{fmt}_elem")(_p(b), int(i))


def dequant(fmt: str, w, rows: int, k: int) -> np.ndarray:
    """Exact decoded weights [rows, k] (f64) of packed rows ``w``."""
    w = _u8(w)
    assert w.size == rows * (k // QK[fmt]) * BLOCK_BYTES[fmt]
    out = np.empty((rows, k), dtype=np.float64)
    rc = _lib().orc_dequant(FMT[fmt], _p(w), rows, k, _p(out))
    assert rc == 0
    return out


def qmv(fmt: str, w, x, rows: int, k: int) -> np.ndarray:
    """f64 dequantize-then-dot matvec, y[rows]."""
    w = _u8(w)
    x = _f32(x)
    assert w.size == rows * (k // QK[fmt]) * BLOCK_BYTES[fmt] and x.size == k
    y = np.empty(rows, dtype=np.float64)
    rc = _lib().orc_qmv(FMT[fmt], _p(w), _p(x), rows, k, _p(y))
    assert rc == 0
    return y


def qmm(fmt: str, w, x, m: int, rows: int, k: int) -> np.ndarray:
    """Small-M batch: y[m, rows] (f64) for the m rows of x[m, k]."""
    w = _u8(w)
    x = _f32(x)
    assert w.size == rows * (k // QK[fmt]) * BLOCK_BYTES[fmt] and x.size == m * k
    y = np.empty((m, rows), dtype=np.float64)
    rc = _lib().orc_qmm(FMT[fmt], _p(w), _p(x), m, rows, k, _p(y))
    assert rc == 0
    return y


def moe_qmv(fmt: str, bank, x, ids, rows: int, k: int, n_experts: int) -> np.ndarray:
    """MoE indexed matvec, y[slots, rows] (NaN rows for out-of-range ids)."""
    bank = _u8(bank)
    x = _f32(x)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    slots = ids.size
    assert x.size == slots * k
    y = np.empty((slots, rows), dtype=np.float64)
    rc = _lib().orc_moe_qmv(FMT[fmt], _p(bank), _p(x), _p(ids), slots, rows, k, n_experts, _p(y))
    assert rc == 0
    return y


def quantize_act_q8(x, m: int, k: int):
    """(xq int8 [m, k], xs f32 [m, k/32], xsum f32 [m, k/32])."""
    x = _f32(x)
    assert x.size == m * k
    xq = np.empty((m, k), dtype=np.int8)
    xs = np.empty((m, k // 32), dtype=np.float32)
    xsum = np.empty((m, k // 32), dtype=np.float32)
    rc = _lib().orc_quantize_act_q8(_p(x), m, k, _p(xq), _p(xs), _p(xsum))
    assert rc == 0
    return xq, xs, xsum


def q8_blockdots(w, xq, rows: int, k: int) -> np.ndarray:
    """Exact int32 per-block dots [rows, k/32] of Q8_0 rows with int8 codes."""
    w = _u8(w)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    dots = np.empty((rows, k // 32), dtype=np.int32)
    rc = _lib().orc_q8_blockdots(_p(w), _p(xq), rows, k, _p(dots))
    assert rc == 0
    return dots


def qmv_q8_dp4a(w, xq, xs, rows: int, k: int) -> np.ndarray:
    """dp4a-path matvec in f64: y[r] = sum_b d_w * d_x * dot."""
    w = _u8(w)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    xs = _f32(xs)
    y = np.empty(rows, dtype=np.float64)
    rc = _lib().orc_qmv_q8_dp4a(_p(w), _p(xq), _p(xs), rows, k, _p(y))
    assert rc == 0
    return y


def q4k_dp4a_blockdots(w, xq, rows: int, k: int) -> np.ndarray:
    """Exact int32 dots [rows, k/32] of every 32-weight Q4_K sub-block's 4-bit
    codes with the int8 activation codes of the same positions."""
    w = _u8(w)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    dots = np.empty((rows, k // 32), dtype=np.int32)
    rc = _lib().orc_q4k_dp4a_blockdots(_p(w), _p(xq), rows, k, _p(dots))
    assert rc == 0
    return dots


def qmv_q4k_dp4a(w, xq, xs, rows: int, k: int) -> np.ndarray:
    """Q4_K dp4a-path matvec in f64: y[r] = sum_t xs_t (d sc dot_t - dmin m sumq_t)."""
    w = _u8(w)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    xs = _f32(xs)
    y = np.empty(rows, dtype=np.float64)
    rc = _lib().orc_qmv_q4k_dp4a(_p(w), _p(xq), _p(xs), rows, k, _p(y))
    assert rc == 0
    return y


def moe_qmv_q4k_dp4a(bank, xq, xs, ids, rows: int, k: int, n_experts: int) -> np.ndarray:
    """MoE on the Q4_K dp4a path, y[slots, rows]: slot s uses expert ids[s]
    and its own codes xq[s] / scales xs[s] (NaN rows for out-of-range ids)."""
    bank = _u8(bank)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    xs = _f32(xs)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    slots = ids.size
    assert xq.size == slots * k and xs.size == slots * (k // 32)
    y = np.empty((slots, rows), dtype=np.float64)
    rc = _lib().orc_moe_qmv_q4k_dp4a(_p(bank), _p(xq), _p(xs), _p(ids), slots, rows, k, n_experts, _p(y))
    assert rc == 0
    return y


def q6k_dp4a_groupdots(w, xq, rows: int, k: int) -> np.ndarray:
    """int32 [rows, k/16]: (q - 32) . xq over every 16-weight scale group."""
    w = _u8(w)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    assert xq.size == k
    out = np.empty((rows, k // 16), dtype=np.int32)
    assert _lib().orc_q6k_dp4a_groupdots(_p(w), _p(xq), rows, k, _p(out)) == 0
    return out


def qmv_q6k_dp4a(w, xq, xs, rows: int, k: int) -> np.ndarray:
    """Q6_K x int8 activation matvec (f64)."""
    w = _u8(w)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    xs = _f32(xs)
    assert xq.size == k and xs.size == k // 32
    y = np.empty(rows, dtype=np.float64)
    assert _lib().orc_qmv_q6k_dp4a(_p(w), _p(xq), _p(xs), rows, k, _p(y)) == 0
    return y


def moe_qmv_q6k_dp4a(bank, xq, xs, ids, rows: int, k: int, n_experts: int) -> np.ndarray:
    """MoE on the Q6_K dp4a path, y[slots, rows] (NaN rows for bad ids)."""
    bank = _u8(bank)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    xs = _f32(xs)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    slots = ids.size
    assert xq.size == slots * k and xs.size == slots * (k // 32)
    y = np.empty((slots, rows), dtype=np.float64)
    rc = _lib().orc_moe_qmv_q6k_dp4a(_p(bank), _p(xq), _p(xs), _p(ids), slots, rows, k, n_experts, _p(y))
    assert rc == 0
    return y


def qmv_threaded(fmt: str, w, x, rows: int, k: int, threads: int) -> np.ndarray:
    """The same oracle matvec, rows split into ``threads`` contiguous ranges run
    on Python threads (ctypes releases the GIL during the C call)."""
    w = _u8(w).reshape(rows, -1)
    x = _f32(x)
    y = np.empty(rows, dtype=np.float64)
    bounds = [rows * t // threads for t in range(threads + 1)]

    def run(t):
        r0, r1 = bounds[t], bounds[t + 1]
        if r1 > r0:
            part = np.ascontiguousarray(w[r0:r1])
            out = np.empty(r1 - r0, dtype=np.float64)
            _lib().orc_qmv(FMT[fmt], _p(part), _p(x), r1 - r0, k, _p(out))
            y[r0:r1] = out

    ths = [threading.Thread(target=run, args=(t,)) for t in range(threads)]
    for th in ths:
        th.start()
    for th in ths:
        th.join()
    return y
