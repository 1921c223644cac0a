"""Seeded generators for raw Q4_K / Q6_K / Q8_0 / Q4_0 / Q5_K weight rows, f32
activations and MoE expert ids.

The block byte layouts follow the GGML/GGUF block structs the pages upload
verbatim (hanzo-ml ``vulkan_backend.rs``: ``quantize_q4k`` for the 144-byte
``block_q4_K``, ``quantize_q6k`` for the 210-byte ``block_q6_K`` and
``quantize_q8_blocks`` for the 34-byte ``block_q8_0``, ``matvec_q4_0_gpu`` for
the native 18-byte ``block_q4_0`` and ``quantize_q5k`` for the 176-byte
``block_q5_K``). Only the field sizes and
their order matter here; how the fields decode is the oracle's business.

Draw order (this repository's choice): blocks in row-major order, and inside a
block one or more 64-bit draws per field in byte order; the activation comes
after all weight draws. Per block:

* Q4_K (20 draws): d, dmin (one draw each), 2 draws -> 16 bytes of which the
  first 12 are the packed scales/mins, 16 draws -> the 128 ``qs`` bytes.
* Q6_K (41 draws): 16 draws -> ``ql[128]``, 8 draws -> ``qh[64]``, 16 draws ->
  one int8 scale each, 1 draw -> d.
* Q8_0 (33 draws): 1 draw -> d, 32 draws -> one int8 weight each.
* Q4_0 (3 draws): 1 draw -> d (either sign), 2 draws -> the 16 ``qs`` bytes.
* Q5_K (24 draws): d, dmin (one draw each), 2 draws -> 16 bytes of which the
  first 12 are the packed scales/mins, 4 draws -> the 32 ``qh`` bytes, 16 draws
  -> the 128 ``qs`` bytes.

A value U[a, b] is ``a + (b - a) * u53`` in f64 with ``u53 = (z >> 11) * 2**-53``,
then rounded to f32 and to f16 (numpy's round-to-nearest-even conversions).
N(0, 1) values come from the Box-Muller transform in f64, rounded to f32.
"""

from __future__ import annotations

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

Q4K_BLOCK_BYTES = 144
Q6K_BLOCK_BYTES = 210
Q8_0_BLOCK_BYTES = 34
Q4_0_BLOCK_BYTES = 18
Q5K_BLOCK_BYTES = 176
QK_K = 256
QK8_0 = 32


def row_bytes(fmt: str, k: int) -> int:
    """Packed bytes of one weight row of length ``k`` in format ``fmt``."""
    if fmt == "q4k":
        return (k // QK_K) * Q4K_BLOCK_BYTES
    if fmt == "q6k":
        return (k // QK_K) * Q6K_BLOCK_BYTES
    if fmt == "q8_0":
        return (k // QK8_0) * Q8_0_BLOCK_BYTES
    if fmt == "q4_0":
        return (k // QK8_0) * Q4_0_BLOCK_BYTES
    if fmt == "q5k":
        return (k // QK_K) * Q5K_BLOCK_BYTES
    raise ValueError(fmt)


class Stream:
    """A splitmix64 stream; ``draw(n)`` returns the next ``n`` 64-bit outputs."""

    def __init__(self, seed: int):
        self.seed = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
        self.pos = 0

    def draw(self, n: int) -> np.ndarray:
        idx = np.arange(self.pos + 1, self.pos + 1 + n, dtype=np.uint64)
        self.pos += n
        with np.errstate(over="ignore"):
            z = self.seed + idx * GOLDEN_GAMMA
            z = (z ^ (z >> np.uint64(30))) * _M1
            z = (z ^ (z >> np.uint64(27))) * _M2
            z = z ^ (z >> np.uint64(31))
        return z


def _u53(z: np.ndarray) -> np.ndarray:
    """Uniform in [0, 1) with 53 random bits."""
    return (z >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _uniform_f16_bits(z: np.ndarray, a: float, b: float) -> np.ndarray:
    v = (a + (b - a) * _u53(z)).astype(np.float32).astype(np.float16)
    return v.view(np.uint16)


def _bytes_of(z: np.ndarray, nbytes: int) -> np.ndarray:
    """Little-endian bytes of consecutive draws, ``z`` shaped [..., ndraws]."""
    b = z.astype("<u8").view(np.uint8).reshape(z.shape[:-1] + (z.shape[-1] * 8,))
    return b[..., :nbytes]


def _uniform_int(z: np.ndarray, lo: int, hi: int) -> np.ndarray:
    """Integer uniform on [lo, hi] from the top 32 bits (multiply-shift)."""
    span = np.uint64(hi - lo + 1)
    top = z >> np.uint64(32)
    return ((top * span) >> np.uint64(32)).astype(np.int64) + lo


def gen_q4k_rows(st: Stream, rows: int, k: int,
                 d_range=(1e-3, 4e-3), dmin_range=(0.0, 2e-3)) -> np.ndarray:
    """Raw Q4_K rows, uint8 [rows, k/256*144]."""
    nb = k // QK_K
    z = st.draw(rows * nb * 20).reshape(rows * nb, 20)
    blk = np.empty((rows * nb, Q4K_BLOCK_BYTES), dtype=np.uint8)
    blk[:, 0:2] = _uniform_f16_bits(z[:, 0], *d_range).view(np.uint8).reshape(-1, 2)
    blk[:, 2:4] = _uniform_f16_bits(z[:, 1], *dmin_range).view(np.uint8).reshape(-1, 2)
    blk[:, 4:16] = _bytes_of(z[:, 2:4], 12)
    blk[:, 16:144] = _bytes_of(z[:, 4:20], 128)
    return blk.reshape(rows, nb * Q4K_BLOCK_BYTES)


def gen_q6k_rows(st: Stream, rows: int, k: int, d_range=(1e-4, 5e-4)) -> np.ndarray:
    """Raw Q6_K rows, uint8 [rows, k/256*210]; int8 scales uniform in [-64, 63]."""
    nb = k // QK_K
    z = st.draw(rows * nb * 41).reshape(rows * nb, 41)
    blk = np.empty((rows * nb, Q6K_BLOCK_BYTES), dtype=np.uint8)
    blk[:, 0:128] = _bytes_of(z[:, 0:16], 128)
    blk[:, 128:192] = _bytes_of(z[:, 16:24], 64)
    blk[:, 192:208] = _uniform_int(z[:, 24:40], -64, 63).astype(np.int8).view(np.uint8)
    blk[:, 208:210] = _uniform_f16_bits(z[:, 40], *d_range).view(np.uint8).reshape(-1, 2)
    return blk.reshape(rows, nb * Q6K_BLOCK_BYTES)


def gen_q8_0_rows(st: Stream, rows: int, k: int, d_range=(1e-3, 1e-2),
                  q_range=(-127, 127)) -> np.ndarray:
    """Raw Q8_0 rows, uint8 [rows, k/32*34]; int8 weights uniform in ``q_range``."""
    nb = k // QK8_0
    z = st.draw(rows * nb * 33).reshape(rows * nb, 33)
    blk = np.empty((rows * nb, Q8_0_BLOCK_BYTES), dtype=np.uint8)
    blk[:, 0:2] = _uniform_f16_bits(z[:, 0], *d_range).view(np.uint8).reshape(-1, 2)
    blk[:, 2:34] = _uniform_int(z[:, 1:33], *q_range).astype(np.int8).view(np.uint8)
    return blk.reshape(rows, nb * Q8_0_BLOCK_BYTES)


def gen_q4_0_rows(st: Stream, rows: int, k: int, d_range=(-1e-2, 1e-2)) -> np.ndarray:
    """Raw Q4_0 rows, uint8 [rows, k/32*18]; d uniform in ``d_range`` (GGML's
    quantizer gives d either sign, so both occur)."""
    nb = k // QK8_0
    z = st.draw(rows * nb * 3).reshape(rows * nb, 3)
    blk = np.empty((rows * nb, Q4_0_BLOCK_BYTES), dtype=np.uint8)
    blk[:, 0:2] = _uniform_f16_bits(z[:, 0], *d_range).view(np.uint8).reshape(-1, 2)
    blk[:, 2:18] = _bytes_of(z[:, 1:3], 16)
    return blk.reshape(rows, nb * Q4_0_BLOCK_BYTES)


def gen_q5k_rows(st: Stream, rows: int, k: int,
                 d_range=(5e-4, 2e-3), dmin_range=(0.0, 2e-3)) -> np.ndarray:
    """Raw Q5_K rows, uint8 [rows, k/256*176]."""
    nb = k // QK_K
    z = st.draw(rows * nb * 24).reshape(rows * nb, 24)
    blk = np.empty((rows * nb, Q5K_BLOCK_BYTES), dtype=np.uint8)
    blk[:, 0:2] = _uniform_f16_bits(z[:, 0], *d_range).view(np.uint8).reshape(-1, 2)
    blk[:, 2:4] = _uniform_f16_bits(z[:, 1], *dmin_range).view(np.uint8).reshape(-1, 2)
    blk[:, 4:16] = _bytes_of(z[:, 2:4], 12)
    blk[:, 16:48] = _bytes_of(z[:, 4:8], 32)
    blk[:, 48:176] = _bytes_of(z[:, 8:24], 128)
    return blk.reshape(rows, nb * Q5K_BLOCK_BYTES)


GEN_ROWS = {"q4k": gen_q4k_rows, "q6k": gen_q6k_rows, "q8_0": gen_q8_0_rows,
            "q4_0": gen_q4_0_rows, "q5k": gen_q5k_rows}


def gen_normal(st: Stream, n: int) -> np.ndarray:
    """``n`` N(0, 1) values (Box-Muller in f64), returned as f32."""
    pairs = (n + 1) // 2
    z = st.draw(2 * pairs).reshape(pairs, 2)
    u1 = ((z[:, 0] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    u2 = _u53(z[:, 1])
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * np.pi * u2
    out = np.empty(2 * pairs, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out[:n].astype(np.float32)


def gen_moe_ids(st: Stream, slots: int, n_experts: int) -> np.ndarray:
    """``slots`` distinct expert ids from 0..n_experts-1 (partial Fisher-Yates)."""
    perm = np.arange(n_experts, dtype=np.int64)
    z = st.draw(slots)
    for i in range(slots):
        span = n_experts - i
        j = i + int((int(z[i]) >> 32) * span >> 32)
        perm[i], perm[j] = perm[j], perm[i]
    return perm[:slots].astype(np.int32)


# The synthetic workloads: name -> (kind, parameters, seed). The first five are
# the suite's; the others are the second and fourth on the dp4a path and a
# Q6_K MoE bank.
CONFIGS = {
    "q4k_256x1024": dict(kind="q4k", rows=256, k=1024, seed=0),
    "q4k_4096x4096": dict(kind="q4k", rows=4096, k=4096, seed=1),
    "q8_0_dp4a_14336x4096": dict(kind="q8_0_dp4a", rows=14336, k=4096, seed=2),
    "moe_q4k_e128_n768_k2048_s8": dict(kind="moe_q4k", rows=768, k=2048, seed=3,
                                       n_experts=128, slots=8),
    "q6k_4096x14336": dict(kind="q6k", rows=4096, k=14336, seed=4),
    # The Q4_K 4096 x 4096 workload (same seed, so the same bytes) on the dp4a
    # path: x is quantized on the device and the codes are dp4a-dotted.
    "q4k_dp4a_4096x4096": dict(kind="q4k_dp4a", rows=4096, k=4096, seed=1),
    # The MoE workload on the dp4a path (same seed: the same bank, ids and x),
    # and the pages' second MoE workload, Q6_K down-projection experts
    # [128, 2048, 768] with 8 routed slots.
    "moe_q4k_dp4a_e128_n768_k2048_s8": dict(kind="moe_q4k_dp4a", rows=768, k=2048, seed=3,
                                            n_experts=128, slots=8),
    "moe_q6k_e128_n2048_k768_s8": dict(kind="moe_q6k", rows=2048, k=768, seed=5, n_experts=128, slots=8),
    # The other formats of the same kernel skeleton: dense Q5_K and Q4_0 at the
    # headline shape, and MoE over Q8_0, Q4_0 and Q5_K banks at the MoE shape.
    "q5k_4096x4096": dict(kind="q5k", rows=4096, k=4096, seed=6),
    "q4_0_4096x4096": dict(kind="q4_0", rows=4096, k=4096, seed=7),
    "moe_q8_0_e128_n768_k2048_s8": dict(kind="moe_q8_0", rows=768, k=2048, seed=8, n_experts=128, slots=8),
    "moe_q4_0_e128_n768_k2048_s8": dict(kind="moe_q4_0", rows=768, k=2048, seed=9, n_experts=128, slots=8),
    "moe_q5k_e128_n768_k2048_s8": dict(kind="moe_q5k", rows=768, k=2048, seed=10, n_experts=128, slots=8),
    # The Q6_K suite matrix and the Q6_K MoE bank on the dp4a path (same seeds:
    # the same bytes, ids and x).
    "q6k_dp4a_4096x14336": dict(kind="q6k_dp4a", rows=4096, k=14336, seed=4),
    "moe_q6k_dp4a_e128_n2048_k768_s8": dict(kind="moe_q6k_dp4a", rows=2048, k=768, seed=5, n_experts=128, slots=8),
    # Small-M batches (m rows of x sharing one weight read) on the headline and
    # the two large suite matrices (same seeds: the same weight bytes; the
    # first row of x is the single-row workload's x).
    "qmm_q4k_4096x4096_m2": dict(kind="qmm_q4k", rows=4096, k=4096, seed=1, m=2),
    "qmm_q4k_4096x4096_m4": dict(kind="qmm_q4k", rows=4096, k=4096, seed=1, m=4),
    "qmm_q4k_4096x4096_m8": dict(kind="qmm_q4k", rows=4096, k=4096, seed=1, m=8),
    "qmm_q6k_4096x14336_m4": dict(kind="qmm_q6k", rows=4096, k=14336, seed=4, m=4),
    "qmm_q8_0_14336x4096_m8": dict(kind="qmm_q8_0", rows=14336, k=4096, seed=2, m=8),
    "qmm_q5k_4096x4096_m4": dict(kind="qmm_q5k", rows=4096, k=4096, seed=6, m=4),
    "qmm_q4_0_4096x4096_m4": dict(kind="qmm_q4_0", rows=4096, k=4096, seed=7, m=4),
}


def make_config(name: str) -> dict:
    """Generate one named workload. Returns a dict with numpy arrays:
    ``w`` (uint8 packed rows or the MoE bank), ``x`` (f32), and for MoE ``ids``."""
    c = dict(CONFIGS[name])
    st = Stream(c["seed"])
    kind, rows, k = c["kind"], c["rows"], c["k"]
    if kind in ("q4k", "q4k_dp4a"):
        c["w"] = gen_q4k_rows(st, rows, k)
        c["x"] = gen_normal(st, k)
    elif kind in ("q6k", "q6k_dp4a"):
        c["w"] = gen_q6k_rows(st, rows, k)
        c["x"] = gen_normal(st, k)
    elif kind == "q8_0_dp4a":
        c["w"] = gen_q8_0_rows(st, rows, k)
        c["x"] = gen_normal(st, k)
    elif kind in ("q5k", "q4_0"):
        c["w"] = GEN_ROWS[kind](st, rows, k)
        c["x"] = gen_normal(st, k)
    elif kind.startswith("qmm_"):
        c["w"] = GEN_ROWS[kind[4:]](st, rows, k)
        c["x"] = gen_normal(st, c["m"] * k).reshape(c["m"], k)
    elif kind in ("moe_q4k", "moe_q4k_dp4a", "moe_q6k", "moe_q6k_dp4a", "moe_q8_0", "moe_q4_0", "moe_q5k"):
        e, s = c["n_experts"], c["slots"]
        fmt = kind[4:].replace("_dp4a", "")
        c["w"] = GEN_ROWS[fmt](st, e * rows, k).reshape(e, rows, -1)
        c["ids"] = gen_moe_ids(st, s, e)
        c["x"] = gen_normal(st, s * k).reshape(s, k)
    else:
        raise ValueError(kind)
    return c
