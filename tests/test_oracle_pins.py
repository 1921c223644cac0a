"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- closed forms on hand-built blocks, numpy's IEEE half conversion,
brute-force dequantize-then-multiply, invariants of a matvec, and the
round-half-even tie cases of the activation quantizer -- so that a dropped term,
a wrong index or sign, or a swapped nibble fails at least one of them.

Block layouts (hanzo-ml src/vulkan_backend.rs): Q4_K super-block of 144 bytes
(quantize_q4k / quantize_q4k_split), Q6_K block of 210 bytes (quantize_q6k /
quantize_q6k_split), Q8_0 block of 34 bytes (quantize_q8_blocks). The bit
mapping inside the blocks is the GGML k-quant layout those passages defer to
(the CPU ``to_float`` dequantizers).
"""

import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ helpers

def f16_bits(v: float) -> int:
    return int(np.array(v, dtype=np.float16).view(np.uint16))


def pack_q4k(d_bits, dmin_bits, sc, m, q):
    """Build a Q4_K block from field values by the inverse of the layout:
    6-bit scale/min of sub-blocks 0..3 in the low 6 bits of bytes 0..3 / 4..7;
    sub-blocks 4..7 keep their low nibbles in bytes 8..11 (scale low, min high)
    and their top two bits in bits 6..7 of bytes 0..3 (scale) / 4..7 (min).
    Element i's 4-bit code goes to qs byte 32*(i//64) + i%32, low nibble for
    sub-blocks of even index, high nibble for odd."""
    b = np.zeros(144, dtype=np.uint8)
    b[0], b[1] = d_bits & 0xFF, d_bits >> 8
    b[2], b[3] = dmin_bits & 0xFF, dmin_bits >> 8
    s = np.zeros(12, dtype=np.int64)
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    b[4:16] = s.astype(np.uint8)
    for i in range(256):
        byte = 16 + 32 * (i // 64) + (i % 32)
        if (i // 32) % 2 == 0:
            b[byte] |= q[i] & 15
        else:
            b[byte] |= (q[i] & 15) << 4
    return b


def pack_q6k(d_bits, scales, q):
    """Build a Q6_K block: element i = 128*H + 32*quad + l takes its low 4 bits
    from ql[64*H + 32*(quad % 2) + l] (low nibble for quad < 2, high otherwise)
    and its top 2 bits from bits 2*quad.. of qh[32*H + l]."""
    b = np.zeros(210, dtype=np.uint8)
    for i in range(256):
        H, quad, l = i // 128, (i % 128) // 32, i % 32
        qli = 64 * H + 32 * (quad % 2) + l
        b[qli] |= (q[i] & 15) << (4 * (quad // 2))
        b[128 + 32 * H + l] |= ((q[i] >> 4) & 3) << (2 * quad)
    b[192:208] = np.array(scales, dtype=np.int8).view(np.uint8)
    b[208], b[209] = d_bits & 0xFF, d_bits >> 8
    return b


def pack_q8_0(d_bits, q):
    b = np.zeros(34, dtype=np.uint8)
    b[0], b[1] = d_bits & 0xFF, d_bits >> 8
    b[2:] = np.array(q, dtype=np.int8).view(np.uint8)
    return b


def pack_q4_0(d_bits, q):
    """Build a Q4_0 block: code i (0..15) of element i < 16 in the low nibble of
    qs byte i, of element i >= 16 in the high nibble of qs byte i-16."""
    b = np.zeros(18, dtype=np.uint8)
    b[0], b[1] = d_bits & 0xFF, d_bits >> 8
    for i in range(32):
        b[2 + i % 16] |= (q[i] & 15) << (4 * (i // 16))
    return b


def pack_q5k(d_bits, dmin_bits, sc, m, q):
    """Build a Q5_K block: the low 4 bits of each code placed as in
    ``pack_q4k`` (qs at byte 48), bit 4 of element i's code as bit i//32 of
    qh byte i%32 (qh at byte 16)."""
    b4 = pack_q4k(d_bits, dmin_bits, sc, m, [v & 15 for v in q])
    b = np.zeros(176, dtype=np.uint8)
    b[0:16] = b4[0:16]
    b[48:176] = b4[16:144]
    for i in range(256):
        b[16 + i % 32] |= ((q[i] >> 4) & 1) << (i // 32)
    return b


def rand_blocks(fmt, n, seed):
    st = synth.Stream(seed)
    if fmt == "q8_0":
        return synth.gen_q8_0_rows(st, n, 32, q_range=(-128, 127))
    return synth.GEN_ROWS[fmt](st, n, oracle.QK[fmt])


# --------------------------------------------------------------- f16 decode

def test_f16_exhaustive_against_numpy():
    """Every binary16 pattern (normals, subnormals, zeros, inf, NaN) decodes to
    the value numpy's IEEE half conversion gives."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(h)) for h in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.f16_to_f64(0x0001) == 2.0 ** -24
    assert oracle.f16_to_f64(0x3C00) == 1.0
    assert oracle.f16_to_f64(0xC000) == -2.0


# --------------------------------------------------------------- Q4_K pins

SC = [1, 2, 3, 4, 21, 38, 55, 63]      # j >= 4 need the high two bits
MN = [5, 9, 13, 17, 33, 47, 61, 62]


def test_q4k_closed_form_scales_and_codes():
    q = [i % 16 for i in range(256)]
    b = pack_q4k(f16_bits(1.0), f16_bits(0.5), SC, MN, q)
    got = oracle.decode_block("q4k", b)
    want = np.array([SC[i // 32] * (i % 16) - 0.5 * MN[i // 32] for i in range(256)])
    assert np.array_equal(got, want)


def test_q4k_min_only():
    b = pack_q4k(f16_bits(0.0), f16_bits(1.0), SC, MN, [7] * 256)
    got = oracle.decode_block("q4k", b)
    assert np.array_equal(got, -np.repeat(np.array(MN, dtype=np.float64), 32))


def test_q4k_subnormal_scale():
    b = pack_q4k(0x0001, 0x0000, [1] * 8, [0] * 8, [1] * 256)
    got = oracle.decode_block("q4k", b)
    assert np.all(got == 2.0 ** -24)


def test_q4k_nibble_positions():
    """A distinct code per element; each must come back at its own index."""
    q = [(i * 7 + (i // 64)) % 16 for i in range(256)]
    b = pack_q4k(f16_bits(1.0), 0, [1] * 8, [0] * 8, q)
    assert np.array_equal(oracle.decode_block("q4k", b), np.array(q, dtype=np.float64))


def test_q4k_field_ranges():
    """Changing one byte of a field touches exactly the elements the layout
    assigns to it (field offsets from the golden layout table)."""
    base = rand_blocks("q4k", 1, 11)[0]
    ref = oracle.decode_block("q4k", base)
    for byte in [16, 16 + 31, 16 + 32 + 5, 16 + 127]:
        b = base.copy()
        b[byte] ^= 0xFF
        changed = np.nonzero(oracle.decode_block("q4k", b) != ref)[0]
        c, l = (byte - 16) // 32, (byte - 16) % 32
        assert set(changed) <= {64 * c + l, 64 * c + 32 + l}
    b = base.copy()
    b[4] ^= 0x3F    # low 6 bits of byte 0 of the scales: scale of sub-block 0
    changed = np.nonzero(oracle.decode_block("q4k", b) != ref)[0]
    assert set(changed) <= set(range(32)) and len(changed) > 0


def test_golden_layout_table_sizes():
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "block_layouts.txt"))
            if ln.strip() and not ln.startswith("#")]
    size = {}
    for fmt, field, off, ln, *_ in rows:
        size.setdefault(fmt, []).append((int(off), int(ln)))
    for fmt, fields in size.items():
        fields.sort()
        pos = 0
        for off, ln in fields:
            assert off == pos
            pos += ln
        assert pos == oracle.BLOCK_BYTES[fmt]


# --------------------------------------------------------------- Q6_K pins

def test_q6k_zero_code():
    b = pack_q6k(f16_bits(1.0), list(range(-8, 8)), [32] * 256)
    assert np.all(oracle.decode_block("q6k", b) == 0.0)


def test_q6k_scale_groups_are_runs_of_16():
    scales = [3, -5, 7, 11, -13, 17, 19, -23, 29, 31, -37, 41, 43, -47, 53, -59]
    b = pack_q6k(f16_bits(0.25), scales, [33] * 256)
    want = np.array([0.25 * scales[i // 16] for i in range(256)])
    assert np.array_equal(oracle.decode_block("q6k", b), want)


def test_q6k_code_extremes_and_positions():
    q = [(i * 5 + 3 * (i // 32)) % 64 for i in range(256)]
    q[0], q[255] = 0, 63
    b = pack_q6k(f16_bits(1.0), [1] * 16, q)
    got = oracle.decode_block("q6k", b)
    assert np.array_equal(got, np.array(q, dtype=np.float64) - 32)
    assert got[0] == -32 and got[255] == 31


def test_q6k_negative_scale_and_subnormal_d():
    b = pack_q6k(0x0001, [-64] * 16, [63] * 256)
    assert np.all(oracle.decode_block("q6k", b) == 2.0 ** -24 * -64 * 31)


# --------------------------------------------------------------- Q8_0 pins

def test_q8_0_closed_form():
    q = list(range(-128, -96)) + []
    b = pack_q8_0(f16_bits(0.5), q)
    assert np.array_equal(oracle.decode_block("q8_0", b), 0.5 * np.array(q, dtype=np.float64))
    q2 = [127 - 8 * i for i in range(32)]
    b2 = pack_q8_0(f16_bits(-3.0), q2)
    assert np.array_equal(oracle.decode_block("q8_0", b2), -3.0 * np.array(q2, dtype=np.float64))


# --------------------------------------------------------------- Q4_0 pins

def test_q4_0_closed_form_and_positions():
    q = [(i * 7 + i // 16) % 16 for i in range(32)]
    b = pack_q4_0(f16_bits(0.5), q)
    assert np.array_equal(oracle.decode_block("q4_0", b), 0.5 * (np.array(q, dtype=np.float64) - 8))
    b2 = pack_q4_0(f16_bits(-3.0), list(range(16)) + list(range(15, -1, -1)))
    got = oracle.decode_block("q4_0", b2)
    assert got[0] == 24.0 and got[15] == -21.0 and got[16] == -21.0 and got[31] == 24.0


def test_q4_0_each_element_is_its_own_nibble():
    """One non-zero code at a time: exactly one output moves, at its index."""
    for i in range(32):
        q = [8] * 32
        q[i] = 9
        got = oracle.decode_block("q4_0", pack_q4_0(f16_bits(1.0), q))
        want = np.zeros(32)
        want[i] = 1.0
        assert np.array_equal(got, want)


def test_q4_0_subnormal_d():
    b = pack_q4_0(0x0001, [0] * 32)
    assert np.all(oracle.decode_block("q4_0", b) == -8 * 2.0 ** -24)


# --------------------------------------------------------------- Q5_K pins

def test_q5k_closed_form_scales_and_codes():
    q = [(i * 3 + i // 32) % 32 for i in range(256)]
    b = pack_q5k(f16_bits(1.0), f16_bits(0.5), SC, MN, q)
    want = np.array([SC[i // 32] * q[i] - 0.5 * MN[i // 32] for i in range(256)])
    assert np.array_equal(oracle.decode_block("q5k", b), want)


def test_q5k_fifth_bit_positions():
    """Code 16 (only the fifth bit set) at one element at a time."""
    for i in range(256):
        q = [0] * 256
        q[i] = 16
        got = oracle.decode_block("q5k", pack_q5k(f16_bits(1.0), 0, [1] * 8, [0] * 8, q))
        want = np.zeros(256)
        want[i] = 16.0
        assert np.array_equal(got, want), i


def test_q5k_without_fifth_bits_is_q4k():
    """With every qh byte zero a Q5_K block decodes as the Q4_K block holding
    the same d, dmin, scales and qs bytes (the pinned Q4_K decoder)."""
    blocks = rand_blocks("q5k", 300, 77)
    for b in blocks:
        b = b.copy()
        b[16:48] = 0
        b4 = np.concatenate([b[0:16], b[48:176]])
        assert np.array_equal(oracle.decode_block("q5k", b), oracle.decode_block("q4k", b4))


def test_q5k_fifth_bit_adds_sixteen_scaled_steps():
    """Setting bit j of qh[l] adds exactly 16*d*sc_j to element 32*j + l."""
    blocks = rand_blocks("q5k", 40, 78)
    for n, b in enumerate(blocks):
        b = b.copy()
        j, l = n % 8, (n * 11) % 32
        b[16 + l] &= ~np.uint8(1 << j)
        base = oracle.decode_block("q5k", b)
        b[16 + l] |= np.uint8(1 << j)
        up = oracle.decode_block("q5k", b)
        d = oracle.f16_to_f64(int(b[0]) | (int(b[1]) << 8))
        s = b[4:16]
        sc = (s[j] & 63) if j < 4 else ((s[j + 4] & 15) | ((s[j - 4] >> 6) << 4))
        diff = up - base
        assert diff[32 * j + l] == 16 * d * int(sc)
        diff[32 * j + l] = 0
        assert not np.any(diff)


# -------------------------------------------- two independent decoders agree

@pytest.mark.parametrize("fmt", ["q4k", "q6k", "q8_0", "q4_0", "q5k"])
def test_two_decoders_agree(fmt):
    n = 10000 if fmt != "q4k" else 10000
    blocks = rand_blocks(fmt, n, 100 + oracle.FMT[fmt])
    qk = oracle.QK[fmt]
    # check a subset of elements per block against the closed-form decoder
    # (all elements for the first 200 blocks)
    for bi in range(n):
        b = blocks[bi]
        loop = oracle.decode_block(fmt, b)
        idx = range(qk) if bi < 200 else [bi % qk, (bi * 37) % qk, qk - 1 - bi % qk]
        for i in idx:
            assert oracle.decode_elem(fmt, b, i) == loop[i]


# -------------------------------------------------- matvec: brute force etc.

@pytest.mark.parametrize("fmt,rows,k", [("q4k", 3, 256), ("q4k", 4, 512), ("q6k", 2, 512),
                                        ("q6k", 4, 256), ("q8_0", 4, 96), ("q8_0", 1, 512),
                                        ("q4_0", 4, 96), ("q4_0", 2, 512), ("q5k", 3, 256),
                                        ("q5k", 2, 768)])
def test_matvec_brute_force(fmt, rows, k):
    st = synth.Stream(7 + rows + k)
    w = synth.GEN_ROWS[fmt](st, rows, k)
    x = synth.gen_normal(st, k)
    W = oracle.dequant(fmt, w, rows, k)
    # brute force: the materialized f64 matrix times x by numpy, element by element
    ref = np.array([sum(W[r, j] * float(x[j]) for j in range(k)) for r in range(rows)])
    got = oracle.qmv(fmt, w, x, rows, k)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-13)
    assert np.allclose(W @ x.astype(np.float64), got, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fmt", ["q4k", "q6k", "q8_0", "q4_0", "q5k"])
def test_matvec_unit_vector_and_row_sums(fmt):
    rows, k = 5, 512
    st = synth.Stream(31)
    w = synth.GEN_ROWS[fmt](st, rows, k)
    W = oracle.dequant(fmt, w, rows, k)
    for j in [0, 1, 31, 32, 100, 255, 256, 511]:
        e = np.zeros(k, dtype=np.float32)
        e[j] = 1.0
        assert np.array_equal(oracle.qmv(fmt, w, e, rows, k), W[:, j])
    ones = np.ones(k, dtype=np.float32)
    assert np.allclose(oracle.qmv(fmt, w, ones, rows, k), W.sum(axis=1), rtol=1e-13, atol=1e-13)


def test_matvec_linearity():
    rows, k = 6, 768
    st = synth.Stream(5)
    w = synth.gen_q4k_rows(st, rows, k)
    x1 = np.round(synth.gen_normal(st, k) * 64).astype(np.float32)   # small integers:
    x2 = np.round(synth.gen_normal(st, k) * 64).astype(np.float32)   # sums stay exact
    y = oracle.qmv("q4k", w, x1 + 3 * x2, rows, k)
    assert np.allclose(y, oracle.qmv("q4k", w, x1, rows, k) + 3 * oracle.qmv("q4k", w, x2, rows, k),
                       rtol=1e-12, atol=1e-9)


def test_matvec_rejects_ragged_k():
    lib = oracle._lib()
    w = np.zeros(144, dtype=np.uint8)
    x = np.zeros(300, dtype=np.float32)
    y = np.zeros(1)
    assert lib.orc_qmv(0, oracle._p(w), oracle._p(x), 1, 300, oracle._p(y)) == -1


# ------------------------------------------------------ activation quantizer

def test_quantize_round_half_even_ties():
    """amax = 127 makes inv = 127/amax exactly 1, so x*inv = x and the halves
    below are exact ties: round-half-even gives 2, 4, -2, 0, 0 (a half-away
    rule would give 3, 4, -3, 1, -1)."""
    x = np.zeros(32, dtype=np.float32)
    x[:6] = [127.0, 2.5, 3.5, -2.5, 0.5, -0.5]
    xq, xs, xsum = oracle.quantize_act_q8(x, 1, 32)
    assert list(xq[0, :6]) == [127, 2, 4, -2, 0, 0]
    assert xs[0, 0] == np.float32(1.0)
    assert xsum[0, 0] == np.float32(127 + 2 + 4 - 2)


def test_quantize_amax_and_zero_blocks():
    x = np.zeros(96, dtype=np.float32)
    x[5] = -3.25
    x[6] = 1.0
    x[64 + 31] = 1e-30
    xq, xs, xsum = oracle.quantize_act_q8(x, 1, 96)
    assert xq[0, 5] == -127 and xs[0, 0] == np.float32(3.25) / np.float32(127.0)
    assert np.all(xq[0, 32:64] == 0) and xs[0, 1] == 0.0 and xsum[0, 1] == 0.0
    assert xq[0, 64 + 31] == 127 and xs[0, 2] == np.float32(1e-30) / np.float32(127.0)


def test_quantize_matches_ieee_f32_restatement():
    """On random rows the codes equal numpy's IEEE binary32 evaluation of the
    same three operations (divide, multiply, rint) with numpy's own rounding."""
    st = synth.Stream(77)
    m, k = 3, 4096
    x = (synth.gen_normal(st, m * k) * np.float32(3.0)).astype(np.float32)
    xq, xs, xsum = oracle.quantize_act_q8(x, m, k)
    xb = x.reshape(-1, 32)
    amax = np.max(np.abs(xb), axis=1)
    inv = np.float32(127.0) / amax
    q = np.clip(np.rint(xb * inv[:, None]), -127, 127).astype(np.int8)
    assert np.array_equal(xq.reshape(-1, 32), q)
    assert np.array_equal(xs.reshape(-1), amax / np.float32(127.0))
    assert np.array_equal(xsum.reshape(-1), (amax / np.float32(127.0)) * q.astype(np.int32).sum(1).astype(np.float32))


# ------------------------------------------------------------ dp4a + blockdots

def test_blockdots_unit_codes_and_brute_force():
    rows, k = 3, 256
    st = synth.Stream(3)
    w = synth.gen_q8_0_rows(st, rows, k, q_range=(-128, 127))
    codes = w.reshape(rows, k // 32, 34)[:, :, 2:].view(np.int8).reshape(rows, k).astype(np.int64)
    for j in [0, 33, 255]:
        xq = np.zeros(k, dtype=np.int8)
        xq[j] = 127
        dots = oracle.q8_blockdots(w, xq, rows, k)
        assert np.array_equal(dots[:, j // 32], 127 * codes[:, j])
        assert np.count_nonzero(np.delete(dots, j // 32, axis=1)) == 0
    xq = np.random.default_rng(0).integers(-127, 128, size=k).astype(np.int8)
    dots = oracle.q8_blockdots(w, xq, rows, k)
    ref = (codes * xq.astype(np.int64)).reshape(rows, k // 32, 32).sum(2)
    assert np.array_equal(dots, ref)


def test_dp4a_matvec_closed_form():
    rows, k = 2, 64
    st = synth.Stream(9)
    w = synth.gen_q8_0_rows(st, rows, k)
    x = synth.gen_normal(st, k)
    xq, xs, _ = oracle.quantize_act_q8(x, 1, k)
    y = oracle.qmv_q8_dp4a(w, xq.reshape(-1), xs.reshape(-1), rows, k)
    dots = oracle.q8_blockdots(w, xq.reshape(-1), rows, k)
    dw = w.reshape(rows, 2, 34)[:, :, :2].copy().view(np.float16).reshape(rows, 2).astype(np.float64)
    ref = (dw * xs.reshape(1, 2).astype(np.float64) * dots).sum(1)
    assert np.allclose(y, ref, rtol=1e-15, atol=0)
    # and it approximates the f32-activation matvec to within the q8 error
    yf = oracle.qmv("q8_0", w, x, rows, k)
    assert np.max(np.abs(y - yf)) <= 0.05 * np.max(np.abs(yf)) + 1e-6


def test_q4k_dp4a_blockdots_of_known_codes():
    """Blocks built by the inverse of the layout with d = 1, dmin = 0 and all
    scales 1 decode (by the pinned decoder) to their codes, so every
    sub-block dot must be that decoded matrix times the activation codes."""
    rng = np.random.default_rng(11)
    rows, k = 3, 512
    blocks = []
    for _ in range(rows * (k // 256)):
        q = rng.integers(0, 16, size=256)
        blocks.append(pack_q4k(f16_bits(1.0), 0, [1] * 8, [0] * 8, q))
    w = np.concatenate(blocks)
    W = oracle.dequant("q4k", w, rows, k)
    assert np.all(W == np.round(W)) and W.min() >= 0 and W.max() <= 15
    xq = rng.integers(-127, 128, size=k).astype(np.int8)
    dots = oracle.q4k_dp4a_blockdots(w, xq, rows, k)
    ref = (W.astype(np.int64) * xq.astype(np.int64)).reshape(rows, k // 32, 32).sum(2)
    assert np.array_equal(dots, ref)
    # a single code 127 at position j isolates column j of the codes
    for j in [0, 31, 32, 63, 64, 200, 511]:
        e = np.zeros(k, dtype=np.int8)
        e[j] = 127
        d1 = oracle.q4k_dp4a_blockdots(w, e, rows, k)
        assert np.array_equal(d1[:, j // 32], 127 * W[:, j].astype(np.int64))
        assert np.count_nonzero(np.delete(d1, j // 32, axis=1)) == 0


def test_q4k_dp4a_matvec_is_the_matvec_of_the_dequantized_activation():
    """With scales and mins, the dp4a-path matvec equals (to f64 rounding) the
    pinned f64 matvec of the decoded weights against xs * xq; a swapped scale
    and min, a dropped min term or a wrong sub-block would not."""
    rows, k = 5, 768
    st = synth.Stream(21)
    w = synth.gen_q4k_rows(st, rows, k)
    x = synth.gen_normal(st, k)
    xq, xs, _ = oracle.quantize_act_q8(x, 1, k)
    xq, xs = xq.reshape(-1), xs.reshape(-1)
    xhat = xs.astype(np.float64).repeat(32) * xq.astype(np.float64)
    ref = oracle.dequant("q4k", w, rows, k) @ xhat
    y = oracle.qmv_q4k_dp4a(w, xq, xs, rows, k)
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(ref))
    # and it approximates the f32-activation matvec to within the q8 error
    yf = oracle.qmv("q4k", w, x, rows, k)
    assert np.max(np.abs(y - yf)) <= 0.05 * np.max(np.abs(yf))


# ------------------------------------------------- Q6_K x int8 (dp4a path)

def test_q6k_dp4a_groupdots_of_known_codes():
    """xq = 127 e_j picks 127 * (q_j - 32) into the 16-group of j, zeros elsewhere."""
    q = [(i * 5 + 3 * (i // 32)) % 64 for i in range(256)]
    b = pack_q6k(f16_bits(1.0), [1] * 16, q)
    for j in [0, 15, 16, 31, 100, 128, 200, 255]:
        xq = np.zeros(256, dtype=np.int8)
        xq[j] = 127
        dots = oracle.q6k_dp4a_groupdots(b, xq, 1, 256)[0]
        want = np.zeros(16, dtype=np.int64)
        want[j // 16] = 127 * (q[j] - 32)
        assert np.array_equal(dots, want)


def test_q6k_dp4a_groupdots_brute_force():
    """With d = 1 and every scale 1 the pinned decoder returns q - 32 itself:
    the group dots are its integer dots with xq, in groups of 16."""
    rows, k = 3, 512
    st = synth.Stream(93)
    w = synth.gen_q6k_rows(st, rows, k)
    w = w.reshape(rows, k // 256, 210).copy()
    w[:, :, 192:208] = 1
    w[:, :, 208], w[:, :, 209] = 0x00, 0x3C
    w = w.reshape(rows, -1)
    codes = oracle.dequant("q6k", w, rows, k).astype(np.int64)
    xq = oracle.quantize_act_q8(synth.gen_normal(st, k), 1, k)[0].reshape(-1)
    want = (codes * xq.astype(np.int64)).reshape(rows, k // 16, 16).sum(axis=2)
    assert np.array_equal(oracle.q6k_dp4a_groupdots(w, xq, rows, k), want)


def test_q6k_dp4a_matvec_is_the_matvec_of_the_dequantized_activation():
    rows, k = 5, 768
    st = synth.Stream(94)
    w = synth.gen_q6k_rows(st, rows, k)
    x = synth.gen_normal(st, k)
    xq, xs, _ = oracle.quantize_act_q8(x, 1, k)
    xdq = (xs.reshape(-1, 1).astype(np.float64) * xq.reshape(-1, 32)).reshape(-1)
    W = oracle.dequant("q6k", w, rows, k)
    assert np.allclose(oracle.qmv_q6k_dp4a(w, xq.reshape(-1), xs.reshape(-1), rows, k), W @ xdq,
                       rtol=1e-12, atol=1e-12)


def test_moe_q6k_dp4a_matches_dense_per_expert_and_flags_bad_ids():
    e, n, k, slots = 4, 3, 512, 4
    st = synth.Stream(95)
    bank = synth.gen_q6k_rows(st, e * n, k)
    x = synth.gen_normal(st, slots * k).reshape(slots, k)
    xq, xs, _ = oracle.quantize_act_q8(x, slots, k)
    ids = np.array([3, 0, 3, 1], dtype=np.int32)
    y = oracle.moe_qmv_q6k_dp4a(bank, xq, xs, ids, n, k, e)
    rb = (k // 256) * 210
    flat = bank.reshape(-1)
    for s_ in range(slots):
        part = flat[ids[s_] * n * rb:(ids[s_] + 1) * n * rb]
        assert np.array_equal(y[s_], oracle.qmv_q6k_dp4a(part, xq[s_], xs[s_], n, k))
    y_bad = oracle.moe_qmv_q6k_dp4a(bank, xq, xs, np.array([1, 4, -1, 0], dtype=np.int32), n, k, e)
    assert np.all(np.isnan(y_bad[1])) and np.all(np.isnan(y_bad[2]))
    assert not np.any(np.isnan(y_bad[0])) and not np.any(np.isnan(y_bad[3]))


# ------------------------------------------------------------- small-M batch

@pytest.mark.parametrize("fmt,m,rows,k", [("q4k", 3, 4, 512), ("q6k", 2, 3, 256), ("q8_0", 8, 5, 96),
                                          ("q5k", 5, 2, 256), ("q4_0", 4, 3, 64)])
def test_batch_brute_force(fmt, m, rows, k):
    """y[i, r] equals an element loop over the materialized f64 matrix and the
    m rows of x, for every (i, r)."""
    st = synth.Stream(300 + m + rows + k)
    w = synth.GEN_ROWS[fmt](st, rows, k)
    x = synth.gen_normal(st, m * k).reshape(m, k)
    W = oracle.dequant(fmt, w, rows, k)
    ref = np.array([[sum(W[r, j] * float(x[i, j]) for j in range(k)) for r in range(rows)] for i in range(m)])
    got = oracle.qmm(fmt, w, x, m, rows, k)
    assert got.shape == (m, rows)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-13)


def test_batch_unit_rows_and_order():
    """Row i of x = e_{j_i} picks column j_i of W into row i of y exactly (the
    output is [m, rows], x rows in order); a row of zeros gives zeros."""
    rows, k = 6, 512
    w = synth.gen_q4k_rows(synth.Stream(51), rows, k)
    W = oracle.dequant("q4k", w, rows, k)
    cols = [0, 511, 37, 256]
    x = np.zeros((5, k), dtype=np.float32)
    for i, j in enumerate(cols):
        x[i, j] = 1.0
    y = oracle.qmm("q4k", w, x, 5, rows, k)
    for i, j in enumerate(cols):
        assert np.array_equal(y[i], W[:, j])
    assert np.all(y[4] == 0.0)


def test_batch_rows_are_independent():
    """Changing one row of x changes only that row of y, and each row equals
    the pinned matvec of that row alone."""
    m, rows, k = 4, 5, 768
    st = synth.Stream(52)
    w = synth.gen_q6k_rows(st, rows, k)
    x = synth.gen_normal(st, m * k).reshape(m, k)
    y = oracle.qmm("q6k", w, x, m, rows, k)
    x2 = x.copy()
    x2[2] = synth.gen_normal(st, k)
    y2 = oracle.qmm("q6k", w, x2, m, rows, k)
    assert np.array_equal(np.delete(y, 2, axis=0), np.delete(y2, 2, axis=0))
    for i in range(m):
        assert np.array_equal(y2[i], oracle.qmv("q6k", w, x2[i], rows, k))


# ------------------------------------------------------------------------ MoE

def test_moe_matches_dense_per_expert_and_flags_bad_ids():
    e, n, k, slots = 5, 3, 256, 4
    st = synth.Stream(13)
    bank = synth.gen_q4k_rows(st, e * n, k)
    x = synth.gen_normal(st, slots * k).reshape(slots, k)
    ids = np.array([4, 0, 4, 2], dtype=np.int32)
    y = oracle.moe_qmv("q4k", bank, x, ids, n, k, e)
    W = oracle.dequant("q4k", bank, e * n, k).reshape(e, n, k)
    for s in range(slots):
        assert np.allclose(y[s], W[ids[s]] @ x[s].astype(np.float64), rtol=1e-12, atol=1e-12)
    y_bad = oracle.moe_qmv("q4k", bank, x, np.array([1, 5, -1, 0], dtype=np.int32), n, k, e)
    assert np.all(np.isnan(y_bad[1])) and np.all(np.isnan(y_bad[2]))
    assert not np.any(np.isnan(y_bad[0])) and not np.any(np.isnan(y_bad[3]))


def test_moe_q6k_matches_dense_per_expert():
    """The MoE oracle on a Q6_K bank (the pages' down-projection layout) is the
    pinned dense matvec of each slot's expert."""
    e, n, k, slots = 4, 3, 512, 3
    st = synth.Stream(14)
    bank = synth.gen_q6k_rows(st, e * n, k)
    x = synth.gen_normal(st, slots * k).reshape(slots, k)
    ids = np.array([3, 3, 0], dtype=np.int32)
    y = oracle.moe_qmv("q6k", bank, x, ids, n, k, e)
    W = oracle.dequant("q6k", bank, e * n, k).reshape(e, n, k)
    for s in range(slots):
        assert np.allclose(y[s], W[ids[s]] @ x[s].astype(np.float64), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_moe_q8_0_and_q4_0_banks_match_dense_per_expert(fmt):
    """The MoE oracle over a Q8_0 or Q4_0 bank equals the pinned dense matvec
    of each slot's expert, and flags ids outside the bank with NaN."""
    e, n, k, slots = 4, 3, 96, 4
    st = synth.Stream(16 + oracle.FMT[fmt])
    bank = synth.GEN_ROWS[fmt](st, e * n, k)
    x = synth.gen_normal(st, slots * k).reshape(slots, k)
    ids = np.array([2, 0, 3, 2], dtype=np.int32)
    y = oracle.moe_qmv(fmt, bank, x, ids, n, k, e)
    W = oracle.dequant(fmt, bank, e * n, k).reshape(e, n, k)
    for s in range(slots):
        assert np.allclose(y[s], W[ids[s]] @ x[s].astype(np.float64), rtol=1e-12, atol=1e-12)
    y_bad = oracle.moe_qmv(fmt, bank, x, np.array([0, 4, -1, 1], dtype=np.int32), n, k, e)
    assert np.all(np.isnan(y_bad[1])) and np.all(np.isnan(y_bad[2]))
    assert not np.any(np.isnan(y_bad[0])) and not np.any(np.isnan(y_bad[3]))


def test_moe_q4k_dp4a_matches_dense_per_expert_and_flags_bad_ids():
    e, n, k, slots = 5, 4, 512, 4
    st = synth.Stream(15)
    bank = synth.gen_q4k_rows(st, e * n, k)
    x = synth.gen_normal(st, slots * k).reshape(slots, k)
    xq, xs, _ = oracle.quantize_act_q8(x, slots, k)
    ids = np.array([4, 0, 4, 2], dtype=np.int32)
    y = oracle.moe_qmv_q4k_dp4a(bank, xq, xs, ids, n, k, e)
    rb = (k // 256) * 144
    flat = bank.reshape(-1)
    for s in range(slots):
        part = flat[ids[s] * n * rb:(ids[s] + 1) * n * rb]
        assert np.array_equal(y[s], oracle.qmv_q4k_dp4a(part, xq[s], xs[s], n, k))
    y_bad = oracle.moe_qmv_q4k_dp4a(bank, xq, xs, np.array([1, 5, -1, 0], dtype=np.int32), n, k, e)
    assert np.all(np.isnan(y_bad[1])) and np.all(np.isnan(y_bad[2]))
    assert not np.any(np.isnan(y_bad[0])) and not np.any(np.isnan(y_bad[3]))


# ------------------------------------------------------------ a planted bug

def test_pins_catch_a_planted_q4k_mistake(monkeypatch):
    """Swap the scale and min of sub-block 5 in the bytes: the closed-form pin
    must notice, i.e. the pin is sensitive to exactly this kind of error."""
    q = [i % 16 for i in range(256)]
    sc, mn = list(SC), list(MN)
    sc[5], mn[5] = mn[5], sc[5]
    b = pack_q4k(f16_bits(1.0), f16_bits(0.5), sc, mn, q)
    got = oracle.decode_block("q4k", b)
    want = np.array([SC[i // 32] * (i % 16) - 0.5 * MN[i // 32] for i in range(256)])
    assert not np.array_equal(got, want)
