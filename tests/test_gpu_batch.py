"""GPU parity of the small-M batched product y[m, rows] = x[m, k] W^T
(qmm_q4k, qmm_q6k, qmm_q8_0, qmm_q5k, qmm_q4_0) against the CPU oracle,
through the C ABI.

Bars: x rows that are unit vectors give y rows equal to the decoded weight
columns bit for bit; otherwise every row of y is within scale-relative error
max|a-b|/max|a| <= 1e-4 of the f64 oracle.
"""

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

SCALE_REL_TOL = 1e-4
FMTS = ["q4k", "q6k", "q8_0", "q5k", "q4_0"]


@pytest.fixture(scope="module")
def q():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    import ggml_format_dequant_gb300 as lib
    lib.qmv_device_status(clear=True)
    return lib


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def scale_rel(ref, got):
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    return float(np.max(np.abs(ref - got)) / max(float(np.max(np.abs(ref))), 1e-30))


def run_qmm(q, fmt, w, x, rows, k, m, cfg=None, overlap=0):
    y = torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda")
    getattr(q, f"qmm_{fmt}")(dev(w), dev(x), y, rows, k, m, cfg=cfg, overlap=overlap)
    return host(y)


def check_rows(ref, y):
    assert not np.any(np.isnan(y))
    for i in range(ref.shape[0]):
        assert scale_rel(ref[i], y[i]) <= SCALE_REL_TOL, i


SHAPES = [("q4k", 300, 768), ("q4k", 1, 256), ("q4k", 97, 4352), ("q4k", 64, 4096), ("q4k", 20, 16384),
          ("q6k", 300, 512), ("q6k", 3, 256), ("q6k", 41, 14336), ("q6k", 130, 2816),
          ("q8_0", 300, 96), ("q8_0", 13, 32), ("q8_0", 7, 4096), ("q8_0", 64, 11008), ("q8_0", 5, 4160),
          ("q5k", 300, 768), ("q5k", 3, 256), ("q5k", 97, 4352), ("q5k", 20, 16384), ("q4_0", 300, 96),
          ("q4_0", 13, 32), ("q4_0", 64, 11008), ("q4_0", 5, 4160)]


@pytest.mark.parametrize("m", [2, 3, 4, 5, 8])
@pytest.mark.parametrize("fmt,rows,k", SHAPES)
def test_batch_matches_oracle(q, fmt, rows, k, m):
    st = synth.Stream(rows * 13 + k + m)
    w = synth.GEN_ROWS[fmt](st, rows, k)
    x = synth.gen_normal(st, m * k).reshape(m, k)
    check_rows(oracle.qmm(fmt, w, x, m, rows, k), run_qmm(q, fmt, w, x, rows, k, m))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [1, 6, 7, 9, 13, 17])
def test_batch_widths_and_tiles(q, fmt, m):
    """m = 1 (the matvec), odd widths, and m > 8 (several tiles)."""
    rows, k = 77, 1024
    st = synth.Stream(900 + m)
    w = synth.GEN_ROWS[fmt](st, rows, k)
    x = synth.gen_normal(st, m * k).reshape(m, k)
    check_rows(oracle.qmm(fmt, w, x, m, rows, k), run_qmm(q, fmt, w, x, rows, k, m))


@pytest.mark.parametrize("fmt", FMTS)
def test_batch_unit_rows_are_exact(q, fmt):
    """Row i of x = e_{j_i}: row i of y is column j_i of the decoded weights
    bit for bit, for every unit position of every tile width."""
    rows, k = 40, 2048
    w = synth.GEN_ROWS[fmt](synth.Stream(61), rows, k)
    W = oracle.dequant(fmt, w, rows, k).astype(np.float32)
    cols = [0, 1, 7, 8, 15, 16, 31, 32, 63, 100, 127, 128, 255, 256, 1000, 2047]
    for m in (2, 3, 8):
        for c0 in range(0, len(cols), m):
            js = cols[c0:c0 + m]
            js = js + [0] * (m - len(js))
            x = np.zeros((m, k), dtype=np.float32)
            for i, j in enumerate(js):
                x[i, j] = 1.0
            y = run_qmm(q, fmt, w, x, rows, k, m)
            for i, j in enumerate(js):
                assert np.array_equal(y[i], W[:, j]), (m, i, j)


@pytest.mark.parametrize("cfg", [dict(ctas=1, chunk_rows=1, chunks=2), dict(ctas=3, chunk_rows=5, chunks=2),
                                 dict(ctas=2, chunk_rows=3, chunks=1), dict(ctas=7, chunks=3),
                                 dict(ctas=2, chunks=1, warps=4), dict(ctas=1, chunk_rows=7, chunks=2, warps=16)])
@pytest.mark.parametrize("fmt,m", [("q4k", 2), ("q4k", 8), ("q6k", 3), ("q8_0", 5), ("q5k", 4), ("q5k", 8), ("q4_0", 6)])
def test_batch_forced_pipelines(q, fmt, m, cfg):
    rows, k = 61, 512
    st = synth.Stream(71 + m)
    w = synth.GEN_ROWS[fmt](st, rows, k)
    x = synth.gen_normal(st, m * k).reshape(m, k)
    check_rows(oracle.qmm(fmt, w, x, m, rows, k), run_qmm(q, fmt, w, x, rows, k, m, cfg=cfg))


def test_batch_extreme_activations(q):
    rows, k, m = 33, 1024, 4
    st = synth.Stream(81)
    w = synth.gen_q4k_rows(st, rows, k)
    x = synth.gen_normal(st, m * k).reshape(m, k)
    x[0, 0:32] = 0.0
    x[1, 32:64] *= np.float32(1e-30)
    x[2, :] *= np.float32(1e30)
    x[3, 96:128] = np.float32(1e-40)
    check_rows(oracle.qmm("q4k", w, x, m, rows, k), run_qmm(q, "q4k", w, x, rows, k, m))


def test_batch_argument_errors(q):
    w = torch.zeros(144 * 4 + 16, dtype=torch.uint8, device="cuda")
    x = torch.zeros(4 * 512, dtype=torch.float32, device="cuda")
    y = torch.zeros(16, dtype=torch.float32, device="cuda")
    assert q.qmm_q4k(w, x, y, 2, 256, 0, check=False) == q.QMV_EINVAL
    assert q.qmm_q4k(w, x, y, 2, 300, 2, check=False) == q.QMV_EINVAL
    assert q.qmm_q4k(w, x.data_ptr() + 4, y, 2, 256, 2, check=False) == q.QMV_EALIGN
    assert q.qmm_q8_0(w, x, y, 2, 48, 2, check=False) == q.QMV_EINVAL
    assert q.qmm_q5k(w, x, y, 2, 300, 2, check=False) == q.QMV_EINVAL       # k not a multiple of 256
    assert q.qmm_q5k(w, x, y, 2, 256, 0, check=False) == q.QMV_EINVAL       # m = 0
    assert q.qmm_q4_0(w, x, y, 2, 48, 2, check=False) == q.QMV_EINVAL       # k not a multiple of 32
    assert q.qmm_q4_0(w, x.data_ptr() + 4, y, 2, 64, 2, check=False) == q.QMV_EALIGN
    assert q.qmm_q4_0(w, x, y, -1, 64, 2, check=False) == q.QMV_EINVAL      # rows < 1


@pytest.mark.parametrize("fmt,rows,k", [("q4k", 300, 4096), ("q6k", 97, 14336), ("q8_0", 500, 4096),
                                        ("q5k", 64, 4352), ("q4_0", 77, 4160)])
@pytest.mark.parametrize("m", [2, 4, 8])
def test_batch_independent_call_plans(q, fmt, rows, k, m):
    """Independent calls (QMV_OVERLAP_INDEPENDENT) take half-SM CTAs of at most 8 warps, so rows
    longer than 2048 weights are cut into more k-chunks than in plain launches:
    every row of y still matches the oracle, unit rows still give the weight
    columns bit for bit."""
    st = synth.Stream(rows + k + 5 * m)
    w = synth.GEN_ROWS[fmt](st, rows, k)
    x = synth.gen_normal(st, m * k).reshape(m, k)
    W = oracle.dequant(fmt, w, rows, k).astype(np.float32)
    js = [3, 1000, k - 1, 2048, 77, 3000, 5, 4000][:m]
    xu = np.zeros((m, k), dtype=np.float32)
    for i, j in enumerate(js):
        xu[i, j] = 1.0
    y = run_qmm(q, fmt, w, x, rows, k, m, overlap=q.OVERLAP_INDEPENDENT)
    yu = run_qmm(q, fmt, w, xu, rows, k, m, overlap=q.OVERLAP_INDEPENDENT)
    check_rows(oracle.qmm(fmt, w, x, m, rows, k), y)
    for i, j in enumerate(js):
        assert np.array_equal(yu[i], W[:, j]), (i, j)


def test_batch_overlap_modes_give_identical_results(q):
    """Rows of 2048 weights (8 slices: one k-chunk in every mode) give the same
    bits in plain, chained and independent calls."""
    st = synth.Stream(91)
    cases = [(fmt, dev(synth.GEN_ROWS[fmt](st, 300, 2048)), dev(synth.gen_normal(st, 5 * 2048)))
             for fmt in FMTS]

    def chain(ov):
        outs = []
        for fmt, w, x in cases:
            y = torch.empty(5, 300, dtype=torch.float32, device="cuda")
            getattr(q, f"qmm_{fmt}")(w, x, y, 300, 2048, 5, overlap=ov)
            outs.append(y)
        torch.cuda.synchronize()
        return [o.cpu().numpy() for o in outs]

    base = chain(q.OVERLAP_NONE)
    for mode in (q.OVERLAP_CHAIN, q.OVERLAP_INDEPENDENT):
        for a, b in zip(base, chain(mode)):
            assert np.array_equal(a, b), mode


@pytest.mark.parametrize("name", ["qmm_q4k_4096x4096_m8", "qmm_q4k_4096x4096_m2", "qmm_q6k_4096x14336_m4",
                                  "qmm_q8_0_14336x4096_m8", "qmm_q5k_4096x4096_m4", "qmm_q4_0_4096x4096_m4"])
def test_full_batch(q, name):
    c = synth.make_config(name)
    fmt = c["kind"][4:]
    y = run_qmm(q, fmt, c["w"], c["x"], c["rows"], c["k"], c["m"])
    check_rows(oracle.qmm(fmt, c["w"], c["x"], c["m"], c["rows"], c["k"]), y)


@pytest.mark.parametrize("fmt,rows,k", [("q4k", 37, 2048), ("q6k", 29, 2560), ("q8_0", 41, 1312), ("q8_0", 19, 96),
                                        ("q5k", 23, 2304), ("q4_0", 31, 1568)])
@pytest.mark.parametrize("warps", [1, 2, 3])
@pytest.mark.parametrize("m", [2, 3, 5, 8])
def test_batch_kchunks(q, fmt, rows, k, warps, m):
    """Rows dealt into several k-chunks inside one launch (a warps bound of
    1-3 slices per chunk; Q8_0 1312 = 41 groups: a ragged last slice and a
    shorter last chunk), packed (m <= 4) and unpacked."""
    st = synth.Stream(rows * 7 + k + 31 * warps + m)
    w = synth.GEN_ROWS[fmt](st, rows, k)
    x = synth.gen_normal(st, m * k).reshape(m, k)
    cfg = dict(warps=warps, chunks=2)
    check_rows(oracle.qmm(fmt, w, x, m, rows, k), run_qmm(q, fmt, w, x, rows, k, m, cfg=cfg))


@pytest.mark.parametrize("fmt", FMTS)
def test_batch_kchunk_unit_rows_are_exact(q, fmt):
    """Unit rows of x through a four-chunk plan still give the decoded weight
    columns bit for bit (the chunks' partial sums are exact zeros elsewhere)."""
    rows, k, m = 24, 2048, 4
    w = synth.GEN_ROWS[fmt](synth.Stream(63), rows, k)
    W = oracle.dequant(fmt, w, rows, k).astype(np.float32)
    js = [5, 700, 1300, 2047]
    x = np.zeros((m, k), dtype=np.float32)
    for i, j in enumerate(js):
        x[i, j] = 1.0
    y = run_qmm(q, fmt, w, x, rows, k, m, cfg=dict(warps=2))
    for i, j in enumerate(js):
        assert np.array_equal(y[i], W[:, j]), (i, j)


@pytest.mark.parametrize("fmt,rows,k", [("q4k", 4096, 4096), ("q4_0", 2600, 2048), ("q5k", 2500, 4096)])
@pytest.mark.parametrize("m", [2, 5, 8])
def test_batch_independent_streaming_plan(q, fmt, rows, k, m):
    """Independent calls of rows that fill a quarter of the SM count with two
    32-row pieces each stream their share through two ring slots in a
    quarter-SM-count of CTAs (Q4_K and Q4_0 here; the Q5_K rows' two slots do
    not fit half an SM, so they keep the other plan): every row of y matches
    the oracle and unit rows of x still give the weight columns bit for bit."""
    P = q.qmm_tc_plan_detail({"q4k": 0, "q5k": 3, "q4_0": 4}[fmt], rows, k, m, overlap=q.OVERLAP_INDEPENDENT,
                             device=q.GB300_DEVICE)
    if fmt != "q5k":
        assert P["ctas"] == q.GB300_DEVICE[0] // 4 and P["CR"] == 32 and P["S"] == 2
    st = synth.Stream(rows + 3 * k + m)
    w = synth.GEN_ROWS[fmt](st, rows, k)
    x = synth.gen_normal(st, m * k).reshape(m, k)
    y = run_qmm(q, fmt, w, x, rows, k, m, overlap=q.OVERLAP_INDEPENDENT)
    check_rows(oracle.qmm(fmt, w, x, m, rows, k), y)
    js = [5, k - 1, 1000, 17, k // 2, 333, 64, 2047][:m]
    xu = np.zeros((m, k), dtype=np.float32)
    for i, j in enumerate(js):
        xu[i, j] = 1.0
    yu = run_qmm(q, fmt, w, xu, rows, k, m, overlap=q.OVERLAP_INDEPENDENT)
    W = oracle.dequant(fmt, w, rows, k).astype(np.float32)
    for i, j in enumerate(js):
        assert np.array_equal(yu[i], W[:, j]), (i, j)
