"""GPU parity of every entry point against the CPU oracle, through the C ABI.

Bars: decoded weights, quantized
activations, int32 block dots and MoE row gathers are bit-exact; f32 matvec
outputs are within scale-relative error max|a-b|/max|a| <= 1e-4 of the f64
oracle.
"""

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

SCALE_REL_TOL = 1e-4
GEN = {"q4k": synth.gen_q4k_rows, "q6k": synth.gen_q6k_rows, "q8_0": synth.gen_q8_0_rows}
QK = {"q4k": 256, "q6k": 256, "q8_0": 32}


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


def run_matvec(q, fmt, w, x, rows, k, cfg=None):
    y = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    fn = {"q4k": q.qmv_q4k, "q6k": q.qmv_q6k, "q8_0": q.qmv_q8_0}[fmt]
    fn(dev(w), dev(x), y, rows, k, cfg=cfg)
    return host(y)


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("fmt,rows,k", [("q4k", 37, 512), ("q4k", 3, 2304), ("q6k", 37, 512),
                                        ("q6k", 5, 256), ("q8_0", 37, 96), ("q8_0", 3, 4096)])
def test_dequant_bit_exact(q, fmt, rows, k):
    st = synth.Stream(1000 + rows + k)
    w = GEN[fmt](st, rows, k) if fmt != "q8_0" else synth.gen_q8_0_rows(st, rows, k, q_range=(-128, 127))
    out = torch.empty(rows, k, dtype=torch.float32, device="cuda")
    getattr(q, f"qmv_dequant_{fmt}")(dev(w), out, rows, k)
    ref = oracle.dequant(fmt, w, rows, k).astype(np.float32)   # RNE of the exact value
    assert np.array_equal(host(out), ref)


def test_dequant_subnormal_scales(q):
    st = synth.Stream(5)
    w = synth.gen_q4k_rows(st, 4, 256, d_range=(0.0, 6e-8), dmin_range=(0.0, 6e-8))
    out = torch.empty(4, 256, dtype=torch.float32, device="cuda")
    q.qmv_dequant_q4k(dev(w), out, 4, 256)
    assert np.array_equal(host(out), oracle.dequant("q4k", w, 4, 256).astype(np.float32))


# ------------------------------------------------------------------ matvec

SHAPES = [("q4k", 256, 1024), ("q4k", 300, 768), ("q4k", 1, 256), ("q4k", 97, 4352), ("q4k", 20, 16384),
          ("q6k", 300, 512), ("q6k", 3, 256), ("q6k", 41, 14336), ("q6k", 130, 2816),
          ("q8_0", 300, 96), ("q8_0", 7, 4096), ("q8_0", 13, 32), ("q8_0", 64, 11008)]


@pytest.mark.parametrize("fmt,rows,k", SHAPES)
def test_matvec_matches_oracle(q, fmt, rows, k):
    st = synth.Stream(rows * 7 + k)
    w = GEN[fmt](st, rows, k)
    x = synth.gen_normal(st, k)
    y = run_matvec(q, fmt, w, x, rows, k)
    assert scale_rel(oracle.qmv(fmt, w, x, rows, k), y) <= SCALE_REL_TOL


@pytest.mark.parametrize("cfg", [dict(ctas=1, chunk_rows=1, chunks=2), dict(ctas=3, chunk_rows=5, chunks=2),
                                 dict(ctas=2, chunk_rows=3, chunks=1), dict(ctas=7, chunks=3),
                                 dict(ctas=1, chunks=2, unroll=1), dict(ctas=3, chunk_rows=4, chunks=3, unroll=2),
                                 dict(ctas=2, chunks=1, warps=2), dict(ctas=5, chunk_rows=2, chunks=4, warps=4),
                                 dict(ctas=1, chunk_rows=7, chunks=2, warps=16, unroll=1)])
@pytest.mark.parametrize("fmt", ["q4k", "q6k", "q8_0"])
def test_matvec_forced_pipelines(q, fmt, cfg):
    """Small CTA counts and rings force many trips around each row group's
    ring, shared pieces and ragged last pieces; every output must still match."""
    rows, k = 61, 512
    st = synth.Stream(17)
    w = GEN[fmt](st, rows, k)
    x = synth.gen_normal(st, k)
    y = run_matvec(q, fmt, w, x, rows, k, cfg=cfg)
    assert not np.any(np.isnan(y))
    assert scale_rel(oracle.qmv(fmt, w, x, rows, k), y) <= SCALE_REL_TOL


@pytest.mark.parametrize("cfg", [dict(ctas=1, chunk_rows=3, chunks=2), dict(ctas=2, chunk_rows=1, chunks=1),
                                 dict(ctas=3, chunk_rows=2, chunks=3, unroll=1), dict(ctas=1, chunks=2, warps=16)])
@pytest.mark.parametrize("fmt,k", [("q4k", 4352), ("q6k", 2816), ("q8_0", 4096), ("q4k", 16384)])
def test_matvec_forced_pipelines_wide(q, fmt, k, cfg):
    """Rows of several k-slices: the warps of a row group share every piece and
    the last one to finish re-fills the slot; ragged slices and pieces."""
    rows = 29
    st = synth.Stream(k + 5)
    w = GEN[fmt](st, rows, k)
    x = synth.gen_normal(st, k)
    y = run_matvec(q, fmt, w, x, rows, k, cfg=cfg)
    assert not np.any(np.isnan(y))
    assert scale_rel(oracle.qmv(fmt, w, x, rows, k), y) <= SCALE_REL_TOL


@pytest.mark.parametrize("cluster", [2, 4, 8])
@pytest.mark.parametrize("fmt,rows,k", [("q4k", 97, 4352), ("q6k", 41, 2048), ("q8_0", 64, 1024)])
def test_matvec_cluster_shared_prep(q, fmt, rows, k, cluster):
    """CTAs of a cluster each convert part of x and write it into every
    member's shared memory: results must match, and equal the unclustered
    ones bit for bit (the same limbs, the same order of sums)."""
    st = synth.Stream(k + cluster)
    w = GEN[fmt](st, rows, k)
    x = synth.gen_normal(st, k)
    cfg = dict(ctas=8, cluster=cluster)
    assert q.qmv_plan_info({"q4k": 0, "q6k": 1, "q8_0": 2}[fmt], rows, k, cfg=cfg)["ctas"] % cluster == 0
    y = run_matvec(q, fmt, w, x, rows, k, cfg=cfg)
    y1 = run_matvec(q, fmt, w, x, rows, k, cfg=dict(ctas=8))
    assert scale_rel(oracle.qmv(fmt, w, x, rows, k), y) <= SCALE_REL_TOL
    assert np.array_equal(y, y1)


@pytest.mark.parametrize("fmt,rows,k", [("q4k", 64, 1024), ("q6k", 24, 768), ("q8_0", 40, 256),
                                        ("q4k", 9, 16384)])
def test_unit_vector_is_exact(q, fmt, rows, k):
    """x = e_j leaves one nonzero product: y[r] must equal the decoded weight
    W[r, j] bit for bit, through the real matvec kernel."""
    st = synth.Stream(23)
    w = GEN[fmt](st, rows, k)
    W = oracle.dequant(fmt, w, rows, k).astype(np.float32)
    for j in sorted({0, 1, 15, 16, 31, 32, 63, 64, 100, 127, 128, 200, 255, k // 2 + 3, k - 1}):
        e = np.zeros(k, dtype=np.float32)
        e[j] = 1.0
        y = run_matvec(q, fmt, w, e, rows, k)
        assert np.array_equal(y, W[:, j]), f"column {j}"


def test_matvec_scaled_unit_vectors(q):
    """Powers of two other than 1 must stay exact as well (limb scaling)."""
    rows, k = 16, 512
    w = synth.gen_q4k_rows(synth.Stream(3), rows, k)
    W = oracle.dequant("q4k", w, rows, k)
    for j, v in [(5, 0.125), (300, 1024.0), (511, -2.0 ** -20)]:
        e = np.zeros(k, dtype=np.float32)
        e[j] = v
        y = run_matvec(q, "q4k", w, e, rows, k)
        assert np.array_equal(y, (W[:, j] * v).astype(np.float32))


def test_matvec_deterministic_and_stream(q):
    rows, k = 512, 4096
    st = synth.Stream(8)
    w = dev(synth.gen_q4k_rows(st, rows, k))
    x = dev(synth.gen_normal(st, k))
    s = torch.cuda.Stream()
    y1 = torch.empty(rows, device="cuda")
    y2 = torch.empty(rows, device="cuda")
    with torch.cuda.stream(s):
        q.qmv_q4k(w, x, y1, rows, k)
        q.qmv_q4k(w, x, y2, rows, k, stream=s)
    s.synchronize()
    assert torch.equal(y1, y2)


def test_matvec_extreme_activations(q):
    """Groups of tiny, huge and zero activations next to ordinary ones."""
    rows, k = 33, 1024
    st = synth.Stream(41)
    w = synth.gen_q4k_rows(st, rows, k)
    x = synth.gen_normal(st, k)
    x[0:32] = 0.0
    x[32:64] *= np.float32(1e-30)
    x[64:96] *= np.float32(1e30)
    x[96:128] = np.float32(1e-40)   # subnormal
    x[200] = np.float32(1e36)    # sum(q*x) of its sub-block must stay finite in f32
    ref = oracle.qmv("q4k", w, x, rows, k)
    y = run_matvec(q, "q4k", w, x, rows, k)
    assert scale_rel(ref, y) <= SCALE_REL_TOL


# ------------------------------------------------- activation quant + dp4a

def test_quantize_act_bit_exact(q):
    m, k = 3, 4096
    x = synth.gen_normal(synth.Stream(12), m * k).astype(np.float32) * np.float32(2.5)
    x[0:32] = 0.0                                     # amax == 0 block
    x[32:64] = 0.0
    x[32:38] = [127.0, 2.5, 3.5, -2.5, 0.5, -0.5]     # exact ties
    x[64:96] *= np.float32(1e-38)
    xq = torch.empty(m * k, dtype=torch.int8, device="cuda")
    xs = torch.empty(m * k // 32, dtype=torch.float32, device="cuda")
    xsum = torch.empty(m * k // 32, dtype=torch.float32, device="cuda")
    q.quantize_act_q8(dev(x), xq, xs, xsum, m, k)
    oq, os_, osum = oracle.quantize_act_q8(x, m, k)
    assert np.array_equal(host(xq), oq.reshape(-1))
    assert np.array_equal(host(xs), os_.reshape(-1))
    assert np.array_equal(host(xsum), osum.reshape(-1))
    # without the optional sum
    q.quantize_act_q8(dev(x), xq, xs, None, m, k)
    assert np.array_equal(host(xq), oq.reshape(-1))


@pytest.mark.parametrize("rows,k", [(300, 4096), (7, 96), (1, 32)])
def test_blockdots_bit_exact(q, rows, k):
    st = synth.Stream(rows + k)
    w = synth.gen_q8_0_rows(st, rows, k, q_range=(-128, 127))
    xq, xs, _ = oracle.quantize_act_q8(synth.gen_normal(st, k), 1, k)
    dots = torch.empty(rows, k // 32, dtype=torch.int32, device="cuda")
    q.qmv_q8_dp4a_blockdots(dev(w), dev(xq.reshape(-1)), dots, rows, k)
    assert np.array_equal(host(dots), oracle.q8_blockdots(w, xq.reshape(-1), rows, k))


@pytest.mark.parametrize("rows,k,cfg", [(300, 4096, None), (61, 256, dict(ctas=2, chunk_rows=3, chunks=2)),
                                        (5, 32, None)])
def test_dp4a_matvec(q, rows, k, cfg):
    st = synth.Stream(99 + rows)
    w = synth.gen_q8_0_rows(st, rows, k)
    x = synth.gen_normal(st, k)
    xq = torch.empty(k, dtype=torch.int8, device="cuda")
    xs = torch.empty(k // 32, dtype=torch.float32, device="cuda")
    q.quantize_act_q8(dev(x), xq, xs, None, 1, k)
    y = torch.empty(rows, dtype=torch.float32, device="cuda")
    q.qmv_q8_dp4a(dev(w), xq, xs, y, rows, k, cfg=cfg)
    oq, os_, _ = oracle.quantize_act_q8(x, 1, k)
    ref = oracle.qmv_q8_dp4a(w, oq.reshape(-1), os_.reshape(-1), rows, k)
    assert scale_rel(ref, host(y)) <= SCALE_REL_TOL


# ------------------------------------------------- Q4_K x q8 activation (dp4a)

def _q4k_dp4a_inputs(q, rows, k, seed):
    st = synth.Stream(seed)
    w = synth.gen_q4k_rows(st, rows, k)
    x = synth.gen_normal(st, k)
    xq = torch.empty(k, dtype=torch.int8, device="cuda")
    xs = torch.empty(k // 32, dtype=torch.float32, device="cuda")
    q.quantize_act_q8(dev(x), xq, xs, None, 1, k)
    oq, os_, _ = oracle.quantize_act_q8(x, 1, k)
    assert np.array_equal(host(xq), oq.reshape(-1)) and np.array_equal(host(xs), os_.reshape(-1))
    return w, xq, xs, oq.reshape(-1), os_.reshape(-1)


@pytest.mark.parametrize("rows,k,cfg", [(300, 4096, None), (61, 512, None), (1, 256, None), (97, 4352, None),
                                        (29, 16384, None), (61, 512, dict(ctas=2, chunk_rows=3, chunks=2)),
                                        (29, 4352, dict(ctas=1, chunk_rows=1, chunks=1)),
                                        (300, 768, dict(ctas=3, unroll=1, warps=4))])
def test_q4k_dp4a_matvec(q, rows, k, cfg):
    w, xq, xs, oq, os_ = _q4k_dp4a_inputs(q, rows, k, 5000 + rows + k)
    y = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    q.qmv_q4k_dp4a(dev(w), xq, xs, y, rows, k, cfg=cfg)
    assert scale_rel(oracle.qmv_q4k_dp4a(w, oq, os_, rows, k), host(y)) <= SCALE_REL_TOL


@pytest.mark.parametrize("rows,k", [(300, 4096), (7, 256), (33, 4352)])
def test_q4k_dp4a_blockdots_bit_exact(q, rows, k):
    w, xq, xs, oq, _ = _q4k_dp4a_inputs(q, rows, k, 6000 + rows)
    dots = torch.empty(rows, k // 32, dtype=torch.int32, device="cuda")
    q.qmv_q4k_dp4a_blockdots(dev(w), xq, dots, rows, k)
    assert np.array_equal(host(dots), oracle.q4k_dp4a_blockdots(w, oq, rows, k))


def test_full_q4k_dp4a_4096(q):
    c = synth.make_config("q4k_dp4a_4096x4096")
    rows, k = 4096, 4096
    xq = torch.empty(k, dtype=torch.int8, device="cuda")
    xs = torch.empty(k // 32, dtype=torch.float32, device="cuda")
    q.quantize_act_q8(dev(c["x"]), xq, xs, None, 1, k)
    y = torch.empty(rows, dtype=torch.float32, device="cuda")
    q.qmv_q4k_dp4a(dev(c["w"]), xq, xs, y, rows, k)
    oq, os_, _ = oracle.quantize_act_q8(c["x"], 1, k)
    assert scale_rel(oracle.qmv_q4k_dp4a(c["w"], oq.reshape(-1), os_.reshape(-1), rows, k), host(y)) <= SCALE_REL_TOL


# --------------------------------------------------------------------- MoE

def moe_run(q, bank, x, ids, rows, k, n_experts, cfg=None):
    slots = len(ids)
    y = torch.full((slots, rows), 7.0, dtype=torch.float32, device="cuda")
    q.moe_qmv_q4k(dev(bank), dev(x), y, rows, k, dev(np.asarray(ids, dtype=np.int32)), slots, n_experts, cfg=cfg)
    return host(y)


@pytest.mark.parametrize("e,n,k,ids", [(16, 96, 512, [3, 15, 0, 3]), (4, 768, 512, [1, 2]),
                                       (8, 7, 256, [7, 6, 5, 4, 3, 2, 1, 0, 7])])
def test_moe_matches_oracle(q, e, n, k, ids):
    st = synth.Stream(e * n + k)
    bank = synth.gen_q4k_rows(st, e * n, k)
    x = synth.gen_normal(st, len(ids) * k).reshape(len(ids), k)
    y = moe_run(q, bank, x, ids, n, k, e)
    ref = oracle.moe_qmv("q4k", bank, x, np.array(ids, dtype=np.int32), n, k, e)
    for s in range(len(ids)):
        assert scale_rel(ref[s], y[s]) <= SCALE_REL_TOL


def test_moe_gather_exact(q):
    """x[s] = e_j in every slot: y[s] must be column j of expert ids[s] exactly,
    so any wrong expert or row shows up bit-wise."""
    e, n, k = 12, 40, 512
    bank = synth.gen_q4k_rows(synth.Stream(4), e * n, k)
    W = oracle.dequant("q4k", bank, e * n, k).reshape(e, n, k).astype(np.float32)
    ids = [11, 0, 5, 5, 3]
    for j in [0, 77, 511]:
        x = np.zeros((len(ids), k), dtype=np.float32)
        x[:, j] = 1.0
        y = moe_run(q, bank, x, ids, n, k, e, cfg=dict(ctas=2, chunk_rows=3, chunks=2))
        for s, eid in enumerate(ids):
            assert np.array_equal(y[s], W[eid, :, j])


def test_moe_bad_ids_give_nan_and_status(q):
    e, n, k = 4, 16, 256
    st = synth.Stream(6)
    bank = synth.gen_q4k_rows(st, e * n, k)
    x = synth.gen_normal(st, 4 * k).reshape(4, k)
    q.qmv_device_status(clear=True)
    y = moe_run(q, bank, x, [1, 4, -1, 2], n, k, e)
    assert np.all(np.isnan(y[1])) and np.all(np.isnan(y[2]))
    ref = oracle.moe_qmv("q4k", bank, x, np.array([1, 0, 0, 2], dtype=np.int32), n, k, e)
    assert scale_rel(ref[0], y[0]) <= SCALE_REL_TOL and scale_rel(ref[3], y[3]) <= SCALE_REL_TOL
    assert q.qmv_device_status(clear=True) & q.QMV_STATUS_BAD_EXPERT_ID
    assert q.qmv_device_status(clear=True) == 0


# ------------------------------------------- MoE: Q6_K bank, Q4_K dp4a path

def moe6_run(q, bank, x, ids, rows, k, n_experts, cfg=None):
    slots = len(ids)
    y = torch.full((slots, rows), 7.0, dtype=torch.float32, device="cuda")
    q.moe_qmv_q6k(dev(bank), dev(x), y, rows, k, dev(np.asarray(ids, dtype=np.int32)), slots, n_experts, cfg=cfg)
    return host(y)


@pytest.mark.parametrize("e,n,k,ids,cfg", [(16, 96, 512, [3, 15, 0, 3], None), (8, 257, 768, [1, 2], None),
                                           (8, 7, 256, [7, 6, 5, 4, 3, 2, 1, 0, 7], None),
                                           (6, 40, 768, [5, 1, 1], dict(ctas=2, chunk_rows=3, chunks=2))])
def test_moe_q6k_matches_oracle(q, e, n, k, ids, cfg):
    st = synth.Stream(e * n + k + 1)
    bank = synth.gen_q6k_rows(st, e * n, k)
    x = synth.gen_normal(st, len(ids) * k).reshape(len(ids), k)
    y = moe6_run(q, bank, x, ids, n, k, e, cfg=cfg)
    ref = oracle.moe_qmv("q6k", bank, x, np.array(ids, dtype=np.int32), n, k, e)
    for s in range(len(ids)):
        assert scale_rel(ref[s], y[s]) <= SCALE_REL_TOL


def test_moe_q6k_gather_exact(q):
    e, n, k = 10, 24, 768
    bank = synth.gen_q6k_rows(synth.Stream(44), e * n, k)
    W = oracle.dequant("q6k", bank, e * n, k).reshape(e, n, k).astype(np.float32)
    ids = [9, 0, 4, 4]
    for j in [0, 100, 767]:
        x = np.zeros((len(ids), k), dtype=np.float32)
        x[:, j] = 1.0
        y = moe6_run(q, bank, x, ids, n, k, e)
        for s, eid in enumerate(ids):
            assert np.array_equal(y[s], W[eid, :, j])


def _moe_dp4a_run(q, bank, x, ids, rows, k, n_experts, cfg=None):
    slots = len(ids)
    xq = torch.empty(slots * k, dtype=torch.int8, device="cuda")
    xs = torch.empty(slots * (k // 32), dtype=torch.float32, device="cuda")
    q.quantize_act_q8(dev(x), xq, xs, None, slots, k)
    y = torch.full((slots, rows), 7.0, dtype=torch.float32, device="cuda")
    q.moe_qmv_q4k_dp4a(dev(bank), xq, xs, y, rows, k, dev(np.asarray(ids, dtype=np.int32)), slots, n_experts, cfg=cfg)
    oq, os_, _ = oracle.quantize_act_q8(x, slots, k)
    assert np.array_equal(host(xq), oq.reshape(-1))
    return host(y), oq, os_


@pytest.mark.parametrize("e,n,k,ids,cfg", [(16, 96, 512, [3, 15, 0, 3], None), (4, 768, 2048, [1, 2], None),
                                           (8, 7, 256, [7, 6, 5, 4, 3, 2, 1, 0, 7], None),
                                           (12, 40, 512, [11, 0, 5], dict(ctas=2, chunk_rows=3, chunks=2))])
def test_moe_q4k_dp4a_matches_oracle(q, e, n, k, ids, cfg):
    st = synth.Stream(e * n + k + 2)
    bank = synth.gen_q4k_rows(st, e * n, k)
    x = synth.gen_normal(st, len(ids) * k).reshape(len(ids), k)
    y, oq, os_ = _moe_dp4a_run(q, bank, x, ids, n, k, e, cfg=cfg)
    ref = oracle.moe_qmv_q4k_dp4a(bank, oq, os_, np.array(ids, dtype=np.int32), n, k, e)
    for s in range(len(ids)):
        assert scale_rel(ref[s], y[s]) <= SCALE_REL_TOL


def test_moe_variants_bad_ids_give_nan_and_status(q):
    e, n, k = 4, 16, 256
    st = synth.Stream(61)
    bank4 = synth.gen_q4k_rows(st, e * n, k)
    bank6 = synth.gen_q6k_rows(st, e * n, k)
    x = synth.gen_normal(st, 4 * k).reshape(4, k)
    ids = [1, 4, -1, 2]
    q.qmv_device_status(clear=True)
    y6 = moe6_run(q, bank6, x, ids, n, k, e)
    assert np.all(np.isnan(y6[1])) and np.all(np.isnan(y6[2])) and not np.any(np.isnan(y6[0]))
    assert q.qmv_device_status(clear=True) & q.QMV_STATUS_BAD_EXPERT_ID
    y4, _, _ = _moe_dp4a_run(q, bank4, x, ids, n, k, e)
    assert np.all(np.isnan(y4[1])) and np.all(np.isnan(y4[2])) and not np.any(np.isnan(y4[3]))
    assert q.qmv_device_status(clear=True) & q.QMV_STATUS_BAD_EXPERT_ID
    assert q.qmv_device_status(clear=True) == 0


def test_full_moe_q6k(q):
    c = synth.make_config("moe_q6k_e128_n2048_k768_s8")
    y = moe6_run(q, c["w"], c["x"], c["ids"], 2048, 768, 128)
    ref = oracle.moe_qmv("q6k", c["w"], c["x"], c["ids"], 2048, 768, 128)
    assert scale_rel(ref, y) <= SCALE_REL_TOL


def test_full_moe_q4k_dp4a(q):
    c = synth.make_config("moe_q4k_dp4a_e128_n768_k2048_s8")
    y, oq, os_ = _moe_dp4a_run(q, c["w"], c["x"], c["ids"], 768, 2048, 128)
    ref = oracle.moe_qmv_q4k_dp4a(c["w"], oq, os_, c["ids"], 768, 2048, 128)
    assert scale_rel(ref, y) <= SCALE_REL_TOL


# ----------------------------------------------------------- argument errors

def test_argument_errors(q):
    w = torch.zeros(144 * 4 + 16, dtype=torch.uint8, device="cuda")
    x = torch.zeros(512, dtype=torch.float32, device="cuda")
    y = torch.zeros(8, dtype=torch.float32, device="cuda")
    assert q.qmv_q4k(w, x, y, 2, 300, check=False) == q.QMV_EINVAL
    assert q.qmv_q4k(w, x, y, 0, 256, check=False) == q.QMV_EINVAL
    assert q.qmv_q4k(None, x, y, 2, 256, check=False) == q.QMV_EINVAL
    assert q.qmv_q4k(w.data_ptr() + 2, x, y, 2, 256, check=False) == q.QMV_EALIGN
    assert q.qmv_q8_0(w, x, y, 2, 48, check=False) == q.QMV_EINVAL
    ids = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert q.moe_qmv_q4k(w, x, y, 2, 256, ids, 0, 2, check=False) == q.QMV_EINVAL
    assert q.moe_qmv_q4k(w, x, y, 2, 256, ids, 2, 0, check=False) == q.QMV_EINVAL
    assert q.quantize_act_q8(x, w, y, None, 1, 40, check=False) == q.QMV_EINVAL
    assert q.qmv_q8_dp4a(w, w.data_ptr() + 4, y, y, 2, 32, check=False) == q.QMV_EALIGN


# ------------------------------------------------- full-size workloads

def _full(q, name):
    c = synth.make_config(name)
    return c


def test_full_q4k_4096(q):
    c = synth.make_config("q4k_4096x4096")
    y = run_matvec(q, "q4k", c["w"], c["x"], 4096, 4096)
    assert scale_rel(oracle.qmv("q4k", c["w"], c["x"], 4096, 4096), y) <= SCALE_REL_TOL


def test_full_q4k_256(q):
    c = synth.make_config("q4k_256x1024")
    y = run_matvec(q, "q4k", c["w"], c["x"], 256, 1024)
    assert scale_rel(oracle.qmv("q4k", c["w"], c["x"], 256, 1024), y) <= SCALE_REL_TOL


def test_full_q6k_4096x14336(q):
    c = synth.make_config("q6k_4096x14336")
    y = run_matvec(q, "q6k", c["w"], c["x"], 4096, 14336)
    assert scale_rel(oracle.qmv("q6k", c["w"], c["x"], 4096, 14336), y) <= SCALE_REL_TOL


def test_full_q8_dp4a_14336x4096(q):
    c = synth.make_config("q8_0_dp4a_14336x4096")
    rows, k = 14336, 4096
    xq = torch.empty(k, dtype=torch.int8, device="cuda")
    xs = torch.empty(k // 32, dtype=torch.float32, device="cuda")
    wd = dev(c["w"])
    q.quantize_act_q8(dev(c["x"]), xq, xs, None, 1, k)
    y = torch.empty(rows, dtype=torch.float32, device="cuda")
    q.qmv_q8_dp4a(wd, xq, xs, y, rows, k)
    dots = torch.empty(rows, k // 32, dtype=torch.int32, device="cuda")
    q.qmv_q8_dp4a_blockdots(wd, xq, dots, rows, k)
    oq, os_, _ = oracle.quantize_act_q8(c["x"], 1, k)
    assert np.array_equal(host(xq), oq.reshape(-1)) and np.array_equal(host(xs), os_.reshape(-1))
    assert np.array_equal(host(dots), oracle.q8_blockdots(c["w"], oq.reshape(-1), rows, k))
    ref = oracle.qmv_q8_dp4a(c["w"], oq.reshape(-1), os_.reshape(-1), rows, k)
    assert scale_rel(ref, host(y)) <= SCALE_REL_TOL


def test_full_moe(q):
    c = synth.make_config("moe_q4k_e128_n768_k2048_s8")
    y = moe_run(q, c["w"], c["x"], c["ids"], 768, 2048, 128)
    ref = oracle.moe_qmv("q4k", c["w"], c["x"], c["ids"], 768, 2048, 128)
    assert scale_rel(ref, y) <= SCALE_REL_TOL


# ------------------------------------------------- decode-chain overlap mode

def test_weight_prefetch_chain_matches(q):
    """With programmatic dependent launch enabled, each call streams weights
    while the previous kernel finishes but must still see that kernel's output
    as its input. Run a chain y1 = W1 x, y2 = W2 y1, ... (square matrices,
    every call reading the previous call's output, plus an MoE call reading
    ids written by a torch kernel just before) with and without the overlap:
    the results must be bitwise identical."""
    n = 2048
    st = synth.Stream(77)
    ws = [dev(synth.gen_q4k_rows(st, n, n)) for _ in range(6)]
    w6 = dev(synth.gen_q6k_rows(st, n, n))
    bank = dev(synth.gen_q4k_rows(st, 8 * n, n))
    x0 = dev(synth.gen_normal(st, n) / np.float32(16))

    def chain(ov):
        bufs = [torch.empty(n, device="cuda") for _ in range(8)]
        cur = x0
        for i, w in enumerate(ws):
            q.qmv_q4k(w, cur, bufs[i], n, n, overlap=ov)
            cur = bufs[i]
        q.qmv_q6k(w6, cur, bufs[6], n, n, overlap=ov)
        ids = (torch.arange(2, device="cuda", dtype=torch.int32) * 3 + 1)   # written by a torch kernel
        ym = torch.empty(2, n, device="cuda")
        xm = torch.stack([bufs[6], bufs[5]])
        q.moe_qmv_q4k(bank, xm, ym, n, n, ids, 2, 8, overlap=ov)
        torch.cuda.synchronize()
        return [b.clone() for b in bufs[:7]] + [ym.clone()]

    ref = chain(q.OVERLAP_NONE)
    for _ in range(3):
        got = chain(q.OVERLAP_CHAIN)
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
    assert torch.isfinite(ref[-1]).all()


def test_independent_inputs_mode_matches(q):
    """QMV_OVERLAP_INDEPENDENT (inputs read before the dependency wait): a stream of calls that
    share one activation (like Q, K, V projections), with every output buffer
    reused by the next-but-one call, must give bitwise the results of plain
    launches; the MoE call reads ids written long before."""
    n = 2048
    st = synth.Stream(78)
    ws = [dev(synth.gen_q4k_rows(st, n, n)) for _ in range(5)]
    w6 = dev(synth.gen_q6k_rows(st, n, n))
    bank = dev(synth.gen_q4k_rows(st, 8 * n, n))
    x = dev(synth.gen_normal(st, n))
    xm = dev(synth.gen_normal(st, 2 * n).reshape(2, n))
    ids = dev(np.array([3, 6], dtype=np.int32))
    torch.cuda.synchronize()

    def stream_of_calls(ov):
        bufs = [torch.full((n,), float("nan"), device="cuda") for _ in range(2)]
        outs = []
        for i, w in enumerate(ws):
            q.qmv_q4k(w, x, bufs[i % 2], n, n, overlap=ov)
            outs.append(bufs[i % 2].clone())   # a torch kernel between calls
        q.qmv_q6k(w6, x, bufs[0], n, n, overlap=ov)
        ym = torch.empty(2, n, device="cuda")
        q.moe_qmv_q4k(bank, xm, ym, n, n, ids, 2, 8, overlap=ov)
        torch.cuda.synchronize()
        return outs + [bufs[0].clone(), ym.clone()]

    ref = stream_of_calls(q.OVERLAP_NONE)
    for mode in (2, 1, 2):
        got = stream_of_calls(mode)
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
    assert all(torch.isfinite(t).all() for t in ref)
