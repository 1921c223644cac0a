"""GPU parity of the Q5_K and Q4_0 matvecs and of the MoE matvecs over Q8_0,
Q4_0 and Q5_K banks against the CPU oracle, through the C ABI.

Bars as for the other formats: decoded weights and MoE gathers (x = e_j)
bit-exact; f32 outputs within scale-relative error max|a-b|/max|a| <= 1e-4
of the f64 oracle.
"""

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

SCALE_REL_TOL = 1e-4
PLAN_FMT = {"q5k": 8, "q4_0": 9}
MOE_FMT = ["q8_0", "q4_0", "q5k"]


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
    getattr(q, f"qmv_{fmt}")(dev(w), dev(x), y, rows, k, cfg=cfg)
    return host(y)


def moe_run(q, fmt, bank, x, ids, rows, k, n_experts, cfg=None):
    slots = len(ids)
    y = torch.full((slots, rows), 7.0, dtype=torch.float32, device="cuda")
    getattr(q, f"moe_qmv_{fmt}")(dev(bank), dev(x), y, rows, k, dev(np.asarray(ids, dtype=np.int32)), slots,
                                 n_experts, cfg=cfg)
    return host(y)


def gen(fmt, st, rows, k):
    return synth.GEN_ROWS[fmt](st, rows, k)


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("fmt,rows,k", [("q5k", 37, 512), ("q5k", 3, 2304), ("q4_0", 37, 96), ("q4_0", 3, 4096)])
def test_dequant_bit_exact(q, fmt, rows, k):
    w = gen(fmt, synth.Stream(2000 + rows + k), rows, k)
    out = torch.empty(rows, k, dtype=torch.float32, device="cuda")
    getattr(q, f"qmv_dequant_{fmt}")(dev(w), out, rows, k)
    assert np.array_equal(host(out), oracle.dequant(fmt, w, rows, k).astype(np.float32))


def test_dequant_subnormal_scales(q):
    w5 = synth.gen_q5k_rows(synth.Stream(9), 4, 256, d_range=(0.0, 6e-8), dmin_range=(0.0, 6e-8))
    w0 = synth.gen_q4_0_rows(synth.Stream(10), 4, 64, d_range=(-6e-8, 6e-8))
    o5 = torch.empty(4, 256, dtype=torch.float32, device="cuda")
    o0 = torch.empty(4, 64, dtype=torch.float32, device="cuda")
    q.qmv_dequant_q5k(dev(w5), o5, 4, 256)
    q.qmv_dequant_q4_0(dev(w0), o0, 4, 64)
    assert np.array_equal(host(o5), oracle.dequant("q5k", w5, 4, 256).astype(np.float32))
    assert np.array_equal(host(o0), oracle.dequant("q4_0", w0, 4, 64).astype(np.float32))


# ------------------------------------------------------------------ matvec

SHAPES = [("q5k", 256, 1024), ("q5k", 300, 768), ("q5k", 1, 256), ("q5k", 97, 4352), ("q5k", 20, 16384),
          ("q4_0", 300, 96), ("q4_0", 7, 4096), ("q4_0", 13, 32), ("q4_0", 64, 11008), ("q4_0", 33, 1056),
          ("q4_0", 5, 14336)]


@pytest.mark.parametrize("fmt,rows,k", SHAPES)
def test_matvec_matches_oracle(q, fmt, rows, k):
    st = synth.Stream(rows * 11 + k)
    w = gen(fmt, st, rows, k)
    x = synth.gen_normal(st, k)
    y = run_matvec(q, fmt, w, x, rows, k)
    assert scale_rel(oracle.qmv(fmt, w, x, rows, k), y) <= SCALE_REL_TOL


@pytest.mark.parametrize("cfg", [dict(ctas=1, chunk_rows=1, chunks=2), dict(ctas=3, chunk_rows=5, chunks=2),
                                 dict(ctas=2, chunk_rows=3, chunks=1), dict(ctas=7, chunks=3),
                                 dict(ctas=1, chunks=2, unroll=1), dict(ctas=3, chunk_rows=4, chunks=3, unroll=2),
                                 dict(ctas=2, chunks=1, warps=2), dict(ctas=5, chunk_rows=2, chunks=4, warps=4),
                                 dict(ctas=1, chunk_rows=7, chunks=2, warps=16, unroll=1)])
@pytest.mark.parametrize("fmt", ["q5k", "q4_0"])
def test_matvec_forced_pipelines(q, fmt, cfg):
    rows, k = 61, 512
    st = synth.Stream(19)
    w = gen(fmt, st, rows, k)
    x = synth.gen_normal(st, k)
    y = run_matvec(q, fmt, w, x, rows, k, cfg=cfg)
    assert not np.any(np.isnan(y))
    assert scale_rel(oracle.qmv(fmt, w, x, rows, k), y) <= SCALE_REL_TOL


@pytest.mark.parametrize("cfg", [dict(ctas=1, chunk_rows=3, chunks=2), dict(ctas=2, chunk_rows=1, chunks=1),
                                 dict(ctas=3, chunk_rows=2, chunks=3, unroll=1), dict(ctas=1, chunks=2, warps=16)])
@pytest.mark.parametrize("fmt,k", [("q5k", 4352), ("q4_0", 4096), ("q4_0", 1056)])
def test_matvec_forced_pipelines_wide(q, fmt, k, cfg):
    rows = 29
    st = synth.Stream(k + 9)
    w = gen(fmt, st, rows, k)
    x = synth.gen_normal(st, k)
    y = run_matvec(q, fmt, w, x, rows, k, cfg=cfg)
    assert not np.any(np.isnan(y))
    assert scale_rel(oracle.qmv(fmt, w, x, rows, k), y) <= SCALE_REL_TOL


@pytest.mark.parametrize("cluster", [2, 4])
@pytest.mark.parametrize("fmt,rows,k", [("q5k", 97, 4352), ("q4_0", 64, 1024)])
def test_matvec_cluster_shared_prep(q, fmt, rows, k, cluster):
    st = synth.Stream(k + cluster + 1)
    w = gen(fmt, st, rows, k)
    x = synth.gen_normal(st, k)
    cfg = dict(ctas=8, cluster=cluster)
    assert q.qmv_plan_info(PLAN_FMT[fmt], rows, k, cfg=cfg)["ctas"] % cluster == 0
    y = run_matvec(q, fmt, w, x, rows, k, cfg=cfg)
    y1 = run_matvec(q, fmt, w, x, rows, k, cfg=dict(ctas=8))
    assert scale_rel(oracle.qmv(fmt, w, x, rows, k), y) <= SCALE_REL_TOL
    assert np.array_equal(y, y1)


@pytest.mark.parametrize("fmt,rows,k", [("q5k", 64, 1024), ("q5k", 9, 16384), ("q4_0", 40, 256),
                                        ("q4_0", 9, 4096)])
def test_unit_vector_is_exact(q, fmt, rows, k):
    """x = e_j: y[r] must be the decoded weight W[r, j] bit for bit (every
    code position, both nibbles and, for Q5_K, every fifth-bit position)."""
    st = synth.Stream(29)
    w = gen(fmt, st, rows, k)
    W = oracle.dequant(fmt, w, rows, k).astype(np.float32)
    cols = {0, 1, 15, 16, 17, 31, 32, 33, 63, 64, 100, 127, 128, 200, 255, k // 2 + 3, k - 1}
    for j in sorted(c for c in cols if c < k):
        e = np.zeros(k, dtype=np.float32)
        e[j] = 1.0
        y = run_matvec(q, fmt, w, e, rows, k)
        assert np.array_equal(y, W[:, j]), f"column {j}"


def test_q5k_every_fifth_bit_position(q):
    """All 256 positions of a super-block with the fifth bit forced on, then
    off: each column equals the decoded weight exactly."""
    rows, k = 8, 256
    w = synth.gen_q5k_rows(synth.Stream(31), rows, k)
    for fill in (0xFF, 0x00):
        w2 = w.copy()
        w2[:, 16:48] = fill
        W = oracle.dequant("q5k", w2, rows, k).astype(np.float32)
        for j in range(0, 256, 3):
            e = np.zeros(k, dtype=np.float32)
            e[j] = 1.0
            assert np.array_equal(run_matvec(q, "q5k", w2, e, rows, k), W[:, j]), (fill, j)


def test_matvec_extreme_activations(q):
    for fmt, k in (("q5k", 1024), ("q4_0", 1024)):
        rows = 33
        st = synth.Stream(43)
        w = gen(fmt, st, rows, k)
        x = synth.gen_normal(st, k)
        x[0:32] = 0.0
        x[32:64] *= np.float32(1e-30)
        x[64:96] *= np.float32(1e30)
        x[96:128] = np.float32(1e-40)
        x[200] = np.float32(1e36)
        y = run_matvec(q, fmt, w, x, rows, k)
        assert scale_rel(oracle.qmv(fmt, w, x, rows, k), y) <= SCALE_REL_TOL, fmt


# --------------------------------------------------------------------- MoE

@pytest.mark.parametrize("fmt", MOE_FMT)
@pytest.mark.parametrize("e,n,k,ids,cfg", [(16, 96, 512, [3, 15, 0, 3], None), (4, 768, 512, [1, 2], None),
                                           (8, 7, 256, [7, 6, 5, 4, 3, 2, 1, 0, 7], None),
                                           (6, 40, 768, [5, 1, 1], dict(ctas=2, chunk_rows=3, chunks=2))])
def test_moe_matches_oracle(q, fmt, e, n, k, ids, cfg):
    st = synth.Stream(e * n + k + 3)
    bank = gen(fmt, st, e * n, k)
    x = synth.gen_normal(st, len(ids) * k).reshape(len(ids), k)
    y = moe_run(q, fmt, bank, x, ids, n, k, e, cfg=cfg)
    ref = oracle.moe_qmv(fmt, bank, x, np.array(ids, dtype=np.int32), n, k, e)
    for s in range(len(ids)):
        assert scale_rel(ref[s], y[s]) <= SCALE_REL_TOL


@pytest.mark.parametrize("fmt", MOE_FMT)
def test_moe_gather_exact(q, fmt):
    """x[s] = e_j in every slot: y[s] is column j of expert ids[s] exactly."""
    e, n, k = 10, 24, 512
    bank = gen(fmt, synth.Stream(47), e * n, k)
    W = oracle.dequant(fmt, bank, e * n, k).reshape(e, n, k).astype(np.float32)
    ids = [9, 0, 4, 4]
    for j in [0, 100, 511]:
        x = np.zeros((len(ids), k), dtype=np.float32)
        x[:, j] = 1.0
        y = moe_run(q, fmt, bank, x, ids, n, k, e, cfg=dict(ctas=2, chunk_rows=3, chunks=2))
        for s, eid in enumerate(ids):
            assert np.array_equal(y[s], W[eid, :, j])


@pytest.mark.parametrize("fmt", MOE_FMT)
def test_moe_bad_ids_give_nan_and_status(q, fmt):
    e, n, k = 4, 16, 256
    st = synth.Stream(63)
    bank = gen(fmt, st, e * n, k)
    x = synth.gen_normal(st, 4 * k).reshape(4, k)
    q.qmv_device_status(clear=True)
    y = moe_run(q, fmt, bank, x, [1, 4, -1, 2], n, k, e)
    assert np.all(np.isnan(y[1])) and np.all(np.isnan(y[2]))
    ref = oracle.moe_qmv(fmt, bank, x, np.array([1, 0, 0, 2], dtype=np.int32), n, k, e)
    assert scale_rel(ref[0], y[0]) <= SCALE_REL_TOL and scale_rel(ref[3], y[3]) <= SCALE_REL_TOL
    assert q.qmv_device_status(clear=True) & q.QMV_STATUS_BAD_EXPERT_ID
    assert q.qmv_device_status(clear=True) == 0


# ------------------------------------------------- full-size workloads

@pytest.mark.parametrize("name,fmt", [("q5k_4096x4096", "q5k"), ("q4_0_4096x4096", "q4_0")])
def test_full_dense(q, name, fmt):
    c = synth.make_config(name)
    y = run_matvec(q, fmt, c["w"], c["x"], c["rows"], c["k"])
    assert scale_rel(oracle.qmv(fmt, c["w"], c["x"], c["rows"], c["k"]), y) <= SCALE_REL_TOL


@pytest.mark.parametrize("fmt", MOE_FMT)
def test_full_moe(q, fmt):
    c = synth.make_config(f"moe_{fmt}_e128_n768_k2048_s8")
    y = moe_run(q, fmt, c["w"], c["x"], c["ids"], 768, 2048, 128)
    ref = oracle.moe_qmv(fmt, c["w"], c["x"], c["ids"], 768, 2048, 128)
    assert scale_rel(ref, y) <= SCALE_REL_TOL


# ------------------------------------------------- decode-chain overlap modes

def test_overlap_modes_give_identical_results(q):
    """The chain and independent overlaps change only when a call waits for the
    previous kernel: back-to-back calls of every new entry point give the
    plain-launch results bit
    for bit (inputs written before the chain, none shared with an output)."""
    st = synth.Stream(71)
    cases = []
    for fmt, rows, k in (("q5k", 300, 2048), ("q4_0", 300, 2048)):
        cases.append(("dense", fmt, dev(gen(fmt, st, rows, k)), dev(synth.gen_normal(st, k)), rows, k))
    ids = dev(np.array([3, 0, 5, 3], dtype=np.int32))
    for fmt in MOE_FMT:
        cases.append(("moe", fmt, dev(gen(fmt, st, 6 * 96, 512)), dev(synth.gen_normal(st, 4 * 512)), 96, 512))

    def chain(ov):
        outs = []
        for kind, fmt, w, x, rows, k in cases:
            if kind == "dense":
                y = torch.empty(rows, dtype=torch.float32, device="cuda")
                getattr(q, f"qmv_{fmt}")(w, x, y, rows, k, overlap=ov)
            else:
                y = torch.empty(4, rows, dtype=torch.float32, device="cuda")
                getattr(q, f"moe_qmv_{fmt}")(w, x, y, rows, k, ids, 4, 6, overlap=ov)
            outs.append(y)
        torch.cuda.synchronize()
        return [o.cpu().numpy() for o in outs]

    base = chain(q.OVERLAP_NONE)
    for mode in (q.OVERLAP_CHAIN, q.OVERLAP_INDEPENDENT):
        for a, b in zip(base, chain(mode)):
            assert np.array_equal(a, b), mode
