"""The largest row length every matvec entry point takes (sixteen warps of
k-slices), one row past it (refused on the host with QMV_ETOOBIG, nothing
launched), degenerate MoE shapes, and batched products over rows of 65536
weights, through the C ABI against the oracle."""

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

SCALE_REL_TOL = 1e-4

# (entry, format, largest k): units per row <= 16 warps x 32 lanes
F32_MAX = [("qmv_q4k", "q4k", 32768), ("qmv_q6k", "q6k", 32768), ("qmv_q8_0", "q8_0", 16384),
           ("qmv_q5k", "q5k", 32768), ("qmv_q4_0", "q4_0", 16384)]
DP4A_MAX = [("qmv_q8_dp4a", "q8_0", 65536), ("qmv_q4k_dp4a", "q4k", 32768), ("qmv_q6k_dp4a", "q6k", 32768)]
STEP = {"q4k": 256, "q6k": 256, "q5k": 256, "q8_0": 32, "q4_0": 32}


@pytest.fixture(scope="module")
def q():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    import ggml_format_dequant_gb300 as lib
    return lib


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def scale_rel(ref, got):
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    return float(np.max(np.abs(ref - got)) / max(float(np.max(np.abs(ref))), 1e-30))


@pytest.mark.parametrize("entry,fmt,kmax", F32_MAX)
def test_f32_largest_k_and_one_block_more(q, entry, fmt, kmax):
    rows = 9
    st = synth.Stream(kmax + 1)
    w = synth.GEN_ROWS[fmt](st, rows, kmax)
    x = synth.gen_normal(st, kmax)
    y = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    getattr(q, entry)(dev(w), dev(x), y, rows, kmax)
    torch.cuda.synchronize()
    assert scale_rel(oracle.qmv(fmt, w, x, rows, kmax), y.cpu().numpy()) <= SCALE_REL_TOL
    k2 = kmax + STEP[fmt]
    w2 = torch.zeros(rows * (k2 // oracle.QK[fmt]) * oracle.BLOCK_BYTES[fmt] + 16, dtype=torch.uint8, device="cuda")
    x2 = torch.zeros(k2, dtype=torch.float32, device="cuda")
    assert getattr(q, entry)(w2, x2, y, rows, k2, check=False) == q.QMV_ETOOBIG


@pytest.mark.parametrize("entry,fmt,kmax", DP4A_MAX)
def test_dp4a_largest_k(q, entry, fmt, kmax):
    rows = 5
    st = synth.Stream(kmax + 3)
    w = synth.GEN_ROWS[fmt](st, rows, kmax)
    x = synth.gen_normal(st, kmax)
    xq = torch.empty(kmax, dtype=torch.int8, device="cuda")
    xs = torch.empty(kmax // 32, dtype=torch.float32, device="cuda")
    q.quantize_act_q8(dev(x), xq, xs, None, 1, kmax)
    oq, os_, _ = oracle.quantize_act_q8(x, 1, kmax)
    y = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    getattr(q, entry)(dev(w), xq, xs, y, rows, kmax)
    torch.cuda.synchronize()
    ref = {"q8_0": oracle.qmv_q8_dp4a, "q4k": oracle.qmv_q4k_dp4a, "q6k": oracle.qmv_q6k_dp4a}[fmt](
        w, oq.reshape(-1), os_.reshape(-1), rows, kmax)
    assert scale_rel(ref, y.cpu().numpy()) <= SCALE_REL_TOL


@pytest.mark.parametrize("slots,ids", [(1, [0]), (3, [0, 0, 0])])
def test_moe_single_expert_bank(q, slots, ids):
    """A bank of one expert, one slot or every slot on it."""
    e, n, k = 1, 33, 512
    st = synth.Stream(7 + slots)
    bank = synth.gen_q4k_rows(st, e * n, k)
    x = synth.gen_normal(st, slots * k).reshape(slots, k)
    y = torch.full((slots, n), 7.0, dtype=torch.float32, device="cuda")
    q.moe_qmv_q4k(dev(bank), dev(x), y, n, k, dev(np.array(ids, dtype=np.int32)), slots, e)
    torch.cuda.synchronize()
    ref = oracle.moe_qmv("q4k", bank, x, np.array(ids, dtype=np.int32), n, k, e)
    for s in range(slots):
        assert scale_rel(ref[s], y[s].cpu().numpy()) <= SCALE_REL_TOL


@pytest.mark.parametrize("fmt", ["q4k", "q6k", "q8_0", "q5k", "q4_0"])
@pytest.mark.parametrize("m,mode", [(3, 0), (8, 0), (8, 2)])
def test_batch_long_rows(q, fmt, m, mode):
    """The batched product has no row-length limit: 65536 weights a row run as
    16 k-chunks of 16 slices (32 of 8 for independent calls) inside one
    launch, against the oracle."""
    rows, k = 40, 65536
    st = synth.Stream(777 + m)
    w = synth.GEN_ROWS[fmt](st, rows, k)
    x = synth.gen_normal(st, m * k).reshape(m, k)
    y = torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda")
    getattr(q, f"qmm_{fmt}")(dev(w), dev(x), y, rows, k, m, overlap=mode)
    torch.cuda.synchronize()
    ref = oracle.qmm(fmt, w, x, m, rows, k)
    got = y.cpu().numpy()
    assert not np.any(np.isnan(got))
    for i in range(m):
        assert scale_rel(ref[i], got[i]) <= SCALE_REL_TOL, i
