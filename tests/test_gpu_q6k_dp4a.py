"""GPU parity of the Q6_K x int8-activation (dp4a) path -- qmv_q6k_dp4a,
qmv_q6k_dp4a_blockdots and moe_qmv_q6k_dp4a -- against the CPU oracle, through
the C ABI. Bars: the int32 group dots bit-exact, the quantized activation
bit-exact, f32 outputs within scale-relative 1e-4 of the f64 oracle on the
same codes."""

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

SCALE_REL_TOL = 1e-4


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


def quantized(q, x, m, k):
    """x quantized on the device, checked bit-exact against the oracle's
    quantizer; returns (device codes, device scales, oracle codes, oracle scales)."""
    xq = torch.empty(m * k, dtype=torch.int8, device="cuda")
    xs = torch.empty(m * (k // 32), dtype=torch.float32, device="cuda")
    q.quantize_act_q8(dev(x), xq, xs, None, m, k)
    oq, os_, _ = oracle.quantize_act_q8(x, m, k)
    assert np.array_equal(host(xq), oq.reshape(-1)) and np.array_equal(host(xs), os_.reshape(-1))
    return xq, xs, oq, os_


@pytest.mark.parametrize("rows,k,cfg", [(300, 4096, None), (61, 512, None), (1, 256, None), (41, 14336, None),
                                        (130, 2816, None), (61, 512, dict(ctas=2, chunk_rows=3, chunks=2)),
                                        (29, 2816, dict(ctas=1, chunk_rows=3, chunks=2)),
                                        (61, 512, dict(ctas=1, chunks=2, unroll=1))])
def test_q6k_dp4a_matvec(q, rows, k, cfg):
    st = synth.Stream(rows * 3 + k)
    w = synth.gen_q6k_rows(st, rows, k)
    x = synth.gen_normal(st, k)
    xq, xs, oq, os_ = quantized(q, x, 1, k)
    y = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    q.qmv_q6k_dp4a(dev(w), xq, xs, y, rows, k, cfg=cfg)
    ref = oracle.qmv_q6k_dp4a(w, oq.reshape(-1), os_.reshape(-1), rows, k)
    assert scale_rel(ref, host(y)) <= SCALE_REL_TOL


@pytest.mark.parametrize("rows,k", [(300, 4096), (7, 256), (33, 2816)])
def test_q6k_dp4a_groupdots_bit_exact(q, rows, k):
    st = synth.Stream(rows + k + 7)
    w = synth.gen_q6k_rows(st, rows, k)
    x = synth.gen_normal(st, k)
    xq, _, oq, _ = quantized(q, x, 1, k)
    dots = torch.full((rows, k // 16), -7, dtype=torch.int32, device="cuda")
    q.qmv_q6k_dp4a_blockdots(dev(w), xq, dots, rows, k)
    assert np.array_equal(host(dots), oracle.q6k_dp4a_groupdots(w, oq.reshape(-1), rows, k))


def _moe(q, bank, x, ids, rows, k, e, cfg=None):
    slots = len(ids)
    xq, xs, oq, os_ = quantized(q, x, slots, k)
    y = torch.full((slots, rows), 7.0, dtype=torch.float32, device="cuda")
    q.moe_qmv_q6k_dp4a(dev(bank), xq, xs, y, rows, k, dev(np.asarray(ids, dtype=np.int32)), slots, e, cfg=cfg)
    return host(y), oq, os_


@pytest.mark.parametrize("e,n,k,ids,cfg", [(16, 96, 512, [3, 15, 0, 3], None), (8, 257, 768, [1, 2], None),
                                           (8, 7, 256, [7, 6, 5, 4, 3, 2, 1, 0, 7], None),
                                           (6, 40, 768, [5, 1, 1], dict(ctas=2, chunk_rows=3, chunks=2))])
def test_moe_q6k_dp4a_matches_oracle(q, e, n, k, ids, cfg):
    st = synth.Stream(e * n + k + 9)
    bank = synth.gen_q6k_rows(st, e * n, k)
    x = synth.gen_normal(st, len(ids) * k).reshape(len(ids), k)
    y, oq, os_ = _moe(q, bank, x, ids, n, k, e, cfg)
    ref = oracle.moe_qmv_q6k_dp4a(bank, oq, os_, np.array(ids, dtype=np.int32), n, k, e)
    for s in range(len(ids)):
        assert scale_rel(ref[s], y[s]) <= SCALE_REL_TOL


def test_moe_q6k_dp4a_bad_ids_give_nan_and_status(q):
    e, n, k = 4, 16, 256
    st = synth.Stream(65)
    bank = synth.gen_q6k_rows(st, e * n, k)
    x = synth.gen_normal(st, 4 * k).reshape(4, k)
    q.qmv_device_status(clear=True)
    y, oq, os_ = _moe(q, bank, x, [1, 4, -1, 2], n, k, e)
    assert np.all(np.isnan(y[1])) and np.all(np.isnan(y[2]))
    ref = oracle.moe_qmv_q6k_dp4a(bank, oq, os_, np.array([1, 0, 0, 2], dtype=np.int32), n, k, e)
    assert scale_rel(ref[0], y[0]) <= SCALE_REL_TOL and scale_rel(ref[3], y[3]) <= SCALE_REL_TOL
    assert q.qmv_device_status(clear=True) & q.QMV_STATUS_BAD_EXPERT_ID
    assert q.qmv_device_status(clear=True) == 0


def test_q6k_dp4a_argument_errors(q):
    w = torch.zeros(210 * 4 + 16, dtype=torch.uint8, device="cuda")
    xq = torch.zeros(512, dtype=torch.int8, device="cuda")
    xs = torch.zeros(16, dtype=torch.float32, device="cuda")
    y = torch.zeros(8, dtype=torch.float32, device="cuda")
    assert q.qmv_q6k_dp4a(w, xq, xs, y, 2, 300, check=False) == q.QMV_EINVAL
    assert q.qmv_q6k_dp4a(w, xq.data_ptr() + 4, xs, y, 2, 256, check=False) == q.QMV_EALIGN
    assert q.qmv_q6k_dp4a(w, xq, None, y, 2, 256, check=False) == q.QMV_EINVAL
    ids = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert q.moe_qmv_q6k_dp4a(w, xq, xs, y, 2, 256, ids, 0, 2, check=False) == q.QMV_EINVAL


def test_full_q6k_dp4a_4096x14336(q):
    c = synth.make_config("q6k_dp4a_4096x14336")
    rows, k = c["rows"], c["k"]
    xq, xs, oq, os_ = quantized(q, c["x"], 1, k)
    wd = dev(c["w"])
    y = torch.empty(rows, dtype=torch.float32, device="cuda")
    q.qmv_q6k_dp4a(wd, xq, xs, y, rows, k)
    ref = oracle.qmv_q6k_dp4a(c["w"], oq.reshape(-1), os_.reshape(-1), rows, k)
    assert scale_rel(ref, host(y)) <= SCALE_REL_TOL
    # the integer dots of a sample of rows, bit-exact
    dots = torch.empty(rows, k // 16, dtype=torch.int32, device="cuda")
    q.qmv_q6k_dp4a_blockdots(wd, xq, dots, rows, k)
    sample = np.arange(0, rows, 97)
    want = oracle.q6k_dp4a_groupdots(c["w"][sample], oq.reshape(-1), len(sample), k)
    assert np.array_equal(host(dots)[sample], want)


def test_full_moe_q6k_dp4a(q):
    c = synth.make_config("moe_q6k_dp4a_e128_n2048_k768_s8")
    y, oq, os_ = _moe(q, c["w"], c["x"], c["ids"], 2048, 768, 128)
    ref = oracle.moe_qmv_q6k_dp4a(c["w"], oq, os_, c["ids"], 2048, 768, 128)
    assert scale_rel(ref, y) <= SCALE_REL_TOL
