"""The activation quantization and the Q8_0 dp4a matvec in one launch
(qmv_q8_dp4a_quant), against the two separate entry points and the oracle:
the in-kernel codes are the standalone quantizer's bit for bit, so the output
equals quantize_act_q8 + qmv_q8_dp4a exactly (same plan family, same dot and
reduction order) and is within scale-relative 1e-4 of the f64 oracle fed the
oracle's codes."""

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


def scale_rel(ref, got):
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    return float(np.max(np.abs(ref - got)) / max(float(np.max(np.abs(ref))), 1e-30))


def separate(q, wd, xd, rows, k, overlap=0):
    xq = torch.empty(k, dtype=torch.int8, device="cuda")
    xs = torch.empty(k // 32, dtype=torch.float32, device="cuda")
    q.quantize_act_q8(xd, xq, xs, None, 1, k)
    y = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    q.qmv_q8_dp4a(wd, xq, xs, y, rows, k, overlap=overlap)
    return y


def fused(q, wd, xd, rows, k, overlap=0, cfg=None):
    y = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    q.qmv_q8_dp4a_quant(wd, xd, y, rows, k, overlap=overlap, cfg=cfg)
    return y


@pytest.mark.parametrize("rows,k", [(300, 4096), (37, 96), (5, 32), (129, 1376), (64, 8192), (17, 16384),
                                    (1, 4096), (1000, 512)])
def test_fused_equals_separate_and_oracle(q, rows, k):
    st = synth.Stream(rows * 7 + k)
    w = synth.gen_q8_0_rows(st, rows, k)
    x = synth.gen_normal(st, k)
    wd, xd = dev(w), dev(x)
    ys = separate(q, wd, xd, rows, k)
    yf = fused(q, wd, xd, rows, k)
    torch.cuda.synchronize()
    assert torch.equal(ys, yf)
    oq, os_, _ = oracle.quantize_act_q8(x, 1, k)
    ref = oracle.qmv_q8_dp4a(w, oq.reshape(-1), os_.reshape(-1), rows, k)
    assert scale_rel(ref, yf.cpu().numpy()) <= SCALE_REL_TOL


def test_fused_quantizer_edge_blocks(q):
    """Zero blocks (d = 0), blocks with a single large value, tiny and huge
    magnitudes, and exact half-way products (amax = 127 makes inv = 1, so x =
    k + 0.5 rounds to even): the fused codes equal the standalone ones, so the
    two outputs agree bit for bit."""
    rows, k = 96, 1024
    st = synth.Stream(4711)
    w = synth.gen_q8_0_rows(st, rows, k)
    x = synth.gen_normal(st, k).astype(np.float32)
    x[0:32] = 0.0
    x[32:64] = 0.0
    x[40] = 3.0e4
    x[64:96] *= np.float32(1e-30)
    x[96:128] *= np.float32(1e30)
    x[128:160] = np.arange(32, dtype=np.float32) - np.float32(15.5)
    x[159] = 127.0
    wd, xd = dev(w), dev(x)
    ys = separate(q, wd, xd, rows, k)
    yf = fused(q, wd, xd, rows, k)
    torch.cuda.synchronize()
    assert torch.equal(ys, yf)


@pytest.mark.parametrize("mode", [1, 2])
def test_fused_overlap_modes(q, mode):
    """The chain and independent overlaps give the plain-launch bits."""
    rows, k = 2048, 4096
    st = synth.Stream(990 + mode)
    ws = [dev(synth.gen_q8_0_rows(st, rows, k)) for _ in range(3)]
    xd = dev(synth.gen_normal(st, k))
    base = [fused(q, w, xd, rows, k) for w in ws]
    got = [fused(q, w, xd, rows, k, overlap=mode) for w in ws]
    torch.cuda.synchronize()
    for a, b in zip(base, got):
        assert torch.equal(a, b)


def test_fused_full_c2(q):
    """The configured dp4a workload (Q8_0 14336 x 4096, seed 2) in one launch."""
    c = synth.make_config("q8_0_dp4a_14336x4096")
    rows, k = 14336, 4096
    wd, xd = dev(c["w"]), dev(c["x"])
    ys = separate(q, wd, xd, rows, k)
    yf = fused(q, wd, xd, rows, k)
    torch.cuda.synchronize()
    assert torch.equal(ys, yf)
    oq, os_, _ = oracle.quantize_act_q8(c["x"], 1, k)
    ref = oracle.qmv_q8_dp4a(c["w"], oq.reshape(-1), os_.reshape(-1), rows, k)
    assert scale_rel(ref, yf.cpu().numpy()) <= SCALE_REL_TOL
    assert q.qmv_device_status(clear=True) == 0


@pytest.mark.parametrize("xoff,qoff", [(0, 0), (1, 0), (0, 3), (3, 5)])
def test_quantizer_alignments(q, xoff, qoff):
    """quantize_act_q8 with x and xq at 4-byte / 1-byte offsets from a
    16-byte boundary (the element-wise path) and aligned (the vector path):
    codes, scales and sums equal the oracle's bit for bit."""
    m, k = 3, 1024
    st = synth.Stream(31 + xoff + 7 * qoff)
    x = synth.gen_normal(st, m * k).astype(np.float32)
    xbuf = torch.zeros(m * k + 8, dtype=torch.float32, device="cuda")
    xbuf[xoff:xoff + m * k] = torch.from_numpy(x).cuda()
    qbuf = torch.zeros(m * k + 32, dtype=torch.int8, device="cuda")
    xs = torch.empty(m * k // 32, dtype=torch.float32, device="cuda")
    xsum = torch.empty(m * k // 32, dtype=torch.float32, device="cuda")
    q.quantize_act_q8(xbuf.data_ptr() + 4 * xoff, qbuf.data_ptr() + qoff, xs, xsum, m, k)
    torch.cuda.synchronize()
    oq, os_, osum = oracle.quantize_act_q8(x, m, k)
    assert np.array_equal(qbuf.cpu().numpy()[qoff:qoff + m * k], oq.reshape(-1))
    assert np.array_equal(xs.cpu().numpy(), os_.reshape(-1))
    assert np.array_equal(xsum.cpu().numpy(), osum.reshape(-1))
