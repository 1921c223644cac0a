"""Seeded random shapes and launch configurations for every matvec family,
against the oracle: rows, k and the forced plan (CTAs, rows per slot, ring
depth, unroll, warps) drawn from a fixed stream, so the same cases run every
time."""

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

SCALE_REL_TOL = 1e-4
FAMILIES = ["q4k", "q6k", "q8_0", "q5k", "q4_0", "q8d", "q4d", "q6d"]
QK = {"q4k": 256, "q6k": 256, "q8_0": 32, "q5k": 256, "q4_0": 32, "q8d": 32, "q4d": 256, "q6d": 256}
FMT = {"q8d": "q8_0", "q4d": "q4k", "q6d": "q6k"}


def cases(n=6):
    out = []
    z = synth.Stream(4242).draw(len(FAMILIES) * n * 8).reshape(len(FAMILIES), n, 8)
    for fi, fam in enumerate(FAMILIES):
        for ci in range(n):
            d = [int(v >> np.uint64(33)) for v in z[fi, ci]]
            nb_max = 8192 // QK[fam]
            nb = 1 + d[0] % nb_max
            rows = 1 + d[1] % 200
            cfg = None
            if d[2] % 2:
                cfg = dict(ctas=1 + d[3] % 9, chunk_rows=d[4] % 6, chunks=d[5] % 4, unroll=d[6] % 3,
                           warps=[0, 4, 8, 16][d[7] % 4])
            out.append((fam, rows, nb * QK[fam], cfg))
    return out


@pytest.fixture(scope="module")
def q():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    import ggml_format_dequant_gb300 as lib
    return lib


@pytest.mark.parametrize("fam,rows,k,cfg", cases())
def test_random_shape(q, fam, rows, k, cfg):
    fmt = FMT.get(fam, fam)
    st = synth.Stream(rows * 131 + k)
    w = synth.GEN_ROWS[fmt](st, rows, k)
    x = synth.gen_normal(st, k)
    wd = torch.from_numpy(w).cuda()
    y = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    if fam in FMT:
        xq = torch.empty(k, dtype=torch.int8, device="cuda")
        xs = torch.empty(k // 32, dtype=torch.float32, device="cuda")
        q.quantize_act_q8(torch.from_numpy(x).cuda(), xq, xs, None, 1, k)
        oq, os_, _ = oracle.quantize_act_q8(x, 1, k)
        entry = {"q8d": q.qmv_q8_dp4a, "q4d": q.qmv_q4k_dp4a, "q6d": q.qmv_q6k_dp4a}[fam]
        rc = entry(wd, xq, xs, y, rows, k, cfg=cfg, check=False)
        ref = {"q8d": oracle.qmv_q8_dp4a, "q4d": oracle.qmv_q4k_dp4a, "q6d": oracle.qmv_q6k_dp4a}[fam](
            w, oq.reshape(-1), os_.reshape(-1), rows, k)
    else:
        rc = getattr(q, f"qmv_{fam}")(wd, torch.from_numpy(x).cuda(), y, rows, k, cfg=cfg, check=False)
        ref = oracle.qmv(fam, w, x, rows, k)
    if rc == q.QMV_ETOOBIG:
        # a forced plan that cannot hold the rows it was given: refused on the
        # host, nothing launched
        assert cfg is not None
        return
    assert rc == q.QMV_OK, q.strerror(rc)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    assert not np.any(np.isnan(got))
    assert float(np.max(np.abs(ref - got)) / max(np.max(np.abs(ref)), 1e-30)) <= SCALE_REL_TOL


# ------------------------------------------------ small-M batched products

BATCH_FMTS = ["q4k", "q6k", "q8_0", "q5k", "q4_0"]


def batch_cases(n=8):
    """(fmt, rows, k, m, cfg, mode) drawn from a fixed stream: k up to 16384
    weights (several k-chunks), m = 2..12 (one or two tiles of x rows), a forced
    plan half of the time, and the plain or independent-call launch mode."""
    out = []
    z = synth.Stream(5151).draw(len(BATCH_FMTS) * n * 8).reshape(len(BATCH_FMTS), n, 8)
    for fi, fmt in enumerate(BATCH_FMTS):
        qk = QK[fmt]
        for ci in range(n):
            d = [int(v >> np.uint64(33)) for v in z[fi, ci]]
            k = (1 + d[0] % (16384 // qk)) * qk
            rows = 1 + d[1] % 160
            m = 2 + d[2] % 11
            cfg = None
            if d[3] % 2:
                cfg = dict(ctas=1 + d[4] % 9, chunk_rows=d[5] % 20, chunks=d[6] % 4, warps=[0, 1, 3, 8][d[7] % 4])
            mode = 2 if d[7] % 3 == 0 else 0
            out.append((fmt, rows, k, m, cfg, mode))
    return out


@pytest.mark.parametrize("fmt,rows,k,m,cfg,mode", batch_cases())
def test_random_batch(q, fmt, rows, k, m, cfg, mode):
    st = synth.Stream(rows * 17 + k + m)
    w = synth.GEN_ROWS[fmt](st, rows, k)
    x = synth.gen_normal(st, m * k).reshape(m, k)
    y = torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda")
    rc = getattr(q, f"qmm_{fmt}")(torch.from_numpy(w).cuda(), torch.from_numpy(x).cuda(), y, rows, k, m,
                                  cfg=cfg, overlap=mode, check=False)
    torch.cuda.synchronize()
    if rc == q.QMV_ETOOBIG:
        assert cfg is not None   # a forced plan refused on the host, nothing launched
        return
    assert rc == q.QMV_OK, q.strerror(rc)
    ref = oracle.qmm(fmt, w, x, m, rows, k)
    got = y.cpu().numpy().astype(np.float64)
    assert not np.any(np.isnan(got))
    for i in range(m):
        e = float(np.max(np.abs(ref[i] - got[i])) / max(np.max(np.abs(ref[i])), 1e-30))
        assert e <= SCALE_REL_TOL, (i, e)


def independent_cases(n=3):
    """(fam, rows, k) drawn from a fixed stream, with rows large enough that
    independent calls take the streaming plan (a fifth of the SM count in
    CTAs, each streaming a long share through a two-slot ring)."""
    fams = ("q4k", "q6k", "q8_0", "q5k", "q4_0", "q8d", "q4d", "q6d")
    z = synth.Stream(20261203).draw(len(fams) * n * 2).reshape(len(fams), n, 2)
    out = []
    for fi, fam in enumerate(fams):
        for ci in range(n):
            d = [int(v >> np.uint64(33)) for v in z[fi, ci]]
            nb = 1 + d[0] % (8 if QK[fam] == 256 else 64)
            rows = 600 + d[1] % 2400
            out.append((fam, rows, nb * QK[fam]))
    return out


@pytest.mark.parametrize("fam,rows,k", independent_cases())
def test_random_shape_independent_calls(q, fam, rows, k):
    """Independent calls (QMV_OVERLAP_INDEPENDENT, the streaming plan) give the
    plain launch's bits, back to back with buffers reused, and the oracle's
    result within the bound."""
    fmt = FMT.get(fam, fam)
    st = synth.Stream(rows * 977 + k)
    w = synth.GEN_ROWS[fmt](st, rows, k)
    x = synth.gen_normal(st, k)
    wd = torch.from_numpy(w).cuda()
    xd = torch.from_numpy(x).cuda()
    if fam in FMT:
        xq = torch.empty(k, dtype=torch.int8, device="cuda")
        xs = torch.empty(k // 32, dtype=torch.float32, device="cuda")
        q.quantize_act_q8(xd, xq, xs, None, 1, k)
        entry = {"q8d": q.qmv_q8_dp4a, "q4d": q.qmv_q4k_dp4a, "q6d": q.qmv_q6k_dp4a}[fam]

        def call(y, ov):
            entry(wd, xq, xs, y, rows, k, overlap=ov)
        oq, os_, _ = oracle.quantize_act_q8(x, 1, k)
        ref = {"q8d": oracle.qmv_q8_dp4a, "q4d": oracle.qmv_q4k_dp4a, "q6d": oracle.qmv_q6k_dp4a}[fam](
            w, oq.reshape(-1), os_.reshape(-1), rows, k)
    else:
        def call(y, ov):
            getattr(q, f"qmv_{fam}")(wd, xd, y, rows, k, overlap=ov)
        ref = oracle.qmv(fam, w, x, rows, k)
    plain = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    call(plain, q.OVERLAP_NONE)
    bufs = [torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda") for _ in range(2)]
    outs = []
    for i in range(4):
        call(bufs[i % 2], q.OVERLAP_INDEPENDENT)
        outs.append(bufs[i % 2].clone())
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, plain)
    got = plain.cpu().numpy().astype(np.float64)
    assert float(np.max(np.abs(ref - got)) / max(float(np.max(np.abs(ref))), 1e-30)) <= 1e-4
