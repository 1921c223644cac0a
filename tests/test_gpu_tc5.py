"""GPU parity of the batched product on the fifth-generation tensor cores
(qmm_q4k_tc5: tcgen05.mma with tensor-memory accumulators, 2-D TMA tensor
copies, k-chunks reduced across a thread-block cluster) against the CPU
oracle, through the C ABI.

Bars as for the other batch kernels: unit rows of x give the weight columns
bit for bit; otherwise every row of y is within scale-relative error
max|a-b|/max|a| <= 1e-4 of the f64 oracle. Shapes cover one and several
128-row tiles, a ragged last tile, k-chunks of unequal length (k / 256 not a
multiple of the cluster size), every cluster size, every ring depth, and
m > 8 (two launches).
"""

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


def run(q, w, x, rows, k, m, cfg=None, overlap=0):
    y = torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda")
    q.qmm_q4k_tc5(dev(w), dev(x), y, rows, k, m, cfg=cfg, overlap=overlap)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def case(rows, k, m, seed):
    st = synth.Stream(seed)
    w = synth.gen_q4k_rows(st, rows, k)
    x = synth.gen_normal(st, m * k).reshape(m, k)
    return w, x


@pytest.mark.parametrize("rows,k,m", [(128, 256, 1), (300, 1024, 3), (256, 4096, 8), (1000, 14336, 4),
                                      (4096, 2048, 5), (517, 2560, 9), (4096, 4096, 2)])
def test_matches_oracle(q, rows, k, m):
    w, x = case(rows, k, m, rows + 7 * k + m)
    y = run(q, w, x, rows, k, m)
    ref = oracle.qmm("q4k", w, x, m, rows, k)
    assert not np.any(np.isnan(y))
    for i in range(m):
        assert scale_rel(ref[i], y[i]) <= SCALE_REL_TOL, i
    assert q.qmv_device_status() == 0


@pytest.mark.parametrize("rows,k", [(256, 1024), (4096, 4096), (200, 2560)])
def test_unit_rows_give_weight_columns(q, rows, k):
    st = synth.Stream(11 + rows)
    w = synth.gen_q4k_rows(st, rows, k)
    js = [5, k - 1, 300, 17, k // 2, 333, 64, 1023]
    xu = np.zeros((8, k), dtype=np.float32)
    for i, j in enumerate(js):
        xu[i, j] = 1.0
    y = run(q, w, xu, rows, k, 8)
    W = oracle.dequant("q4k", w, rows, k).astype(np.float32)
    for i, j in enumerate(js):
        assert np.array_equal(y[i], W[:, j]), (i, j)


@pytest.mark.parametrize("cluster", [1, 2, 4, 8])
def test_every_cluster_size_and_ring_depth(q, cluster):
    """The cluster size sets how k is split (the rounding of the chunk sums
    changes, so each is checked against the oracle); the ring depth only
    schedules the same arithmetic, so every depth gives the same bits."""
    rows, k, m = 384, 3072, 4
    w, x = case(rows, k, m, 99)
    ref = oracle.qmm("q4k", w, x, m, rows, k)
    ys = [run(q, w, x, rows, k, m, cfg={"cluster": cluster, "chunks": s}) for s in (1, 2, 4)]
    for y in ys:
        for i in range(m):
            assert scale_rel(ref[i], y[i]) <= SCALE_REL_TOL, (cluster, i)
    assert np.array_equal(ys[0], ys[1]) and np.array_equal(ys[0], ys[2])


def test_launch_overlap_modes_are_bitwise_equal(q):
    """The overlap mode only changes when a launch may start: with the plan
    held (a forced cluster size keeps independent calls on the cluster plan)
    every mode gives the same bits."""
    rows, k, m = 4096, 4096, 4
    w, x = case(rows, k, m, 5)
    ys = [run(q, w, x, rows, k, m, cfg={"cluster": 8}, overlap=o)
          for o in (q.OVERLAP_NONE, q.OVERLAP_CHAIN, q.OVERLAP_INDEPENDENT)]
    assert np.array_equal(ys[0], ys[1]) and np.array_equal(ys[0], ys[2])
    assert np.array_equal(ys[0], run(q, w, x, rows, k, m))


def test_same_as_chained_calls_in_a_stream(q):
    """Ten calls in a row on one stream, chained (each call's x is the
    previous call's y, rows == k), all within the tolerance of the oracle fed
    the inputs each call read."""
    n, m = 2048, 2
    st = synth.Stream(77)
    ws = [synth.gen_q4k_rows(st, n, n) for _ in range(10)]
    x0 = (synth.gen_normal(st, m * n) / np.float32(16)).astype(np.float32).reshape(m, n)
    cur = dev(x0)
    outs = []
    for w in ws:
        y = torch.empty((m, n), dtype=torch.float32, device="cuda")
        q.qmm_q4k_tc5(dev(w), cur, y, n, n, m, overlap=q.OVERLAP_CHAIN)
        outs.append(y)
        cur = y
    torch.cuda.synchronize()
    inputs = [x0] + [o.cpu().numpy() for o in outs[:-1]]
    for w, xin, o in zip(ws, inputs, outs):
        ref = oracle.qmm("q4k", w, xin, m, n, n)
        got = o.cpu().numpy()
        for i in range(m):
            assert scale_rel(ref[i], got[i]) <= SCALE_REL_TOL


def test_rejects_unaligned_operands(q):
    rows, k, m = 128, 256, 2
    w, x = case(rows, k, m, 3)
    wd = torch.zeros(w.nbytes + 16, dtype=torch.uint8, device="cuda")
    wd[2:2 + w.nbytes] = dev(w.reshape(-1))
    y = torch.empty((m, rows), dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmvError):
        q.qmm_q4k_tc5(wd[2:], dev(x), y, rows, k, m)


@pytest.mark.parametrize("rows,k,m", [(256, 2048, 2), (300, 1024, 8)])
def test_timeout_path_marks_outputs_nan(q, rows, k, m):
    """Every CTA's decoders take the path of a weight copy that did not land:
    all outputs are NaN, the status word says so, and the next call on the
    same context is correct again."""
    w, x = case(rows, k, m, 41 + rows)
    q.qmv_device_status(clear=True)
    y = torch.zeros((m, rows), dtype=torch.float32, device="cuda")
    q.qmm_q4k_tc5_selftest_timeout_path(dev(w), dev(x), y, rows, k, m)
    torch.cuda.synchronize()
    assert np.all(np.isnan(y.cpu().numpy()))
    assert q.qmv_device_status(clear=True) & q.QMV_STATUS_WAIT_TIMEOUT
    y2 = run(q, w, x, rows, k, m)
    ref = oracle.qmm("q4k", w, x, m, rows, k)
    for i in range(m):
        assert scale_rel(ref[i], y2[i]) <= SCALE_REL_TOL
    assert q.qmv_device_status() == 0


@pytest.mark.parametrize("rows,k,m", [(128, 256, 1), (300, 1024, 3), (256, 4096, 8), (4096, 4096, 2),
                                      (4096, 2048, 5), (517, 2560, 9), (1, 512, 8), (4096, 4096, 8),
                                      (1000, 14336, 4), (300, 16384, 8), (129, 768, 2)])
def test_streaming_plan_matches_oracle(q, rows, k, m):
    """Independent calls take the streaming plan (one CTA a 128-row tile over
    the whole of k, the MMAs of each super-block's halves issued by two
    threads into two accumulators). It is within the tolerance of the oracle,
    and the ring depth only schedules the same arithmetic, so every depth
    gives the same bits."""
    P = q.qmm_q4k_tc5_plan_detail(rows, k, min(m, 8), overlap=q.OVERLAP_INDEPENDENT)
    assert P["streaming"] == 1
    w, x = case(rows, k, m, 3 * rows + k + m)
    y = run(q, w, x, rows, k, m, overlap=q.OVERLAP_INDEPENDENT)
    ref = oracle.qmm("q4k", w, x, m, rows, k)
    assert not np.any(np.isnan(y))
    for i in range(m):
        assert scale_rel(ref[i], y[i]) <= SCALE_REL_TOL, i
    ys = [run(q, w, x, rows, k, m, cfg={"chunks": s}, overlap=q.OVERLAP_INDEPENDENT) for s in (1, 2, 3)]
    for ysd in ys:
        assert np.array_equal(ysd, y)
    assert q.qmv_device_status() == 0


def test_streaming_plan_unit_rows_give_weight_columns(q):
    rows, k = 4096, 4096
    st = synth.Stream(12)
    w = synth.gen_q4k_rows(st, rows, k)
    js = [5, k - 1, 300, 17, k // 2, 333, 64, 1023]
    xu = np.zeros((8, k), dtype=np.float32)
    for i, j in enumerate(js):
        xu[i, j] = 1.0
    y = run(q, w, xu, rows, k, 8, overlap=q.OVERLAP_INDEPENDENT)
    W = oracle.dequant("q4k", w, rows, k).astype(np.float32)
    for i, j in enumerate(js):
        assert np.array_equal(y[i], W[:, j]), (i, j)


def test_streaming_plan_in_a_stream_of_independent_calls(q):
    """Twenty independent calls on one stream (each may start before the one
    before it ends), each with its own weights, x and y."""
    rows, k, m = 2048, 4096, 4
    st = synth.Stream(313)
    ws = [synth.gen_q4k_rows(st, rows, k) for _ in range(4)]
    xs = [synth.gen_normal(st, m * k).reshape(m, k) for _ in range(5)]
    wd = [dev(w) for w in ws]
    xd = [dev(x) for x in xs]
    ys = [torch.empty((m, rows), dtype=torch.float32, device="cuda") for _ in range(20)]
    for i in range(20):
        q.qmm_q4k_tc5(wd[i % 4], xd[i % 5], ys[i], rows, k, m, overlap=q.OVERLAP_INDEPENDENT)
    torch.cuda.synchronize()
    for i in range(20):
        ref = oracle.qmm("q4k", ws[i % 4], xs[i % 5], m, rows, k)
        got = ys[i].cpu().numpy()
        for j in range(m):
            assert scale_rel(ref[j], got[j]) <= SCALE_REL_TOL, (i, j)
    assert q.qmv_device_status() == 0


def test_streaming_plan_timeout_path_marks_outputs_nan(q):
    rows, k, m = 300, 2048, 8
    w, x = case(rows, k, m, 43)
    q.qmv_device_status(clear=True)
    y = torch.zeros((m, rows), dtype=torch.float32, device="cuda")
    q.qmm_q4k_tc5_selftest_timeout_path(dev(w), dev(x), y, rows, k, m, overlap=q.OVERLAP_INDEPENDENT)
    torch.cuda.synchronize()
    assert np.all(np.isnan(y.cpu().numpy()))
    assert q.qmv_device_status(clear=True) & q.QMV_STATUS_WAIT_TIMEOUT
    y2 = run(q, w, x, rows, k, m, overlap=q.OVERLAP_INDEPENDENT)
    ref = oracle.qmm("q4k", w, x, m, rows, k)
    for i in range(m):
        assert scale_rel(ref[i], y2[i]) <= SCALE_REL_TOL
    assert q.qmv_device_status() == 0


def random_cases(n=12):
    """Seeded random shapes: rows 1..3000 (ragged last tiles), k a multiple of
    256 up to 16384, m 1..12, a forced cluster size or the default."""
    z = synth.Stream(20261204).draw(n * 4).reshape(n, 4)
    out = []
    for i in range(n):
        d = [int(v >> np.uint64(33)) for v in z[i]]
        rows = 1 + d[0] % 3000
        k = 256 * (1 + d[1] % 64)
        m = 1 + d[2] % 12
        cl = [0, 1, 2, 3, 4, 5, 6, 7, 8][d[3] % 9]
        out.append((rows, k, m, cl))
    return out


@pytest.mark.parametrize("rows,k,m,cluster", random_cases())
def test_random_shapes(q, rows, k, m, cluster):
    w, x = case(rows, k, m, rows * 31 + k + m)
    cfg = {"cluster": cluster} if cluster else None
    try:
        y = run(q, w, x, rows, k, m, cfg=cfg)
    except q.QmvError as e:
        # a forced cluster size whose chunks do not fit one CTA's shared
        # memory is refused on the host, never launched
        assert e.code == q.QMV_ETOOBIG and cluster and k // 256 > cluster
        return
    ref = oracle.qmm("q4k", w, x, m, rows, k)
    assert not np.any(np.isnan(y))
    for i in range(m):
        assert scale_rel(ref[i], y[i]) <= SCALE_REL_TOL, i


def streaming_cases(n=10):
    """Seeded random shapes for the streaming plan: rows 1..3000 (ragged last
    tiles), k a multiple of 256 up to 16384, m 1..16 (two launches past 8)."""
    z = synth.Stream(20261205).draw(n * 3).reshape(n, 3)
    out = []
    for i in range(n):
        d = [int(v >> np.uint64(33)) for v in z[i]]
        out.append((1 + d[0] % 3000, 256 * (1 + d[1] % 64), 1 + d[2] % 16))
    return out


@pytest.mark.parametrize("rows,k,m", streaming_cases())
def test_streaming_plan_random_shapes(q, rows, k, m):
    w, x = case(rows, k, m, rows * 17 + k + 3 * m)
    y = run(q, w, x, rows, k, m, overlap=q.OVERLAP_INDEPENDENT)
    ref = oracle.qmm("q4k", w, x, m, rows, k)
    assert not np.any(np.isnan(y))
    for i in range(m):
        assert scale_rel(ref[i], y[i]) <= SCALE_REL_TOL, i
    assert q.qmv_device_status() == 0


def test_streaming_and_cluster_plans_interleaved_in_one_stream(q):
    """Independent calls (streaming plan) alternating with chained calls
    (cluster plan) in one stream: a CTA of either plan never shares an SM with
    another tensor-memory CTA that could hold columns it waits for, so the
    sequence completes, and every call is within the tolerance of the oracle."""
    rows, k, m = 1024, 2048, 4
    st = synth.Stream(4242)
    ws = [synth.gen_q4k_rows(st, rows, k) for _ in range(3)]
    xs = [synth.gen_normal(st, m * k).reshape(m, k) for _ in range(3)]
    wd = [dev(w) for w in ws]
    xd = [dev(x) for x in xs]
    ys = [torch.empty((m, rows), dtype=torch.float32, device="cuda") for _ in range(12)]
    for i in range(12):
        mode = q.OVERLAP_INDEPENDENT if i % 2 == 0 else q.OVERLAP_CHAIN
        q.qmm_q4k_tc5(wd[i % 3], xd[(i + 1) % 3], ys[i], rows, k, m, overlap=mode)
    torch.cuda.synchronize()
    for i in range(12):
        ref = oracle.qmm("q4k", ws[i % 3], xs[(i + 1) % 3], m, rows, k)
        got = ys[i].cpu().numpy()
        for j in range(m):
            assert scale_rel(ref[j], got[j]) <= SCALE_REL_TOL, (i, j)
    assert q.qmv_device_status() == 0


def test_both_plans_on_two_streams_at_once(q):
    """Chained cluster-plan calls on one stream and independent streaming-plan
    calls on another, enqueued alternately so that their CTAs share the GPU:
    at most two cluster-plan CTAs (256 tensor-memory columns each) fit an SM,
    and a streaming CTA (512 columns) shares its SM with neither, so no
    allocation waits on another stream. Every call matches the oracle."""
    rows, k, m = 2048, 2048, 4
    st = synth.Stream(5151)
    ws = [synth.gen_q4k_rows(st, rows, k) for _ in range(2)]
    x0 = (synth.gen_normal(st, m * k) / np.float32(16)).astype(np.float32).reshape(m, k)
    xs = synth.gen_normal(st, m * k).reshape(m, k)
    wd = [dev(w) for w in ws]
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    chain_out, ind_out = [], []
    cur = dev(x0)
    xsd = dev(xs)
    # the inputs were copied on the current stream
    sa.wait_stream(torch.cuda.current_stream())
    sb.wait_stream(torch.cuda.current_stream())
    for i in range(8):
        with torch.cuda.stream(sa):
            y = torch.empty((m, rows), dtype=torch.float32, device="cuda")
            q.qmm_q4k_tc5(wd[0], cur, y, rows, k, m, stream=sa, overlap=q.OVERLAP_CHAIN)
            chain_out.append(y)
            cur = y
        with torch.cuda.stream(sb):
            y2 = torch.empty((m, rows), dtype=torch.float32, device="cuda")
            q.qmm_q4k_tc5(wd[1], xsd, y2, rows, k, m, stream=sb, overlap=q.OVERLAP_INDEPENDENT)
            ind_out.append(y2)
    torch.cuda.synchronize()
    inputs = [x0] + [o.cpu().numpy() for o in chain_out[:-1]]
    for xin, o in zip(inputs, chain_out):
        ref = oracle.qmm("q4k", ws[0], xin, m, rows, k)
        got = o.cpu().numpy()
        for j in range(m):
            assert scale_rel(ref[j], got[j]) <= SCALE_REL_TOL
    ref = oracle.qmm("q4k", ws[1], xs, m, rows, k)
    for o in ind_out:
        got = o.cpu().numpy()
        for j in range(m):
            assert scale_rel(ref[j], got[j]) <= SCALE_REL_TOL
    assert q.qmv_device_status() == 0


@pytest.mark.parametrize("overlap", [0, 2])
def test_many_tiles(q, overlap):
    """20000 rows: 157 tiles (more CTAs than SMs in either plan, a ragged last
    tile), k = 4096, m = 8; the cluster plan (plain launch) and the streaming
    plan (independent call)."""
    rows, k, m = 20000, 4096, 8
    w, x = case(rows, k, m, 2026)
    y = run(q, w, x, rows, k, m, overlap=overlap)
    ref = oracle.qmm("q4k", w, x, m, rows, k)
    assert not np.any(np.isnan(y))
    for i in range(m):
        assert scale_rel(ref[i], y[i]) <= SCALE_REL_TOL, i
    assert q.qmv_device_status() == 0
