"""Several host threads calling the library at once, each on its own stream
(the entry points are reentrant): every result matches the oracle. The first
launches of each kernel (device query, shared-memory opt-in) happen under
contention here as well."""

import threading

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def test_concurrent_host_threads():
    import __graft_entry__
    __graft_entry__.build()
    import ggml_format_dequant_gb300 as q

    cases = []
    for i, (fmt, rows, k) in enumerate([("q4k", 300, 2048), ("q6k", 200, 1536), ("q8_0", 260, 1024),
                                        ("q5k", 120, 2304), ("q4_0", 310, 992), ("q4k", 77, 4352)]):
        st = synth.Stream(500 + i)
        w = synth.GEN_ROWS[fmt](st, rows, k)
        x = synth.gen_normal(st, k)
        cases.append((fmt, rows, k, w, x, oracle.qmv(fmt, w, x, rows, k)))
    errors = []

    def worker(case):
        fmt, rows, k, w, x, ref = case
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                wd = torch.from_numpy(w).cuda()
                xd = torch.from_numpy(x).cuda()
                ys = [torch.empty(rows, dtype=torch.float32, device="cuda") for _ in range(20)]
                for y in ys:
                    getattr(q, f"qmv_{fmt}")(wd, xd, y, rows, k, stream=s)
            s.synchronize()
            for y in ys:
                got = y.cpu().numpy().astype(np.float64)
                e = float(np.max(np.abs(ref - got)) / np.max(np.abs(ref)))
                if e > 1e-4:
                    errors.append((fmt, e))
                    return
        except Exception as exc:   # reported below
            errors.append((fmt, repr(exc)))

    threads = [threading.Thread(target=worker, args=(c,)) for c in cases]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors


def test_concurrent_threads_with_different_overlap_modes():
    """Launch options belong to the call: one host thread runs a dependent
    decode chain (QMV_OVERLAP_CHAIN, every call reading the previous call's y)
    on its stream while another runs independent projections of one activation
    (QMV_OVERLAP_INDEPENDENT) on its own. Both give bitwise the results of
    plain launches, and every call is within 1e-4 of the oracle given its
    inputs."""
    import __graft_entry__
    __graft_entry__.build()
    import ggml_format_dequant_gb300 as q

    n, steps = 2048, 6
    st = synth.Stream(4242)
    wc = [synth.gen_q4k_rows(st, n, n) for _ in range(steps)]
    wi = [synth.gen_q4k_rows(st, n, n) for _ in range(steps)]
    x0 = (synth.gen_normal(st, n) / np.float32(16)).astype(np.float32)
    xi = synth.gen_normal(st, n)
    dwc = [torch.from_numpy(w).cuda() for w in wc]
    dwi = [torch.from_numpy(w).cuda() for w in wi]
    dx0 = torch.from_numpy(x0).cuda()
    dxi = torch.from_numpy(xi).cuda()

    def chain(ov, s):
        with torch.cuda.stream(s):
            bufs = [torch.empty(n, dtype=torch.float32, device="cuda") for _ in range(steps)]
            cur = dx0
            for i in range(steps):
                q.qmv_q4k(dwc[i], cur, bufs[i], n, n, stream=s, overlap=ov)
                cur = bufs[i]
        s.synchronize()
        return [b.cpu().numpy() for b in bufs]

    def projections(ov, s):
        with torch.cuda.stream(s):
            bufs = [torch.full((n,), float("nan"), dtype=torch.float32, device="cuda") for _ in range(2)]
            outs = []
            for i in range(steps):
                q.qmv_q4k(dwi[i], dxi, bufs[i % 2], n, n, stream=s, overlap=ov)
                outs.append(bufs[i % 2].clone())
        s.synchronize()
        return [o.cpu().numpy() for o in outs]

    s0 = torch.cuda.Stream()
    ref_chain = chain(q.OVERLAP_NONE, s0)
    ref_proj = projections(q.OVERLAP_NONE, s0)
    # the oracle, fed the inputs each call actually read
    inputs = [x0] + ref_chain[:-1]
    for i in range(steps):
        r = oracle.qmv("q4k", wc[i], inputs[i], n, n)
        assert float(np.max(np.abs(r - ref_chain[i])) / np.max(np.abs(r))) <= 1e-4, ("chain", i)
        r = oracle.qmv("q4k", wi[i], xi, n, n)
        assert float(np.max(np.abs(r - ref_proj[i])) / np.max(np.abs(r))) <= 1e-4, ("proj", i)

    results, errors = {}, []
    start = threading.Barrier(2)

    def run(name, fn, ov):
        try:
            s = torch.cuda.Stream()
            start.wait(timeout=60)
            results[name] = [fn(ov, s) for _ in range(3)]
        except Exception as exc:   # reported below
            errors.append((name, repr(exc)))

    ta = threading.Thread(target=run, args=("chain", chain, q.OVERLAP_CHAIN))
    tb = threading.Thread(target=run, args=("proj", projections, q.OVERLAP_INDEPENDENT))
    ta.start()
    tb.start()
    ta.join(timeout=120)
    tb.join(timeout=120)
    assert not errors, errors
    for got in results["chain"]:
        for a, b in zip(ref_chain, got):
            assert np.array_equal(a, b)
    for got in results["proj"]:
        for a, b in zip(ref_proj, got):
            assert np.array_equal(a, b)
