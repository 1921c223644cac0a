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
