"""Run by tests/test_gpu_bounds_check.py in a process of its own: loads the
checking build of the library (every shared- and global-memory access of the
matvec and batch kernels tested against its region, QMV_STATUS_OUT_OF_BOUNDS
raised instead of an access outside it) and drives it over a seeded sweep of
shapes, launch modes and forced plans of every matvec family, the dp4a,
block-dot and fused-quantization entry points, MoE banks (one bad id among the
slots) and the small-M batched products.
Every result is checked against the oracle as well. Prints one JSON line:
calls made, calls refused on the host, the status word, and the failures."""

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402
from ggml_format_dequant_gb300 import _build  # noqa: E402
import ggml_format_dequant_gb300 as q  # noqa: E402

TOL = 1e-4
QK = {"q4k": 256, "q6k": 256, "q8_0": 32, "q5k": 256, "q4_0": 32}
DP4A = {"q8d": "q8_0", "q4d": "q4k", "q6d": "q6k"}


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def scale_rel(ref, got):
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    return float(np.max(np.abs(ref - got)) / max(float(np.max(np.abs(ref))), 1e-30))


def draws(seed, n, width):
    z = synth.Stream(seed).draw(n * width).reshape(n, width)
    return [[int(v >> np.uint64(33)) for v in row] for row in z]


def forced(d):
    """A forced plan half of the time (the same fields the planner takes)."""
    if d[0] % 2 == 0:
        return None
    return dict(ctas=1 + d[1] % 9, chunk_rows=d[2] % 6, chunks=d[3] % 4, unroll=d[4] % 3,
                warps=[0, 4, 8, 16][d[5] % 4])


def planted():
    """The build with ring slots half as long as planned: a few Q4_K matvec
    and batch calls whose pieces hold several rows; the checks of each kernel
    must raise the bit (results are undefined, so they are not compared)."""
    q.load(_build.lib_path("check_planted"))
    q.qmv_device_status(clear=True)
    calls = 0
    for rows, k in ((300, 2048), (1500, 4096)):
        st = synth.Stream(rows + k)
        w = synth.GEN_ROWS["q4k"](st, rows, k)
        x = synth.gen_normal(st, k)
        y = torch.zeros(rows, device="cuda")
        for cfg in (None, dict(chunk_rows=4, chunks=2)):
            if q.qmv_q4k(dev(w), dev(x), y, rows, k, cfg=cfg, check=False) == q.QMV_OK:
                calls += 1
    torch.cuda.synchronize()
    matvec_status = q.qmv_device_status(clear=True)
    # the batch kernel with the same planted fault
    for rows, k, m in ((300, 2048, 2), (700, 4096, 8)):
        st = synth.Stream(rows + k + m)
        w = synth.GEN_ROWS["q4k"](st, rows, k)
        x = synth.gen_normal(st, m * k).reshape(m, k)
        y = torch.zeros((m, rows), device="cuda")
        if q.qmm_q4k(dev(w), dev(x), y, rows, k, m, check=False) == q.QMV_OK:
            calls += 1
    torch.cuda.synchronize()
    batch_status = q.qmv_device_status(clear=True)
    print(json.dumps({"calls": calls, "status": matvec_status, "batch_status": batch_status}))


def main():
    q.load(_build.lib_path("check"))
    q.qmv_device_status(clear=True)
    calls, refused, fails = 0, 0, []

    def record(rc, name, check):
        nonlocal calls, refused
        if rc == q.QMV_ETOOBIG:
            refused += 1
            return
        if rc != q.QMV_OK:
            fails.append(f"{name}: rc {rc}")
            return
        calls += 1
        torch.cuda.synchronize()
        err = check()
        if err:
            fails.append(f"{name}: {err}")

    # dense matvecs, f32 activation
    for fi, fam in enumerate(QK):
        for d in draws(7100 + fi, 9, 9):
            qk = QK[fam]
            k = qk * (1 + d[0] % (8192 // qk))
            rows = 1 + d[1] % 1500
            mode = d[2] % 3
            cfg = forced(d[3:])
            st = synth.Stream(rows * 7 + k)
            w = synth.GEN_ROWS[fam](st, rows, k)
            x = synth.gen_normal(st, k)
            y = torch.full((rows,), float("nan"), device="cuda")
            rc = getattr(q, f"qmv_{fam}")(dev(w), dev(x), y, rows, k, cfg=cfg, overlap=mode, check=False)
            record(rc, f"qmv_{fam} {rows}x{k} mode {mode} {cfg}",
                   lambda: None if scale_rel(oracle.qmv(fam, w, x, rows, k), y.cpu().numpy()) <= TOL else "parity")

    # dp4a matvecs and their block / group dots, and the fused quantization
    for fi, fam in enumerate(DP4A):
        fmt = DP4A[fam]
        for d in draws(7200 + fi, 7, 9):
            qk = QK[fmt]
            k = qk * (1 + d[0] % (8192 // qk))
            rows = 1 + d[1] % 1500
            mode = d[2] % 3
            cfg = forced(d[3:])
            st = synth.Stream(rows * 11 + k)
            w = synth.GEN_ROWS[fmt](st, rows, k)
            x = synth.gen_normal(st, k)
            xq = torch.empty(k, dtype=torch.int8, device="cuda")
            xs = torch.empty(k // 32, dtype=torch.float32, device="cuda")
            q.quantize_act_q8(dev(x), xq, xs, None, 1, k)
            oq, os_, _ = oracle.quantize_act_q8(x, 1, k)
            oq, os_ = oq.reshape(-1), os_.reshape(-1)
            y = torch.full((rows,), float("nan"), device="cuda")
            entry = {"q8d": q.qmv_q8_dp4a, "q4d": q.qmv_q4k_dp4a, "q6d": q.qmv_q6k_dp4a}[fam]
            ref_fn = {"q8d": oracle.qmv_q8_dp4a, "q4d": oracle.qmv_q4k_dp4a, "q6d": oracle.qmv_q6k_dp4a}[fam]
            rc = entry(dev(w), xq, xs, y, rows, k, cfg=cfg, overlap=mode, check=False)
            record(rc, f"{fam} {rows}x{k} mode {mode} {cfg}",
                   lambda: None if scale_rel(ref_fn(w, oq, os_, rows, k), y.cpu().numpy()) <= TOL else "parity")
            # the exact integer dots of every block
            dots_fn = {"q8d": (q.qmv_q8_dp4a_blockdots, oracle.q8_blockdots, 32),
                       "q4d": (q.qmv_q4k_dp4a_blockdots, oracle.q4k_dp4a_blockdots, 32),
                       "q6d": (q.qmv_q6k_dp4a_blockdots, oracle.q6k_dp4a_groupdots, 16)}[fam]
            dots = torch.full((rows * (k // dots_fn[2]),), -7, dtype=torch.int32, device="cuda")
            rc = dots_fn[0](dev(w), xq, dots, rows, k, check=False)
            record(rc, f"{fam} dots {rows}x{k}",
                   lambda: None if np.array_equal(dots.cpu().numpy().reshape(-1),
                                                  np.asarray(dots_fn[1](w, oq, rows, k)).reshape(-1)) else "dots")
            if fam == "q8d":
                y2 = torch.full((rows,), float("nan"), device="cuda")
                rc = q.qmv_q8_dp4a_quant(dev(w), dev(x), y2, rows, k, cfg=cfg, overlap=mode, check=False)
                record(rc, f"q8_dp4a_quant {rows}x{k} mode {mode} {cfg}",
                       lambda: None if scale_rel(ref_fn(w, oq, os_, rows, k), y2.cpu().numpy()) <= TOL else "parity")

    # MoE banks: slots of routed experts, one slot with an id outside the bank
    moe = [("q4k", q.moe_qmv_q4k, False), ("q6k", q.moe_qmv_q6k, False), ("q8_0", q.moe_qmv_q8_0, False),
           ("q4_0", q.moe_qmv_q4_0, False), ("q5k", q.moe_qmv_q5k, False), ("q4k", q.moe_qmv_q4k_dp4a, True),
           ("q6k", q.moe_qmv_q6k_dp4a, True)]
    for mi, (fmt, fn, dp4a) in enumerate(moe):
        for d in draws(7300 + mi, 4, 13):
            qk = QK[fmt]
            k = qk * (1 + d[0] % (4096 // qk))
            rows = 1 + d[1] % 700
            ne = 2 + d[2] % 6
            slots = 1 + d[3] % min(8, ne)   # distinct experts per token
            mode = d[4] % 3
            cfg = forced(d[5:11])
            st = synth.Stream(rows * 13 + k + ne)
            bank = synth.GEN_ROWS[fmt](st, ne * rows, k).reshape(ne, rows, -1)
            ids = synth.gen_moe_ids(st, slots, ne).astype(np.int32)
            if slots > 1:
                ids[d[11] % slots] = ne + d[12] % 3   # an unroutable slot
            x = synth.gen_normal(st, slots * k).reshape(slots, k)
            y = torch.full((slots, rows), 5.0, device="cuda")
            if dp4a:
                xq = torch.empty(slots * k, dtype=torch.int8, device="cuda")
                xs = torch.empty(slots * (k // 32), dtype=torch.float32, device="cuda")
                q.quantize_act_q8(dev(x), xq, xs, None, slots, k)
                oq, os_, _ = oracle.quantize_act_q8(x, slots, k)
                ref_fn = oracle.moe_qmv_q4k_dp4a if fmt == "q4k" else oracle.moe_qmv_q6k_dp4a
                rc = fn(dev(bank), xq, xs, y, rows, k, dev(ids), slots, ne, cfg=cfg, overlap=mode, check=False)
                ref = lambda: ref_fn(bank, oq, os_, ids, rows, k, ne)  # noqa: E731
            else:
                rc = fn(dev(bank), dev(x), y, rows, k, dev(ids), slots, ne, cfg=cfg, overlap=mode, check=False)
                ref = lambda: oracle.moe_qmv(fmt, bank, x, ids, rows, k, ne)  # noqa: E731

            def moe_check():
                r = np.asarray(ref(), dtype=np.float64).reshape(slots, rows)
                g = y.cpu().numpy().astype(np.float64)
                for s in range(slots):
                    bad = not (0 <= ids[s] < ne)
                    if bad:
                        if not np.all(np.isnan(g[s])):
                            return f"slot {s}: bad id not NaN"
                    elif scale_rel(r[s], g[s]) > TOL:
                        return f"slot {s}: parity"
                return None
            record(rc, f"moe {fn.__name__} {rows}x{k} e{ne} s{slots} mode {mode} {cfg}", moe_check)

    # small-M batched products (the tensor-core batch kernel): m = 2..12 rows
    # of x (one or two launches), forced plans, every launch mode
    for fi, fmt in enumerate(QK):
        for d in draws(7400 + fi, 5, 10):
            qk = QK[fmt]
            k = qk * (1 + d[0] % (8192 // qk))
            rows = 1 + d[1] % 600
            m = 2 + d[2] % 11
            mode = d[3] % 3
            cfg = None if d[4] % 2 == 0 else dict(ctas=1 + d[5] % 9, chunk_rows=d[6] % 20, chunks=d[7] % 4,
                                                   warps=[0, 1, 3, 8][d[8] % 4])
            st = synth.Stream(rows * 19 + k + m)
            w = synth.GEN_ROWS[fmt](st, rows, k)
            x = synth.gen_normal(st, m * k).reshape(m, k)
            y = torch.full((m, rows), float("nan"), device="cuda")
            rc = getattr(q, f"qmm_{fmt}")(dev(w), dev(x), y, rows, k, m, cfg=cfg, overlap=mode, check=False)

            def qmm_check():
                r = oracle.qmm(fmt, w, x, m, rows, k)
                g = y.cpu().numpy()
                return None if all(scale_rel(r[i], g[i]) <= TOL for i in range(m)) else "parity"
            record(rc, f"qmm_{fmt} {rows}x{k} m {m} mode {mode} {cfg}", qmm_check)

    # the path of a staged copy that did not land: NaN outputs
    for rows, k in ((300, 2048), (4096, 4096)):
        st = synth.Stream(rows + k)
        w = synth.GEN_ROWS["q4k"](st, rows, k)
        x = synth.gen_normal(st, k)
        y = torch.zeros(rows, device="cuda")
        rc = q.qmv_selftest_timeout_path(dev(w), dev(x), y, rows, k, check=False)
        record(rc, f"timeout path {rows}x{k}",
               lambda: None if np.all(np.isnan(y.cpu().numpy())) else "timeout outputs not NaN")

    torch.cuda.synchronize()
    status = q.qmv_device_status(clear=True)
    print(json.dumps({"calls": calls, "refused": refused, "status": status, "failures": fails[:20],
                      "n_failures": len(fails)}))


if __name__ == "__main__":
    if sys.argv[1:] == ["planted"]:
        planted()
    else:
        main()
