"""Benchmark of the GB300 quantized matvec library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one call of the hot path on the Q4_K 4096x4096 workload (rows =
k = 4096, seed 1): qmv_q4k reads the packed weight straight from HBM, decodes
it in registers and writes y. Consecutive steps cycle through enough distinct
copies of the weight (more than 3x the L2 size in total) that every call reads
its weight HBM-cold. The steps are independent (each reads the same x), and
are launched as such (QMV_OVERLAP_INDEPENDENT: a call overlaps the previous
one and waits for it only before writing y); ``--chain`` times a dependent
decode chain instead (QMV_OVERLAP_CHAIN) and ``--isolated`` plain launches.
The K timed steps are one CUDA-graph replay bracketed by CUDA events on the
launching stream, with a barrier and a device synchronize on both sides; the
line reports the max over ranks.

Before the headline, one short JSON line per workload of the suite gives its
us per call and fraction of the measured HBM copy bandwidth in all three
launch modes (the metric's five workloads last). The headline line, printed
last, carries the five workloads' figures in ``config.us_per_call``, the
roofline of the timed kernel against the measured HBM copy bandwidth, the
end-to-end number through the public API with host buffers, the CPU oracle as
a baseline (whose output also checks the timed calls' and the end-to-end
calls' y), and the SM clocks seen while timing.

``--impl reference`` times the CPU oracle (plain C, f64) on the same workload
on the host cores: the only other implementation of the method available here
(the pages' Vulkan kernels cannot run on this machine).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = ("packed-weight GB/s and % of GB300 HBM peak per quant matvec (µs/call, HBM-cold)")
HEADLINE = "q4k_4096x4096"
NOMINAL_HBM_GBS = 7900.0
FALLBACK_HBM_GBS = 6800.0

# ncu DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one
# qmv_q4k launch on the headline workload, per launch mode, valid only for the
# kernel sources whose hash it is recorded under.
NCU_TRAFFIC = {"0a9c75a7ace08efe": {2: 9496576}}

KERNEL_SOURCES = ["qmv_device.cuh", "qmv_formats.cuh", "qmv_kernel.cuh", "qmv_launch.cuh", "qmv_q4k.cu"]


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "ggml_format_dequant_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Block format of each workload kind's weights.
KIND_FMT = {"q4k": "q4k", "q4k_dp4a": "q4k", "q6k": "q6k", "q6k_dp4a": "q6k", "moe_q6k_dp4a": "q6k",
            "q8_0_dp4a": "q8_0", "q5k": "q5k", "q4_0": "q4_0",
            "moe_q4k": "q4k", "moe_q4k_dp4a": "q4k", "moe_q6k": "q6k", "moe_q8_0": "q8_0", "moe_q4_0": "q4_0",
            "moe_q5k": "q5k", "qmm_q4k": "q4k", "qmm_q6k": "q6k", "qmm_q8_0": "q8_0",
            "qmm_q5k": "q5k", "qmm_q4_0": "q4_0"}
# MoE kinds with an f32 activation (one entry point each, same arguments).
MOE_F32 = ("moe_q4k", "moe_q6k", "moe_q8_0", "moe_q4_0", "moe_q5k")


def weight_bytes(name: str) -> int:
    c = synth.CONFIGS[name]
    rb = synth.row_bytes(KIND_FMT[c["kind"]], c["k"]) * c["rows"]
    if c["kind"].startswith("moe_"):
        return rb * c["slots"]   # routed rows only
    return rb


def algorithmic_bytes(name: str) -> int:
    """Bytes a call must move at minimum: packed weight rows read, activation
    read, output written."""
    c = synth.CONFIGS[name]
    wb = weight_bytes(name)
    if c["kind"] in MOE_F32:
        return wb + 4 * c["slots"] * c["k"] + 4 * c["slots"] * c["rows"] + 4 * c["slots"]
    if c["kind"].startswith("qmm_"):
        return wb + 4 * c["m"] * c["k"] + 4 * c["m"] * c["rows"]   # W read once for all m rows
    if c["kind"] in ("moe_q4k_dp4a", "moe_q6k_dp4a"):
        return wb + c["slots"] * (c["k"] + 4 * (c["k"] // 32)) + 4 * c["slots"] * c["rows"] + 4 * c["slots"]
    if c["kind"] in ("q8_0_dp4a", "q4k_dp4a", "q6k_dp4a"):
        return wb + c["k"] + 4 * (c["k"] // 32) + 4 * c["rows"]
    return wb + 4 * c["k"] + 4 * c["rows"]


# --------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,power.draw")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return

        def reader():
            for ln in self.proc.stdout:
                self.lines.append((time.time(), ln.strip()))

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float) -> dict:
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if ts < t0 or ts > t1:
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                power.append(float(parts[7]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------ GPU side

class Workload:
    """Device buffers of one named workload, rotated over `copies` weights."""

    def __init__(self, q, torch, name: str, l2_bytes: int, device, copies: int = 0):
        self.name = name
        c = synth.make_config(name)
        self.c = c
        self.kind = c["kind"]
        self.rows, self.k = c["rows"], c["k"]
        dev = device
        wb = c["w"].nbytes
        self.copies = copies if copies > 0 else max(4, math.ceil(3 * l2_bytes / wb) + 1)
        # one pinned host copy, `copies` device copies (content identical; the
        # addresses differ, which is what makes each call read from HBM)
        w0 = torch.from_numpy(c["w"].reshape(-1))
        self.w = [w0.to(dev) for _ in range(self.copies)]
        self.x = torch.from_numpy(np.ascontiguousarray(c["x"])).to(dev)
        # one output buffer per weight copy: consecutive calls write different
        # outputs, as the Q, K and V projections of one activation do
        if self.kind.startswith("moe_"):
            self.ys = [torch.empty(c["slots"], self.rows, dtype=torch.float32, device=dev) for _ in range(self.copies)]
            # a cycle of seeded id sets so no (bank, expert) slice repeats within 3x L2
            st = synth.Stream(1003)
            self.ids = [torch.from_numpy(c["ids"]).to(dev)]
            for _ in range(15):
                self.ids.append(torch.from_numpy(synth.gen_moe_ids(st, c["slots"], c["n_experts"])).to(dev))
        elif self.kind.startswith("qmm_"):
            self.ys = [torch.empty(c["m"], self.rows, dtype=torch.float32, device=dev) for _ in range(self.copies)]
        else:
            self.ys = [torch.empty(self.rows, dtype=torch.float32, device=dev) for _ in range(self.copies)]
        self.y = self.ys[0]
        if self.kind in ("q8_0_dp4a", "q4k_dp4a", "q6k_dp4a", "moe_q4k_dp4a", "moe_q6k_dp4a"):
            m = c.get("slots", 1) if self.kind.startswith("moe_") else 1
            self.m = m
            self.xq = torch.empty(m * self.k, dtype=torch.int8, device=dev)
            self.xs = torch.empty(m * (self.k // 32), dtype=torch.float32, device=dev)
            q.quantize_act_q8(self.x, self.xq, self.xs, None, m, self.k)
        self.q = q
        self.cfg = None   # optional forced launch configuration (dict), for tuning sweeps
        self.overlap = 0  # launch overlap of every call (q.OVERLAP_*)
        self.fused = False  # q8_0_dp4a: quantize x inside the matvec launch (qmv_q8_dp4a_quant)
        self.tc5 = False    # qmm_q4k: the fifth-generation tensor-core kernel (qmm_q4k_tc5)

    def call(self, i: int, stream: int, with_quant: bool = False) -> int:
        """Enqueue call i; returns the number of kernels it launched."""
        q, w, cfg, ov = self.q, self.w[i % self.copies], self.cfg, self.overlap
        self.y = self.ys[i % self.copies]
        if self.kind == "q4k":
            q.qmv_q4k(w, self.x, self.y, self.rows, self.k, stream=stream, cfg=cfg, overlap=ov)
        elif self.kind in ("q6k", "q5k", "q4_0"):
            getattr(q, f"qmv_{self.kind}")(w, self.x, self.y, self.rows, self.k, stream=stream, cfg=cfg, overlap=ov)
        elif self.kind == "qmm_q4k" and self.tc5:
            m = self.c["m"]
            q.qmm_q4k_tc5(w, self.x, self.y, self.rows, self.k, m, stream=stream, cfg=cfg, overlap=ov)
            return (m + 7) // 8
        elif self.kind.startswith("qmm_"):
            m = self.c["m"]
            getattr(q, self.kind)(w, self.x, self.y, self.rows, self.k, m, stream=stream, cfg=cfg, overlap=ov)
            return q.qmm_launches(self.kind[4:], self.k, m)
        elif self.kind == "q8_0_dp4a" and self.fused:
            q.qmv_q8_dp4a_quant(w, self.x, self.y, self.rows, self.k, stream=stream, cfg=cfg, overlap=ov)
            return 1
        elif self.kind in ("q8_0_dp4a", "q4k_dp4a", "q6k_dp4a"):
            n = 1
            if with_quant:
                q.quantize_act_q8(self.x, self.xq, self.xs, None, 1, self.k, stream=stream)
                n = 2
            fn = {"q8_0_dp4a": q.qmv_q8_dp4a, "q4k_dp4a": q.qmv_q4k_dp4a, "q6k_dp4a": q.qmv_q6k_dp4a}[self.kind]
            fn(w, self.xq, self.xs, self.y, self.rows, self.k, stream=stream, cfg=cfg, overlap=ov)
            return n
        elif self.kind in MOE_F32:
            c = self.c
            fn = getattr(q, f"moe_qmv_{self.kind[4:]}")
            fn(w, self.x, self.y, self.rows, self.k, self.ids[i % len(self.ids)], c["slots"],
               c["n_experts"], stream=stream, cfg=cfg, overlap=ov)
        elif self.kind in ("moe_q4k_dp4a", "moe_q6k_dp4a"):
            c = self.c
            n = 1
            if with_quant:
                q.quantize_act_q8(self.x, self.xq, self.xs, None, self.m, self.k, stream=stream)
                n = 2
            fn = q.moe_qmv_q4k_dp4a if self.kind == "moe_q4k_dp4a" else q.moe_qmv_q6k_dp4a
            fn(w, self.xq, self.xs, self.y, self.rows, self.k, self.ids[i % len(self.ids)],
               c["slots"], c["n_experts"], stream=stream, cfg=cfg, overlap=ov)
            return n
        return 1


def max_over_ranks(torch, ms: float, dist, device) -> float:
    """The slowest rank's timed region (every rank calls it; one process, or
    no process group: its own)."""
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if dist is not None and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, steps: int, bytes_per_step: int, ms_max: float) -> float:
    """Packed-weight GB/s of the whole job: every rank ran `steps` steps of
    `bytes_per_step` (replicas, weak scaling) within the slowest rank's time."""
    return world * steps * bytes_per_step / (ms_max * 1e-3) / 1e9


def time_graph(torch, wl: Workload, n_calls: int, with_quant=False, replays=1, barrier=None):
    """Capture n_calls rotated calls into one CUDA graph; return (ms per call,
    kernels per call, graph). Times `replays` replays with CUDA events."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        # eager warm-up outside capture (sets kernel attributes, loads modules)
        for i in range(min(4, n_calls)):
            wl.call(i, s.cuda_stream, with_quant)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    launches = 0
    with torch.cuda.graph(g, stream=s):
        for i in range(n_calls):
            launches += wl.call(i, s.cuda_stream, with_quant)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if barrier:
        barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(replays):
            g.replay()
        e1.record(s)
    e1.synchronize()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    ms = e0.elapsed_time(e1) / (replays * n_calls)
    return ms, launches / n_calls, g, s


# The five workloads the metric is quoted on, in order (the first is the small
# case; the second the headline).
METRIC_CONFIGS = ["q4k_256x1024", "q4k_4096x4096", "q8_0_dp4a_14336x4096", "moe_q4k_e128_n768_k2048_s8",
                  "q6k_4096x14336"]
MODE_NAMES = {0: "isolated", 1: "chain", 2: "independent"}
DP4A_KINDS = ("q8_0_dp4a", "q4k_dp4a", "q6k_dp4a", "moe_q4k_dp4a", "moe_q6k_dp4a")


def workload_line(name, times, peak):
    """One short JSON line per workload: us per call and fraction of the
    measured HBM peak in each launch mode (and with the activation
    quantization for the dp4a kinds)."""
    wb = weight_bytes(name)
    d = {"workload": name, "packed_weight_bytes": wb}
    for key, ms in times.items():
        d[key] = {"us": round(ms * 1e3, 3), "frac": round(wb / (ms * 1e-3) / 1e9 / peak, 4)}
    return d


def run_ours(args):
    import torch

    import __graft_entry__
    import ggml_format_dequant_gb300 as q

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    __graft_entry__.build()
    q.load()
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20)
    peak, peak_kind = measured_peak()

    def barrier():
        if dist is not None:
            dist.barrier()

    sampler = ClockSampler(local)
    sampler.start()

    # ------------------------------------------------ the headline workload
    # The timed calls are independent of one another (every call reads the
    # same x, like the Q / K / V projections of one activation), so they are
    # launched with QMV_OVERLAP_INDEPENDENT: each call is scheduled while the
    # previous one runs, streams its weights and decodes at once, and waits
    # for the previous call only before it writes y. --chain times a
    # dependent decode chain (QMV_OVERLAP_CHAIN: x is read only after the
    # previous call is done), --isolated plain launches; the per-workload
    # lines report all three.
    head_mode = args.headline_mode if args.headline_mode is not None else (0 if args.isolated else (1 if args.chain else 2))
    wl = Workload(q, torch, HEADLINE, l2, device)
    wl.overlap = head_mode
    K, W = args.steps, args.warmup
    # warm-up steps (untimed)
    _, _, gw, sw = time_graph(torch, wl, max(W, 1))
    # pre-roll: keep the GPU busy with the same work so clock samples exist
    # even when the K-step region is short
    _, _, gk, sk = time_graph(torch, wl, K)
    pre_t0 = time.time()
    while time.time() - pre_t0 < 0.5:
        with torch.cuda.stream(sk):
            gk.replay()
        torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(sk):
        # a short device-side delay ahead of the start event, so that the
        # graph launch is queued on the device before the timed region opens
        # (the region then holds the K steps alone, not the host's launch)
        torch.cuda._sleep(100000)
        e0.record(sk)
        gk.replay()
        e1.record(sk)
    e1.synchronize()
    torch.cuda.synchronize()
    barrier()
    ms_total = e0.elapsed_time(e1)
    head_y = wl.y.detach().cpu().numpy().copy()   # the last call's output (kept for the parity check)
    post_t0 = time.time()
    while time.time() - post_t0 < 0.5:
        with torch.cuda.stream(sk):
            gk.replay()
        torch.cuda.synchronize()
    clock_window = (pre_t0, time.time())

    ms_max = max_over_ranks(torch, ms_total, dist, device)
    wbytes = weight_bytes(HEADLINE)
    value = whole_job_gbs(world, K, wbytes, ms_max)
    ms_step = ms_max / K
    alg = algorithmic_bytes(HEADLINE)
    achieved = alg / (ms_step * 1e-3) / 1e9

    # ------------------------------------------------ end to end (host buffers)
    e2e, e2e_y = end_to_end(torch, q, wl, device, K)

    # ------------------------------------------------ every workload, three modes
    # A stream of independent calls (they share no inputs with the call
    # before, like the Q / K / V projections of one activation), a dependent
    # decode chain, and isolated calls.
    lines = {}
    del wl, gk, gw
    torch.cuda.empty_cache()
    names = [HEADLINE] if args.headline_only else list(synth.CONFIGS)
    if args.only:
        names = [n for n in synth.CONFIGS if n == HEADLINE or any(n.startswith(o) for o in args.only.split(","))]
    # the metric's five workloads last, so that they end up next to the headline
    names = [n for n in names if n not in METRIC_CONFIGS] + [n for n in METRIC_CONFIGS if n in names]
    for name in names:
        w2 = Workload(q, torch, name, l2, device)
        # graphs of at least 256 calls: a graph boundary serialises calls, so
        # short graphs under-state independent calls (Q4_K dp4a 4096 x 4096
        # measured 1.77 / 1.67 / 1.63 us a call in graphs of 64 / 256 / 1000)
        n = max(256, w2.copies)
        times = {}
        for mode in (2, 1, 0):
            w2.overlap = mode
            ms, _, g2, _ = time_graph(torch, w2, n, replays=4)
            del g2
            times[MODE_NAMES[mode]] = ms
            if w2.kind in DP4A_KINDS and mode in (1, 0):
                msq, _, g3, _ = time_graph(torch, w2, n, with_quant=True, replays=4)
                times[MODE_NAMES[mode] + "_with_quantize"] = msq
                del g3
            if w2.kind == "qmm_q4k":
                # the same product on the fifth-generation tensor cores
                w2.tc5 = True
                mst, _, g5, _ = time_graph(torch, w2, n, replays=4)
                times[MODE_NAMES[mode] + "_tcgen05"] = mst
                w2.tc5 = False
                del g5
            if w2.kind == "q8_0_dp4a":
                # the quantization inside the matvec launch
                w2.fused = True
                msf, _, g4, _ = time_graph(torch, w2, n, replays=4)
                times[MODE_NAMES[mode] + "_quantize_fused"] = msf
                w2.fused = False
                del g4
        lines[name] = workload_line(name, times, peak)
        if rank == 0:
            print(json.dumps(lines[name]), flush=True)
        del w2
        torch.cuda.empty_cache()
    sampler.stop()
    clocks = sampler.summary(*clock_window)
    clocks["window"] = "nvidia-smi every 50 ms over a 0.5 s pre-roll, the timed region and a 0.5 s post-roll of the same graph"

    traffic = NCU_TRAFFIC.get(kernel_hash(), {}).get(head_mode)
    cpu, ref_y = cpu_baseline(args) if rank == 0 else (None, None)
    if rank == 0:
        def srel(a, b):
            return float(np.max(np.abs(a.astype(np.float64) - b)) / max(float(np.max(np.abs(b))), 1e-30))
        parity = {"scale_rel_timed_calls": round(srel(head_y, ref_y), 9),
                  "scale_rel_e2e": round(srel(e2e_y, ref_y), 9), "bound": 1e-4}
        parity["ok"] = parity["scale_rel_timed_calls"] <= 1e-4 and parity["scale_rel_e2e"] <= 1e-4
        e2e["matches_oracle"] = parity["scale_rel_e2e"] <= 1e-4
        summary = {}
        for nm in METRIC_CONFIGS:
            if nm in lines:
                summary[nm] = {m: lines[nm][m]["us"] for m in ("independent", "chain", "isolated") if m in lines[nm]}
                summary[nm]["independent_frac"] = lines[nm]["independent"]["frac"]
                summary[nm]["chain_frac"] = lines[nm]["chain"]["frac"]
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": K,
            "warmup": W,
            "ms_per_step": round(ms_step, 6),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32 activation as 3 exact int8 limbs, int32 dp4a dots, f32 sums",
            "data": "synthetic (seeded splitmix64 Q4_K blocks and N(0,1) activations; no model weights)",
            "config": {
                "workload": "q4k_4096x4096: Q4_K matvec rows=4096 k=4096 (attention-projection shape), seed 1",
                "rows": 4096, "k": 4096, "format": "Q4_K", "packed_weight_bytes": wbytes,
                "l2": f"inputs larger than L2: rotated weight copies ({lines[HEADLINE]['packed_weight_bytes']} B "
                      f"each, >3x the {l2 / 2**20:.0f} MiB L2 in total)" if HEADLINE in lines else "",
                "timing": "K calls captured in one CUDA graph, CUDA events on the launching stream",
                "launch": {0: "isolated calls (plain launches)",
                           1: "dependent decode chain (QMV_OVERLAP_CHAIN): each call streams its weights while the "
                              "previous call finishes and reads x after it",
                           2: "independent calls (QMV_OVERLAP_INDEPENDENT): each call streams its weights and "
                              "decodes while the previous call finishes and writes y after it"}[head_mode],
                "us_per_call": summary,
                "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
            },
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "peak_kind": f"{peak_kind} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_kind == "measured" else "fallback 6.8 TB/s",
                         "algorithmic_bytes_per_launch": alg},
            "e2e": e2e,
            "gpu_launches": K,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "parity": parity,
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def end_to_end(torch, q, wl, device, K):
    """Public API with host buffers: per step, copy the step's inputs (the
    weight and x, laid end to end in one pinned host buffer, so one copy moves
    both) to the device, run qmv_q4k on them, copy y back. The steps are
    enqueued on two streams that alternate, each with its own device buffers,
    so that one step's host-to-device copy overlaps the previous step's kernel
    and read-back (every step still moves its own inputs and result). Plain
    launches: each call follows the copy of its own inputs, which no overlap
    mode may run ahead of. Returns the record and the last step's output."""
    c = wl.c
    wb = np.ascontiguousarray(c["w"]).reshape(-1).view(np.uint8)
    xb = np.ascontiguousarray(c["x"], dtype=np.float32).reshape(-1).view(np.uint8)
    nw = wb.size   # a multiple of 16 (whole 144-byte blocks x rows of 16), so x stays 16-byte aligned
    assert nw % 16 == 0
    h = torch.from_numpy(np.concatenate([wb, xb])).pin_memory()
    hy = [torch.empty(wl.rows, dtype=torch.float32).pin_memory() for _ in range(2)]
    d = [torch.empty_like(h, device=device) for _ in range(2)]
    dy = [torch.empty(wl.rows, dtype=torch.float32, device=device) for _ in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    main = torch.cuda.Stream()
    steps = max(2, min(K, 200))

    def step(i):
        b = i & 1
        s = streams[b]
        with torch.cuda.stream(s):
            d[b].copy_(h, non_blocking=True)
            q.qmv_q4k(d[b].data_ptr(), d[b].data_ptr() + nw, dy[b], wl.rows, wl.k, stream=s.cuda_stream)
            hy[b].copy_(dy[b], non_blocking=True)

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for s in streams:
        s.wait_event(e0)
    for i in range(steps):
        step(i)
    for s in streams:
        main.wait_stream(s)
    e1.record(main)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    last = hy[(steps - 1) & 1].numpy().copy()
    return ({"value": round(weight_bytes(HEADLINE) / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
             "h2d_bytes_per_step": int(h.numel()), "d2h_bytes_per_step": 4 * wl.rows,
             "ms_per_step": round(ms, 4), "steps": steps,
             "pipelining": "two streams alternate steps: a step's host-to-device copy (weight and x in one "
                           "pinned buffer) overlaps the previous step's kernel and read-back"}, last)


# ------------------------------------------------------------- CPU side

def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(args, seconds: float = 10.0) -> dict:
    """The oracle as it stands, rows split over the host cores, repeated on the
    full headline workload for about `seconds` of wall time."""
    import oracle

    c = synth.make_config(HEADLINE)
    n = cpu_cores()
    ref_y = oracle.qmv_threaded("q4k", c["w"], c["x"], 4096, 4096, n)   # load + warm; the expected output
    calls = 0
    t0 = time.perf_counter()
    while True:
        oracle.qmv_threaded("q4k", c["w"], c["x"], 4096, 4096, n)
        calls += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    # the same oracle on one thread, for about a fifth of the time
    calls1 = 0
    t1 = time.perf_counter()
    while True:
        oracle.qmv("q4k", c["w"], c["x"], 4096, 4096)
        calls1 += 1
        if time.perf_counter() - t1 >= seconds / 5:
            break
    dt1 = time.perf_counter() - t1
    return ({"value": round(calls * weight_bytes(HEADLINE) / dt / 1e9, 4), "unit": "GB/s", "cores": n,
             "kind": "oracle",
             "sample": f"{calls} full 4096x4096 Q4_K matvecs (f64 dequantize-then-dot), rows split over {n} threads, "
                       f"{dt:.1f} s",
             "single_thread": {"value": round(calls1 * weight_bytes(HEADLINE) / dt1 / 1e9, 4), "unit": "GB/s",
                               "sample": f"{calls1} full matvecs on one thread, {dt1:.1f} s"}},
            np.asarray(ref_y, dtype=np.float64))


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle

    c = synth.make_config(HEADLINE)
    n = cpu_cores()
    for _ in range(args.warmup):
        oracle.qmv_threaded("q4k", c["w"], c["x"], 4096, 4096, n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.qmv_threaded("q4k", c["w"], c["x"], 4096, 4096, n)
    dt = time.perf_counter() - t0
    value = args.steps * weight_bytes(HEADLINE) / dt / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded splitmix64 Q4_K blocks and N(0,1) activations; no model weights)",
        "config": {"workload": "q4k_4096x4096: Q4_K matvec rows=4096 k=4096 (attention-projection shape), seed 1",
                   "rows": 4096, "k": 4096, "format": "Q4_K"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": n, "kind": "oracle",
                         "sample": f"each step one full 4096x4096 Q4_K matvec, rows split over {n} threads"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "the reference is the CPU oracle: the pages' own kernels are Vulkan/SPIR-V and cannot run here",
    }
    print(json.dumps(line))


def run_profile(args):
    """A few eager calls of one workload and nothing else: the command ncu
    captures (ncu flushes the caches between its replay passes, so one weight
    copy suffices)."""
    import torch

    import __graft_entry__
    import ggml_format_dequant_gb300 as q

    __graft_entry__.build()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    wl = Workload(q, torch, args.profile_workload, 0, device, copies=1)
    if args.headline_mode is not None:
        wl.overlap = args.headline_mode   # the launch mode (and plan) the bench times
    wl.tc5 = args.tcgen05
    s = torch.cuda.current_stream().cuda_stream
    for i in range(args.warmup + args.steps):
        wl.call(i, s, with_quant=True)
    torch.cuda.synchronize()
    print(json.dumps({"profile_workload": args.profile_workload, "calls": args.warmup + args.steps,
                      "y_finite": bool(torch.isfinite(wl.y).all().item())}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true", help="skip the per-config table")
    ap.add_argument("--headline-mode", type=int, choices=[0, 1, 2], default=None,
                    help="launch overlap of the headline calls (0 none, 1 chain, 2 independent); default 2")
    ap.add_argument("--only", default="", help="per-config table for the workloads whose names start with one of "
                                               "these comma-separated prefixes")
    ap.add_argument("--chain", action="store_true",
                    help="time the headline as a dependent decode chain (mode 1)")
    ap.add_argument("--isolated", action="store_true",
                    help="time the headline without decode-chain overlap (programmatic dependent launch off)")
    ap.add_argument("--profile-workload", choices=list(synth.CONFIGS),
                    help="only run warmup+steps eager calls of this workload (the command ncu captures)")
    ap.add_argument("--tcgen05", action="store_true",
                    help="with --profile-workload qmm_q4k_*: run the fifth-generation tensor-core kernel")
    args = ap.parse_args()
    if args.profile_workload:
        run_profile(args)
        return
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
