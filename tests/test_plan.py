"""The launch planners without a GPU: for each shape (the configured
workloads, the GPU test shapes, forced configurations and the seeded random
cases) the plan is taken from the library for a described GB300 and the
kernel's work assignment is replayed here, so that every index the kernel
forms is checked before it runs. For the matvec kernel:

* every (row, unit) pair of every matrix is decoded exactly once;
* every shared-memory read of a unit (including the bytes a format's loads
  read past its block) stays inside its ring slot, and every slot holds the
  16-byte-aligned cover its bulk copy writes;
* unit addresses have the alignment their loads need (16 bytes for Q4_K and Q5_K, 8 for
  the aligned Q8_0 dp4a path, 2 otherwise);
* parked partials stay inside the CTA's table, and the shared-memory regions
  are disjoint and fit the device.

For the tensor-core batch kernel (qmm_tc.cuh): the k-chunks tile every row,
every row's chunk copy fits its slot row, every staged-row read of a tile
(spare rows included) stays inside its slot, and the shared-memory regions
are disjoint and fit the device; independent-call plans also fit in half an
SM.

The replays restate the kernels' arithmetic (qmv_kernel.cuh, qmm_tc.cuh) in
numpy; they check index bounds, not numerics."""

import numpy as np
import pytest

DEVICE = (152, 232448, 233472, 1024)
FMT_ID = {"q4k": 0, "q6k": 1, "q8_0": 2, "q8d": 3, "moe": 4, "q4d": 5, "moe6": 6, "moe4d": 7, "q5k": 8,
          "q4_0": 9, "moe8": 10, "moe40": 11, "moe5": 12,
          "q6d": 16, "moe6d": 17, "q8dq": 18}


# Per format: weights per block, bytes per block, blocks per warp slice,
# units per row, a unit's block offset in its slice, and the byte range a
# unit's loads touch relative to its address a (lo may depend on a & 3).
def fmt_info(fmt, m=1):
    if fmt in ("q4k", "moe", "q4d", "moe4d"):
        return dict(qk=256, bb=144, sb=8, units=lambda nb: 4 * nb, ubyte=lambda u: (u >> 2) * 144,
                    extent=lambda a: (a, a + 144), align=16)
    if fmt in ("q5k", "moe5"):
        return dict(qk=256, bb=176, sb=8, units=lambda nb: 4 * nb, ubyte=lambda u: (u >> 2) * 176,
                    extent=lambda a: (a, a + 176), align=16)
    if fmt in ("q4_0", "moe40"):
        # five 32-bit loads from the word below the 2-byte aligned block
        return dict(qk=32, bb=18, sb=32, units=lambda nb: nb, ubyte=lambda u: u * 18,
                    extent=lambda a: (a - (a & 3), a - (a & 3) + 20), align=2)
    if fmt in ("q6k", "moe6", "q6d", "moe6d"):
        return dict(qk=256, bb=210, sb=8, units=lambda nb: 4 * nb, ubyte=lambda u: (u >> 2) * 210,
                    extent=lambda a: (a - (a & 3), a - (a & 3) + 212), align=2)
    if fmt in ("q8_0", "moe8"):
        return dict(qk=32, bb=34, sb=32, units=lambda nb: nb, ubyte=lambda u: u * 34,
                    extent=lambda a: (a - (a & 3), a - (a & 3) + 40), align=2)
    if fmt in ("q8d", "q8dq"):
        # aligned path: [a, a + 136); block-by-block path: up to a + 142
        return dict(qk=32, bb=34, sb=128, units=lambda nb: (nb + 3) // 4, ubyte=lambda u: u * 136,
                    extent=lambda a: (a - (a & 3), a - (a & 3) + 144), align=2)
    raise ValueError(fmt)


@pytest.fixture(scope="module")
def q():
    import __graft_entry__
    __graft_entry__.build()
    import ggml_format_dequant_gb300 as lib
    return lib


def replay(q, fmt, rows, k, slots=1, cfg=None, mode=0):
    """Replay the plan computed under launch mode `mode` (0: plain, 2:
    independent calls)."""
    P = q.qmv_plan_detail(FMT_ID[fmt], rows, k, slots, cfg, DEVICE, overlap=mode)
    f = fmt_info(fmt, slots)
    nb = k // f["qk"]
    U = f["units"](nb)
    KS, GS, NG, CR, S, R, W = P["KS"], P["GS"], P["NG"], P["CR"], P["S"], P["unroll"], P["W"]
    rowbytes, stride, parts = P["rowbytes"], P["slot_stride"], P["ctas"]
    assert rowbytes == nb * f["bb"] and U == P["U"]
    early = 1 if mode == 2 else 0
    assert KS == (U + 31) // 32 and W == (KS if KS > 1 else early) and GS & (GS - 1) == 0 and U <= KS * GS
    assert 32 * NG * KS == P["threads"] <= 512
    assert P["rq"] * parts + P["rrem"] == rows and 0 <= P["rrem"] < parts
    # clusters share the activation prep: the CTAs of a matrix fill whole
    # clusters, every CTA converts an even number of 16-element halves, and the
    # integer-activation path has no prep to share
    CL = P["CL"]
    assert CL in (1, 2, 4, 8) and parts % CL == 0 and (k // 16) % (2 * CL) == 0
    assert P["rq"] >= 1
    if fmt in ("q8d", "q4d", "moe4d", "q6d", "moe6d", "q8dq"):
        assert CL == 1
    lg = GS.bit_length() - 1
    rpw = 32 >> lg
    aligned8 = P["aligned8"] == 1
    if fmt in ("q8d", "q8dq"):
        assert aligned8 == (rowbytes % 8 == 0)

    # shared-memory layout: disjoint, ordered regions inside the device limit
    regions = []
    if fmt == "q8dq":
        # the CTA's own codes and scales of x
        regions += [(P["off_la"], k), (P["off_xs"], 4 * (k // 32))]
    elif fmt not in ("q8d", "q4d", "moe4d", "q6d", "moe6d"):
        regions += [(P["off_la"], k), (P["off_lb"], k), (P["off_lc"], k), (P["off_xs"], 4 * (k // 32)),
                    (P["off_xsum16"], 4 * (k // 16))]
        for o, _ in regions:
            assert o % 16 == 0
    rpc = P["rq"] + (1 if P["rrem"] else 0)
    regions += [(P["off_red"], 4 * rpc * W), (P["off_ring"], NG * S * stride), (P["off_bars"], 8 * NG * S),
                (P["off_cnt"], 4 * (NG * S + NG + 1))]
    regions.sort()
    for (o1, n1), (o2, _) in zip(regions, regions[1:]):
        assert o1 + n1 <= o2
    assert regions[-1][0] + regions[-1][1] <= P["smem"] <= DEVICE[1]
    assert P["off_ring"] % 128 == 0 and stride % 128 == 0 and P["off_bars"] % 8 == 0

    lanes = np.arange(32)
    covered = np.zeros((rows, U), dtype=np.int32)
    for part in range(parts):
        big = part < P["rrem"]
        nrows = P["rq"] + (1 if big else 0)
        R0 = part * P["rq"] + min(part, P["rrem"])
        gq, grem = (P["gq1"], P["grem1"]) if big else (P["gq0"], P["grem0"])
        assert gq * NG + grem == nrows
        for rg in range(NG):
            glo = rg * gq + min(rg, grem)
            gn = gq + (1 if rg < grem else 0)
            npc = -(-gn // CR)
            for pc in range(npc):
                nr = min(CR, gn - pc * CR)
                rl0 = glo + pc * CR
                gs = (R0 + rl0) * rowbytes          # the weight base is 16-byte aligned
                d0 = gs & 15
                a0, a1 = gs & ~15, (gs + nr * rowbytes + 15) & ~15
                assert a1 - a0 <= stride               # the bulk copy's cover fits its slot
                for ks in range(KS):
                    u = (lanes & (GS - 1)) if KS == 1 else lanes
                    sub = (lanes >> lg) if KS == 1 else np.zeros(32, dtype=int)
                    ug = ks * 32 + u
                    has = ug < U
                    # lanes past the last unit decode the last unit (result dropped)
                    uc = np.where(has, u, U - 1 - ks * 32)
                    assert np.all(uc >= 0)
                    ubyte = ks * f["sb"] * f["bb"] + np.array([f["ubyte"](int(v)) for v in uc])
                    # R-row steps, then single steps for the remainder
                    steps, jb = [], 0
                    while jb + R * rpw <= nr:
                        steps.append((jb, R))
                        jb += R * rpw
                    while jb < nr:
                        steps.append((jb, 1))
                        jb += rpw
                    for jb, nq in steps:
                        for qq in range(nq):
                            j = jb + qq * rpw + sub
                            valid = j < nr
                            jj = np.where(valid, j, 0)
                            a = d0 + jj * rowbytes + ubyte
                            for ai in a:
                                lo, hi = f["extent"](int(ai))
                                assert 0 <= lo and hi <= stride, (ai, lo, hi, stride)
                                assert ai % f["align"] == 0
                                if fmt in ("q8d", "q8dq") and aligned8:
                                    assert ai % 8 == 0
                            sel = valid & has
                            np.add.at(covered, (R0 + rl0 + j[sel], ug[sel]), 1)
                            # parked slice sum of every valid row (rows of several slices)
                            if KS > 1:
                                idx = (rl0 + j[valid]) * W + ks
                                assert idx.size == 0 or (idx.min() >= 0 and idx.max() < nrows * W)
    assert np.all(covered == 1), np.argwhere(covered != 1)[:5]
    return P


WORKLOADS = [("q4k", 4096, 4096, 1), ("q4k", 256, 1024, 1), ("q8d", 14336, 4096, 1), ("q8dq", 14336, 4096, 1),
             ("q6k", 4096, 14336, 1),
             ("moe", 768, 2048, 8), ("q4d", 4096, 4096, 1), ("moe6", 2048, 768, 8), ("moe4d", 768, 2048, 8),
             ("q5k", 4096, 4096, 1), ("q4_0", 4096, 4096, 1), ("moe8", 768, 2048, 8), ("moe40", 768, 2048, 8),
             ("moe5", 768, 2048, 8), ("q6d", 4096, 14336, 1), ("moe6d", 2048, 768, 8)]


@pytest.mark.parametrize("fmt,rows,k,slots", WORKLOADS)
def test_workload_plans(q, fmt, rows, k, slots):
    P = replay(q, fmt, rows, k, slots)
    assert P["S"] >= 1
    if (fmt, rows) in (("q4k", 4096), ("moe", 768)):
        # the whole share in flight at once, in small CTAs that leave room for
        # the next call's CTA on every SM
        assert P["S"] == 1 and P["CR"] * P["NG"] >= P["rq"]
        assert P["threads"] <= 256 and P["smem"] <= (DEVICE[2] - 2 * DEVICE[3]) // 2
    if (fmt, rows) in (("q8d", 14336), ("q6k", 4096)):
        # streamed through a ring at least two slots deep
        assert P["S"] >= 2


SHAPES = [("q4k", 300, 768), ("q4k", 1, 256), ("q4k", 97, 4352), ("q4k", 20, 16384), ("q6k", 300, 512),
          ("q6k", 3, 256), ("q6k", 41, 14336), ("q6k", 130, 2816), ("q8_0", 300, 96), ("q8_0", 7, 4096),
          ("q8_0", 13, 32), ("q8_0", 64, 11008), ("q8d", 300, 4096), ("q8d", 7, 96), ("q8d", 1, 32),
          ("q8d", 61, 256), ("q8d", 5, 4160), ("moe", 96, 512, ), ("moe", 7, 256), ("q4d", 300, 768), ("q4d", 1, 256),
          ("q4d", 97, 4352), ("q4d", 20, 16384), ("moe6", 96, 512), ("moe6", 7, 256), ("moe4d", 40, 512),
          ("q5k", 300, 768), ("q5k", 1, 256), ("q5k", 97, 4352), ("q5k", 20, 16384), ("q4_0", 300, 96),
          ("q4_0", 7, 4096), ("q4_0", 13, 32), ("q4_0", 64, 11008), ("q4_0", 33, 1056), ("moe8", 96, 512),
          ("moe8", 7, 96), ("moe40", 96, 512), ("moe40", 7, 96), ("moe5", 40, 512), ("moe5", 7, 256),
          ("q6d", 300, 512), ("q6d", 3, 256), ("q6d", 41, 14336), ("q6d", 130, 2816), ("moe6d", 96, 512),
          ("moe6d", 7, 256)]


@pytest.mark.parametrize("shape", SHAPES)
def test_shape_plans(q, shape):
    fmt, rows, k = shape
    replay(q, fmt, rows, k, 4 if fmt.startswith("moe") else 1)


CFGS = [dict(ctas=1, chunk_rows=1, chunks=2), dict(ctas=3, chunk_rows=5, chunks=2), dict(ctas=2, chunk_rows=3, chunks=1),
        dict(ctas=7, chunks=3), dict(ctas=1, chunks=2, unroll=1), dict(ctas=3, chunk_rows=4, chunks=3, unroll=2),
        dict(ctas=2, chunks=1, warps=2), dict(ctas=5, chunk_rows=2, chunks=4, warps=4),
        dict(ctas=1, chunk_rows=7, chunks=2, warps=16, unroll=1)]


@pytest.mark.parametrize("cfg", CFGS)
@pytest.mark.parametrize("fmt", ["q4k", "q6k", "q8_0", "q8d", "q4d", "q5k", "q4_0", "q6d"])
def test_forced_plans(q, fmt, cfg):
    replay(q, fmt, 61, 512 if fmt != "q8d" else 256, 1, cfg)


WIDE_CFGS = [dict(ctas=1, chunk_rows=3, chunks=2), dict(ctas=2, chunk_rows=1, chunks=1),
             dict(ctas=3, chunk_rows=2, chunks=3, unroll=1), dict(ctas=1, chunks=2, warps=16)]


@pytest.mark.parametrize("cfg", WIDE_CFGS)
@pytest.mark.parametrize("fmt,k", [("q4k", 4352), ("q6k", 2816), ("q8_0", 4096), ("q4k", 16384), ("q5k", 4352),
                                   ("q4_0", 4096), ("q4_0", 1056)])
def test_forced_wide_plans(q, fmt, k, cfg):
    replay(q, fmt, 29, k, 1, cfg)


def test_moe_forced_plan(q):
    replay(q, "moe", 40, 512, 5, dict(ctas=2, chunk_rows=3, chunks=2))
    for fmt in ("moe8", "moe40", "moe5", "moe6d"):
        replay(q, fmt, 40, 512, 5, dict(ctas=2, chunk_rows=3, chunks=2))


def test_retired_batch_plan_ids(q):
    """Batches of two or more rows run on the tensor cores: plan ids 13-15 are
    refused."""
    for fid in (13, 14, 15):
        with pytest.raises(q.QmvError):
            q.qmv_plan_detail(fid, 64, 512, 2, None, DEVICE)


@pytest.mark.parametrize("fmt,rows,k,slots", WORKLOADS)
def test_independent_call_plans(q, fmt, rows, k, slots):
    """Independent calls: a fifth of the SM count in CTAs (shared by the
    slots of an MoE call) of at most 8 warps, in half an SM's shared memory,
    each streaming its share of the rows through two ring slots (one when a
    row group has a single piece); every index is replayed as for the default
    plans."""
    P = replay(q, fmt, rows, k, slots, mode=2)
    per = max(slots, 1)
    half = (DEVICE[2] - 2 * DEVICE[3]) // 2
    want = max(1, -(-(DEVICE[0] // 5) // per))
    default = q.qmv_plan_detail(FMT_ID[fmt], rows, k, slots, None, DEVICE)
    if want < default["ctas"]:
        assert P["ctas"] == want
        assert P["smem"] <= half and P["threads"] <= 256
        gmax = P["gq1"] + (1 if P["grem1"] else 0)
        assert P["S"] == min(2, -(-gmax // P["CR"]))
    else:   # small shapes keep the default CTAs and pieces (y then parked until the wait)
        assert (P["ctas"], P["CR"], P["S"], P["W"]) == (default["ctas"], default["CR"], default["S"],
                                                          max(default["W"], 1))


def test_chain_shapes(q):
    for fmt in ("q4k", "q6k"):
        replay(q, fmt, 2048, 2048)
    replay(q, "moe", 2048, 2048, 2)


def test_planner_rejects(q):
    assert q.qmv_plan_detail.__name__
    with pytest.raises(q.QmvError):
        q.qmv_plan_detail(FMT_ID["q4k"], 10, 256 * 1024, 1, None, DEVICE)   # 64 k-slices per row
    with pytest.raises(q.QmvError):
        q.qmv_plan_detail(FMT_ID["q4k"], 10, 8192, 1, dict(warps=2), DEVICE)   # 4 slices, 2 warps


# ------------------------------------------- tensor-core batch plan (qmm_tc)

TC_FMT = {"q4k": (0, 256, 144), "q6k": (1, 256, 210), "q8_0": (2, 32, 34), "q5k": (3, 256, 176), "q4_0": (4, 32, 18)}


def tc_max_read(fmt, slices, groups):
    """Last byte (exclusive) a lane may read past the first byte of a staged
    row's k-chunk of `slices` slices and `groups` groups."""
    if fmt == "q4k":
        return slices * 144
    if fmt == "q5k":
        return slices * 176
    if fmt == "q6k":
        return (slices - 1) * 210 + 216   # funnel loads of d at 208: 8 bytes from the word below
    if fmt == "q4_0":
        return (groups - 1) * 18 + 22     # codes at 2 + 4t: 8 bytes from the word below
    return (groups - 1) * 34 + 38          # codes at 18 + 4t: 8 bytes from the word below


def tc_replay(q, fmt, rows, k, m, cfg=None, mode=0):
    """Replay the tensor-core plan computed under launch mode `mode` (0:
    plain, 2: independent calls, where CTAs of at most 8 warps take at most
    half an SM's shared memory unless that plan does not fit)."""
    fid, qk, bb = TC_FMT[fmt]
    P = q.qmm_tc_plan_detail(fid, rows, k, m, cfg, DEVICE, overlap=mode)
    ng = k // 32
    NS = -(-ng // 8)
    kmax = min(cfg["warps"], 16) if cfg and cfg.get("warps") else 16
    half = (DEVICE[2] - 2 * DEVICE[3]) // 2
    if mode == 2 and not (cfg and cfg.get("warps")) and P["threads"] <= 32 * 8:
        kmax = 8
        assert P["smem"] <= half
    nch = -(-NS // kmax)
    KS = -(-NS // nch)
    assert P["KS"] == KS and P["nchunks"] == nch and P["threads"] == 32 * KS <= 512 and P["ngroups"] == ng
    rowbytes = (k // qk) * bb
    cgroups = 8 * KS
    chunk = min(cgroups * 32 // qk * bb, rowbytes)
    stride, CR, S, parts = P["stride"], P["CR"], P["S"], P["ctas"]
    assert P["chunk_bytes"] == chunk
    assert stride % 128 == 16 and stride >= chunk + 16
    cap = -(-CR // 16) * 16
    assert P["slot_stride"] >= cap * stride and P["slot_stride"] % 128 == 0
    assert P["rq"] * parts + P["rrem"] == rows and P["rq"] >= 1
    rpc = P["rq"] + (1 if P["rrem"] else 0)
    sums = 32 * 32 * KS if fmt in ("q4k", "q5k") else 0   # 32 bytes a thread (min-term fragments)
    regions = [(P["off_red"], 4 * rpc * KS * 8), (P["off_sums"], sums), (P["off_ring"], S * P["slot_stride"]),
               (P["off_bars"], 8 * S), (P["off_cnt"], 4 * (S + 2))]
    regions.sort()
    for (o1, n1), (o2, _) in zip(regions, regions[1:]):
        assert o1 + n1 <= o2
    assert regions[-1][0] + regions[-1][1] <= P["smem"] <= DEVICE[1]
    assert P["off_ring"] % 128 == 0 and P["off_bars"] % 8 == 0 and P["off_red"] % 16 == 0 and P["off_sums"] % 16 == 0
    # the chunks tile each row: chunk c holds groups [c * cgroups, ...), every
    # chunk non-empty, the last one ending at the row's end
    ends = []
    for c in range(nch):
        gc = min(cgroups, ng - c * cgroups)
        assert gc > 0
        cb = gc * 32 // qk * bb
        woff = c * chunk
        assert woff == c * cgroups * 32 // qk * bb and woff + cb <= rowbytes
        ends.append((woff, cb, -(-gc // 8), gc))
    assert ends[-1][0] + ends[-1][1] == rowbytes
    wbytes = rows * rowbytes
    covered = np.zeros(rows, dtype=np.int64)
    for woff, cb, slices, gc in ends:
        last = tc_max_read(fmt, slices, gc)
        for part in range(parts):
            nrows = P["rq"] + (1 if part < P["rrem"] else 0)
            R0 = part * P["rq"] + min(part, P["rrem"])
            for pc in range(-(-nrows // CR)):
                nr = min(CR, nrows - pc * CR)
                for i in range(nr):
                    gs = (R0 + pc * CR + i) * rowbytes + woff   # the weight base is 16-byte aligned
                    a0, a1 = gs & ~15, (gs + cb + 15) & ~15
                    if a1 > wbytes:
                        a1 = (gs + cb) & ~15
                    assert a1 - a0 <= stride
                    covered[R0 + pc * CR + i] += cb
                # every row a tile touches (spare rows included) stays in the slot
                for r in range(0, nr, 16):
                    for ia in range(r, r + 16):
                        assert ia < cap
                        ph = ((R0 + pc * CR + ia) * rowbytes + woff) & 15
                        assert ia * stride + ph + last <= P["slot_stride"]
    assert np.all(covered == rowbytes)
    return P


TC_SHAPES = [("q4k", 4096, 4096), ("q4k", 300, 768), ("q4k", 1, 256), ("q4k", 97, 2304), ("q6k", 4096, 4096),
             ("q6k", 300, 512), ("q6k", 3, 256), ("q6k", 41, 3840), ("q8_0", 14336, 4096), ("q8_0", 300, 96),
             ("q8_0", 13, 32), ("q8_0", 7, 4064), ("q8_0", 64, 1056), ("q4k", 20, 16384), ("q4k", 97, 4352),
             ("q6k", 4096, 14336), ("q6k", 41, 14336), ("q8_0", 64, 11008), ("q8_0", 5, 4160), ("q8_0", 3, 12320),
             ("q5k", 4096, 4096), ("q5k", 37, 512), ("q5k", 3, 4352), ("q5k", 1, 256), ("q4_0", 4096, 4096),
             ("q4_0", 300, 96), ("q4_0", 13, 32), ("q4_0", 64, 11008), ("q4_0", 7, 4160), ("q4k", 40, 65536),
             ("q6k", 40, 65536), ("q8_0", 40, 65536), ("q5k", 40, 65536), ("q4_0", 40, 65536)]


@pytest.mark.parametrize("m", [1, 2, 5, 8])
@pytest.mark.parametrize("shape", TC_SHAPES)
def test_tc_plans(q, shape, m):
    fmt, rows, k = shape
    tc_replay(q, fmt, rows, k, m)


@pytest.mark.parametrize("cfg", [dict(ctas=1, chunk_rows=1, chunks=2), dict(ctas=3, chunk_rows=5, chunks=2),
                                 dict(ctas=2, chunk_rows=20, chunks=1), dict(ctas=7, chunks=3),
                                 dict(ctas=1, chunk_rows=16, chunks=2), dict(ctas=2, chunks=2, warps=1),
                                 dict(ctas=3, chunk_rows=7, chunks=3, warps=3)])
@pytest.mark.parametrize("fmt", ["q4k", "q6k", "q8_0", "q5k", "q4_0"])
def test_tc_forced_plans(q, fmt, cfg):
    tc_replay(q, fmt, 61, 512, 3, cfg)


@pytest.mark.parametrize("shape", TC_SHAPES)
@pytest.mark.parametrize("m", [2, 4, 8])
def test_tc_independent_call_plans(q, shape, m):
    """Independent calls: every index replayed as for the default plans; the
    suite's large matrices take CTAs of at most 8 warps in half an SM."""
    fmt, rows, k = shape
    P = tc_replay(q, fmt, rows, k, m, mode=2)
    if rows >= 4096 and k >= 4096:
        assert P["threads"] <= 256 and P["smem"] <= (DEVICE[2] - 2 * DEVICE[3]) // 2


def test_tc_long_rows_take_kchunks(q):
    """Rows longer than 16 slices are dealt into balanced k-chunks of one
    launch: 14336 weights = 56 slices = 4 chunks of 14, 4352 = 17 slices = 2
    chunks of 9 (the second one 8); a warps bound forces more chunks."""
    assert tc_replay(q, "q6k", 4096, 14336, 4)["nchunks"] == 4
    P = tc_replay(q, "q4k", 64, 4352, 4)
    assert (P["nchunks"], P["KS"]) == (2, 9)
    P = tc_replay(q, "q8_0", 13, 1056, 5, dict(warps=2))
    assert (P["nchunks"], P["KS"]) == (3, 2)
    with pytest.raises(q.QmvError):
        q.qmm_tc_plan_detail(0, 64, 4100, 4, None, DEVICE)   # k not a multiple of 256


def _random_cases():
    from test_gpu_random_shapes import cases
    return cases()


@pytest.mark.parametrize("fam,rows,k,cfg", _random_cases())
def test_random_shape_plans(q, fam, rows, k, cfg):
    """The seeded random shapes and forced plans of the GPU test, replayed on
    the host before they run (a plan the host refuses is never launched)."""
    try:
        replay(q, fam, rows, k, 1, cfg)
    except q.QmvError as e:
        assert cfg is not None and e.code == q.QMV_ETOOBIG


def _random_batch_cases():
    from test_gpu_random_shapes import batch_cases
    return batch_cases()


@pytest.mark.parametrize("fmt,rows,k,m,cfg,mode", _random_batch_cases())
def test_random_batch_plans(q, fmt, rows, k, m, cfg, mode):
    """The seeded random batches of the GPU test, every tile's plan replayed on
    the host before they run (a plan the host refuses is never launched)."""
    tiles = -(-m // 8)
    for mt in sorted({m // tiles + (1 if t < m % tiles else 0) for t in range(tiles)}):
        try:
            tc_replay(q, fmt, rows, k, mt, cfg, mode=mode)
        except q.QmvError as e:
            assert cfg is not None and e.code == q.QMV_ETOOBIG


def _tc_sweep(n=240):
    import synth
    fmts = list(TC_FMT)
    z = synth.Stream(9090).draw(n * 8).reshape(n, 8)
    out = []
    for i in range(n):
        d = [int(v >> np.uint64(33)) for v in z[i]]
        fmt = fmts[d[0] % len(fmts)]
        qk = TC_FMT[fmt][1]
        k = (1 + d[1] % (20000 // qk)) * qk
        rows = 1 + d[2] % 3000
        m = 1 + d[3] % 8
        cfg = None
        if d[4] % 3 == 0:
            cfg = dict(ctas=d[5] % 200, chunk_rows=d[6] % 40, chunks=d[7] % 6, warps=[0, 1, 2, 5, 8, 16][d[4] % 6])
        mode = 2 if d[6] % 2 else 0
        out.append((fmt, rows, k, m, cfg, mode))
    return out


@pytest.mark.parametrize("fmt,rows,k,m,cfg,mode", _tc_sweep())
def test_tc_plan_sweep(q, fmt, rows, k, m, cfg, mode):
    """A wider seeded sweep of tensor-core plans (rows up to 3000, k up to
    20000, forced configurations, both launch modes), replayed on the host
    only: every plan the planner returns keeps its copies and reads in bounds;
    a forced plan may be refused, never a default one."""
    try:
        tc_replay(q, fmt, rows, k, m, cfg, mode=mode)
    except q.QmvError as e:
        assert cfg is not None and e.code == q.QMV_ETOOBIG


MV_QK = {"q4k": 256, "q6k": 256, "q8_0": 32, "q5k": 256, "q4_0": 32, "q8d": 32, "q4d": 256, "q6d": 256,
         "moe": 256, "moe6": 256, "moe4d": 256, "moe8": 32, "moe40": 32, "moe5": 256, "moe6d": 256}


def _mv_sweep(n=240):
    import synth
    fams = list(MV_QK)
    z = synth.Stream(8080).draw(n * 8).reshape(n, 8)
    out = []
    for i in range(n):
        d = [int(v >> np.uint64(33)) for v in z[i]]
        fam = fams[d[0] % len(fams)]
        qk = MV_QK[fam]
        k = (1 + d[1] % (8192 // qk)) * qk
        rows = 1 + d[2] % 2500
        slots = 1 + d[3] % 8 if fam.startswith("moe") else 1
        cfg = None
        if d[4] % 3 == 0:
            cfg = dict(ctas=d[5] % 200, chunk_rows=d[6] % 12, chunks=d[7] % 5, unroll=d[4] % 3,
                       warps=[0, 2, 4, 8, 16][d[5] % 5])
        mode = 2 if d[6] % 2 else 0
        out.append((fam, rows, k, slots, cfg, mode))
    return out


@pytest.mark.parametrize("fam,rows,k,slots,cfg,mode", _mv_sweep())
def test_matvec_plan_sweep(q, fam, rows, k, slots, cfg, mode):
    """A wider seeded sweep of matvec and MoE plans (rows up to 2500, k up to
    8192, 1-8 slots, forced configurations, both launch modes), replayed on the
    host only: every (row, unit) decoded once, every read inside its slot; a
    forced plan may be refused, never a default one."""
    try:
        replay(q, fam, rows, k, slots, cfg, mode=mode)
    except q.QmvError as e:
        assert cfg is not None and e.code == q.QMV_ETOOBIG
