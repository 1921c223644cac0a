"""Host replay of the tcgen05 batch kernel's plan (qmm_q4k_tc5_plan_detail,
no GPU): for a sweep of shapes and forced plans, every index the kernel
derives from the plan stays inside its buffer. Checked here:
* every rank's k-chunk, the rows it adds up, and its inbox slot;
* the shared-memory regions the kernel writes (ring, B, B', scales, staged x,
  inbox, barriers) do not overlap and fit the CTA's allocation;
* the MMA descriptors' B reads and the TMA tensor coordinates stay in range.
"""

import itertools

import pytest

import ggml_format_dequant_gb300 as q

DEV = q.GB300_DEVICE
SLOT = 128 * 144          # one super-block column of a 128-row tile
STATIC_SMEM_MARGIN = 1024


def shapes():
    ks = [256, 512, 768, 1024, 1280, 1536, 1792, 2560, 3072, 4096, 5632, 7168, 14336]
    rows = [1, 127, 128, 129, 1578, 4096]
    for k, r, m in itertools.product(ks, rows, (1, 3, 8)):
        for cl in (0, 1, 2, 3, 5, 6, 7, 8):
            yield r, k, m, cl


def replay(rows, k, m, cl, chunks=0):
    cfg = {}
    if cl:
        cfg["cluster"] = cl
    if chunks:
        cfg["chunks"] = chunks
    try:
        P = q.qmm_q4k_tc5_plan_detail(rows, k, m, cfg=cfg or None, device=DEV)
    except q.QmvError as e:
        assert e.code == q.QMV_ETOOBIG
        return None
    nsb = k // 256
    CL, S = P["CL"], P["S"]
    assert P["nsb"] == nsb
    # power of two, within the cluster limit, the super-blocks, and the request
    assert CL & (CL - 1) == 0 and 1 <= CL <= 8 and CL <= nsb
    if cl:
        assert CL <= cl
    assert 128 % CL == 0
    nq_max = -(-nsb // CL)
    for c in range(CL):
        q0 = c * nsb // CL
        nq = (c + 1) * nsb // CL - q0
        assert 1 <= nq <= nq_max
        # TMA tensor coordinates (8-byte elements) of the chunk's super-blocks
        assert (q0 + nq) * 18 <= nsb * 18
        # B descriptors: the last step's second k-block, rows 8..15
        assert (32 * nq - 1) * 256 + 128 + 128 <= nq_max * 32 * 256
    rpr = 128 // CL
    for r in range(128):
        dst, rl = r // rpr, r % rpr
        assert dst < CL
        for c in range(CL):
            assert (c * rpr + rl) * 32 + 32 <= 128 * 8 * 4
    assert 1 <= S <= max(1, nq_max)
    # regions in order, each large enough, aligned as the copies need
    assert P["off_b"] >= S * SLOT and P["off_b"] % 128 == 0
    assert P["off_bm"] >= P["off_b"] + nq_max * 32 * 256 and P["off_bm"] % 16 == 0
    assert P["off_sc"] >= P["off_bm"] + nq_max * 512
    assert P["off_x"] >= P["off_sc"] + nq_max * 8 * 2 * 4 and P["off_x"] % 16 == 0
    assert P["off_in"] >= P["off_x"] + m * nq_max * 256 * 4 and P["off_in"] % 16 == 0
    assert P["off_bars"] >= P["off_in"] + 128 * 8 * 4 and P["off_bars"] % 8 == 0
    assert P["smem"] >= P["off_bars"] + 8 * (2 * S + 10)
    assert P["smem"] <= DEV[1] - STATIC_SMEM_MARGIN
    # at least 80 KB keeps two CTAs an SM at most (two tensor-memory allocations)
    assert P["smem"] >= 80 * 1024
    assert 3 * (P["smem"] + DEV[3]) > DEV[2]
    assert P["ctas"] == -(-rows // 128) * CL and P["threads"] == 160
    return P


def test_plans_stay_in_bounds():
    n = 0
    for r, k, m, cl in shapes():
        if replay(r, k, m, cl) is not None:
            n += 1
    assert n > 1000


@pytest.mark.parametrize("chunks", [1, 2, 3, 4, 8])
def test_forced_ring_depths(chunks):
    for k in (1024, 4096, 14336):
        for cl in (1, 2, 4, 8):
            replay(1000, k, 8, cl, chunks)


def test_default_cluster_sizes():
    """The default splits a tile's k into the most power-of-two chunks up to
    eight: k / 256 = 6 super-blocks give 4 chunks, 22 give 8."""
    assert q.qmm_q4k_tc5_plan_detail(4096, 1536, 4)["CL"] == 4
    assert q.qmm_q4k_tc5_plan_detail(1578, 5632, 8)["CL"] == 8
    assert q.qmm_q4k_tc5_plan_detail(1578, 5632, 8, cfg={"cluster": 6})["CL"] == 4
    assert q.qmm_q4k_tc5_plan_detail(300, 256, 2)["CL"] == 1


def test_streaming_plans_stay_in_bounds():
    """Independent calls take the streaming plan for every k (one CTA a
    128-row tile; rings of weight copies, of B / B' / scales for 4
    super-blocks, and of the rows' d / dmin for 8); every region the kernel
    writes fits, in order, and the plan keeps every other tensor-memory CTA
    off its SM."""
    SB, SD, NBARS_FIXED = 4, 8, 33
    for k in (256, 512, 1024, 2048, 3072, 4096, 5632, 6144, 7168, 14336, 65536):
        for rows in (1, 128, 300, 4096):
            for m in (1, 4, 8):
                for chunks in (0, 1, 2, 4, 6, 8, 12):
                    cfg = {"chunks": chunks} if chunks else None
                    P = q.qmm_q4k_tc5_plan_detail(rows, k, m, cfg=cfg, device=DEV, overlap=q.OVERLAP_INDEPENDENT)
                    assert P["streaming"] == 1
                    nsb, S = k // 256, P["S"]
                    assert P["CL"] == 1 and P["nsb"] == nsb and 1 <= S <= min(nsb, chunks or 6)
                    assert P["ctas"] == -(-rows // 128) and P["threads"] == 19 * 32
                    assert P["off_b"] >= S * SLOT and P["off_b"] % 128 == 0
                    assert P["off_bm"] >= P["off_b"] + SB * 32 * 256 and P["off_bm"] % 16 == 0
                    assert P["off_sc"] >= P["off_bm"] + SB * 512 and P["off_sc"] % 16 == 0
                    off_dm = P["off_x"]
                    assert off_dm >= P["off_sc"] + SB * 8 * 2 * 4 and off_dm % 8 == 0
                    assert P["off_in"] == 0
                    assert P["off_bars"] >= off_dm + SD * 128 * 8 and P["off_bars"] % 8 == 0
                    assert P["smem"] >= P["off_bars"] + 8 * (2 * S + NBARS_FIXED)
                    assert P["smem"] <= DEV[1] - STATIC_SMEM_MARGIN
                    # one CTA an SM, and no CTA of the cluster plan (at least 80 KB)
                    # beside it: nothing else on the SM holds tensor memory
                    assert 2 * (P["smem"] + DEV[3]) > DEV[2]
                    assert P["smem"] + DEV[3] + 80 * 1024 + DEV[3] > DEV[2]
    # a forced cluster size keeps the cluster plan, and so do the other modes
    assert q.qmm_q4k_tc5_plan_detail(4096, 4096, 8, cfg={"cluster": 8}, device=DEV,
                                     overlap=q.OVERLAP_INDEPENDENT)["streaming"] == 0
    assert q.qmm_q4k_tc5_plan_detail(4096, 4096, 8, device=DEV)["streaming"] == 0
    assert q.qmm_q4k_tc5_plan_detail(4096, 4096, 8, device=DEV, overlap=q.OVERLAP_CHAIN)["streaming"] == 0
