// qmv_kernel.cuh -- the streaming matvec kernel shared by every format (the
// launch plan is in qmv_launch.cuh).
//
// Shape of the computation (y[r] = sum_j W[r, j] x[j], W in packed GGML blocks):
//  * A row is cut into k-slices of 32 "units" (one unit per lane, see
//    qmv_formats.cuh); KS warps, one per slice, cover a row. A CTA owns a
//    contiguous run of rows, split evenly over NG row groups of KS warps.
//  * Every row group streams its rows through its own ring of S shared-memory
//    slots. A slot holds a piece of CR whole rows, which are contiguous in
//    memory, so one bulk TMA copy (cp.async.bulk ... mbarrier::complete_tx)
//    fills it. The first S pieces are requested before anything else, before
//    the kernel even waits for the previous one on the stream (the packed
//    weights are constant). The group's warps wait on the slot's mbarrier,
//    decode their slice of every row of the piece against the activation they
//    keep in registers, and count themselves done; the last of them re-fills
//    the slot with the group's next piece. No producer warp, no CTA barrier in
//    the stream.
//  * Rows narrower than a warp (fewer than 32 units) put 32/GS rows side by
//    side in one warp.
//  * A warp reduces its lanes' partial sums of every row with a fixed shuffle
//    tree right after decoding it, while other warps keep the memory busy. A
//    row of one slice is written to y at once; a row of several slices parks
//    its slice sums in shared memory and they are added in slice order once
//    the CTA is done (deterministic, no atomics on the data, no memory beyond
//    the inputs and the output).
//  * MoE: grid.y is the slot; the CTA reads ids[slot] once and streams rows of
//    expert ids[slot]'s matrix, so only routed rows are read.
//  * Every wait is bounded (WAIT_LIMIT_NS): a copy that never lands raises
//    STATUS_WAIT_TIMEOUT, and the CTA still waits (bounded) for the copies it
//    issued before it exits.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "qmv_formats.cuh"

namespace qmv {

// Device status word of the translation unit that instantiates the kernels.
static __device__ unsigned int g_status;

// The checking build's test of one access (see BOUNDS_CHECK): whether it may
// go ahead. Always true in the normal build, where `ok` is never evaluated.
__device__ __forceinline__ bool in_bounds(bool ok) {
    if constexpr (BOUNDS_CHECK) {
        if (!ok) atomicOr(&g_status, STATUS_OUT_OF_BOUNDS);
        return ok;
    } else {
        return true;
    }
}

enum Mode : int { MODE_MATVEC = 0, MODE_BLOCKDOTS = 1 };

struct KParams {
    const uint8_t* w;           // packed rows (dense) or the [E, rows] bank (MoE)
    const float* x;             // f32 activation: [k] dense, [slots, k] MoE
    const int8_t* xq;           // dp4a activation codes: [k] dense, [slots, k] MoE
    const float* xqs;           // dp4a activation scales: [k/32] dense, [slots, k/32] MoE
    float* y;                   // [rows] dense, [slots, rows] MoE
    int32_t* dots;              // [rows, k / F::DOT_WEIGHTS] integer dots (MODE_BLOCKDOTS)
    const int32_t* ids;         // [slots] expert ids (MoE)
    int n_experts;
    int rows, k, nb;            // rows per matrix, k, blocks per row
    uint32_t rowbytes;
    unsigned long long matbytes;   // bytes of one matrix (MoE expert stride)
    unsigned long long wbytes;     // readable bytes starting at w (tail clipping)
    int U;                      // units per row
    int KS;                     // k-slices (warps) per row
    int GS;                     // lanes per row inside a warp: 32, or a smaller power of two when KS == 1
    int lgGS;                   // log2(GS)
    int NG;                     // row groups per CTA (working warps = NG * KS)
    int CR;                     // rows per piece (one ring slot)
    int S;                      // ring slots per row group
    int rq, rrem;               // rows per CTA: rq or rq + 1 (the first rrem CTAs)
    int gq[2], grem[2];         // rows per row group for a CTA of rq ([0]) or rq + 1 ([1]) rows
    int npc4[4];                // pieces of a row group: [2 * (CTA of rq + 1 rows) + (group of gq + 1 rows)]
    uint8_t wmap[16];           // warp w works on row group wmap[w] >> 4, k-slice wmap[w] & 15 (0xff: idle)
    int W;                      // parked sums per row: KS, or 1 (early inputs), or 0 (rows written at once)
    int aligned8;               // every unit starts 8-byte aligned in shared memory (Q8_0 dp4a)
    int CL;                     // CTAs per cluster sharing the activation prep (1: no cluster)
    int early_inputs;           // x / ids may be read before waiting for the previous kernel (only y waits)
    int force_timeout;          // failure-path test: every first wait reports a copy that did not land
    uint32_t slot_stride;
    LimbTables lt;              // activation limb tables (f32-activation formats)
    uint32_t off_red;           // parked slice sums [rows of the CTA][W]
    uint32_t off_ring;          // NG * S slots
    uint32_t off_bars;          // NG * S mbarriers
    uint32_t off_cnt;           // NG * S done-counters, NG issued-piece counts, 1 timeout flag
};

// Copy bytes [gs, gs + bytes) of global memory into the slot at shared
// address dst (128-byte aligned), the data starting at dst + (gs & 15). The
// bulk engine takes the 16-byte-aligned cover of the range; if that cover would
// run past the caller's buffer, the ragged last bytes are copied one by one
// before the barrier is armed (so the arrive releases them to the waiters).
__device__ __forceinline__ void issue_copy(const KParams& p, uint8_t* dst_ptr, uint32_t dst, uint32_t bar,
                                           uintptr_t gs, uintptr_t bytes) {
    const uintptr_t ge = gs + bytes;
    const uintptr_t a0 = gs & ~uintptr_t(15);
    uintptr_t a1 = (ge + 15) & ~uintptr_t(15);
    const uintptr_t lim = reinterpret_cast<uintptr_t>(p.w) + static_cast<uintptr_t>(p.wbytes);
    // (the whole 16-byte cover fits the slot; it reads only the weights)
    if (!in_bounds(a1 - a0 <= p.slot_stride && a0 >= (reinterpret_cast<uintptr_t>(p.w) & ~uintptr_t(15)) &&
                   ge <= lim)) {
        mbar_arrive(bar);   // nothing copied; the waiters go on
        return;
    }
    if (a1 > lim) {
        a1 = ge & ~uintptr_t(15);
        for (uintptr_t b = (a1 > a0 ? a1 : a0); b < ge; b++) dst_ptr[b - a0] = *reinterpret_cast<const uint8_t*>(b);
    }
    if (a1 > a0) {
        const uint32_t n = static_cast<uint32_t>(a1 - a0);
        mbar_arrive_expect_tx(bar, n);
        tma_bulk_g2s(dst, reinterpret_cast<const void*>(a0), n, bar);
    } else {
        mbar_arrive(bar);
    }
}

// The lane's dot for the unit at shared address a.
template <class F>
__device__ __forceinline__ float dot_of(uint32_t a, const typename F::L& lc, const typename F::X& xr, bool aligned8) {
    if constexpr (F::LIMBS)
        return F::dot(a, lc, xr, 0.0f);
    else
        return F::dot(a, lc, xr, 0.0f, aligned8);
}

// Sum of v over each aligned group of GS lanes (a fixed xor tree); every lane
// of the group ends with the group's sum.
template <bool WIDE>
__device__ __forceinline__ float group_sum(float v, int GS) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        if (WIDE || off < GS) v += __shfl_xor_sync(FULL, v, off);
    }
    return v;
}

// Sums over all 32 lanes of two values at once: lanes 0..15 end with the sum
// of a, lanes 16..31 with the sum of b (one exchange splits the pair, then a
// 16-lane tree), 12 instructions instead of 20.
__device__ __forceinline__ float pair_sum(float a, float b, int lane) {
    const bool hi = (lane & 16) != 0;
    float keep = hi ? b : a;
    const float send = hi ? a : b;
    keep += __shfl_xor_sync(FULL, send, 16);
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) keep += __shfl_xor_sync(FULL, keep, off);
    return keep;
}

template <class F, int R, bool MOE, int MODE, bool WIDE>
__global__ void __launch_bounds__(512, 1) qmv_stream_kernel(const KParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    // ---- rows of this CTA (balanced split precomputed on the host)
    const int slot = MOE ? static_cast<int>(blockIdx.y) : 0;
    const int part = blockIdx.x;
    const int big = part < p.rrem ? 1 : 0;
    const int nrows = p.rq + big;
    const int R0 = part * p.rq + min(part, p.rrem);
    const long long yoff = MOE ? static_cast<long long>(slot) * p.rows : 0;

    // The next call on the stream may be scheduled now; it still waits for
    // this one before it touches anything this one writes.
    pdl_launch_dependents();

    const uint8_t* wbase = p.w;
    const float* xrow = p.x;
    const int8_t* xqrow = p.xq;      // integer-activation formats: this slot's codes and scales
    const float* xqsrow = p.xqs;
    if (MOE) {
        // ids may come from the kernel just before (the router), unless the
        // caller declared this call's inputs independent of it.
        if (!p.early_inputs) pdl_dependency_wait();
        const int e = __ldg(p.ids + slot);
        if (e < 0 || e >= p.n_experts) {
            // Unroutable slot: NaN marks every output of it, and the status
            // word records the fact. No byte of the bank is touched.
            pdl_dependency_wait();
            for (int r = R0 + tid; r < R0 + nrows; r += blockDim.x)
                if (in_bounds(r >= 0 && r < p.rows)) p.y[yoff + r] = __int_as_float(0x7fc00000);
            if (tid == 0) atomicOr(&g_status, STATUS_BAD_EXPERT_ID);
            return;
        }
        wbase = p.w + static_cast<unsigned long long>(e) * p.matbytes;
        xrow = p.x + static_cast<long long>(slot) * p.k;
        xqrow = p.xq + static_cast<long long>(slot) * p.k;
        xqsrow = p.xqs + static_cast<long long>(slot) * (p.k >> 5);
    }
    // (The planner never gives a CTA zero rows, and the MoE check above is the
    // same for every CTA of a cluster, which all serve one slot: no CTA leaves
    // before the cluster barrier below unless all of its cluster do.)
    if (nrows <= 0) return;

    // ---- this warp: row group rg, k-slice ks (mapping and piece counts
    // precomputed on the host)
    const uint32_t wm = p.wmap[warp];
    const bool working = wm != 0xffu;
    const int rg = static_cast<int>(wm >> 4);
    const int ks = static_cast<int>(wm & 15u);
    const int gq = p.gq[big], grem = p.grem[big];
    const int glo = rg * gq + min(rg, grem);          // first row of the group, CTA-local
    const int longer = rg < grem ? 1 : 0;
    const int gn = working ? gq + longer : 0;
    const int npc = working ? p.npc4[2 * big + longer] : 0;   // pieces of the group

    const uint32_t sbase = smem_u32(smem);
    const uint32_t ring = sbase + p.off_ring + static_cast<uint32_t>(rg * p.S) * p.slot_stride;
    uint8_t* ring_ptr = smem + p.off_ring + static_cast<uint32_t>(rg * p.S) * p.slot_stride;
    const uint32_t bars = sbase + p.off_bars + 8u * static_cast<uint32_t>(rg * p.S);
    int* cnt = reinterpret_cast<int*>(smem + p.off_cnt);
    int* done = cnt + rg * p.S;                       // this group's per-slot done-counters
    int* issued = cnt + p.NG * p.S + rg;              // pieces requested so far by this group
    int* timeout = cnt + p.NG * p.S + p.NG;           // CTA-wide flag

    // Request piece pc of the group into slot s (one thread).
    auto issue = [&](int pc, int s) {
        const int r0 = R0 + glo + pc * p.CR;
        const int nr = min(p.CR, gn - pc * p.CR);
        // the piece's rows are the matrix's, its slot lies in the ring
        if (!in_bounds(rg < p.NG && s < p.S && nr > 0 && r0 >= 0 && r0 + nr <= p.rows &&
                       static_cast<uint32_t>(rg * p.S + s + 1) * p.slot_stride <= p.off_bars - p.off_ring)) {
            if (rg < p.NG && s < p.S) mbar_arrive(bars + 8u * s);
            return;
        }
        const uintptr_t gs = reinterpret_cast<uintptr_t>(wbase) + static_cast<uintptr_t>(r0) * p.rowbytes;
        issue_copy(p, ring_ptr + static_cast<uint32_t>(s) * p.slot_stride, ring + static_cast<uint32_t>(s) * p.slot_stride,
                   bars + 8u * s, gs, static_cast<uintptr_t>(nr) * p.rowbytes);
    };

    // ---- first requests, before anything else
    if (working && ks == 0 && lane == 0) {
        for (int s = 0; s < p.S; s++) {
            mbar_init(bars + 8u * s, 1);
            done[s] = 0;
        }
        fence_mbar_init();
        const int first = npc < p.S ? npc : p.S;
        for (int pc = 0; pc < first; pc++) issue(pc, pc);
        *issued = first;
    }
    if (tid == 0) *timeout = 0;

    // The packed weights are constant, so they were requested above without
    // waiting for the previous kernel; x (and y, written below) may be shared
    // with it. With early inputs only the writes of y wait (at the end).
    if (!MOE && (!p.early_inputs || MODE == MODE_BLOCKDOTS)) pdl_dependency_wait();

    if constexpr (F::LIMBS) {
        // The activation limb tables, shared among the CTAs of a cluster (all
        // of them work on the same x: the same matrix, or the same MoE slot).
        if (p.CL > 1)
            prep_limbs<2>(xrow, p.k, smem, p.lt, tid, static_cast<int>(blockDim.x), p.CL, cluster_rank());
        else
            prep_limbs_cta<4>(xrow, p.k, smem, p.lt, tid, static_cast<int>(blockDim.x));
    } else if constexpr (quantizes_x<F>::value) {
        // the dp4a codes of x, quantized by this CTA into its own tables
        int8_t* tq = reinterpret_cast<int8_t*>(smem + p.lt.la);
        float* ts = reinterpret_cast<float*>(smem + p.lt.xs);
        quantize_x_cta(xrow, p.k, tq, ts, tid, static_cast<int>(blockDim.x));
        xqrow = tq;
        xqsrow = ts;
    }
    if (p.CL > 1)
        cluster_sync();   // every CTA's limb tables complete; barriers and counters initialized
    else
        __syncthreads();

    float* red = reinterpret_cast<float*>(smem + p.off_red);

    if (working) {
        // ---- this lane's unit: unit u of slice ks (KS > 1), or of the row
        const int u = (p.KS == 1) ? (lane & (p.GS - 1)) : lane;
        const int sub = (p.KS == 1) ? (lane >> p.lgGS) : 0;   // which of the side-by-side rows
        const int ug = ks * 32 + u;                 // unit index within the row
        const bool has_unit = ug < p.U;
        // Lanes past the row's last unit decode that unit too (valid data and
        // activation) and drop the result, so every dot is unconditional and
        // the unrolled dots of a step can be interleaved.
        const int ugc = has_unit ? ug : p.U - 1;
        const int uc = ugc - ks * 32;
        const int rpw = 32 >> p.lgGS;               // rows side by side in a warp step
        typename F::X xr;
        const typename F::L lc = F::lane_consts(uc, p.nb, ugc);
        in_bounds(rg < p.NG);
        {
            const int e0 = ks * F::SLICE_BLOCKS * F::QK + F::unit_elem(uc);
            in_bounds(e0 >= 0 && e0 < p.k);
            if constexpr (F::LIMBS)
                F::load_x(xr, smem, p.lt, e0);
            else
                F::load_xq(xr, lc, xqrow, xqsrow, e0);
        }
        // Byte offset of the lane's unit inside a row, and 16-byte phase of the
        // group's rows in memory (pieces may start off a 16-byte boundary).
        const uint32_t ubyte = static_cast<uint32_t>(ks) * (F::SLICE_BLOCKS * F::BLOCK_BYTES) + F::unit_byte(uc);
        in_bounds(ubyte < p.rowbytes && ks < p.KS);
        const uint32_t gphase = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(wbase)) +
                                static_cast<uint32_t>(R0 + glo) * p.rowbytes;
        const uint32_t piece_bytes = static_cast<uint32_t>(p.CR) * p.rowbytes;
        const uint32_t rstep = static_cast<uint32_t>(rpw) * p.rowbytes;   // bytes between warp steps
        const bool aligned8 = p.aligned8 != 0;
        // A finished row sum: to y (rows of one slice, no early inputs) or
        // parked by slice until the CTA is done.
        auto store_row = [&](int rl, float v) {
            if (p.W == 0) {
                if (in_bounds(rl >= 0 && R0 + rl < p.rows)) p.y[yoff + R0 + rl] = v;
            } else {
                if (in_bounds(rl >= 0 && static_cast<uint32_t>(rl * p.W + ks + 1) * 4u <= p.off_ring - p.off_red))
                    red[rl * p.W + ks] = v;
            }
        };

        int s = 0;
        uint32_t par = 0;
        for (int pc = 0; pc < npc; pc++) {
            const bool landed = !p.force_timeout && __all_sync(FULL, mbar_wait_bounded(bars + 8u * s, par));
            if (!landed) {
                if (lane == 0) {
                    atomicOr(&g_status, STATUS_WAIT_TIMEOUT);
                    atomicExch(timeout, 1);
                }
                break;
            }
            const int nr = min(p.CR, gn - pc * p.CR);
            const int rl0 = glo + pc * p.CR;                     // CTA-local row of the piece's first row
            const uint32_t d0 = (gphase + static_cast<uint32_t>(pc) * piece_bytes) & 15u;
            const uint32_t prow0 = ring + static_cast<uint32_t>(s) * p.slot_stride + d0 + ubyte;   // unit, row 0
            uint32_t a = prow0 + static_cast<uint32_t>(sub) * p.rowbytes;                     // unit, step 0
            // The checking build: the piece (from its 16-byte phase on, with
            // the format's read slack) fits its slot, and every unit a lane
            // reads starts inside one of the piece's rows.
            const uint32_t piece_lo = ring + static_cast<uint32_t>(s) * p.slot_stride + d0;
            in_bounds(d0 + static_cast<uint32_t>(nr) * p.rowbytes + F::SLACK <= p.slot_stride);
            auto unit_at = [&](uint32_t aa) -> uint32_t {
                return in_bounds(aa >= piece_lo && aa - piece_lo < static_cast<uint32_t>(nr) * p.rowbytes) ? aa : piece_lo;
            };
            int jb = 0;
            if constexpr (MODE == MODE_MATVEC) {
                // Whole steps of R * rpw rows: R independent dots, then the
                // row sums (every row of such a step lies inside the piece).
                for (; jb + R * rpw <= nr; jb += R * rpw, a += R * rstep) {
                    float acc[R];
#pragma unroll
                    for (int q = 0; q < R; q++) {
                        acc[q] = dot_of<F>(unit_at(a + q * rstep), lc, xr, aligned8);
                        acc[q] = has_unit ? acc[q] : 0.0f;
                    }
                    if constexpr (WIDE && R == 2) {
                        const float v = pair_sum(acc[0], acc[1], lane);
                        if ((lane & 15) == 0) store_row(rl0 + jb + (lane >> 4), v);
                    } else {
#pragma unroll
                        for (int q = 0; q < R; q++) {
                            const float v = group_sum<WIDE>(acc[q], p.GS);
                            if (u == 0) store_row(rl0 + jb + q * rpw + sub, v);
                        }
                    }
                }
                // The piece's remaining rows, one step at a time; lanes whose
                // row lies past the piece decode row 0 and drop the result.
                for (; jb < nr; jb += rpw, a += rstep) {
                    const bool valid = jb + sub < nr;
                    float v = dot_of<F>(unit_at(valid ? a : prow0), lc, xr, aligned8);
                    v = has_unit ? v : 0.0f;
                    v = group_sum<WIDE>(v, p.GS);
                    if (u == 0 && valid) store_row(rl0 + jb + sub, v);
                }
            } else {
                // MODE_BLOCKDOTS: the exact int32 dots of every block.
                if constexpr (!F::LIMBS) {
                    for (; jb < nr; jb += rpw, a += rstep) {
                        if (has_unit && jb + sub < nr &&
                                in_bounds(R0 + rl0 + jb + sub < p.rows && F::dot_base(ug) < p.k / F::DOT_WEIGHTS))
                            F::block_dots(unit_at(a), lc, xr, aligned8,
                                          p.dots + static_cast<long long>(R0 + rl0 + jb + sub) * (p.k / F::DOT_WEIGHTS) +
                                              F::dot_base(ug));
                    }
                }
            }
            __syncwarp();   // the whole warp is done with slot s
            if (pc + p.S < npc) {
                // The group's piece pc + S goes into this slot once every warp of
                // the group is done with it; the last one to finish requests it.
                if (lane == 0) {
                    bool last = true;
                    if (p.KS > 1) {
                        __threadfence_block();
                        last = atomicAdd(&done[s], 1) == p.KS - 1;
                        if (last) done[s] = 0;
                    }
                    if (last) {
                        fence_proxy_async();
                        issue(pc + p.S, s);
                        atomicMax(issued, pc + p.S + 1);
                    }
                }
            }
            if (++s == p.S) {
                s = 0;
                par ^= 1u;
            }
        }
    }

    __syncthreads();
    if (*timeout) {
        // A copy did not land in time: give every copy this group still has in
        // flight a bounded chance to land before the shared memory is released,
        // and mark every output of the CTA NaN (as an unroutable MoE slot is),
        // so that no caller reads a stale y as a result.
        if (working && ks == 0 && lane == 0) {
            const int n = *issued;
            for (int pc = n - p.S > 0 ? n - p.S : 0; pc < n; pc++)
                if (!mbar_wait_bounded(bars + 8u * (pc % p.S), static_cast<uint32_t>((pc / p.S) & 1))) break;
        }
        if constexpr (MODE == MODE_MATVEC) {
            pdl_dependency_wait();
            for (int r = tid; r < nrows; r += blockDim.x)
                if (in_bounds(R0 + r < p.rows)) p.y[yoff + R0 + r] = __int_as_float(0x7fc00000);
        }
        return;
    }

    if (MODE == MODE_MATVEC && p.W > 0) {
        // Parked rows (several k-slices, or early inputs): add the slice sums
        // in slice order, once the previous kernel is done with y.
        if (p.early_inputs) pdl_dependency_wait();
        for (int r = tid; r < nrows; r += blockDim.x) {
            if (!in_bounds(R0 + r < p.rows && static_cast<uint32_t>((r + 1) * p.W) * 4u <= p.off_ring - p.off_red))
                continue;
            float v = 0.0f;
            for (int q = 0; q < p.W; q++) v += red[r * p.W + q];
            p.y[yoff + R0 + r] = v;
        }
    }
}

}  // namespace qmv
