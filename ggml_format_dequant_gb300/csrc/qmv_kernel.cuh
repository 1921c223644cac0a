// qmv_kernel.cuh -- the streaming matvec kernel shared by every format (the
// launch plan is in qmv_launch.cuh).
//
// Shape of the computation (y[r] = sum_j W[r, j] x[j], W in packed GGML blocks):
//  * A row is cut into k-slices of 32 "units" (one unit per lane, see
//    qmv_formats.cuh). For every format a slice is a whole number of blocks
//    whose byte length is a multiple of 16 (Q4_K 8 blocks = 1152 B, Q6_K 8
//    blocks = 1680 B, Q8_0 32 blocks = 1088 B, Q8_0 dp4a 128 blocks = 4352 B),
//    so one bulk TMA copy (cp.async.bulk ... mbarrier::complete_tx) brings one
//    slice of one row into shared memory.
//  * Each CTA owns a contiguous range of rows; its warps form NG row groups x
//    KS k-slices. Every warp runs its own pipeline: lane 0 requests the warp's
//    next S slots, the warp waits on the slot's mbarrier, decodes its 32 units
//    in registers against the activation it keeps in registers, and lane 0
//    re-fills the slot after a __syncwarp. No producer warp, no cross-warp
//    barrier in the stream; copy issue is spread over all warps.
//  * Rows narrower than a warp (fewer than 32 units) put 32/GS rows side by
//    side in one warp. A warp reduces its lanes' partial sums with a fixed
//    shuffle tree; when a row spans several k-slices the per-slice partials
//    wait in shared memory and are summed in a fixed order once the CTA is
//    done, so results are deterministic and no scratch memory or atomics are
//    needed.
//  * MoE: grid.y is the slot; the CTA reads ids[slot] once and streams rows of
//    expert ids[slot]'s slice of the bank, so only routed rows are read.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "qmv_formats.cuh"

namespace qmv {

// Device status word of the translation unit that instantiates the kernels.
static __device__ unsigned int g_status;

enum Mode : int { MODE_MATVEC = 0, MODE_BLOCKDOTS = 1 };

struct KParams {
    const uint8_t* w;           // packed rows (dense) or the [E, rows] bank (MoE)
    const float* x;             // f32 activation: [k] dense, [slots, k] MoE
    const int8_t* xq;           // dp4a activation codes [k]
    const float* xqs;           // dp4a activation scales [k/32]
    float* y;                   // [rows] dense, [slots, rows] MoE
    int32_t* dots;              // [rows, k/32] block dots (MODE_BLOCKDOTS)
    const int32_t* ids;         // [slots] expert ids (MoE)
    int n_experts;
    int rows, k, nb;            // rows per matrix, k, blocks per row
    long long rowbytes;
    unsigned long long wbytes;  // readable bytes starting at w (tail clipping)
    int U;                      // units per row
    int KS;                     // k-slices per row
    int GS;                     // lanes per row inside a warp: 32, or a smaller power of two when KS == 1
    int NG;                     // row groups per CTA (working warps = NG * KS)
    int R;                      // row steps per slot (KS == 1); 1 otherwise
    int S;                      // slots per warp
    int lgGS;                   // log2(GS)
    int rq, rrem;               // rows per CTA: rq or rq + 1 (the first rrem CTAs)
    int gq[2], grem[2];         // rows per row group for a CTA of rq ([0]) or rq + 1 ([1]) rows
    int defer;                  // 1: lanes park partial sums in shared memory, reduced once at the end
    int W;                      // units per row rounded up (KS * GS): the width of a parked row
    uint32_t off_la, off_lb, off_lc, off_xs, off_xsum;   // activation limb tables
    uint32_t off_red;           // parked lane partials [rows][W] (defer), else slice partials [rows][KS]
    uint32_t off_slots, slot_stride, off_bars;
};

// Copy bytes [gs, gs + bytes) of global memory into the slot at `dst`
// (16-byte aligned), starting the data at dst + (gs & 15). The bulk engine
// takes the 16-byte-aligned cover of the range; if that cover would run past
// the caller's buffer, the ragged last bytes are copied one by one before the
// barrier is armed (so the arrive releases them to the waiting lanes).
__device__ __forceinline__ void issue_copy(const KParams& p, uint8_t* dst, uint32_t bar, uintptr_t gs,
                                           uintptr_t bytes) {
    const uintptr_t ge = gs + bytes;
    const uintptr_t a0 = gs & ~uintptr_t(15);
    uintptr_t a1 = (ge + 15) & ~uintptr_t(15);
    const uintptr_t lim = reinterpret_cast<uintptr_t>(p.w) + static_cast<uintptr_t>(p.wbytes);
    if (a1 > lim) {
        a1 = ge & ~uintptr_t(15);
        for (uintptr_t b = (a1 > a0 ? a1 : a0); b < ge; b++) dst[b - a0] = *reinterpret_cast<const uint8_t*>(b);
    }
    if (a1 > a0) {
        const uint32_t n = static_cast<uint32_t>(a1 - a0);
        mbar_arrive_expect_tx(bar, n);
        tma_bulk_g2s(smem_u32(dst), reinterpret_cast<const void*>(a0), n, bar);
    } else {
        mbar_arrive(bar);
    }
}

// The same copy as issue_copy done by the 32 lanes of a warp with 16-byte
// cp.async (LDGSTS) requests, committed as one group per call.
__device__ __forceinline__ void issue_copy_async(const KParams& p, uint8_t* dst, uintptr_t gs, uintptr_t bytes,
                                                 int lane) {
    const uintptr_t ge = gs + bytes;
    const uintptr_t a0 = gs & ~uintptr_t(15);
    uintptr_t a1 = (ge + 15) & ~uintptr_t(15);
    const uintptr_t lim = reinterpret_cast<uintptr_t>(p.w) + static_cast<uintptr_t>(p.wbytes);
    if (a1 > lim) {
        a1 = ge & ~uintptr_t(15);
        if (lane == 0)
            for (uintptr_t b = (a1 > a0 ? a1 : a0); b < ge; b++) dst[b - a0] = *reinterpret_cast<const uint8_t*>(b);
    }
    const int n16 = a1 > a0 ? static_cast<int>((a1 - a0) >> 4) : 0;
    const uint32_t d0 = smem_u32(dst);
    for (int i = lane; i < n16; i += 32) cp_async16(d0 + 16u * i, reinterpret_cast<const void*>(a0 + 16u * i));
    cp_async_commit();
}

template <class F, int R, bool MOE, int MODE, bool BULK>
__global__ void __launch_bounds__(F::MAX_THREADS, 1) qmv_stream_kernel(const KParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    // ---- rows of this CTA
    const int slot = MOE ? static_cast<int>(blockIdx.y) : 0;
    // Balanced split precomputed on the host: no integer division here (a
    // 64-bit division is a long serial routine right where latency matters).
    const int part = blockIdx.x;
    const int big = part < p.rrem ? 1 : 0;
    const int nrows = p.rq + big;
    const int R0 = part * p.rq + min(part, p.rrem);
    const int R1 = R0 + nrows;
    const long long yoff = MOE ? static_cast<long long>(slot) * p.rows : 0;

    // The next call on the stream may be scheduled now; it still waits for
    // this one before it touches anything this one writes.
    pdl_launch_dependents();

    const uint8_t* wbase = p.w;
    const float* xrow = p.x;
    if (MOE) {
        // ids may come from the kernel just before (the router).
        pdl_dependency_wait();
        const int e = __ldg(p.ids + slot);
        if (e < 0 || e >= p.n_experts) {
            // Unroutable slot: NaN marks every output of it, and the status
            // word records the fact. No byte of the bank is touched.
            for (int r = R0 + tid; r < R1; r += blockDim.x) p.y[yoff + r] = __int_as_float(0x7fc00000);
            if (tid == 0) atomicOr(&g_status, STATUS_BAD_EXPERT_ID);
            return;
        }
        wbase = p.w + static_cast<long long>(e) * p.rows * p.rowbytes;
        xrow = p.x + static_cast<long long>(slot) * p.k;
    }
    if (nrows <= 0) return;

    // ---- this warp's tile: row group rg (a contiguous run of the CTA's rows) x k-slice ks
    const bool working = warp < p.NG * p.KS;
    const int rg = warp / p.KS;
    const int ks = warp - rg * p.KS;
    const int gq = p.gq[big], grem = p.grem[big];
    const int row_lo = R0 + rg * gq + min(rg, grem);
    const int row_hi = row_lo + gq + (rg < grem ? 1 : 0);
    const int lg_rpw = 5 - p.lgGS;                       // log2 of the rows side by side in a warp
    const int rpw = 1 << lg_rpw;
    constexpr int LG_R = R == 4 ? 2 : (R == 2 ? 1 : 0);
    const int lg_rps = (p.KS == 1) ? LG_R + lg_rpw : 0;  // log2 of the rows per slot
    const int rows_per_slot = 1 << lg_rps;
    const int nslot = working ? (row_hi - row_lo + rows_per_slot - 1) >> lg_rps : 0;
    // bytes of the slice inside a row
    const int blk0 = ks * F::SLICE_BLOCKS;
    const int nblk = min(F::SLICE_BLOCKS, p.nb - blk0);
    const uintptr_t slice_off = static_cast<uintptr_t>(blk0) * F::BLOCK_BYTES;
    const uintptr_t slice_len = static_cast<uintptr_t>(nblk) * F::BLOCK_BYTES;

    uint8_t* myslots = smem + p.off_slots + static_cast<uint32_t>(warp) * p.S * p.slot_stride;
    const uint32_t mybars = smem_u32(smem + p.off_bars) + 8u * static_cast<uint32_t>(warp * p.S);

    // Request slot t: bulk TMA from lane 0, or cp.async from every lane.
    auto issue = [&](int t, int sl) {
        const int r = row_lo + (t << lg_rps);
        const int nr = min(rows_per_slot, row_hi - r);
        const uintptr_t gs = reinterpret_cast<uintptr_t>(wbase) + static_cast<uintptr_t>(r) * p.rowbytes + slice_off;
        const uintptr_t bytes = (p.KS == 1) ? static_cast<uintptr_t>(nr) * p.rowbytes : slice_len;
        if constexpr (BULK) {
            if (lane == 0) issue_copy(p, myslots + sl * p.slot_stride, mybars + 8u * sl, gs, bytes);
        } else {
            issue_copy_async(p, myslots + sl * p.slot_stride, gs, bytes, lane);
        }
    };

    // ---- first requests, before anything else
    if (working) {
        if (BULK && lane == 0) {
            for (int s = 0; s < p.S; s++) mbar_init(mybars + 8u * s, 1);
            fence_mbar_init();
        }
        const int first = nslot < p.S ? nslot : p.S;
        for (int t = 0; t < first; t++) issue(t, t);
    }
    int issued = nslot < p.S ? nslot : p.S;

    // The packed weights are constant, so they were requested above without
    // waiting for the previous kernel; x (and y, written below) may be shared
    // with it.
    if (!MOE) pdl_dependency_wait();

    // ---- activation limbs into shared memory (f32 formats), all threads
    XPrepSmem P;
    P.la = smem + p.off_la;
    P.lb = smem + p.off_lb;
    P.lc = smem + p.off_lc;
    P.xs = reinterpret_cast<float*>(smem + p.off_xs);
    P.xsum16 = reinterpret_cast<float*>(smem + p.off_xsum);
    if constexpr (F::LIMBS) prep_limbs<4>(xrow, p.k, P, tid, static_cast<int>(blockDim.x));
    __syncthreads();   // limb tables written; every warp's barriers initialized

    float* red = reinterpret_cast<float*>(smem + p.off_red);

    if (working) {
        // ---- this lane's unit: unit u of slice ks (KS > 1), or of the row
        const int u = (p.KS == 1) ? (lane & (p.GS - 1)) : lane;
        const int ug = ks * 32 + u;                 // unit index within the row
        const bool has_unit = ug < p.U;
        const int sub = (p.KS == 1) ? (lane >> p.lgGS) : 0;   // which of the side-by-side rows
        const int wcol = ks * p.GS + u;             // this lane's column in a parked row
        typename F::X xr;
        typename F::L lc = F::lane_consts(u, p.nb, ug);
        if (has_unit) {
            const int e0 = blk0 * F::QK + F::unit_elem(u);
            if constexpr (F::LIMBS)
                F::load_x(xr, P, e0);
            else
                F::load_xq(xr, lc, p.xq, p.xqs, e0);
        }
        const int ubyte = F::unit_byte(u);

        int sl = 0;          // slot of step t
        uint32_t ph = 0;     // its barrier phase
        for (int t = 0; t < nslot; t++) {
            bool landed = true;
            if constexpr (BULK) {
                landed = __all_sync(FULL, mbar_wait_bounded(mybars + 8u * sl, ph));
                if (!landed && lane == 0) atomicOr(&g_status, STATUS_WAIT_TIMEOUT);
            } else {
                // slots t+1 .. min(t+S-1, nslot-1) may still be in flight
                cp_async_wait(min(p.S - 1, nslot - 1 - t));
                __syncwarp();
            }
            const int r = row_lo + (t << lg_rps);
            const int nr = min(rows_per_slot, row_hi - r);
            const uintptr_t gs = reinterpret_cast<uintptr_t>(wbase) + static_cast<uintptr_t>(r) * p.rowbytes + slice_off;
            const uint8_t* data = myslots + sl * p.slot_stride + static_cast<uint32_t>(gs & 15u);

            if constexpr (MODE == MODE_BLOCKDOTS) {
                if constexpr (!F::LIMBS) {
                    for (int i = 0; i < R; i++) {
                        const int j = (i << lg_rpw) + sub;
                        if (has_unit && j < nr) {
                            const uint8_t* ub = data + static_cast<long long>(j) * p.rowbytes + ubyte;
                            for (int b = 0; b < lc.nblk; b++)
                                p.dots[static_cast<long long>(r + j) * p.nb + blk0 + 4 * u + b] =
                                    F::block_dot(ub + b * F::BLOCK_BYTES, xr.q[b]);
                        }
                    }
                }
            } else {
                float acc[R];
#pragma unroll
                for (int i = 0; i < R; i++) {
                    // Row j of the slot; steps past the slot's rows recompute
                    // the lane's row of step 0 (valid data) and are dropped, so
                    // the unrolled dots carry no control dependence.
                    int j = (i << lg_rpw) + sub;
                    j = j < nr ? j : sub;
                    acc[i] = has_unit ? F::dot(data + static_cast<long long>(j) * p.rowbytes + ubyte, lc, xr, 0.0f)
                                      : 0.0f;
                }
                if (p.defer) {
                    // Park the lane partials; the rows are reduced once, at the end.
#pragma unroll
                    for (int i = 0; i < R; i++) {
                        const int j = (i << lg_rpw) + sub;
                        if (j < nr) red[static_cast<long long>(r + j - R0) * p.W + wcol] = acc[i];
                    }
                } else {
                    for (int off = p.GS >> 1; off > 0; off >>= 1) {
#pragma unroll
                        for (int i = 0; i < R; i++) acc[i] += __shfl_xor_sync(FULL, acc[i], off);
                    }
                    if (u == 0) {
#pragma unroll
                        for (int i = 0; i < R; i++) {
                            const int j = (i << lg_rpw) + sub;
                            if (j < nr) {
                                if (p.KS == 1)
                                    p.y[yoff + r + j] = acc[i];
                                else
                                    red[static_cast<long long>(r + j - R0) * p.KS + ks] = acc[i];
                            }
                        }
                    }
                }
            }
            __syncwarp();   // the whole warp is done with slot sl
            if (landed && t + p.S < nslot) {
                issue(t + p.S, sl);
                issued = t + p.S + 1;
            }
            if (!landed) {
                // A copy did not land in time: stop, but give the copies this
                // warp still has in flight a bounded chance to land before the
                // shared memory is released.
                if (lane == 0) {
                    int s2 = sl;
                    uint32_t ph2 = ph;
                    for (int tt = t + 1; tt < issued; tt++) {
                        if (++s2 == p.S) {
                            s2 = 0;
                            ph2 ^= 1u;
                        }
                        if (!mbar_wait_bounded(mybars + 8u * s2, ph2)) break;
                    }
                }
                break;
            }
            if (++sl == p.S) {
                sl = 0;
                ph ^= 1u;
            }
        }
    }

    if (MODE == MODE_MATVEC && p.defer) {
        // One warp per row: strided lane sums over the parked partials, then a
        // fixed shuffle tree.
        __syncthreads();
        const int nwarps = blockDim.x >> 5;
        for (int r = warp; r < nrows; r += nwarps) {
            float s = 0.0f;
            for (int c = lane; c < p.W; c += 32) s += red[static_cast<long long>(r) * p.W + c];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(FULL, s, off);
            if (lane == 0) p.y[yoff + R0 + r] = s;
        }
    } else if (MODE == MODE_MATVEC && p.KS > 1) {
        // Rows spanning several k-slices: sum the slice partials in a fixed order.
        __syncthreads();
        for (int r = tid; r < nrows; r += blockDim.x) {
            float s = 0.0f;
            for (int q = 0; q < p.KS; q++) s += red[static_cast<long long>(r) * p.KS + q];
            p.y[yoff + R0 + r] = s;
        }
    }
}

}  // namespace qmv
