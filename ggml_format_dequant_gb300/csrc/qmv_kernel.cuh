// qmv_kernel.cuh -- the persistent streaming matvec kernel shared by every
// format (the launch plan is in qmv_launch.cuh).
//
// Shape of the computation (y[r] = sum_j W[r, j] x[j], W in packed GGML blocks):
//  * Each CTA owns a contiguous range of output rows. Contiguous rows are one
//    contiguous byte range of the packed weight, so the CTA streams it through
//    a ring of S shared-memory stages with 1-D bulk TMA copies
//    (cp.async.bulk ... mbarrier::complete_tx), G rows per stage. All S stages
//    are requested before anything else happens, so a CTA's DRAM requests are
//    in flight from its first instruction.
//  * The CTA's threads form NG groups of GS lanes. Lane i of a group owns unit i
//    of every row (a fixed k-slice) and keeps that slice of the activation in
//    registers for the whole kernel; group g handles rows g, g+NG, ... of each
//    stage. Per row a lane decodes its unit in registers and forms integer dp4a
//    dots (see qmv_formats.cuh); the group then reduces its lanes' partial sums
//    with a fixed shuffle tree (and, for groups wider than a warp, a fixed-order
//    sum of per-warp partials in shared memory), so results are deterministic.
//  * Split-k happens only inside a CTA (across the lanes of a group); rows are
//    never split across CTAs, so no atomics and no scratch memory are needed.
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
    int U, GS, NG, G, S, UPL;   // units per row, group size/count, rows per stage, stages, units per lane
    uint32_t off_la, off_lb, off_lc, off_xs, off_xsum, off_stage, stage_stride, off_red, off_bar;
};

template <class F>
__device__ __forceinline__ void issue_stage(const KParams& p, uint8_t* smem, const uint8_t* wbase,
                                            long long row0, int nr, int slot, uint64_t policy) {
    const uint32_t bar = smem_u32(smem + p.off_bar + 8 * slot);
    uint8_t* dst = smem + p.off_stage + static_cast<uint32_t>(slot) * p.stage_stride;
    const uintptr_t gs = reinterpret_cast<uintptr_t>(wbase) + static_cast<uintptr_t>(row0 * p.rowbytes);
    const uintptr_t ge = gs + static_cast<uintptr_t>(nr) * static_cast<uintptr_t>(p.rowbytes);
    const uintptr_t a0 = gs & ~uintptr_t(15);
    uintptr_t a1 = (ge + 15) & ~uintptr_t(15);
    const uintptr_t lim = reinterpret_cast<uintptr_t>(p.w) + static_cast<uintptr_t>(p.wbytes);
    if (a1 > lim) {
        // The last 16-byte word would run past the caller's buffer: copy the
        // aligned part with the bulk engine and the ragged tail byte by byte.
        a1 = ge & ~uintptr_t(15);
        for (uintptr_t b = (a1 > a0 ? a1 : a0); b < ge; b++)
            dst[b - a0] = *reinterpret_cast<const uint8_t*>(b);
    }
    if (a1 > a0) {
        const uint32_t bytes = static_cast<uint32_t>(a1 - a0);
        mbar_arrive_expect_tx(bar, bytes);
        tma_bulk_g2s(smem_u32(dst), reinterpret_cast<const void*>(a0), bytes, bar, policy);
    } else {
        mbar_arrive(bar);
    }
}

template <class F, int RG, bool RESIDENT, bool MOE, int MODE>
__global__ void __launch_bounds__(256, 1) qmv_stream_kernel(const KParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;

    // ---- rows of this CTA
    const int slot = MOE ? static_cast<int>(blockIdx.y) : 0;
    const int part = blockIdx.x, nparts = gridDim.x;
    const int R0 = static_cast<int>(static_cast<long long>(p.rows) * part / nparts);
    const int R1 = static_cast<int>(static_cast<long long>(p.rows) * (part + 1) / nparts);
    const int nrows = R1 - R0;
    const int nst = (nrows + p.G - 1) / p.G;
    const long long yoff = MOE ? static_cast<long long>(slot) * p.rows : 0;

    const uint8_t* wbase = p.w;
    const float* xrow = p.x;
    if (MOE) {
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

    // ---- request the first stages
    __shared__ uint64_t policy_s;
    __shared__ int issued_s;   // stages requested so far (written and read by thread 0 only)
    if (tid == 0) {
        for (int s = 0; s < p.S; s++) mbar_init(smem_u32(smem + p.off_bar + 8 * s), 1);
        fence_mbar_init();
        const uint64_t pol = l2_evict_first_policy();
        policy_s = pol;
        const int first = nst < p.S ? nst : p.S;
        for (int t = 0; t < first; t++) {
            const int nr = min(p.G, nrows - t * p.G);
            issue_stage<F>(p, smem, wbase, R0 + static_cast<long long>(t) * p.G, nr, t, pol);
        }
        issued_s = first;
    }

    // ---- activation: integer limbs into shared memory (f32 formats)
    XPrepSmem P;
    P.la = smem + p.off_la;
    P.lb = smem + p.off_lb;
    P.lc = smem + p.off_lc;
    P.xs = reinterpret_cast<float*>(smem + p.off_xs);
    P.xsum16 = reinterpret_cast<float*>(smem + p.off_xsum);
    if constexpr (F::LIMBS) prep_limbs(xrow, p.k, P, warp, nwarps, lane);
    __syncthreads();

    // ---- this lane's unit(s)
    const int g = tid / p.GS;
    const int lig = tid - g * p.GS;
    typename F::X xr;
    typename F::L lc;
    auto load_unit = [&](int u) {
        const int b = u / F::UNITS_PER_BLOCK;
        const int v = u - b * F::UNITS_PER_BLOCK;
        lc = F::lane_consts(v);
        int e0;
        if constexpr (F::UNITS_PER_BLOCK == 1) {
            e0 = b * F::QK;
        } else if constexpr (F::BLOCK_BYTES == 144) {
            e0 = b * F::QK + 64 * v;                          // Q4_K chunk v
        } else {
            e0 = b * F::QK + 128 * (v >> 1) + 16 * (v & 1);   // Q6_K (half, 16-slice)
        }
        if constexpr (F::LIMBS)
            F::load_x(xr, P, e0);
        else
            F::load_xq(xr, p.xq, p.xqs, e0);
    };
    const bool resident_active = RESIDENT && lig < p.U;
    if (resident_active) load_unit(lig);

    float* red = reinterpret_cast<float*>(smem + p.off_red);
    const int wpg = p.GS >> 5;   // warps per group when GS > 32

    int abort_at = -1;
    for (int t = 0; t < nst; t++) {
        const int sl = t % p.S;
        const uint32_t par = static_cast<uint32_t>(t / p.S) & 1u;
        const bool timed_out = !mbar_wait_bounded(smem_u32(smem + p.off_bar + 8 * sl), par);
        if (timed_out) atomicOr(&g_status, STATUS_WAIT_TIMEOUT);
        const long long row0 = R0 + static_cast<long long>(t) * p.G;
        const int rows_here = min(p.G, nrows - t * p.G);
        const uintptr_t gstart = reinterpret_cast<uintptr_t>(wbase) + static_cast<uintptr_t>(row0 * p.rowbytes);
        const uint8_t* st = smem + p.off_stage + static_cast<uint32_t>(sl) * p.stage_stride +
                            static_cast<uint32_t>(gstart & 15u);

        float acc[RG];
#pragma unroll
        for (int i = 0; i < RG; i++) acc[i] = 0.0f;

        for (int vv = 0; vv < (RESIDENT ? 1 : p.UPL); vv++) {
            const int u = RESIDENT ? lig : lig + p.GS * vv;
            if (u >= p.U) break;
            if (!RESIDENT) load_unit(u);
            const int b = u / F::UNITS_PER_BLOCK;
#pragma unroll
            for (int i = 0; i < RG; i++) {
                const int j = g + p.NG * i;
                if (j < rows_here) {
                    const uint8_t* blk = st + static_cast<long long>(j) * p.rowbytes + b * F::BLOCK_BYTES;
                    if constexpr (MODE == MODE_BLOCKDOTS) {
                        if constexpr (!F::LIMBS) {
                            const int dv = F::block_dot(blk, xr);
                            p.dots[(row0 + j) * p.nb + b] = dv;
                        }
                    } else {
                        acc[i] = F::dot(blk, lc, xr, acc[i]);
                    }
                }
            }
        }

        if constexpr (MODE == MODE_MATVEC) {
            if (p.GS <= 32) {
                for (int off = p.GS >> 1; off > 0; off >>= 1) {
#pragma unroll
                    for (int i = 0; i < RG; i++) acc[i] += __shfl_xor_sync(FULL, acc[i], off);
                }
                if (lig == 0) {
#pragma unroll
                    for (int i = 0; i < RG; i++) {
                        const int j = g + p.NG * i;
                        if (j < rows_here) p.y[yoff + row0 + j] = acc[i];
                    }
                }
            } else {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
                    for (int i = 0; i < RG; i++) acc[i] += __shfl_xor_sync(FULL, acc[i], off);
                }
                if (lane == 0) {
                    float* rb = red + (t & 1) * (p.G * wpg);
#pragma unroll
                    for (int i = 0; i < RG; i++) {
                        const int j = g + p.NG * i;
                        if (j < rows_here) rb[j * wpg + (lig >> 5)] = acc[i];
                    }
                }
            }
        }

        // Every lane is done with stage slot `sl`; all threads learn together
        // whether any of them gave up waiting.
        const int aborted = __syncthreads_or(timed_out ? 1 : 0);

        if (tid == 0 && t + p.S < nst && !aborted) {
            const int tn = t + p.S;
            issue_stage<F>(p, smem, wbase, R0 + static_cast<long long>(tn) * p.G,
                           min(p.G, nrows - tn * p.G), sl, policy_s);
            issued_s = tn + 1;
        }
        if (MODE == MODE_MATVEC && p.GS > 32 && tid < rows_here) {
            const float* rb = red + (t & 1) * (p.G * wpg);
            float s = 0.0f;
            for (int w = 0; w < wpg; w++) s += rb[tid * wpg + w];
            p.y[yoff + row0 + tid] = s;
        }
        if (aborted) {
            abort_at = t;
            break;
        }
    }

    if (abort_at >= 0 && tid == 0) {
        // Stages t+1 .. issued-1 were requested but never waited for: give each
        // a bounded chance to land before the shared memory is released.
        for (int s = abort_at + 1; s < issued_s; s++) {
            const uint32_t bar = smem_u32(smem + p.off_bar + 8 * (s % p.S));
            if (!mbar_wait_bounded(bar, static_cast<uint32_t>(s / p.S) & 1u)) break;
        }
    }
}

}  // namespace qmv
