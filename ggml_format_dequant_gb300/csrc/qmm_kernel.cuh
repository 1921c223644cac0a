// qmm_kernel.cuh -- the small-M batched product y[m, rows] = x[m, k] W^T on
// the streaming skeleton of qmv_kernel.cuh (same row split, row groups, bulk
// TMA rings with last-finisher refill, bounded waits and status word).
//
// Differences from the matvec kernel: the activation is M rows of f32 x held
// in registers as they are (no limbs); each lane decodes its unit of every row
// into f32 weights once and forms M dot products; a row's M lane partials are
// reduced across the warp with a transposing shuffle tree (M values in
// M - 1 + (5 - log2 M) exchanges, each lane ending with one of them) and
// written as y[i, row] (one slice per row) or parked per (row, slice, i) and
// summed in slice order after the CTA barrier.
#pragma once

#include "qmm_formats.cuh"
#include "qmv_launch.cuh"

namespace qmv {

constexpr int pow2_at_least(int v) { return v <= 1 ? 1 : 2 * pow2_at_least((v + 1) / 2); }

template <class F, int M, bool WIDE>
__global__ void __launch_bounds__(512, 1) qmm_stream_kernel(const KParams p) {
    constexpr int UW = F::UW;
    constexpr int MP = pow2_at_least(M);
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    const int part = blockIdx.x;
    const int big = part < p.rrem ? 1 : 0;
    const int nrows = p.rq + big;
    const int R0 = part * p.rq + min(part, p.rrem);

    pdl_launch_dependents();
    if (nrows <= 0) return;

    const int nwork = p.NG * p.KS;
    const bool working = warp < nwork;
    const int rg = warp / p.KS;
    const int ks = warp - rg * p.KS;
    const int gq = p.gq[big], grem = p.grem[big];
    const int glo = rg * gq + min(rg, grem);
    const int gn = working ? gq + (rg < grem ? 1 : 0) : 0;
    const int npc = (gn + p.CR - 1) / p.CR;

    const uint32_t sbase = smem_u32(smem);
    const uint32_t ring = sbase + p.off_ring + static_cast<uint32_t>(rg * p.S) * p.slot_stride;
    uint8_t* ring_ptr = smem + p.off_ring + static_cast<uint32_t>(rg * p.S) * p.slot_stride;
    const uint32_t bars = sbase + p.off_bars + 8u * static_cast<uint32_t>(rg * p.S);
    int* cnt = reinterpret_cast<int*>(smem + p.off_cnt);
    int* done = cnt + rg * p.S;
    int* issued = cnt + p.NG * p.S + rg;
    int* timeout = cnt + p.NG * p.S + p.NG;

    auto issue = [&](int pc, int s) {
        const int r0 = R0 + glo + pc * p.CR;
        const int nr = min(p.CR, gn - pc * p.CR);
        const uintptr_t gs = reinterpret_cast<uintptr_t>(p.w) + static_cast<uintptr_t>(r0) * p.rowbytes;
        issue_copy(p, ring_ptr + static_cast<uint32_t>(s) * p.slot_stride, ring + static_cast<uint32_t>(s) * p.slot_stride,
                   bars + 8u * s, gs, static_cast<uintptr_t>(nr) * p.rowbytes);
    };

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
    if (!p.early_inputs) pdl_dependency_wait();
    __syncthreads();

    float* red = reinterpret_cast<float*>(smem + p.off_red);

    if (working) {
        const int u = (p.KS == 1) ? (lane & (p.GS - 1)) : lane;
        const int sub = (p.KS == 1) ? (lane >> p.lgGS) : 0;
        const int ug = ks * 32 + u;
        const bool has_unit = ug < p.U;
        const int ugc = has_unit ? ug : p.U - 1;
        const int uc = ugc - ks * 32;
        const int rpw = 32 >> p.lgGS;
        const typename F::L lc = F::lane_consts(uc, p.nb, ugc);
        // This lane's activations of all M rows: x[i, e0 .. e0 + UW).
        float2 xr[M][UW / 2];
        {
            const int e0 = ks * F::SLICE_BLOCKS * F::QK + F::unit_elem(uc);
#pragma unroll
            for (int i = 0; i < M; i++) {
                const float4* src = reinterpret_cast<const float4*>(p.x + static_cast<long long>(i) * p.k + e0);
#pragma unroll
                for (int v = 0; v < UW / 4; v++) {
                    const float4 t = __ldg(src + v);
                    xr[i][2 * v] = make_float2(t.x, t.y);
                    xr[i][2 * v + 1] = make_float2(t.z, t.w);
                }
            }
        }
        const uint32_t ubyte = static_cast<uint32_t>(ks) * (F::SLICE_BLOCKS * F::BLOCK_BYTES) + F::unit_byte(uc);
        const uint32_t gphase = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(p.w)) +
                                static_cast<uint32_t>(R0 + glo) * p.rowbytes;
        const uint32_t piece_bytes = static_cast<uint32_t>(p.CR) * p.rowbytes;
        const uint32_t rstep = static_cast<uint32_t>(rpw) * p.rowbytes;

        int s = 0;
        uint32_t par = 0;
        for (int pc = 0; pc < npc; pc++) {
            const bool landed = __all_sync(FULL, mbar_wait_bounded(bars + 8u * s, par));
            if (!landed) {
                if (lane == 0) {
                    atomicOr(&g_status, STATUS_WAIT_TIMEOUT);
                    atomicExch(timeout, 1);
                }
                break;
            }
            const int nr = min(p.CR, gn - pc * p.CR);
            const int rl0 = glo + pc * p.CR;
            const uint32_t d0 = (gphase + static_cast<uint32_t>(pc) * piece_bytes) & 15u;
            const uint32_t prow0 = ring + static_cast<uint32_t>(s) * p.slot_stride + d0 + ubyte;
            uint32_t a = prow0 + static_cast<uint32_t>(sub) * p.rowbytes;
            for (int jb = 0; jb < nr; jb += rpw, a += rstep) {
                const bool valid = jb + sub < nr;
                float2 wv[UW / 2];
                F::decode(valid ? a : prow0, lc, wv);
                float v[MP];
#pragma unroll
                for (int i = 0; i < M; i++) {
                    float2 acc = mul2(wv[0], xr[i][0]);
#pragma unroll
                    for (int q = 1; q < UW / 2; q++) acc = fma2(wv[q], xr[i][q], acc);
                    v[i] = has_unit ? acc.x + acc.y : 0.0f;
                }
#pragma unroll
                for (int i = M; i < MP; i++) v[i] = 0.0f;
                const int rl = rl0 + jb + sub;
                if constexpr (WIDE) {
                    // Transposing reduction: at offset 16 >> t the lanes whose
                    // bit is clear keep the lower half of their values and
                    // the others the upper half, each adding its partner's.
#pragma unroll
                    for (int t = 0, half = MP / 2; half >= 1; t++, half >>= 1) {
                        const int off = 16 >> t;
                        const bool upper = (lane & off) != 0;
#pragma unroll
                        for (int c = 0; c < half; c++) {
                            const float send = upper ? v[c] : v[c + half];
                            const float keep = upper ? v[c + half] : v[c];
                            v[c] = keep + __shfl_xor_sync(FULL, send, off);
                        }
                    }
#pragma unroll
                    for (int off = 16 / MP; off >= 1; off >>= 1) v[0] += __shfl_xor_sync(FULL, v[0], off);
                    // lane holds output index sum over t of upper_t * (MP >> (t + 1))
                    int idx = 0;
#pragma unroll
                    for (int t = 0, half = MP / 2; half >= 1; t++, half >>= 1)
                        if (lane & (16 >> t)) idx += half;
                    if ((lane & (32 / MP - 1)) == 0 && idx < M && valid) {
                        if (p.W == 0)
                            p.y[static_cast<long long>(idx) * p.rows + R0 + rl] = v[0];
                        else
                            red[(rl * p.W + ks) * M + idx] = v[0];
                    }
                } else {
                    // Rows narrower than a warp: GS lanes per row, each value
                    // summed over its group; the group's first lane stores.
#pragma unroll
                    for (int i = 0; i < M; i++) v[i] = group_sum<false>(v[i], p.GS);
                    if (u == 0 && valid) {
#pragma unroll
                        for (int i = 0; i < M; i++) {
                            if (p.W == 0)
                                p.y[static_cast<long long>(i) * p.rows + R0 + rl] = v[i];
                            else
                                red[(rl * p.W + ks) * M + i] = v[i];
                        }
                    }
                }
            }
            __syncwarp();
            if (pc + p.S < npc) {
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
        if (working && ks == 0 && lane == 0) {
            const int n = *issued;
            for (int pc = n - p.S > 0 ? n - p.S : 0; pc < n; pc++)
                if (!mbar_wait_bounded(bars + 8u * (pc % p.S), static_cast<uint32_t>((pc / p.S) & 1))) break;
        }
        return;
    }

    if (p.W > 0) {
        if (p.early_inputs) pdl_dependency_wait();
        for (int e = tid; e < nrows * M; e += blockDim.x) {
            const int r = e / M, i = e - (e / M) * M;
            float v = 0.0f;
            for (int q = 0; q < p.W; q++) v += red[(r * p.W + q) * M + i];
            p.y[static_cast<long long>(i) * p.rows + R0 + r] = v;
        }
    }
}

template <class F, int M, bool WIDE>
inline int launch_qmm_one(const KParams& kp, const Plan& pl, cudaStream_t stream) {
    auto kern = qmm_stream_kernel<F, M, WIDE>;
    static SmemOptIn opted;
    int dev = 0;
    DevInfo di;
    if (dev_info(&di, &dev)) return QMV_ECUDA;
    if (const int rc = ensure_smem(kern, opted, dev, static_cast<int>(pl.smem))) return rc;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(pl.parts, 1, 1);
    lc.blockDim = dim3(pl.T, 1, 1);
    lc.dynamicSmemBytes = pl.smem;
    lc.stream = stream;
    cudaLaunchAttribute at[1];
    int na = 0;
    if (__atomic_load_n(&weight_prefetch_flag(), __ATOMIC_RELAXED)) {
        at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[na].val.programmaticStreamSerializationAllowed = 1;
        na++;
    }
    lc.attrs = at;
    lc.numAttrs = na;
    return cuda_rc(cudaLaunchKernelEx(&lc, kern, kp));
}

template <class F, int M>
inline int launch_qmm(const KParams& kp, const Plan& pl, cudaStream_t stream) {
    return kp.GS == 32 ? launch_qmm_one<F, M, true>(kp, pl, stream) : launch_qmm_one<F, M, false>(kp, pl, stream);
}

// Rows of x one launch of FB can take for this k: the largest tile of 2..8
// rows whose units per row fit the 16 warps of a CTA (a lane keeps UW * tile
// activations in registers, so wider tiles mean smaller units and more of
// them); 1 if none does.
template <template <int> class FB>
inline int qmm_max_tile(int k) {
    const int nb = k / FB<2>::QK;
    if (FB<8>::units(nb) <= 32 * MAX_WARPS) return 8;
    if (FB<4>::units(nb) <= 32 * MAX_WARPS) return 4;
    if (FB<2>::units(nb) <= 32 * MAX_WARPS) return 2;
    return 1;
}

// A matvec entry of the same format, for tiles of one row.
using MatvecFn = int (*)(const void*, const float*, float*, int, int, const qmv_cfg*, cudaStream_t);

// y[m, rows] = x[m, k] W^T for format template FB (Q4KB):
// ceil(m / tile) balanced tiles of rows of x, one launch each (every launch
// reads W once); tiles of one row go through the matvec. kp carries w, rows,
// k, nb, rowbytes, matbytes, wbytes.
template <template <int> class FB>
inline int qmm_run(KParams kp, const float* x, float* y, int m, const qmv_cfg* cfg, cudaStream_t s,
                   MatvecFn matvec) {
    const int tmax = qmm_max_tile<FB>(kp.k);
    const int tiles = (m + tmax - 1) / tmax;
    for (int t0 = 0, m0 = 0; t0 < tiles; t0++) {
        const int mt = m / tiles + (t0 < m % tiles ? 1 : 0);
        KParams t = kp;
        t.x = x + static_cast<long long>(m0) * kp.k;
        t.y = y + static_cast<long long>(m0) * kp.rows;
        Plan pl;
        int rc = QMV_OK;
        switch (mt) {
#define QMM_CASE(MM)                                                    \
    case MM:                                                            \
        rc = make_plan<FB<MM>>(kp.rows, kp.k, 1, cfg, &t, &pl);         \
        if (!rc) rc = launch_qmm<FB<MM>, MM>(t, pl, s);                 \
        break;
            QMM_CASE(2) QMM_CASE(3) QMM_CASE(4) QMM_CASE(5) QMM_CASE(6) QMM_CASE(7) QMM_CASE(8)
#undef QMM_CASE
        default:
            rc = matvec(kp.w, t.x, t.y, kp.rows, kp.k, cfg, s);
        }
        if (rc) return rc;
        m0 += mt;
    }
    return QMV_OK;
}

}  // namespace qmv
