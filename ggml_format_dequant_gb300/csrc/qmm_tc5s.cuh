// qmm_tc5s.cuh -- the streaming form of the fifth-generation tensor-core batch
// kernel (qmm_tc5.cuh), for streams of independent calls: one CTA an SM owns
// a 128-row tile for the whole of k, so there is no cross-CTA reduction and
// the CTA's fixed costs (tensor-memory allocation, barrier set-up, building
// B) are paid once per tile instead of once per k-chunk.
//
//  * B (x as hi / lo f16 parts, and B' the group sums) is built once, for the
//    whole of k, from x in global memory by the decoder warps, while the
//    first weight copies land. It takes k x 32 bytes of shared memory, so the
//    plan is made for rows of up to a few thousand weights (Q4_K 4096).
//  * Eight decoder warps, two a lane quarter: warp w decodes half hh = w / 4
//    of every super-block (sub-blocks 4hh .. 4hh+3) for rows 32 (w % 4) .. +31.
//    Each half's A operand is double-buffered in tensor memory, so a warp
//    decodes super-block q + 1 while the MMAs of q run.
//  * One thread of a ninth warp issues the TMA copies and the MMAs, as in
//    qmm_tc5.cuh. The accumulators alternate between two pairs; decoder warp w
//    reads back the columns of rows j = 4hh .. 4hh+3 of x and writes them.
//  * Every wait is bounded; a wait that gives up marks the CTA's outputs NaN
//    and sets STATUS_WAIT_TIMEOUT. Tensor memory (512 columns) is allocated
//    and released by the issuing warp; the shared memory the plan asks for
//    keeps one CTA an SM, so the allocation never waits.
#pragma once

#include "qmm_tc5.cuh"

namespace qmv {

constexpr int T5S_DECODERS = 8;                        // decoder warps
constexpr int T5S_THREADS = 32 * (T5S_DECODERS + 1);   // and the issuing warp
constexpr int T5S_TMEM_COLS = 512;
// Tensor-memory columns: A operand [half][buffer] (64 columns each), the
// min-term operand [buffer] (8 used of 16), accumulators D and D' [buffer].
__host__ __device__ constexpr uint32_t t5s_col_a(int h, int b) {
    return 64u * static_cast<uint32_t>(2 * h + b);
}
__host__ __device__ constexpr uint32_t t5s_col_am(int b) { return 256u + 16u * static_cast<uint32_t>(b); }
__host__ __device__ constexpr uint32_t t5s_col_d(int b) { return 288u + 16u * static_cast<uint32_t>(b); }
__host__ __device__ constexpr uint32_t t5s_col_dm(int b) { return 320u + 16u * static_cast<uint32_t>(b); }

struct T5SParams {
    const float* x;       // [m, k]
    float* y;             // [m, rows]
    int rows, k, m;
    int nsb;              // super-blocks per row
    int S;                // ring slots
    int early_inputs;     // x read before waiting for the previous kernel (only y waits)
    int force_timeout;    // failure-path test
    uint32_t slot_bytes;  // 128 rows x 144 bytes
    uint32_t off_ring, off_b, off_bm, off_sc, off_bars;
};

__device__ __forceinline__ void tmem_ld4(uint32_t t, uint32_t (&r)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(t)
                 : "memory");
}

__global__ void __launch_bounds__(T5S_THREADS, 1)
    qmm_tc5s_q4k_kernel(const __grid_constant__ CUtensorMap wmap, const T5SParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint32_t s_tmem;
    __shared__ int s_tmo;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int row0 = static_cast<int>(blockIdx.x) * T5_ROWS;
    const int nq = p.nsb;
    const uint32_t sb = smem_u32(smem);
    const uint32_t ring = sb + p.off_ring;
    const uint32_t bars = sb + p.off_bars;
    // barriers: full[S], empty[S], afull[half][buffer], afree[half][buffer], dfull[2], dfree[2], fin
    const uint32_t full0 = bars, empty0 = bars + 8u * p.S, afull0 = bars + 16u * p.S;
    const uint32_t afree0 = afull0 + 32u, dfull0 = afull0 + 64u, dfree0 = afull0 + 80u, fin = afull0 + 96u;

    pdl_launch_dependents();

    if (warp == T5S_DECODERS) {
        if (lane == 0) {
            for (int s = 0; s < p.S; s++) {
                mbar_init(full0 + 8u * s, 1);
                mbar_init(empty0 + 8u * s, 32 * T5S_DECODERS);
            }
            for (int i = 0; i < 4; i++) {
                mbar_init(afull0 + 8u * i, 32 * T5S_DECODERS / 2);
                mbar_init(afree0 + 8u * i, 1);
            }
            for (int b = 0; b < 2; b++) {
                mbar_init(dfull0 + 8u * b, 1);
                mbar_init(dfree0 + 8u * b, 32 * T5S_DECODERS);
            }
            mbar_init(fin, 1);
            s_tmo = 0;
            fence_mbar_init();
            // the weights are constant: the first slots are requested at once
            const int first = nq < p.S ? nq : p.S;
            for (int i = 0; i < first; i++) {
                mbar_arrive_expect_tx(full0 + 8u * i, p.slot_bytes);
                tma_load_2d(ring + static_cast<uint32_t>(i) * p.slot_bytes, &wmap, i * (T5_SBBYTES / 8), row0,
                            full0 + 8u * i);
            }
        }
        __syncwarp();
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(T5S_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // every barrier is initialized (and the tensor-memory address written)
    // before any thread waits on one
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // x may come from the kernel just before, unless the caller declared it
    // independent of it
    if (!p.early_inputs) pdl_dependency_wait();

    // ---- B and B' for the whole of k, by the decoder warps, from x in global
    // memory (while the first weight copies land)
    float* scl = reinterpret_cast<float*>(smem + p.off_sc);
    if (warp < T5S_DECODERS) {
        t5_build_b(p.x, p.k, nq, p.m, warp, T5S_DECODERS, lane, smem + p.off_b, smem + p.off_bm, scl);
        fence_proxy_async();   // B is read by the tensor cores (async proxy)
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int* tmo = &s_tmo;

    if (warp == T5S_DECODERS) {
        // ---- the issuing thread: per super-block, the MMAs of its two halves
        // (each in the buffer of its parity) and the min term, then the refill
        // of the ring slot every row has read
        int next = p.S < nq ? p.S : nq;   // next super-block to request
        if (lane == 0 && !p.force_timeout) {
            const uint32_t bbase = sb + p.off_b, bmbase = sb + p.off_bm;
            bool ok = true;
            for (int q = 0; q < nq && ok; q++) {
                const int db = q & 1, ab = q & 1;
                if (q >= 2 && !mbar_wait_bounded(dfree0 + 8u * db, static_cast<uint32_t>(((q - 2) >> 1) & 1))) {
                    ok = false;
                    break;
                }
                for (int h = 0; h < 2; h++) {
                    const uint32_t ai = static_cast<uint32_t>(2 * h + ab);
                    if (!mbar_wait_bounded(afull0 + 8u * ai, static_cast<uint32_t>((q >> 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int t = 0; t < 8; t++) {
                        const uint32_t kb = static_cast<uint32_t>(32 * q + 16 * h + 2 * t);   // first k-block of the step
                        mma_f16_ts(tmem + t5s_col_d(db), tmem + t5s_col_a(h, ab) + 8u * t,
                                   smem_desc(bbase + kb * 256u, 256u, 128u), T5_IDESC, h > 0 || t > 0);
                    }
                    if (h == 1)
                        mma_f16_ts(tmem + t5s_col_dm(db), tmem + t5s_col_am(ab),
                                   smem_desc(bmbase + static_cast<uint32_t>(q) * 512u, 256u, 128u), T5_IDESC, false);
                    mma_commit(afree0 + 8u * ai);
                }
                if (!ok) break;
                mma_commit(dfull0 + 8u * db);
                if (next < nq) {
                    const int s = q % p.S;
                    if (!mbar_wait_bounded(empty0 + 8u * s, static_cast<uint32_t>((q / p.S) & 1))) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async();
                    mbar_arrive_expect_tx(full0 + 8u * s, p.slot_bytes);
                    tma_load_2d(ring + static_cast<uint32_t>(s) * p.slot_bytes, &wmap, next * (T5_SBBYTES / 8), row0,
                                full0 + 8u * s);
                    next++;
                }
            }
            if (!ok) atomicExch(const_cast<int*>(tmo), 1);
            // every MMA issued is complete before tensor memory is released
            mma_commit(fin);
            if (!mbar_wait_bounded(fin, 0u)) atomicExch(const_cast<int*>(tmo), 1);
            // copies still in flight (a failed run) land before the CTA ends
            for (int i = next - p.S > 0 ? next - p.S : 0; i < next; i++)
                if (!mbar_wait_bounded(full0 + 8u * (i % p.S), static_cast<uint32_t>((i / p.S) & 1))) break;
        } else if (lane == 0) {
            // failure-path test: no MMA issued; the copies still land
            for (int i = 0; i < next; i++)
                if (!mbar_wait_bounded(full0 + 8u * i, 0u)) break;
        }
        __syncwarp();
        __syncthreads();   // every decoder is done with tensor memory
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(T5S_TMEM_COLS)
                     : "memory");
        return;
    }

    // ---- decoder warps: half hh of every super-block of row r of the tile,
    // and the read-back of rows j = 4hh .. 4hh+3 of x
    const int lq = warp & 3, hh = warp >> 2;
    const int r = 32 * lq + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * lq) << 16;
    float yacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    float dprev = 0.0f, mprev = 0.0f;   // d and dmin of the super-block read back next
    bool ok = !p.force_timeout;
    const uint32_t K1024 = 0x64006400u;   // f16x2 (1024, 1024)
    for (int q = 0; q <= nq && ok; q++) {
        float dcur = 0.0f, mcur = 0.0f;
        if (q < nq) {
            const int s = q % p.S;
            // (every decision a warp takes is a vote: the tensor-memory
            // instructions below are warp-collective)
            if (!__all_sync(FULL, mbar_wait_bounded(full0 + 8u * s, static_cast<uint32_t>((q / p.S) & 1)) &&
                                      *tmo == 0)) {
                ok = false;
                break;
            }
            const uint32_t a = ring + static_cast<uint32_t>(s) * p.slot_bytes + static_cast<uint32_t>(r) * T5_SBBYTES;
            const uint4 hd = lds128<0>(a);
            uint32_t qs[16];   // the half's two 32-byte chunks of codes
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const uint4 v = lds128<0>(a + 16u + 64u * static_cast<uint32_t>(hh) + 16u * i);
                qs[4 * i] = v.x; qs[4 * i + 1] = v.y; qs[4 * i + 2] = v.z; qs[4 * i + 3] = v.w;
            }
            mbar_arrive(empty0 + 8u * s);   // this row's half is done with the slot
            {
                const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hd.x));
                dcur = dd.x;
                mcur = dd.y;
            }
            // the 6-bit scales of sub-blocks 4hh .. 4hh+3, one per byte
            const uint32_t scw = hh ? ((hd.w & 0x0f0f0f0fu) | ((hd.y >> 2) & 0x30303030u)) : (hd.y & 0x3f3f3f3fu);
            const int ab = q & 1;
            const uint32_t ai = static_cast<uint32_t>(2 * hh + ab);
            if (q >= 2 &&
                !__all_sync(FULL, mbar_wait_bounded(afree0 + 8u * ai, static_cast<uint32_t>(((q - 2) >> 1) & 1)))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t acol = tmem + lane_base + t5s_col_a(hh, ab);
#pragma unroll
            for (int gg = 0; gg < 4; gg++) {
                // sub-block 4hh + gg: the half's chunk gg / 2, low (even) or high nibbles
                const uint32_t bsel = static_cast<uint32_t>(gg) | (static_cast<uint32_t>(gg) << 8) | 0x4040u;
                const uint32_t sc2 = hsub2_5(prmt(scw, 0x64646464u, bsel), K1024);   // (sc, sc)
                const uint32_t nb2 = hmul2(sc2, 0xE400E400u);                       // (-1024 sc, -1024 sc)
                uint32_t av[16];
#pragma unroll
                for (int w = 0; w < 8; w++) {
                    const uint32_t wv = qs[8 * (gg >> 1) + w];
                    const uint32_t n = (gg & 1) ? ((wv >> 4) & 0x0f0f0f0fu) : (wv & 0x0f0f0f0fu);
                    av[2 * w] = hfma2(prmt(n, 0x64646464u, 0x4140u), sc2, nb2);
                    av[2 * w + 1] = hfma2(prmt(n, 0x64646464u, 0x4342u), sc2, nb2);
                }
                tmem_st16(acol + 16u * gg, av);
            }
            if (hh == 1) {
                // the min-term operand: m_0 .. m_7 at k = 0..7, zeros at 8..15
                const uint32_t m_lo = hd.z & 0x3f3f3f3fu;
                const uint32_t m_hi = ((hd.w >> 4) & 0x0f0f0f0fu) | ((hd.z >> 2) & 0x30303030u);
                uint32_t mv[8];
                mv[0] = hsub2_5(prmt(m_lo, 0x64646464u, 0x4140u), K1024);
                mv[1] = hsub2_5(prmt(m_lo, 0x64646464u, 0x4342u), K1024);
                mv[2] = hsub2_5(prmt(m_hi, 0x64646464u, 0x4140u), K1024);
                mv[3] = hsub2_5(prmt(m_hi, 0x64646464u, 0x4342u), K1024);
                mv[4] = mv[5] = mv[6] = mv[7] = 0u;
                tmem_st8(tmem + lane_base + t5s_col_am(ab), mv);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(afull0 + 8u * ai);
        }
        if (q >= 1) {
            // read back super-block q - 1: columns 4hh .. 4hh+3 (hi) and 8 + the
            // same (lo) of both accumulators
            const int qb = q - 1, db = qb & 1;
            if (!__all_sync(FULL, mbar_wait_bounded(dfull0 + 8u * db, static_cast<uint32_t>((qb >> 1) & 1)))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t dh[4], dl[4], mh[4], ml[4];
            const uint32_t cj = 4u * static_cast<uint32_t>(hh);
            tmem_ld4(tmem + lane_base + t5s_col_d(db) + cj, dh);
            tmem_ld4(tmem + lane_base + t5s_col_d(db) + 8u + cj, dl);
            tmem_ld4(tmem + lane_base + t5s_col_dm(db) + cj, mh);
            tmem_ld4(tmem + lane_base + t5s_col_dm(db) + 8u + cj, ml);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(dfree0 + 8u * db);
            const float* sq = scl + qb * T5_COLS * 2;
#pragma unroll
            for (int jj = 0; jj < 4; jj++) {
                const int j = 4 * hh + jj;
                if (j < p.m) {
                    const float t = dprev * (__uint_as_float(dh[jj]) + __uint_as_float(dl[jj]));
                    const float u = mprev * (__uint_as_float(mh[jj]) + __uint_as_float(ml[jj]));
                    yacc[jj] = __fmaf_rn(t, sq[2 * j], yacc[jj]);
                    yacc[jj] = __fmaf_rn(-u, sq[2 * j + 1], yacc[jj]);
                }
            }
        }
        dprev = dcur;
        mprev = mcur;
    }
    if (!ok) atomicExch(const_cast<int*>(tmo), 1);
    tc_fence_before();
    __syncthreads();   // with the issuing warp: tensor memory is released after this
    if (*tmo) {
#pragma unroll
        for (int jj = 0; jj < 4; jj++) yacc[jj] = __int_as_float(0x7fc00000);
        if (tid == 0) atomicOr(&g_status, STATUS_WAIT_TIMEOUT);
    }
    // y after the previous kernel is done with it
    if (p.early_inputs) pdl_dependency_wait();
    if (row0 + r < p.rows) {
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
            const int j = 4 * hh + jj;
            if (j < p.m) p.y[static_cast<long long>(j) * p.rows + row0 + r] = yacc[jj];
        }
    }
}

}  // namespace qmv
