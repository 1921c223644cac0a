// qmm_tc5s.cuh -- the streaming form of the fifth-generation tensor-core batch
// kernel (qmm_tc5.cuh), for streams of independent calls: one CTA an SM owns
// a 128-row tile for the whole of k, so there is no cross-CTA reduction and
// the CTA's fixed costs (tensor-memory allocation, barrier set-up) are paid
// once per tile instead of once per k-chunk.
//
// The warps have one role each, and each role waits only on the stage that
// feeds it, so that one super-block's latencies (weight copy, decode, MMA,
// read-back) overlap the neighbouring super-blocks' instead of adding up:
//  * warps 0..7 decode: warp w decodes half hh = w / 4 of every super-block
//    (sub-blocks 4hh .. 4hh+3) of rows 32 (w % 4) .. +31 into the A operand
//    in tensor memory, three buffers per half; warps 0..3 also pass each
//    row's d and dmin to the read-back through a shared-memory ring;
//  * warps 8 and 18 (one thread each) issue the MMAs of each super-block into
//    one of ND accumulator sets: warp 8 those of the first half into D0,
//    warp 18 those of the second half into D1 and the min term into D'. (A
//    thread issues one MMA in 50-100 cycles whatever N, while threads of
//    different warps issue side by side, so two issuers double the rate; the
//    read-back adds D0 + D1.)
//  * warps 9..12 read back and fold each super-block's accumulators for
//    their lane quarter of rows;
//  * warp 13 (one thread) keeps the ring of S weight copies (2-D TMA) full,
//    refilling a slot as soon as every decoder has read it;
//  * warps 14..17 build B and B' (x as hi / lo f16 parts, and the group sums)
//    into a ring of SB super-blocks, as far ahead as the ring allows, from x
//    prefetched into registers two super-blocks earlier.
// B no longer spans k, so any k fits. Every wait is bounded; a wait that gives
// up marks the CTA's outputs NaN and sets STATUS_WAIT_TIMEOUT. Tensor memory
// (512 columns) is allocated and released by warp 8. The shared memory the
// plan asks for keeps any other CTA that uses tensor memory (of this kernel or
// of the cluster plan) off the SM, and the next kernel is let start only once
// the columns are held; this kernel waits for the previous one only after
// releasing them.
#pragma once

#include "qmm_tc5.cuh"

namespace qmv {

constexpr int T5S_DECODERS = 8;                         // decoder warps 0..7
constexpr int T5S_ISSUER = 8;                           // MMA-issuing warp of the first halves
constexpr int T5S_EPI0 = 9;                             // read-back warps 9..12
constexpr int T5S_PRODUCER = 13;                        // weight-copy warp
constexpr int T5S_BUILD0 = 14;                          // B-building warps 14..17
constexpr int T5S_ISSUER1 = 18;                         // MMA-issuing warp of the second halves
constexpr int T5S_THREADS = 32 * 19;
constexpr int T5S_TMEM_COLS = 512;
constexpr int T5S_NA = 3;   // A buffers per half
constexpr int T5S_SB = 4;   // B ring
constexpr int T5S_ND = 2;   // accumulator sets
constexpr int T5S_SD = 8;   // d / dmin ring (at least NA + ND deep: see the decoders)
constexpr uint32_t T5S_BSLOT = 32u * 256u;   // one super-block of B: 32 k-blocks x 16 rows x 16 bytes
constexpr uint32_t T5S_BMSLOT = 512u;        // one super-block of B': two k-blocks, the second zeros
constexpr int T5S_NBARS_FIXED = 4 * T5S_NA + 2 * T5S_SB + T5S_SD + 2 * T5S_ND + 1;
static_assert(T5S_SD >= T5S_NA + T5S_ND, "the d / dmin ring");

// Tensor-memory columns: A operand [half][buffer] (64 columns each), the
// min-term operand [buffer] (8 columns: 16 f16 of k), then on a 16-column
// boundary the accumulators D0 [ND], D1 [ND] and D' [ND] (16 columns each).
constexpr uint32_t T5S_COL_AM0 = 128u * T5S_NA;
constexpr uint32_t T5S_COL_D0 = (T5S_COL_AM0 + 8u * T5S_NA + 15u) & ~15u;
__host__ __device__ constexpr uint32_t t5s_col_a(int h, int b) {
    return 64u * static_cast<uint32_t>(T5S_NA * h + b);
}
__host__ __device__ constexpr uint32_t t5s_col_am(int b) { return T5S_COL_AM0 + 8u * static_cast<uint32_t>(b); }
__host__ __device__ constexpr uint32_t t5s_col_d(int h, int b) {
    return T5S_COL_D0 + 16u * static_cast<uint32_t>(h * T5S_ND + b);
}
__host__ __device__ constexpr uint32_t t5s_col_dm(int b) {
    return T5S_COL_D0 + 16u * static_cast<uint32_t>(2 * T5S_ND + b);
}
static_assert(t5s_col_dm(T5S_ND - 1) + 16u <= static_cast<uint32_t>(T5S_TMEM_COLS), "tensor-memory columns");

struct T5SParams {
    const float* x;       // [m, k]
    float* y;             // [m, rows]
    int rows, k, m;
    int nsb;              // super-blocks per row
    int S;                // weight ring slots
    int early_inputs;     // x read before waiting for the previous kernel (only y waits)
    int force_timeout;    // failure-path test
    uint32_t slot_bytes;  // 128 rows x 144 bytes
    uint32_t off_ring, off_b, off_bm, off_sc, off_dm, off_bars;
};

// Barriers, in order: full[S], empty[S], afull[2 NA], afree[2 NA], bfull[SB],
// sfree[SB], hfull[SD], dfull[ND], dfree[ND], fin (8 bytes each).
struct T5SBars {
    uint32_t full0, empty0, afull0, afree0, bfull0, sfree0, hfull0, dfull0, dfree0, fin;
    __device__ __forceinline__ explicit T5SBars(uint32_t bars, int S) {
        full0 = bars;
        empty0 = full0 + 8u * S;
        afull0 = empty0 + 8u * S;
        afree0 = afull0 + 16u * T5S_NA;
        bfull0 = afree0 + 16u * T5S_NA;
        sfree0 = bfull0 + 8u * T5S_SB;
        hfull0 = sfree0 + 8u * T5S_SB;
        dfull0 = hfull0 + 8u * T5S_SD;
        dfree0 = dfull0 + 8u * T5S_ND;
        fin = dfree0 + 8u * T5S_ND;
    }
};

// This lane's 8 values of row j of x in super-block q (k = 256 q + 8 lane ..).
__device__ __forceinline__ void t5s_load_x(const float* x, int k, int q, int j, int lane, float (&v)[8]) {
    const float4* src = reinterpret_cast<const float4*>(x + static_cast<long long>(j) * k + q * T5_SB + 8 * lane);
    const float4 a = src[0], c4 = src[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = c4.x; v[5] = c4.y; v[6] = c4.z; v[7] = c4.w;
}

// B and B' of rows j0 and j1 of x for one super-block (its slot at bptr /
// bmptr, scales at scl[2 j + {0, 1}]), from the lanes' 8 values each: the
// arithmetic of t5_build_b, two pairs interleaved; row `j1` < 0 is skipped.
__device__ __forceinline__ void t5s_convert2(const float (&v)[2][8], int j0, int j1, int lane, uint8_t* bptr,
                                             uint8_t* bmptr, float* scl) {
    float mx[2], part[2], ms[2];
#pragma unroll
    for (int b = 0; b < 2; b++) {
        mx[b] = 0.0f;
        part[b] = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; e++) {
            mx[b] = fmaxf(mx[b], fabsf(v[b][e]));
            part[b] += v[b][e];
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int b = 0; b < 2; b++) mx[b] = fmaxf(mx[b], __shfl_xor_sync(FULL, mx[b], o));
#pragma unroll
    for (int b = 0; b < 2; b++) part[b] += __shfl_xor_sync(FULL, part[b], 1);
#pragma unroll
    for (int b = 0; b < 2; b++) part[b] += __shfl_xor_sync(FULL, part[b], 2);
#pragma unroll
    for (int b = 0; b < 2; b++) ms[b] = fabsf(part[b]);
#pragma unroll
    for (int o2 = 4; o2 < 32; o2 <<= 1)
#pragma unroll
        for (int b = 0; b < 2; b++) ms[b] = fmaxf(ms[b], __shfl_xor_sync(FULL, ms[b], o2));
#pragma unroll
    for (int b = 0; b < 2; b++) {
        const int j = b ? j1 : j0;
        if (j < 0) break;   // uniform across the warp
        float inv;
        const float p2 = t5_scale(mx[b], inv);
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const float x0 = v[b][2 * e] * p2, x1 = v[b][2 * e + 1] * p2;
            const __half2 h = __floats2half2_rn(x0, x1);
            const float2 hf = __half22float2(h);
            const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
            hi[e] = *reinterpret_cast<const uint32_t*>(&h);
            lo[e] = *reinterpret_cast<const uint32_t*>(&l);
        }
        // k = 8 lane ..: core matrix (k-block lane), row j (hi) / 8 + j (lo)
        const uint32_t o = static_cast<uint32_t>(lane) * 256u + 16u * j;
        *reinterpret_cast<uint4*>(bptr + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(bptr + o + 128u) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        // group sums (lanes 4g .. 4g + 3 hold group g) under their own scale
        float sinv;
        const float s2 = t5_scale(ms[b], sinv);
        const float sp = part[b] * s2;
        const __half sh = __float2half_rn(sp);
        const __half sl = __float2half_rn(sp - __half2float(sh));
        if ((lane & 3) == 0) {
            const uint32_t om = 16u * j + 2u * static_cast<uint32_t>(lane >> 2);
            *reinterpret_cast<__half*>(bmptr + om) = sh;
            *reinterpret_cast<__half*>(bmptr + om + 128u) = sl;
        }
        if (lane == 0) {
            scl[2 * j] = inv;
            scl[2 * j + 1] = sinv;
        }
    }
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
    const T5SBars B(sb + p.off_bars, p.S);
    float yacc[T5_COLS];   // the read-back warps' row sums
#pragma unroll
    for (int j = 0; j < T5_COLS; j++) yacc[j] = 0.0f;

    if (warp == T5S_ISSUER) {
        if (lane == 0) {
            for (int s = 0; s < p.S; s++) {
                mbar_init(B.full0 + 8u * s, 1);
                mbar_init(B.empty0 + 8u * s, 32 * T5S_DECODERS);
            }
            for (int i = 0; i < 2 * T5S_NA; i++) {
                mbar_init(B.afull0 + 8u * i, 32 * T5S_DECODERS / 2);
                mbar_init(B.afree0 + 8u * i, 1);
            }
            for (int i = 0; i < T5S_SB; i++) {
                mbar_init(B.bfull0 + 8u * i, 128);
                mbar_init(B.sfree0 + 8u * i, 128);
            }
            for (int i = 0; i < T5S_SD; i++) mbar_init(B.hfull0 + 8u * i, 128);
            for (int i = 0; i < T5S_ND; i++) {
                mbar_init(B.dfull0 + 8u * i, 2);   // one commit from each issuer
                mbar_init(B.dfree0 + 8u * i, 128);
            }
            mbar_init(B.fin, 2);
            s_tmo = 0;
            fence_mbar_init();
        }
        __syncwarp();
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(T5S_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // every barrier is initialized (and the tensor-memory address written)
    // before any thread uses one
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int* tmo = &s_tmo;
    // The next kernel may start only now that this CTA holds its tensor
    // memory: a later kernel's CTA on this SM that took columns first, and
    // then waited for this kernel while holding them, would leave this CTA's
    // allocation waiting forever.
    pdl_launch_dependents();
    // x may come from the kernel just before, unless the caller declared it
    // independent of it
    if (!p.early_inputs) pdl_dependency_wait();

    if (warp == T5S_PRODUCER) {
        // ---- the weight copies: the weights are constant, so the first S
        // are requested at once; then each slot is refilled as soon as every
        // decoder has read it
        if (lane == 0) {
            const int first = nq < p.S ? nq : p.S;
            int next = 0;
            for (; next < first; next++) {
                mbar_arrive_expect_tx(B.full0 + 8u * next, p.slot_bytes);
                tma_load_2d(ring + static_cast<uint32_t>(next) * p.slot_bytes, &wmap, next * (T5_SBBYTES / 8), row0,
                            B.full0 + 8u * next);
            }
            if (!p.force_timeout) {
                for (; next < nq; next++) {
                    const int q = next - p.S, s = q % p.S;   // the slot super-block q used
                    if (!mbar_wait_bounded(B.empty0 + 8u * s, static_cast<uint32_t>((q / p.S) & 1))) {
                        atomicExch(const_cast<int*>(tmo), 1);
                        break;
                    }
                    fence_proxy_async();
                    mbar_arrive_expect_tx(B.full0 + 8u * s, p.slot_bytes);
                    tma_load_2d(ring + static_cast<uint32_t>(s) * p.slot_bytes, &wmap, next * (T5_SBBYTES / 8), row0,
                                B.full0 + 8u * s);
                }
            }
            // every copy requested lands before the CTA ends (a failed run
            // leaves the last S unread)
            for (int i = next - p.S > 0 ? next - p.S : 0; i < next; i++)
                if (!mbar_wait_bounded(B.full0 + 8u * (i % p.S), static_cast<uint32_t>((i / p.S) & 1))) break;
        }
        __syncwarp();
    } else if (warp == T5S_ISSUER || warp == T5S_ISSUER1) {
        // ---- the MMAs of half h of every super-block, once its B is built
        // and its accumulator set is free: the 8 steps (in A buffer q % NA)
        // into D_h, and for h = 1 the min term
        const int h = warp == T5S_ISSUER ? 0 : 1;
        if (lane == 0 && !p.force_timeout) {
            const uint32_t bbase = sb + p.off_b, bmbase = sb + p.off_bm;
            bool ok = true;
            for (int q = 0; q < nq; q++) {
                const int bs = q % T5S_SB, db = q % T5S_ND, ab = q % T5S_NA;
                const uint32_t ai = static_cast<uint32_t>(T5S_NA * h + ab);
                if (!mbar_wait_bounded(B.bfull0 + 8u * bs, static_cast<uint32_t>((q / T5S_SB) & 1)) ||
                    (q >= T5S_ND &&
                     !mbar_wait_bounded(B.dfree0 + 8u * db, static_cast<uint32_t>(((q - T5S_ND) / T5S_ND) & 1))) ||
                    !mbar_wait_bounded(B.afull0 + 8u * ai, static_cast<uint32_t>((q / T5S_NA) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t bq = bbase + static_cast<uint32_t>(bs) * T5S_BSLOT;
#pragma unroll
                for (int t = 0; t < 8; t++) {
                    const uint32_t kb = static_cast<uint32_t>(16 * h + 2 * t);   // first k-block of the step
                    mma_f16_ts(tmem + t5s_col_d(h, db), tmem + t5s_col_a(h, ab) + 8u * t,
                               smem_desc(bq + kb * 256u, 256u, 128u), T5_IDESC, t > 0);
                }
                if (h == 1)
                    mma_f16_ts(tmem + t5s_col_dm(db), tmem + t5s_col_am(ab),
                               smem_desc(bmbase + static_cast<uint32_t>(bs) * T5S_BMSLOT, 256u, 128u), T5_IDESC, false);
                mma_commit(B.afree0 + 8u * ai);
                mma_commit(B.dfull0 + 8u * db);
            }
            if (!ok) atomicExch(const_cast<int*>(tmo), 1);
            // every MMA issued is complete before tensor memory is released
            mma_commit(B.fin);
            if (!mbar_wait_bounded(B.fin, 0u)) atomicExch(const_cast<int*>(tmo), 1);
        }
        __syncwarp();
    } else if (warp < T5S_DECODERS) {
        // ---- decoders: half hh of every super-block of row r of the tile
        const int lq = warp & 3, hh = warp >> 2;
        const int r = 32 * lq + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * lq) << 16;
        float2* dmr = reinterpret_cast<float2*>(smem + p.off_dm);
        bool ok = !p.force_timeout;
        const uint32_t K1024 = 0x64006400u;   // f16x2 (1024, 1024)
        for (int q = 0; q < nq && ok; q++) {
            const int s = q % p.S;
            // (every decision a warp takes is a vote: the tensor-memory
            // instructions below are warp-collective)
            if (!__all_sync(FULL, mbar_wait_bounded(B.full0 + 8u * s, static_cast<uint32_t>((q / p.S) & 1)) &&
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
            mbar_arrive(B.empty0 + 8u * s);   // this row's half is done with the slot
            const int ab = q % T5S_NA;
            const uint32_t ai = static_cast<uint32_t>(T5S_NA * hh + ab);
            // A buffer q % NA is free once the MMAs of q - NA are done; those
            // were issued after the accumulators of q - NA - ND were released,
            // so the read-back is done with the d / dmin slot written here
            // (SD >= NA + ND)
            if (q >= T5S_NA &&
                !__all_sync(FULL, mbar_wait_bounded(B.afree0 + 8u * ai,
                                                    static_cast<uint32_t>(((q - T5S_NA) / T5S_NA) & 1)))) {
                ok = false;
                break;
            }
            if (hh == 0) {
                dmr[(q % T5S_SD) * T5_ROWS + r] = __half22float2(*reinterpret_cast<const __half2*>(&hd.x));
                mbar_arrive(B.hfull0 + 8u * (q % T5S_SD));
            }
            tc_fence_after();
            // the 6-bit scales of sub-blocks 4hh .. 4hh+3, one per byte
            const uint32_t scw = hh ? ((hd.w & 0x0f0f0f0fu) | ((hd.y >> 2) & 0x30303030u)) : (hd.y & 0x3f3f3f3fu);
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
            mbar_arrive(B.afull0 + 8u * ai);
        }
        if (!ok) atomicExch(const_cast<int*>(tmo), 1);
    } else if (warp >= T5S_BUILD0) {
        // ---- warps 14..17: B of rows ew and ew + 4 of x, super-block after
        // super-block. B(qb) takes the slot and the scales of qb - SB: both
        // are free once the read-back has read the accumulators (so their
        // MMAs are done) and the scales of qb - SB.
        const int ew = warp - T5S_BUILD0;
        uint8_t* bring = smem + p.off_b;
        uint8_t* bmring = smem + p.off_bm;
        float* scr = reinterpret_cast<float*>(smem + p.off_sc);
        const int j0 = ew < p.m ? ew : -1;
        const int j1 = ew + 4 < p.m ? ew + 4 : -1;
        bool ok = !p.force_timeout;
        // x of the next three super-blocks, in three register sets used in
        // turn (loaded two super-blocks ahead; a copy from one set to another
        // would wait for the loads in flight)
        float xa[2][8] = {}, xb[2][8] = {}, xc[2][8] = {};
        auto load = [&](int qq, float(&v)[2][8]) {
            if (j0 >= 0) t5s_load_x(p.x, p.k, qq, j0, lane, v[0]);
            if (j1 >= 0) t5s_load_x(p.x, p.k, qq, j1, lane, v[1]);
        };
        auto step = [&](int qb, const float(&cur)[2][8], float(&nxt)[2][8]) -> bool {
            // nxt: the set of qb - 1, already built
            if (qb >= T5S_SB) {
                const int qo = qb - T5S_SB;
                if (!__all_sync(FULL, mbar_wait_bounded(B.sfree0 + 8u * (qo % T5S_SB),
                                                        static_cast<uint32_t>((qo / T5S_SB) & 1)) &&
                                          *tmo == 0))
                    return false;
            }
            if (qb + 2 < nq) load(qb + 2, nxt);
            const int bs = qb % T5S_SB;
            if (j0 >= 0)
                t5s_convert2(cur, j0, j1, lane, bring + bs * T5S_BSLOT, bmring + bs * T5S_BMSLOT,
                             scr + bs * 2 * T5_COLS);
            fence_proxy_async();   // B is read by the tensor cores (async proxy)
            mbar_arrive(B.bfull0 + 8u * bs);
            return true;
        };
        if (ok) {
            // the second k-block of every B' slot is zeros (the rows of the
            // first that belong to rows j >= m of x stay unwritten: they reach
            // only columns of D' that are not read)
            for (int i = ew * 32 + lane; i < T5S_SB * 64; i += 128)
                reinterpret_cast<uint32_t*>(bmring)[(i >> 6) * 128 + 64 + (i & 63)] = 0u;
            load(0, xa);
            if (nq > 1) load(1, xb);
        }
        // B(qb) from the set of qb, x of qb + 2 into the set of qb - 1
        for (int qb = 0; qb < nq && ok; qb += 3) {
            ok = step(qb, xa, xc);
            if (ok && qb + 1 < nq) ok = step(qb + 1, xb, xa);
            if (ok && qb + 2 < nq) ok = step(qb + 2, xc, xb);
        }
        if (!ok) atomicExch(const_cast<int*>(tmo), 1);
    } else {
        // ---- warps 9..12: the read-back and fold of every super-block for
        // lane quarter warp % 4 of the rows
        const int lq = warp & 3;
        const int r = 32 * lq + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * lq) << 16;
        const float* scr = reinterpret_cast<const float*>(smem + p.off_sc);
        const float2* dmr = reinterpret_cast<const float2*>(smem + p.off_dm);
        bool ok = !p.force_timeout;
        for (int q = 0; q < nq && ok; q++) {
            const int db = q % T5S_ND, hs = q % T5S_SD, bs = q % T5S_SB;
            // the accumulators, the rows' d / dmin, and (long done) the
            // scales of B(q)
            if (!__all_sync(FULL, mbar_wait_bounded(B.dfull0 + 8u * db, static_cast<uint32_t>((q / T5S_ND) & 1)) &&
                                      mbar_wait_bounded(B.hfull0 + 8u * hs, static_cast<uint32_t>((q / T5S_SD) & 1)) &&
                                      mbar_wait_bounded(B.bfull0 + 8u * bs, static_cast<uint32_t>((q / T5S_SB) & 1)) &&
                                      *tmo == 0)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t dv[16], ev[16], mv[16];
            tmem_ld16(tmem + lane_base + t5s_col_d(0, db), dv);
            tmem_ld16(tmem + lane_base + t5s_col_d(1, db), ev);
            tmem_ld16(tmem + lane_base + t5s_col_dm(db), mv);
            const float2 dd = dmr[hs * T5_ROWS + r];
            float sq[2 * T5_COLS];
#pragma unroll
            for (int i = 0; i < T5_COLS / 2; i++) {
                const float4 v = reinterpret_cast<const float4*>(scr + bs * 2 * T5_COLS)[i];
                sq[4 * i] = v.x; sq[4 * i + 1] = v.y; sq[4 * i + 2] = v.z; sq[4 * i + 3] = v.w;
            }
            tmem_wait_ld();
            tc_fence_before();
            // the accumulators are free, and so are B(q)'s slot and scales
            mbar_arrive(B.dfree0 + 8u * db);
            mbar_arrive(B.sfree0 + 8u * bs);
#pragma unroll
            for (int j = 0; j < T5_COLS; j++) {
                if (j < p.m) {
                    const float hi = __uint_as_float(dv[j]) + __uint_as_float(ev[j]);
                    const float lo = __uint_as_float(dv[8 + j]) + __uint_as_float(ev[8 + j]);
                    const float t = dd.x * (hi + lo);
                    const float u = dd.y * (__uint_as_float(mv[j]) + __uint_as_float(mv[8 + j]));
                    yacc[j] = __fmaf_rn(t, sq[2 * j], yacc[j]);
                    yacc[j] = __fmaf_rn(-u, sq[2 * j + 1], yacc[j]);
                }
            }
        }
        if (!ok) atomicExch(const_cast<int*>(tmo), 1);
    }

    // every role is done: tensor memory is released, and the rows written
    tc_fence_before();
    __syncthreads();
    if (warp == T5S_ISSUER) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(T5S_TMEM_COLS)
                     : "memory");
        return;
    }
    if (warp < T5S_EPI0 || warp >= T5S_EPI0 + 4) return;
    if (*tmo) {
#pragma unroll
        for (int j = 0; j < T5_COLS; j++) yacc[j] = __int_as_float(0x7fc00000);
        if (warp == T5S_EPI0 && lane == 0) atomicOr(&g_status, STATUS_WAIT_TIMEOUT);
    }
    // y after the previous kernel is done with it
    if (p.early_inputs) pdl_dependency_wait();
    const int r = 32 * (warp & 3) + lane;
    if (row0 + r < p.rows) {
#pragma unroll
        for (int j = 0; j < T5_COLS; j++)
            if (j < p.m) p.y[static_cast<long long>(j) * p.rows + row0 + r] = yacc[j];
    }
}

}  // namespace qmv
