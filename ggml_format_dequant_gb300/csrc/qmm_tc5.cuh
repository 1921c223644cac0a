// qmm_tc5.cuh -- the small-M batched product y[m, rows] = x[m, k] W^T on the
// fifth-generation tensor cores (tcgen05.mma, accumulators in tensor memory),
// for Q4_K rows and m <= 8 rows of x.
//
// Shape of the computation:
//  * A CTA owns a tile of 128 rows of W and one k-chunk of them; the CL
//    chunks of a tile are the CL CTAs of one thread-block cluster, which add
//    their partial sums through distributed shared memory at the end (in
//    rank order: deterministic, no atomics, no memory beyond x and y).
//  * The weights arrive by 2-D TMA tensor copies, one super-block column of
//    the tile (128 rows x 144 bytes) per ring slot; a thread of the four
//    decoder warps owns one row, reads its 144 bytes and writes the row's
//    A operand into tensor memory (tcgen05.st, 32x32b: lane = row). A
//    super-block's operand holds the exact integer products sc_j * q (at
//    most 63 * 15 = 945, exact in f16), so one MMA chain of 16 k-steps covers
//    the whole super-block and d is applied once per super-block.
//  * B (the x side, in shared memory, K-major canonical layout without
//    swizzle) holds every row j of x as two f16 parts, hi (column j) and lo
//    (column 8 + j), after a power-of-two scale per (super-block, j) that
//    puts the super-block's largest |x| in [2^14, 2^15): the pair carries
//    about 22 bits of x and each product sc*q*part is exact.
//  * The min term dmin * sum_j m_j S_j (S_j the sum of x over group j) is one
//    more MMA per super-block, A' = the eight 6-bit m_j (k = 0..7, 8..15
//    zero), B' = S_j as hi/lo under its own power-of-two scale, into its own
//    accumulator.
//  * Per super-block and row the four decoder threads read the two
//    accumulators back (tcgen05.ld) and fold y_j += d * D_j * 2^-e -
//    dmin * D'_j * 2^-e'. Two accumulator pairs alternate, so that the MMAs
//    of one super-block run while the previous one is read back.
//  * One thread of a fifth warp issues the TMA copies and the MMAs
//    (tcgen05.mma ... kind::f16, A from tensor memory, B from shared memory)
//    and commits them to mbarriers. Every wait is bounded; a wait that gives
//    up marks the CTA's outputs NaN and sets STATUS_WAIT_TIMEOUT.
//  * x is staged by bulk copies (after the dependency wait in a chain) and
//    converted by the decoder warps. Tensor memory is allocated before
//    anything else and released before the cluster barrier, so a CTA holding
//    it never waits for another CTA. The partial sums travel by remote stores
//    into the owning CTA's shared memory before that one barrier.
#pragma once

#include <cuda.h>   // CUtensorMap (the type only)

#include "qmv_launch.cuh"

namespace qmv {

constexpr int T5_ROWS = 128;         // rows of a tile (MMA M)
constexpr int T5_N = 16;             // MMA N: hi parts in columns 0..7, lo parts in 8..15
constexpr int T5_COLS = 8;           // rows of x a launch takes, at most
constexpr int T5_SB = 256;           // weights of a super-block
constexpr int T5_SBBYTES = 144;      // bytes of a Q4_K super-block
constexpr int T5_THREADS = 160;      // four decoder warps and the issuing warp
constexpr int T5_TMEM_COLS = 256;    // tensor-memory columns a CTA allocates
// Tensor-memory columns: A operand of half a super-block (128 k, 64 columns)
// x 2, the min-term operand (16 k, 8 columns), accumulators 16 columns each.
constexpr uint32_t T5_COL_A0 = 0, T5_COL_A1 = 64, T5_COL_AM = 128;
__host__ __device__ constexpr uint32_t t5_col_d(int b) { return 160u + 16u * static_cast<uint32_t>(b); }
__host__ __device__ constexpr uint32_t t5_col_dm(int b) { return 192u + 16u * static_cast<uint32_t>(b); }

struct T5Params {
    const float* x;       // [m, k]
    float* y;             // [m, rows]
    int rows, k, m;
    int nsb;              // super-blocks per row
    int CL;               // k-chunks of a tile = cluster size
    int S;                // ring slots
    int early_inputs;     // x read before waiting for the previous kernel (only y waits)
    int late_alloc;       // tensor memory taken after the wait for the previous kernel (chained launches)
    int force_timeout;    // failure-path test
    uint32_t slot_bytes;  // 128 rows x 144 bytes
    uint32_t off_ring, off_b, off_bm, off_sc, off_x, off_in, off_bars;
};

// ---------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hsub2_5(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_st16(uint32_t t, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(t),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t t, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(t), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t t, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(t)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// D (+)= A (tensor memory, K-major) * B (shared memory descriptor), f16 in,
// f32 accumulate; acc = false overwrites D.
__device__ __forceinline__ void mma_f16_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(idesc), "r"(acc ? 1 : 0)
        : "memory");
}
// Arrive on the mbarrier once every MMA this thread issued so far is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 2-D tensor copy of the box at (x, y) (elements) into shared memory.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor: K-major, no swizzle; core matrices of 8
// rows x 16 bytes, lbo bytes apart along K, sbo bytes apart along M/N.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((addr >> 4) & 0x3fffu) | (static_cast<uint64_t>((lbo >> 4) & 0x3fffu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3fffu) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16: f32 accumulator, f16 A and B, both
// K-major, N = 16, M = 128.
constexpr uint32_t T5_IDESC = (1u << 4) | (static_cast<uint32_t>(T5_N >> 3) << 17) |
                              (static_cast<uint32_t>(T5_ROWS >> 4) << 24);

// Power-of-two scale of a block of values with largest magnitude mx: 2^e puts
// mx in [2^14, 2^15) (2^0 for a zero block); returns 2^e, inv receives 2^-e.
__device__ __forceinline__ float t5_scale(float mx, float& inv) {
    const int E = static_cast<int>(__float_as_uint(mx) >> 23);   // biased exponent; mx < 2^(E - 126)
    int e = mx > 0.0f ? 14 - (E - 127) : 0;
    e = e > 126 ? 126 : (e < -126 ? -126 : e);
    inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    return __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
}

// B and B' of super-blocks 0 .. nq-1 from x (row j of super-block q at
// x + j * xstride + 256 q; any readable memory, global or shared), by warps
// `warp` of `nwarps` that all call it: the (super-block, row of x) pairs are
// dealt over the warps, four at a time a warp so that their shuffle trees
// interleave; rows j >= m are zeros. Scales go to scl[(q * 8 + j) * 2 + {0, 1}].
__device__ __forceinline__ void t5_build_b(const float* x, long long xstride, int nq, int m, int warp, int nwarps,
                                           int lane, uint8_t* bptr, uint8_t* bmptr, float* scl) {
    for (int i = warp * 32 + lane; i < nq * 64; i += nwarps * 32)
        reinterpret_cast<uint32_t*>(bmptr)[(i >> 6) * 128 + 64 + (i & 63)] = 0u;
    for (int base = warp; base < nq * T5_COLS; base += 4 * nwarps) {
        float v[4][8], mx[4], part[4];
#pragma unroll
        for (int b = 0; b < 4; b++) {
            const int pi = base + nwarps * b;
            const int q = pi / T5_COLS, j = pi % T5_COLS;
            if (pi < nq * T5_COLS && j < m) {
                const float4* src =
                    reinterpret_cast<const float4*>(x + static_cast<long long>(j) * xstride + q * T5_SB + 8 * lane);
                const float4 a = src[0], c4 = src[1];
                v[b][0] = a.x; v[b][1] = a.y; v[b][2] = a.z; v[b][3] = a.w;
                v[b][4] = c4.x; v[b][5] = c4.y; v[b][6] = c4.z; v[b][7] = c4.w;
            } else {
#pragma unroll
                for (int e = 0; e < 8; e++) v[b][e] = 0.0f;
            }
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
            for (int b = 0; b < 4; b++) mx[b] = fmaxf(mx[b], __shfl_xor_sync(FULL, mx[b], o));
#pragma unroll
        for (int b = 0; b < 4; b++) {
            part[b] += __shfl_xor_sync(FULL, part[b], 1);
        }
#pragma unroll
        for (int b = 0; b < 4; b++) part[b] += __shfl_xor_sync(FULL, part[b], 2);
        float ms[4];
#pragma unroll
        for (int b = 0; b < 4; b++) ms[b] = fabsf(part[b]);
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1)
#pragma unroll
            for (int b = 0; b < 4; b++) ms[b] = fmaxf(ms[b], __shfl_xor_sync(FULL, ms[b], o2));
#pragma unroll
        for (int b = 0; b < 4; b++) {
            const int pi = base + nwarps * b;
            if (pi >= nq * T5_COLS) break;   // uniform across the warp
            const int q = pi / T5_COLS, j = pi % T5_COLS;
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
            // k = 256q + 8 lane: core matrix (k-block 32q + lane), row j (hi) / 8 + j (lo)
            const uint32_t o = static_cast<uint32_t>(32 * q + lane) * 256u + 16u * j;
            *reinterpret_cast<uint4*>(bptr + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(bptr + o + 128u) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            // group sums (lanes 4g .. 4g + 3 hold group g) under their own scale
            float sinv;
            const float s2 = t5_scale(ms[b], sinv);
            const float sp = part[b] * s2;
            const __half sh = __float2half_rn(sp);
            const __half sl = __float2half_rn(sp - __half2float(sh));
            if ((lane & 3) == 0) {
                const int g = lane >> 2;
                const uint32_t om = static_cast<uint32_t>(q) * 512u + 16u * j + 2u * g;
                *reinterpret_cast<__half*>(bmptr + om) = sh;
                *reinterpret_cast<__half*>(bmptr + om + 128u) = sl;
            }
            if (lane == 0) {
                scl[(q * T5_COLS + j) * 2] = inv;
                scl[(q * T5_COLS + j) * 2 + 1] = sinv;
            }
        }
    }
}

// ------------------------------------------------------------- the kernel

__global__ void __launch_bounds__(T5_THREADS, 1)
    qmm_tc5_q4k_kernel(const __grid_constant__ CUtensorMap wmap, const T5Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint32_t s_tmem;
    __shared__ int s_tmo;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int tile = static_cast<int>(blockIdx.x) / p.CL;
    const int c = static_cast<int>(blockIdx.x) % p.CL;   // cluster rank: the k-chunk
    const int q0 = c * p.nsb / p.CL;
    const int nq = (c + 1) * p.nsb / p.CL - q0;           // super-blocks of the chunk
    const int row0 = tile * T5_ROWS;
    const uint32_t sb = smem_u32(smem);
    const uint32_t ring = sb + p.off_ring;
    const uint32_t bars = sb + p.off_bars;
    // barriers: full[S], empty[S], afull[2], afree[2], dfull[2], dfree[2], fin, xbar
    const uint32_t full0 = bars, empty0 = bars + 8u * p.S, afull0 = bars + 16u * p.S;
    const uint32_t afree0 = afull0 + 16u, dfull0 = afull0 + 32u, dfree0 = afull0 + 48u, fin = afull0 + 64u;
    const uint32_t xbar = fin + 8u;
    const int rpr = T5_ROWS / p.CL;   // rows of the tile whose sums this CTA adds up and writes
    // x of the chunk, rows 0..m-1, staged by bulk copies
    auto request_x = [&]() {
        const uint32_t xb = static_cast<uint32_t>(nq * T5_SB * 4);
        mbar_arrive_expect_tx(xbar, xb * static_cast<uint32_t>(p.m));
        for (int j = 0; j < p.m; j++)
            tma_bulk_g2s(sb + p.off_x + static_cast<uint32_t>(j) * xb,
                         p.x + static_cast<long long>(j) * p.k + static_cast<long long>(q0) * T5_SB, xb, xbar);
    };

    pdl_launch_dependents();

    if (warp == 4) {
        if (lane == 0) {
            for (int s = 0; s < p.S; s++) {
                mbar_init(full0 + 8u * s, 1);
                mbar_init(empty0 + 8u * s, T5_ROWS);
            }
            for (int b = 0; b < 2; b++) {
                mbar_init(afull0 + 8u * b, T5_ROWS);
                mbar_init(afree0 + 8u * b, 1);
                mbar_init(dfull0 + 8u * b, 1);
                mbar_init(dfree0 + 8u * b, T5_ROWS);
            }
            mbar_init(fin, 1);
            mbar_init(xbar, 1);
            s_tmo = 0;
            fence_mbar_init();
            if (p.early_inputs) request_x();
            // the first slots: the weights are constant, request them at once
            const int first = nq < p.S ? nq : p.S;
            for (int i = 0; i < first; i++) {
                mbar_arrive_expect_tx(full0 + 8u * i, p.slot_bytes);
                tma_load_2d(ring + static_cast<uint32_t>(i) * p.slot_bytes, &wmap, (q0 + i) * (T5_SBBYTES / 8), row0,
                            full0 + 8u * i);
            }
        }
        __syncwarp();
        if (!p.late_alloc) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(&s_tmem)),
                         "r"(T5_TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    // every barrier is initialized before any thread waits on one
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // x may come from the kernel just before, unless the caller declared it
    // independent of it.
    if (!p.early_inputs) {
        pdl_dependency_wait();
        if (tid == 4 * 32) request_x();
    }
    // A chained launch takes its tensor memory only now, after its wait for
    // the previous kernel (while warps 0..3 build B): a CTA never holds
    // columns while it waits for another kernel that may still need columns
    // on this SM. (A plain launch starts after the previous kernel has ended;
    // independent calls release their columns before they wait.)
    if (p.late_alloc && warp == 4) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(T5_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }

    // ---- B: x of the chunk as hi / lo f16 (warps 0..3), zero where j >= m
    uint8_t* bptr = smem + p.off_b;
    uint8_t* bmptr = smem + p.off_bm;
    float* scl = reinterpret_cast<float*>(smem + p.off_sc);   // [nq][8][2]: 2^-e of x, 2^-e' of the sums
    if (warp < 4) {
        const bool xok = __all_sync(FULL, mbar_wait_bounded(xbar, 0u));
        if (!xok && lane == 0) atomicExch(&s_tmo, 1);
        t5_build_b(reinterpret_cast<const float*>(smem + p.off_x), static_cast<long long>(nq) * T5_SB, nq, p.m, warp, 4,
                   lane, bptr, bmptr, scl);
        fence_proxy_async();   // B is read by the tensor cores (async proxy)
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int* tmo = &s_tmo;

    if (warp == 4) {
        // ---- the issuing thread: MMAs of every super-block, ring refills
        if (lane == 0 && !p.force_timeout) {
            const uint32_t bbase = sb + p.off_b, bmbase = sb + p.off_bm;
            int next = p.S < nq ? p.S : nq;   // next super-block to request
            bool ok = true;
            for (int q = 0; q < nq && ok; q++) {
                const int db = q & 1;
                if (q >= 2 && !mbar_wait_bounded(dfree0 + 8u * db, static_cast<uint32_t>(((q - 2) >> 1) & 1))) {
                    ok = false;
                    break;
                }
                for (int h = 0; h < 2; h++) {
                    if (!mbar_wait_bounded(afull0 + 8u * h, static_cast<uint32_t>(q & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t acol = h ? T5_COL_A1 : T5_COL_A0;
#pragma unroll
                    for (int t = 0; t < 8; t++) {
                        const uint32_t kb = static_cast<uint32_t>(32 * q + 16 * h + 2 * t);   // first k-block of the step
                        mma_f16_ts(tmem + t5_col_d(db), tmem + acol + 8u * t, smem_desc(bbase + kb * 256u, 256u, 128u),
                                   T5_IDESC, h > 0 || t > 0);
                    }
                    if (h == 1)
                        mma_f16_ts(tmem + t5_col_dm(db), tmem + T5_COL_AM,
                                   smem_desc(bmbase + static_cast<uint32_t>(q) * 512u, 256u, 128u), T5_IDESC, false);
                    mma_commit(afree0 + 8u * h);
                    // refill: the slot of super-block q is free once every row has read it
                    if (h == 0 && next < nq) {
                        const int s = q % p.S;
                        if (!mbar_wait_bounded(empty0 + 8u * s, static_cast<uint32_t>((q / p.S) & 1))) {
                            ok = false;
                            break;
                        }
                        fence_proxy_async();
                        mbar_arrive_expect_tx(full0 + 8u * s, p.slot_bytes);
                        tma_load_2d(ring + static_cast<uint32_t>(s) * p.slot_bytes, &wmap,
                                    (q0 + next) * (T5_SBBYTES / 8), row0, full0 + 8u * s);
                        next++;
                    }
                }
                if (!ok) break;
                mma_commit(dfull0 + 8u * db);
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
            for (int i = 0; i < (nq < p.S ? nq : p.S); i++)
                if (!mbar_wait_bounded(full0 + 8u * i, 0u)) break;
        }
        __syncwarp();
    } else {
        // ---- decoder / reader threads: row r of the tile
        const int r = tid;
        float yacc[T5_COLS];
#pragma unroll
        for (int j = 0; j < T5_COLS; j++) yacc[j] = 0.0f;
        const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
        float dprev = 0.0f, mprev = 0.0f;   // d and dmin of the super-block read back next
        bool ok = !p.force_timeout;
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
                uint32_t qs[32];
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const uint4 v = lds128<0>(a + 16u + 16u * i);
                    qs[4 * i] = v.x; qs[4 * i + 1] = v.y; qs[4 * i + 2] = v.z; qs[4 * i + 3] = v.w;
                }
                mbar_arrive(empty0 + 8u * s);   // this row is done with the slot
                {
                    const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hd.x));
                    dcur = dd.x;
                    mcur = dd.y;
                }
                // 6-bit scales and mins of sub-blocks 0..3 and 4..7, one per byte
                const uint32_t sc_lo = hd.y & 0x3f3f3f3fu;
                const uint32_t m_lo = hd.z & 0x3f3f3f3fu;
                const uint32_t sc_hi = (hd.w & 0x0f0f0f0fu) | ((hd.y >> 2) & 0x30303030u);
                const uint32_t m_hi = ((hd.w >> 4) & 0x0f0f0f0fu) | ((hd.z >> 2) & 0x30303030u);
                const uint32_t K1024 = 0x64006400u;   // f16x2 (1024, 1024)
                for (int h = 0; h < 2; h++) {
                    const int i = 2 * q + h;
                    if (i >= 2 &&
                        !__all_sync(FULL, mbar_wait_bounded(afree0 + 8u * h, static_cast<uint32_t>(((i - 2) >> 1) & 1)))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t scw = h ? sc_hi : sc_lo;
                    const uint32_t acol = tmem + lane_base + (h ? T5_COL_A1 : T5_COL_A0);
#pragma unroll
                    for (int gg = 0; gg < 4; gg++) {
                        // sub-block g = 4h + gg: chunk cc = g / 2, low (even g) or high nibbles
                        const int cc = 2 * h + (gg >> 1);
                        const uint32_t bsel = static_cast<uint32_t>(gg) | (static_cast<uint32_t>(gg) << 8) | 0x4040u;
                        const uint32_t sc2 = hsub2_5(prmt(scw, 0x64646464u, bsel), K1024);   // (sc, sc)
                        const uint32_t nb2 = hmul2(sc2, 0xE400E400u);                       // (-1024 sc, -1024 sc)
                        uint32_t av[16];
#pragma unroll
                        for (int w = 0; w < 8; w++) {
                            const uint32_t wv = qs[8 * cc + w];
                            const uint32_t n = (gg & 1) ? ((wv >> 4) & 0x0f0f0f0fu) : (wv & 0x0f0f0f0fu);
                            av[2 * w] = hfma2(prmt(n, 0x64646464u, 0x4140u), sc2, nb2);
                            av[2 * w + 1] = hfma2(prmt(n, 0x64646464u, 0x4342u), sc2, nb2);
                        }
                        tmem_st16(acol + 16u * gg, av);
                    }
                    if (h == 1) {
                        // the min-term operand: m_0 .. m_7 at k = 0..7, zeros at 8..15
                        uint32_t mv[8];
                        mv[0] = hsub2_5(prmt(m_lo, 0x64646464u, 0x4140u), K1024);
                        mv[1] = hsub2_5(prmt(m_lo, 0x64646464u, 0x4342u), K1024);
                        mv[2] = hsub2_5(prmt(m_hi, 0x64646464u, 0x4140u), K1024);
                        mv[3] = hsub2_5(prmt(m_hi, 0x64646464u, 0x4342u), K1024);
                        mv[4] = mv[5] = mv[6] = mv[7] = 0u;
                        tmem_st8(tmem + lane_base + T5_COL_AM, mv);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(afull0 + 8u * h);
                }
                if (!ok) break;
            }
            if (q >= 1) {
                // read back super-block q - 1 and fold it into the row sums
                const int qb = q - 1, db = qb & 1;
                if (!__all_sync(FULL, mbar_wait_bounded(dfull0 + 8u * db, static_cast<uint32_t>((qb >> 1) & 1)))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t dv[16], mv[16];
                tmem_ld16(tmem + lane_base + t5_col_d(db), dv);
                tmem_ld16(tmem + lane_base + t5_col_dm(db), mv);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(dfree0 + 8u * db);
                const float* sq = scl + qb * T5_COLS * 2;
#pragma unroll
                for (int j = 0; j < T5_COLS; j++) {
                    if (j < p.m) {
                        const float t = dprev * (__uint_as_float(dv[j]) + __uint_as_float(dv[8 + j]));
                        const float u = mprev * (__uint_as_float(mv[j]) + __uint_as_float(mv[8 + j]));
                        yacc[j] = __fmaf_rn(t, sq[2 * j], yacc[j]);
                        yacc[j] = __fmaf_rn(-u, sq[2 * j + 1], yacc[j]);
                    }
                }
            }
            dprev = dcur;
            mprev = mcur;
        }
        if (!ok) atomicExch(const_cast<int*>(tmo), 1);
        tc_fence_before();
        __syncthreads();
        // ---- the end of the row: the row's partial sums go to the CTA that
        // adds up row r (rank r / rpr); after the cluster barrier (which the
        // issuing warp joins once tensor memory is released) that CTA adds the
        // CL chunks' sums in rank order and writes y.
        if (*tmo) {
#pragma unroll
            for (int j = 0; j < T5_COLS; j++) yacc[j] = __int_as_float(0x7fc00000);
            if (r == 0) atomicOr(&g_status, STATUS_WAIT_TIMEOUT);
        }
        const int dst = r / rpr, rl = r - dst * rpr;
        const uint32_t inbox = sb + p.off_in;   // [rank][rpr][8] floats
        if (dst != c) {
            const uint32_t a = cluster_addr(inbox + static_cast<uint32_t>(c * rpr + rl) * 32u, static_cast<uint32_t>(dst));
            st_cluster_v4(a, make_uint4(__float_as_uint(yacc[0]), __float_as_uint(yacc[1]), __float_as_uint(yacc[2]),
                                        __float_as_uint(yacc[3])));
            st_cluster_v4(a + 16u, make_uint4(__float_as_uint(yacc[4]), __float_as_uint(yacc[5]),
                                              __float_as_uint(yacc[6]), __float_as_uint(yacc[7])));
        }
        __syncwarp();
        cluster_sync();   // every rank's partial sums have landed; no remote access follows
        if (dst != c) return;
        if (p.early_inputs) pdl_dependency_wait();
        const float* in = reinterpret_cast<const float*>(smem + p.off_in);
#pragma unroll
        for (int j = 0; j < T5_COLS; j++) {
            if (j < p.m) {
                float v = 0.0f;
                for (int src = 0; src < p.CL; src++)
                    v += src == c ? yacc[j] : in[(src * rpr + rl) * T5_COLS + j];
                if (row0 + r < p.rows) p.y[static_cast<long long>(j) * p.rows + row0 + r] = v;
            }
        }
        return;
    }
    __syncthreads();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(T5_TMEM_COLS) : "memory");
    cluster_sync();
}

}  // namespace qmv
