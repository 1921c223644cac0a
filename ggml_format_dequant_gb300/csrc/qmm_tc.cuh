// qmm_tc.cuh -- the small-M batched product y[m, rows] = x[m, k] W^T on the
// tensor cores (warp-level mma.sync m16n8k16, f16 operands, f32 accumulate);
// one launch covers rows of up to 4096 weights, longer rows go in k-chunks.
//
// The product is a skinny dense contraction (m <= 8 columns), so a warp-level
// MMA with register accumulators fits it: the weights' per-32 (Q4_K, Q8_0) or
// per-16 (Q6_K) scales are applied to each group's partial product in
// registers right after its MMAs, which keeps every operand exact:
//  * A (16 weight rows x 16 k): the integer codes, exact in f16: Q4_K's q as
//    the subnormal q * 2^-24 or 16 q * 2^-24 (one mask, or a shift and a
//    mask, per pair; the power of two goes into the row scale), Q6_K's q - 32 and Q8_0's q made from the code bytes with
//    one byte permute into the f16 pattern of 1024 + v and one f16x2
//    subtraction.
//  * B (16 k x 8 rows of x): x in two f16 parts, hi + lo, after a power-of-two
//    scale per 32-group and row of x that puts the group maximum in
//    [2^14, 2^15); hi + lo carries x to about 22 bits, so the MMA pair
//    A*hi + A*lo is the group's integer-code dot at f32 accuracy.
//  * Per group the accumulator D (16 x 8, four values a lane) is folded into
//    the row sums: y += (d*sc * 2^-s) * D  (- dmin*m * sum(x) for Q4_K).
// The k order inside each 16-column half of a group is permuted identically
// for A and B so that a lane's code bytes are aligned 4-byte runs: MMA
// columns (2t, 2t+1, 2t+8, 2t+9) of lane group t hold positions (4t, 4t+2,
// 4t+1, 4t+3) of the half.
//
// Staging: a CTA owns a run of rows; every row of a piece is copied by its own
// bulk TMA copy into a slot whose row stride is 16 bytes past a multiple of
// 128, so that the 32 lanes of a warp, reading 8 rows x 4 runs, hit 32
// different banks. Warps split k into slices of 8 groups (256 weights); each
// keeps its slice's x fragments (hi and lo, 64 registers) for the whole call.
// Rows are processed in tiles of 16; slice partials are parked per (row,
// slice, column) and summed in slice order at the end. Waits are bounded as in
// qmv_kernel.cuh.
#pragma once

#include "qmv_launch.cuh"

namespace qmv {

struct TParams {
    const uint8_t* w;             // packed rows [rows, K / QK blocks], K the full row length
    const float* x;               // x[i, 0] of this launch's k-chunk (row stride xstride)
    float* y;                     // [m, rows]
    unsigned long long wbytes;    // readable bytes from w (tail clipping)
    int rows, k, m;               // k: the chunk's weights per row; m: rows of x, 1..8
    int xstride;                  // floats between rows of x (the full row length)
    uint32_t wpitch;              // bytes between rows of W
    uint32_t woff;                // byte offset of the chunk inside a row
    int accumulate;               // add to y (a later k-chunk) instead of writing it
    int ngroups;                  // k / 32
    uint32_t rowbytes;            // bytes of one row's chunk
    uint32_t stride;              // shared-memory row stride (16 mod 128)
    int KS;                       // warps, one per slice of 8 groups
    int CR;                       // rows per piece
    int S;                        // ring slots
    int rq, rrem;                 // rows per CTA: rq or rq + 1 (the first rrem CTAs)
    int early_inputs;
    uint32_t slot_stride;         // bytes per slot (rows rounded up to 16)
    uint32_t off_st, off_red, off_ring, off_bars, off_cnt;
};

constexpr int TC_GROUPS_PER_SLICE = 8;   // 32-weight groups per warp slice
constexpr int TC_TILE_ROWS = 16;
constexpr int TC_COLS = 8;               // rows of x per launch, at most

// ----------------------------------------------------------- f16 helpers

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Bytes 0 and 2 (even) or 1 and 3 (odd) of w, each v <= 1023, as the f16
// pair (v - off), bias being the f16x2 pattern of 1024 + off.
__device__ __forceinline__ uint32_t f16_even(uint32_t w, uint32_t bias) {
    return hsub2(prmt(w, 0x64646464u, 0x4240u), bias);
}
__device__ __forceinline__ uint32_t f16_odd(uint32_t w, uint32_t bias) {
    return hsub2(prmt(w, 0x64646464u, 0x4341u), bias);
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float2 unpack_h2(uint32_t v) {
    return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

// 4 bytes at the 2-byte aligned shared address a.
__device__ __forceinline__ uint32_t lds32_a2(uint32_t a) {
    const uint32_t wa = a & ~3u;
    return __funnelshift_r(lds32<0>(wa), lds32<4>(wa), (a & 3u) * 8u);
}

// Four floats at the 16-byte aligned shared address a.
__device__ __forceinline__ float4 lds_f4(uint32_t a) {
    const uint4 v = lds128<0>(a);
    return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
}

// MMA of one 16-column half (A from the code words of rows g and g+8, already
// shifted/masked to one byte per weight, with the f16 bias) against hi and lo.
__device__ __forceinline__ void mma_half(float (&D)[4], uint32_t ka, uint32_t kb, uint32_t bias, uint32_t bh0,
                                         uint32_t bh1, uint32_t bl0, uint32_t bl1) {
    const uint32_t a0 = f16_even(ka, bias), a1 = f16_even(kb, bias);
    const uint32_t a2 = f16_odd(ka, bias), a3 = f16_odd(kb, bias);
    mma16816(D, a0, a1, a2, a3, bh0, bh1);
    mma16816(D, a0, a1, a2, a3, bl0, bl1);
}

// MMA of one 16-column half with A given directly (rows g, g+8; even, odd
// columns) against hi and lo.
__device__ __forceinline__ void mma_half_a(float (&D)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t bh0, uint32_t bh1, uint32_t bl0, uint32_t bl1) {
    mma16816(D, a0, a1, a2, a3, bh0, bh1);
    mma16816(D, a0, a1, a2, a3, bl0, bl1);
}

constexpr float TWO24 = 16777216.0f;

// y4 += scale_row * inv_col * D (columns 2t, 2t+1 for rows g, g+8).
__device__ __forceinline__ void fold(float (&y4)[4], const float (&D)[4], float sa, float sb, float inv0, float inv1) {
    y4[0] = __fmaf_rn(sa * inv0, D[0], y4[0]);
    y4[1] = __fmaf_rn(sa * inv1, D[1], y4[1]);
    y4[2] = __fmaf_rn(sb * inv0, D[2], y4[2]);
    y4[3] = __fmaf_rn(sb * inv1, D[3], y4[3]);
}

// ------------------------------------------------------- format bodies
//
// slice(): one 16-row tile against the warp's slice of groups. ra / rb:
// shared addresses of rows g and g + 8 of the tile (their first byte);
// xh / xl: the lane's B fragments (hi, lo) of the slice's groups, [group][4]
// = MMA0 b0, b1, MMA1 b0, b1; st: shared address of the statistics
// (2^-s, sum x) of columns 2t, 2t + 1 of the slice's group 0 (64 bytes per
// group further); y4: the row sums of (g, 2t), (g, 2t + 1), (g + 8, 2t),
// (g + 8, 2t + 1).

// Q4_K: a slice is one 144-byte block; group j = sub-block j. The code bytes
// of a lane's positions in chunk c (sub-blocks 2c, 2c+1) are qs[32c + 4t ..]
// and qs[32c + 16 + 4t ..]: low nibbles sub-block 2c, high nibbles 2c + 1.
struct Q4KT {
    static constexpr int QK = 256;
    static constexpr int BLOCK_BYTES = 144;
    static constexpr int SLACK = 0;

    __device__ __forceinline__ static void slice(uint32_t ra, uint32_t rb, int ks, int, int t,
                                                 const uint32_t (&xh)[8][4], const uint32_t (&xl)[8][4],
                                                 uint32_t st, float (&y4)[4]) {
        const uint32_t ba = ra + static_cast<uint32_t>(ks) * BLOCK_BYTES;
        const uint32_t bb = rb + static_cast<uint32_t>(ks) * BLOCK_BYTES;
        const uint4 ha = lds128<0>(ba);
        const uint4 hb = lds128<0>(bb);
        const uint32_t sa_lo = ha.y & 0x3f3f3f3fu, ma_lo = ha.z & 0x3f3f3f3fu;
        const uint32_t sa_hi = (ha.w & 0x0f0f0f0fu) | ((ha.y >> 2) & 0x30303030u);
        const uint32_t ma_hi = ((ha.w >> 4) & 0x0f0f0f0fu) | ((ha.z >> 2) & 0x30303030u);
        const uint32_t sb_lo = hb.y & 0x3f3f3f3fu, mb_lo = hb.z & 0x3f3f3f3fu;
        const uint32_t sb_hi = (hb.w & 0x0f0f0f0fu) | ((hb.y >> 2) & 0x30303030u);
        const uint32_t mb_hi = ((hb.w >> 4) & 0x0f0f0f0fu) | ((hb.z >> 2) & 0x30303030u);
        const float dma = f16_hi(ha.x), dmb = f16_hi(hb.x);
#pragma unroll
        for (int c = 0; c < 4; c++) {
            const uint32_t off = 16u + 32u * c + 4u * static_cast<uint32_t>(t);
            const uint32_t wa0 = lds32<0>(ba + off), wa1 = lds32<16>(ba + off);
            const uint32_t wb0 = lds32<0>(bb + off), wb1 = lds32<16>(bb + off);
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int j = 2 * c + h;
                // The 4-bit codes as f16 subnormals, exact: the low nibbles
                // (h = 0) as q * 2^-24, the high nibbles (h = 1) left in place
                // as 16 q * 2^-24; bytes 0 and 2 (even columns) by one mask,
                // bytes 1 and 3 (odd) by a shift and a mask.
                const uint32_t me = h ? 0x00f000f0u : 0x000f000fu;
                float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                mma_half_a(D, wa0 & me, wb0 & me, (wa0 >> 8) & me, (wb0 >> 8) & me, xh[j][0], xh[j][1], xl[j][0],
                           xl[j][1]);
                mma_half_a(D, wa1 & me, wb1 & me, (wa1 >> 8) & me, (wb1 >> 8) & me, xh[j][2], xh[j][3], xl[j][2],
                           xl[j][3]);
                // d * sc_j scaled by 2^24 (2^20 for the high nibbles), exactly
                const float da = f16_lo(ha.x) * (h ? TWO24 / 16.0f : TWO24);
                const float db = f16_lo(hb.x) * (h ? TWO24 / 16.0f : TWO24);
                const uint32_t sel = 0x7440u | static_cast<uint32_t>(j & 3);
                const float dsa = __fmaf_rn(da, __uint_as_float(prmt(j < 4 ? sa_lo : sa_hi, 0x4B000000u, sel)), -da * TWO23);
                const float dna = __fmaf_rn(dma, __uint_as_float(prmt(j < 4 ? ma_lo : ma_hi, 0x4B000000u, sel)), -dma * TWO23);
                const float dsb = __fmaf_rn(db, __uint_as_float(prmt(j < 4 ? sb_lo : sb_hi, 0x4B000000u, sel)), -db * TWO23);
                const float dnb = __fmaf_rn(dmb, __uint_as_float(prmt(j < 4 ? mb_lo : mb_hi, 0x4B000000u, sel)), -dmb * TWO23);
                const float4 s = lds_f4(st + 64u * j);
                fold(y4, D, dsa, dsb, s.x, s.z);
                y4[0] = __fmaf_rn(-dna, s.y, y4[0]);
                y4[1] = __fmaf_rn(-dna, s.w, y4[1]);
                y4[2] = __fmaf_rn(-dnb, s.y, y4[2]);
                y4[3] = __fmaf_rn(-dnb, s.w, y4[3]);
            }
        }
    }
};

// Q6_K: a slice is one 210-byte block (2-byte aligned); group q covers
// weights 32q .. 32q+31 = half H = q/4, quarter qd = q%4, positions l. A
// lane's positions 4t.. and 16 + 4t.. take their low 4 bits from ql[64H +
// 32(qd%2) + l] (high nibbles for qd >= 2) and their top 2 bits from bits 2qd
// of qh[32H + l]; the two 16-column halves have scales 2q and 2q + 1.
struct Q6KT {
    static constexpr int QK = 256;
    static constexpr int BLOCK_BYTES = 210;
    static constexpr int SLACK = 16;

    __device__ __forceinline__ static void slice(uint32_t ra, uint32_t rb, int ks, int, int t,
                                                 const uint32_t (&xh)[8][4], const uint32_t (&xl)[8][4],
                                                 uint32_t st, float (&y4)[4]) {
        const uint32_t ba = ra + static_cast<uint32_t>(ks) * BLOCK_BYTES;
        const uint32_t bb = rb + static_cast<uint32_t>(ks) * BLOCK_BYTES;
        const uint32_t bias = 0x64206420u;   // 1024 + 32: the codes become q - 32
        const float da = f16_lo(lds32_a2(ba + 208u)), db = f16_lo(lds32_a2(bb + 208u));
        const uint32_t lt = 4u * static_cast<uint32_t>(t);
#pragma unroll
        for (int H = 0; H < 2; H++) {
            const uint32_t qha0 = lds32_a2(ba + 128u + 32u * H + lt), qha1 = lds32_a2(ba + 144u + 32u * H + lt);
            const uint32_t qhb0 = lds32_a2(bb + 128u + 32u * H + lt), qhb1 = lds32_a2(bb + 144u + 32u * H + lt);
            // scales 8H .. 8H + 7 of both rows
            const uint32_t sca0 = lds32_a2(ba + 192u + 8u * H), sca1 = lds32_a2(ba + 196u + 8u * H);
            const uint32_t scb0 = lds32_a2(bb + 192u + 8u * H), scb1 = lds32_a2(bb + 196u + 8u * H);
#pragma unroll
            for (int p = 0; p < 2; p++) {   // qd % 2
                const uint32_t o = 64u * H + 32u * p + lt;
                const uint32_t qla0 = lds32_a2(ba + o), qla1 = lds32_a2(ba + o + 16u);
                const uint32_t qlb0 = lds32_a2(bb + o), qlb1 = lds32_a2(bb + o + 16u);
#pragma unroll
                for (int hi = 0; hi < 2; hi++) {
                    const int qd = 2 * hi + p;
                    const int q = 4 * H + qd;
                    const int sh = 2 * qd;
                    const uint32_t ka0 = ((hi ? qla0 >> 4 : qla0) & 0x0f0f0f0fu) | (((qha0 >> sh) & 0x03030303u) << 4);
                    const uint32_t ka1 = ((hi ? qla1 >> 4 : qla1) & 0x0f0f0f0fu) | (((qha1 >> sh) & 0x03030303u) << 4);
                    const uint32_t kb0 = ((hi ? qlb0 >> 4 : qlb0) & 0x0f0f0f0fu) | (((qhb0 >> sh) & 0x03030303u) << 4);
                    const uint32_t kb1 = ((hi ? qlb1 >> 4 : qlb1) & 0x0f0f0f0fu) | (((qhb1 >> sh) & 0x03030303u) << 4);
                    float D0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, D1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    mma_half(D0, ka0, kb0, bias, xh[q][0], xh[q][1], xl[q][0], xl[q][1]);
                    mma_half(D1, ka1, kb1, bias, xh[q][2], xh[q][3], xl[q][2], xl[q][3]);
                    // scale bytes 2qd and 2qd + 1 of this half's 8 (sign-extended)
                    const uint32_t wa = qd < 2 ? sca0 : sca1, wb = qd < 2 ? scb0 : scb1;
                    const uint32_t b0 = static_cast<uint32_t>((2 * qd) & 3), b1 = b0 + 1u;
                    const uint32_t s0 = b0 | ((8u | b0) * 0x1110u), s1 = b1 | ((8u | b1) * 0x1110u);
                    const float nda = -da * THREE22, ndb = -db * THREE22;
                    const float ds0a = __fmaf_rn(da, __uint_as_float(prmt(wa, 0u, s0) + 0x4B400000u), nda);
                    const float ds1a = __fmaf_rn(da, __uint_as_float(prmt(wa, 0u, s1) + 0x4B400000u), nda);
                    const float ds0b = __fmaf_rn(db, __uint_as_float(prmt(wb, 0u, s0) + 0x4B400000u), ndb);
                    const float ds1b = __fmaf_rn(db, __uint_as_float(prmt(wb, 0u, s1) + 0x4B400000u), ndb);
                    const float4 s = lds_f4(st + 64u * q);
                    fold(y4, D0, ds0a, ds0b, s.x, s.z);
                    fold(y4, D1, ds1a, ds1b, s.x, s.z);
                }
            }
        }
    }
};

// Q8_0: a slice is 8 consecutive 34-byte blocks (2-byte aligned), one per
// group; a lane's code bytes sit at 2 + 4t and 18 + 4t of its block, as
// int8 made unsigned by flipping the sign bit (bias 1024 + 128).
struct Q8T {
    static constexpr int QK = 32;
    static constexpr int BLOCK_BYTES = 34;
    static constexpr int SLACK = 16;

    __device__ __forceinline__ static void slice(uint32_t ra, uint32_t rb, int ks, int ng, int t,
                                                 const uint32_t (&xh)[8][4], const uint32_t (&xl)[8][4],
                                                 uint32_t st, float (&y4)[4]) {
        const uint32_t bias = 0x64806480u;
        const uint32_t lt = 4u * static_cast<uint32_t>(t);
#pragma unroll
        for (int j = 0; j < TC_GROUPS_PER_SLICE; j++) {
            if (j < ng) {
                const uint32_t off = static_cast<uint32_t>(ks * TC_GROUPS_PER_SLICE + j) * BLOCK_BYTES;
                const uint32_t ba = ra + off, bb = rb + off;
                const float da = f16_lo(lds32_a2(ba)), db = f16_lo(lds32_a2(bb));
                const uint32_t ka0 = lds32_a2(ba + 2u + lt) ^ 0x80808080u, ka1 = lds32_a2(ba + 18u + lt) ^ 0x80808080u;
                const uint32_t kb0 = lds32_a2(bb + 2u + lt) ^ 0x80808080u, kb1 = lds32_a2(bb + 18u + lt) ^ 0x80808080u;
                float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                mma_half(D, ka0, kb0, bias, xh[j][0], xh[j][1], xl[j][0], xl[j][1]);
                mma_half(D, ka1, kb1, bias, xh[j][2], xh[j][3], xl[j][2], xl[j][3]);
                const float4 s = lds_f4(st + 64u * j);
                fold(y4, D, da, db, s.x, s.z);
            }
        }
    }
};

// ------------------------------------------------------------------ kernel

// Copy rows [r0, r0 + nr) of W into the slot at shared address dst (row i at
// dst + i * stride + (its address & 15)), one bulk copy per row, the rows
// spread over the lanes of the calling warp (all 32 lanes call it). The ragged
// bytes of a row whose 16-byte cover would run past the buffer are copied by
// hand before the barrier is armed.
__device__ __forceinline__ void tc_issue_warp(const TParams& p, uint8_t* dst_ptr, uint32_t dst, uint32_t bar, int r0,
                                              int nr, int lane) {
    const uintptr_t lim = reinterpret_cast<uintptr_t>(p.w) + static_cast<uintptr_t>(p.wbytes);
    uint32_t total = 0;
    for (int i = lane; i < nr; i += 32) {
        const uintptr_t gs = reinterpret_cast<uintptr_t>(p.w) + static_cast<uintptr_t>(r0 + i) * p.wpitch + p.woff;
        const uintptr_t ge = gs + p.rowbytes;
        const uintptr_t a0 = gs & ~uintptr_t(15);
        uintptr_t a1 = (ge + 15) & ~uintptr_t(15);
        if (a1 > lim) {
            a1 = ge & ~uintptr_t(15);
            uint8_t* row = dst_ptr + static_cast<uint32_t>(i) * p.stride;
            for (uintptr_t b = (a1 > a0 ? a1 : a0); b < ge; b++) row[b - a0] = *reinterpret_cast<const uint8_t*>(b);
        }
        if (a1 > a0) total += static_cast<uint32_t>(a1 - a0);
    }
    total = __reduce_add_sync(FULL, total);
    __syncwarp();   // hand-copied bytes are ordered before the arrive below
    if (lane == 0) mbar_arrive_expect_tx(bar, total);
    __syncwarp();
    for (int i = lane; i < nr; i += 32) {
        const uintptr_t gs = reinterpret_cast<uintptr_t>(p.w) + static_cast<uintptr_t>(r0 + i) * p.wpitch + p.woff;
        const uintptr_t ge = gs + p.rowbytes;
        const uintptr_t a0 = gs & ~uintptr_t(15);
        uintptr_t a1 = (ge + 15) & ~uintptr_t(15);
        if (a1 > lim) a1 = ge & ~uintptr_t(15);
        if (a1 > a0)
            tma_bulk_g2s(dst + static_cast<uint32_t>(i) * p.stride, reinterpret_cast<const void*>(a0),
                         static_cast<uint32_t>(a1 - a0), bar);
    }
}

template <class F>
__global__ void __launch_bounds__(512, 1) qmm_tc_kernel(const TParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int ks = tid >> 5;   // this warp's slice
    const int g = lane >> 2, t = lane & 3;

    const int part = blockIdx.x;
    const int nrows = p.rq + (part < p.rrem ? 1 : 0);
    const int R0 = part * p.rq + min(part, p.rrem);

    pdl_launch_dependents();
    if (nrows <= 0) return;

    const int npc = (nrows + p.CR - 1) / p.CR;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t ring = sbase + p.off_ring;
    const uint32_t bars = sbase + p.off_bars;
    int* cnt = reinterpret_cast<int*>(smem + p.off_cnt);
    int* done = cnt;
    int* issued = cnt + p.S;
    int* timeout = cnt + p.S + 1;

    // Request piece pc into slot s (a whole warp).
    auto issue = [&](int pc, int s) {
        tc_issue_warp(p, smem + p.off_ring + static_cast<uint32_t>(s) * p.slot_stride,
                      ring + static_cast<uint32_t>(s) * p.slot_stride, bars + 8u * s, R0 + pc * p.CR,
                      min(p.CR, nrows - pc * p.CR), lane);
    };

    if (ks == 0) {
        if (lane == 0) {
            for (int s = 0; s < p.S; s++) {
                mbar_init(bars + 8u * s, 1);
                done[s] = 0;
            }
            fence_mbar_init();
            *timeout = 0;
        }
        __syncwarp();
        const int first = npc < p.S ? npc : p.S;
        for (int pc = 0; pc < first; pc++) issue(pc, pc);
        if (lane == 0) *issued = first;
    }
    if (!p.early_inputs) pdl_dependency_wait();

    // ---- this lane's x fragments: column m = g of the slice's groups
    const int G0 = ks * TC_GROUPS_PER_SLICE;
    const int ng = min(TC_GROUPS_PER_SLICE, p.ngroups - G0);
    uint32_t xh[8][4], xl[8][4];
    float2* stt = reinterpret_cast<float2*>(smem + p.off_st);
#pragma unroll
    for (int j = 0; j < TC_GROUPS_PER_SLICE; j++) {
        float v[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        const bool live = j < ng && g < p.m;
        if (live) {
            const float* src = p.x + static_cast<long long>(g) * p.xstride + 32 * (G0 + j) + 4 * t;
            const float4 u0 = __ldg(reinterpret_cast<const float4*>(src));
            const float4 u1 = __ldg(reinterpret_cast<const float4*>(src + 16));
            v[0] = u0.x; v[1] = u0.y; v[2] = u0.z; v[3] = u0.w;
            v[4] = u1.x; v[5] = u1.y; v[6] = u1.z; v[7] = u1.w;
        }
        float amax = 0.0f, sum = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            amax = fmaxf(amax, fabsf(v[i]));
            sum += v[i];
        }
        amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 2));
        sum += __shfl_xor_sync(FULL, sum, 1);
        sum += __shfl_xor_sync(FULL, sum, 2);
        // power-of-two scale putting the group maximum in [2^14, 2^15)
        int s = 0;
        if (amax > 0.0f) {
            s = 141 - static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu);
            s = s > 126 ? 126 : (s < -126 ? -126 : s);
        }
        const float p2 = __uint_as_float(static_cast<uint32_t>(s + 127) << 23);
        const float inv = __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
#pragma unroll
        for (int i = 0; i < 8; i++) v[i] *= p2;
        // MMA-k order of a half: (4t, 4t+2) then (4t+1, 4t+3)
        const uint32_t h0 = pack_h2(v[0], v[2]), h1 = pack_h2(v[1], v[3]);
        const uint32_t h2 = pack_h2(v[4], v[6]), h3 = pack_h2(v[5], v[7]);
        const float2 f0 = unpack_h2(h0), f1 = unpack_h2(h1), f2 = unpack_h2(h2), f3 = unpack_h2(h3);
        xh[j][0] = h0; xh[j][1] = h1; xh[j][2] = h2; xh[j][3] = h3;
        xl[j][0] = pack_h2(v[0] - f0.x, v[2] - f0.y);
        xl[j][1] = pack_h2(v[1] - f1.x, v[3] - f1.y);
        xl[j][2] = pack_h2(v[4] - f2.x, v[6] - f2.y);
        xl[j][3] = pack_h2(v[5] - f3.x, v[7] - f3.y);
        if (t == 0 && j < ng) stt[(G0 + j) * TC_COLS + g] = live ? make_float2(inv, sum) : make_float2(0.0f, 0.0f);
    }
    __syncthreads();   // statistics complete; barriers initialized

    float* red = reinterpret_cast<float*>(smem + p.off_red);
    const uint32_t st = sbase + p.off_st + static_cast<uint32_t>((G0 * TC_COLS + 2 * t) * 8);
    const uintptr_t wbase = reinterpret_cast<uintptr_t>(p.w);

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
        const int nr = min(p.CR, nrows - pc * p.CR);
        const int rl0 = pc * p.CR;   // CTA-local row of the piece's first row
        const uint32_t slot = ring + static_cast<uint32_t>(s) * p.slot_stride;
        for (int r = 0; r < nr; r += TC_TILE_ROWS) {
            const int ia = r + g, ib = r + g + 8;
            // rows past the piece read the slot's spare rows (results dropped)
            const uint32_t pa =
                static_cast<uint32_t>((wbase + static_cast<uintptr_t>(R0 + rl0 + ia) * p.wpitch + p.woff) & 15u);
            const uint32_t pb =
                static_cast<uint32_t>((wbase + static_cast<uintptr_t>(R0 + rl0 + ib) * p.wpitch + p.woff) & 15u);
            const uint32_t ra = slot + static_cast<uint32_t>(ia) * p.stride + pa;
            const uint32_t rb = slot + static_cast<uint32_t>(ib) * p.stride + pb;
            float y4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            F::slice(ra, rb, ks, ng, t, xh, xl, st, y4);
            // park this slice's sums of columns 2t, 2t + 1
            if (ia < nr) {
                red[((rl0 + ia) * p.KS + ks) * TC_COLS + 2 * t] = y4[0];
                red[((rl0 + ia) * p.KS + ks) * TC_COLS + 2 * t + 1] = y4[1];
            }
            if (ib < nr) {
                red[((rl0 + ib) * p.KS + ks) * TC_COLS + 2 * t] = y4[2];
                red[((rl0 + ib) * p.KS + ks) * TC_COLS + 2 * t + 1] = y4[3];
            }
        }
        __syncwarp();
        if (pc + p.S < npc) {
            // the last warp done with slot s re-fills it with piece pc + S
            int last = 1;
            if (lane == 0 && p.KS > 1) {
                __threadfence_block();
                last = atomicAdd(&done[s], 1) == p.KS - 1;
                if (last) done[s] = 0;
            }
            last = __shfl_sync(FULL, last, 0);
            if (last) {
                fence_proxy_async();
                issue(pc + p.S, s);
                if (lane == 0) atomicMax(issued, pc + p.S + 1);
            }
        }
        if (++s == p.S) {
            s = 0;
            par ^= 1u;
        }
    }

    __syncthreads();
    if (*timeout) {
        if (tid == 0) {
            const int n = *issued;
            for (int pc = n - p.S > 0 ? n - p.S : 0; pc < n; pc++)
                if (!mbar_wait_bounded(bars + 8u * (pc % p.S), static_cast<uint32_t>((pc / p.S) & 1))) break;
        }
        return;
    }
    if (p.early_inputs) pdl_dependency_wait();
    for (int e = tid; e < nrows * p.m; e += blockDim.x) {
        const int r = e / p.m, i = e - (e / p.m) * p.m;
        float v = 0.0f;
        for (int q = 0; q < p.KS; q++) v += red[(r * p.KS + q) * TC_COLS + i];
        float* dst = p.y + static_cast<long long>(i) * p.rows + R0 + r;
        *dst = p.accumulate ? *dst + v : v;
    }
}

// ------------------------------------------------------------------ plan

// Shared-memory stride of one staged row: its bytes plus the 16-byte cover
// (and the format's read slack), rounded to 16 bytes past a multiple of 128.
inline uint32_t tc_row_stride(uint32_t rowbytes, int slack) {
    uint32_t s = static_cast<uint32_t>(round_up(static_cast<long long>(rowbytes) + 16 + slack, 16));
    return s + ((16u + 128u - (s & 127u)) & 127u);
}

// Launch plan for m (1..8) rows of x on a device described by di.
template <class F>
inline int make_tc_plan_for(const DevInfo& di, int rows, int k, int m, const qmv_cfg* cfg, TParams* tp, Plan* pl) {
    if (m < 1 || m > TC_COLS || rows <= 0 || k <= 0 || k % F::QK) return QMV_EINVAL;
    const int ngroups = k / 32;
    const int KS = (ngroups + TC_GROUPS_PER_SLICE - 1) / TC_GROUPS_PER_SLICE;
    if (KS > MAX_WARPS) return QMV_ETOOBIG;
    const long long rowbytes = static_cast<long long>(k / F::QK) * F::BLOCK_BYTES;
    const uint32_t stride = tc_row_stride(static_cast<uint32_t>(rowbytes), F::SLACK);
    const int mode = __atomic_load_n(&weight_prefetch_flag(), __ATOMIC_RELAXED);
    const long long full = di.smem_optin;

    int parts = (cfg && cfg->ctas > 0) ? cfg->ctas : di.nsm;
    if (!(cfg && cfg->ctas > 0)) {
        const long long by_bytes = std::max<long long>(1, static_cast<long long>(rows) * rowbytes / MIN_CTA_BYTES);
        if (by_bytes < parts) parts = static_cast<int>(by_bytes);
    }
    parts = std::max(1, std::min(parts, rows));
    while (true) {
        const int rpc = (rows + parts - 1) / parts;
        int CR = (cfg && cfg->chunk_rows > 0) ? cfg->chunk_rows : TC_TILE_ROWS;
        CR = std::max(1, std::min(CR, rpc));
        const long long cap = round_up(CR, TC_TILE_ROWS);   // rows a slot holds (tiles of 16)
        const long long slot = round_up(cap * stride, 128);
        const int pieces = (rpc + CR - 1) / CR;
        const long long fixed = round_up(8LL * ngroups * TC_COLS, 128) + round_up(4LL * rpc * KS * TC_COLS, 128);
        int S = (cfg && cfg->chunks > 0) ? std::min(cfg->chunks, pieces) : pieces;
        while (S > 0 && fixed + S * slot + 8LL * S + 4LL * (S + 2) > full) S--;
        if (S >= 1 && slot <= 0x7fffffffLL) {
            long long off = 0;
            tp->off_st = 0;
            off = round_up(8LL * ngroups * TC_COLS, 128);
            tp->off_red = static_cast<uint32_t>(off);
            off = round_up(off + 4LL * rpc * KS * TC_COLS, 128);
            tp->off_ring = static_cast<uint32_t>(off);
            off += S * slot;
            tp->off_bars = static_cast<uint32_t>(off);
            off += 8LL * S;
            tp->off_cnt = static_cast<uint32_t>(off);
            off += 4LL * (S + 2);
            pl->smem = static_cast<size_t>(round_up(off, 16));
            pl->T = 32 * KS;
            pl->parts = parts;
            pl->R = 1;
            pl->CL = 1;
            tp->rows = rows;
            tp->k = k;
            tp->m = m;
            tp->xstride = k;
            tp->wpitch = static_cast<uint32_t>(rowbytes);
            tp->woff = 0;
            tp->accumulate = 0;
            tp->ngroups = ngroups;
            tp->rowbytes = static_cast<uint32_t>(rowbytes);
            tp->stride = stride;
            tp->KS = KS;
            tp->CR = CR;
            tp->S = S;
            tp->rq = rows / parts;
            tp->rrem = rows % parts;
            tp->early_inputs = mode >= 2 ? 1 : 0;
            tp->slot_stride = static_cast<uint32_t>(slot);
            return QMV_OK;
        }
        if (cfg && cfg->ctas > 0) return QMV_ETOOBIG;
        if (parts >= rows) return QMV_ETOOBIG;
        parts = std::min(rows, parts * 2);   // fewer rows per CTA, smaller tables
    }
}

template <class F>
inline int launch_tc(const TParams& tp, const Plan& pl, cudaStream_t stream) {
    auto kern = qmm_tc_kernel<F>;
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
    return cuda_rc(cudaLaunchKernelEx(&lc, kern, tp));
}

// Weights per row one launch takes: 16 warps x 256.
constexpr int TC_MAX_K = TC_GROUPS_PER_SLICE * 32 * MAX_WARPS;

// y[m, rows] = x[m, k] W^T on the tensor cores, m >= 1: ceil(m / 8) balanced
// tiles of rows of x; rows longer than TC_MAX_K weights in k-chunks of
// TC_MAX_K, one launch each, the later chunks adding to y in chunk order
// (each launch reads its chunk of W once).
template <class F>
inline int qmm_tc_run(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_cfg* cfg,
                      cudaStream_t s) {
    const int tiles = (m + TC_COLS - 1) / TC_COLS;
    const long long pitch = static_cast<long long>(k / F::QK) * F::BLOCK_BYTES;
    DevInfo di;
    int rc = dev_info(&di, nullptr);
    if (rc) return rc;
    for (int t0 = 0, m0 = 0; t0 < tiles; t0++) {
        const int mt = m / tiles + (t0 < m % tiles ? 1 : 0);
        for (int k0 = 0; k0 < k; k0 += TC_MAX_K) {
            const int kc = std::min(TC_MAX_K, k - k0);
            TParams tp{};
            Plan pl;
            rc = make_tc_plan_for<F>(di, rows, kc, mt, cfg, &tp, &pl);
            if (rc) return rc;
            tp.w = static_cast<const uint8_t*>(w);
            tp.x = x + static_cast<long long>(m0) * k + k0;
            tp.y = y + static_cast<long long>(m0) * rows;
            tp.xstride = k;
            tp.wpitch = static_cast<uint32_t>(pitch);
            tp.woff = static_cast<uint32_t>(static_cast<long long>(k0 / F::QK) * F::BLOCK_BYTES);
            tp.accumulate = k0 > 0 ? 1 : 0;
            tp.wbytes = static_cast<unsigned long long>(rows) * static_cast<unsigned long long>(pitch);
            rc = launch_tc<F>(tp, pl, s);
            if (rc) return rc;
        }
        m0 += mt;
    }
    return QMV_OK;
}

}  // namespace qmv
