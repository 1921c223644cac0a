// qmm_tc.cuh -- the small-M batched product y[m, rows] = x[m, k] W^T on the
// tensor cores (warp-level mma.sync, f16 operands, f32 accumulate), one launch
// per tile of up to 8 rows of x; rows of any length, in k-chunks inside the
// launch.
//
// The product is a skinny dense contraction (m <= 8 columns), so a warp-level
// MMA with register accumulators fits it: the weights' per-32 (Q4_K, Q5_K,
// Q8_0, Q4_0) or per-16 (Q6_K) scales are applied to each group's partial
// product in registers right after its MMAs, which keeps every operand exact:
//  * A (16 weight rows x 16 k): the integer codes, exact in f16: Q4_K's q as
//    the subnormal q * 2^-24 or 16 q * 2^-24 (one mask, or a shift and a
//    mask, per pair; the power of two goes into the row scale), Q5_K's
//    five-bit q likewise as q * 2^-24; Q6_K's q - 32, Q8_0's q and Q4_0's
//    q - 8 made from the code bytes with one byte permute into the f16
//    pattern of 1024 + v and one f16x2 subtraction.
//  * B (16 k x 8 rows of x): x in two f16 parts, hi + lo, after a power-of-two
//    scale per row of x and warp slice (256 weights) that puts the slice's
//    maximum in [2^14, 2^15); hi + lo carries x to about 22 bits, so the MMA
//    pair A*hi + A*lo is the group's integer-code dot at f32 accuracy, and
//    the scale comes off once per tile when the slice's sums are parked.
//  * Per group the accumulator D (16 x 8, four values a lane) is folded into
//    the row sums: y += d*sc * D. Up to 4 rows of x, hi and lo share one MMA
//    (columns 0-3 hi, 4-7 lo; the final sum adds the halves).
//  * The min term of Q4_K and Q5_K, dmin * sum_j m_j S_j with
//    S_j the sum of x over group j, is one more product per tile: A' = the
//    six-bit m_j of the 16 rows, B' = a lane's partial sums of the groups
//    (hi + lo), over a k made of (group, lane) pairs, so that no lane needs
//    another lane's sums.
// The k order inside each 16-column half of a group is permuted identically
// for A and B so that a lane's code bytes are aligned 4-byte runs: MMA
// columns (2t, 2t+1, 2t+8, 2t+9) of lane group t hold positions (4t, 4t+2,
// 4t+1, 4t+3) of the half.
//
// Staging: a CTA owns a run of rows; the pieces it streams are (k-chunk, rows)
// pairs, k-chunk major; every row of a piece is copied by its own bulk TMA
// copy into a slot whose row stride is 16 bytes past a multiple of 128, so
// that the 32 lanes of a warp, reading 8 rows x 4 runs, hit 32 different
// banks. A k-chunk is one slice of 8 groups (256 weights) per warp; a warp
// converts its slice of x when it enters a chunk and keeps the fragments (hi
// and lo, 64 registers) for the chunk's pieces. Rows are processed in tiles of
// 16; slice partials are parked per (row, slice, column), added over the
// chunks, and summed in slice order at the end. Waits are bounded as in
// qmv_kernel.cuh. The planner (make_tc_plan_for) gives independent calls
// half-SM CTAs of at most 8 warps, so that two calls share an SM.
#pragma once

#include "qmv_launch.cuh"

namespace qmv {

struct TParams {
    const uint8_t* w;             // packed rows [rows, k / QK blocks]
    const float* x;               // [m, k], row-major
    float* y;                     // [m, rows]
    unsigned long long wbytes;    // readable bytes from w (tail clipping)
    int rows, k, m;               // m: rows of x, 1..8
    uint32_t wpitch;              // bytes between rows of W
    int ngroups;                  // k / 32
    int KS;                       // warps; a k-chunk is KS slices of 8 groups
    int nchunks;                  // k-chunks (the last one may hold fewer slices)
    uint32_t chunk_bytes;         // bytes of one row's full k-chunk
    uint32_t stride;              // shared-memory row stride (16 mod 128)
    int CR;                       // rows per piece
    int S;                        // ring slots
    int rq, rrem;                 // rows per CTA: rq or rq + 1 (the first rrem CTAs)
    int early_inputs;
    int force_timeout;            // failure-path test: every first wait reports a copy that did not land
    uint32_t slot_stride;         // bytes per slot (rows rounded up to 16)
    uint32_t off_red, off_sums, off_ring, off_bars, off_cnt;
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

__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// 4 bytes at the 2-byte aligned shared address a.
__device__ __forceinline__ uint32_t lds32_a2(uint32_t a) {
    const uint32_t wa = a & ~3u;
    return __funnelshift_r(lds32<0>(wa), lds32<4>(wa), (a & 3u) * 8u);
}

// 4 bytes at the shared address a whose phase a & 3 is ph: 0 (one load), 2
// (two loads and a constant shift) or unknown (-1: lds32_a2). ph is a
// constant once the callers are inlined and their loops unrolled.
__device__ __forceinline__ uint32_t lds32_ph(uint32_t a, int ph) {
    if (ph == 0) return lds32<0>(a);
    if (ph == 2) return __funnelshift_r(lds32<0>(a - 2u), lds32<4>(a - 2u), 16u);
    return lds32_a2(a);
}

// The f16 at the 2-byte aligned shared address a (phase ph as above), as f32.
__device__ __forceinline__ float ldh_ph(uint32_t a, int ph) {
    if (ph == 0) return f16_lo(lds32<0>(a));
    if (ph == 2) return f16_hi(lds32<0>(a - 2u));
    return f16_lo(lds32_a2(a));
}

// The phase (a & 3) that addresses a and b share in every lane of the warp:
// 0, 2, or -1 when they differ.
__device__ __forceinline__ int warp_phase(uint32_t a, uint32_t b) {
    const uint32_t pa = a & 3u, pb = b & 3u;
    if (__all_sync(FULL, pa == 0u && pb == 0u)) return 0;
    if (__all_sync(FULL, pa == 2u && pb == 2u)) return 2;
    return -1;
}

// MMA of one 16-column half with A given directly (rows g, g+8; even, odd
// columns) against hi and lo; packed (P): the lane's one fragment already
// holds hi (columns 0-3) or lo (columns 4-7), one MMA.
template <bool P>
__device__ __forceinline__ void mma_half_a(float (&D)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t bh0, uint32_t bh1, uint32_t bl0, uint32_t bl1) {
    mma16816(D, a0, a1, a2, a3, bh0, bh1);
    if (!P) mma16816(D, a0, a1, a2, a3, bl0, bl1);
}

// The same with A from the code words of rows g and g+8, already shifted /
// masked to one byte per weight, with the f16 bias.
template <bool P>
__device__ __forceinline__ void mma_half(float (&D)[4], uint32_t ka, uint32_t kb, uint32_t bias, uint32_t bh0,
                                         uint32_t bh1, uint32_t bl0, uint32_t bl1) {
    const uint32_t a0 = f16_even(ka, bias), a1 = f16_even(kb, bias);
    const uint32_t a2 = f16_odd(ka, bias), a3 = f16_odd(kb, bias);
    mma_half_a<P>(D, a0, a1, a2, a3, bh0, bh1, bl0, bl1);
}

constexpr float TWO24 = 16777216.0f;

// y4 += scale_row * D (columns 2t, 2t+1 for rows g, g+8).
__device__ __forceinline__ void fold(float (&y4)[4], const float (&D)[4], float sa, float sb) {
    y4[0] = __fmaf_rn(sa, D[0], y4[0]);
    y4[1] = __fmaf_rn(sa, D[1], y4[1]);
    y4[2] = __fmaf_rn(sb, D[2], y4[2]);
    y4[3] = __fmaf_rn(sb, D[3], y4[3]);
}

// A lane's B fragments for its warp's slice (column g of the MMA, scaled): h /
// l = hi / lo parts, [group][4] = MMA0 b0, b1, MMA1 b0, b1. Packed (m <= 4
// rows of x): MMA column g < 4 is hi of row g of x and column g >= 4 lo of row
// g - 4, all in h; l is unused. sh (Q4_K, packed): the lane's partial sums of
// groups (0, 1), (2, 3), (4, 5), (6, 7) over its eight positions each, times
// 1/8, as f16 pairs (hi or lo as h); unpacked, the same pairs (hi, then lo)
// go to the lane's 32 bytes of shared memory instead, to spare registers.
struct XFrag {
    uint32_t h[8][4], l[8][4];
    uint32_t sh[4];
};

// The slice's power-of-two scale from the maximum |x| a lane holds: 2^s puts
// the maximum over the lanes of the row (xor masks given) in [2^14, 2^15);
// returns 2^s, inv receives 2^-s.
__device__ __forceinline__ float tc_scale(float amax, bool partner, float& inv) {
    amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 2));
    if (partner) amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 16));
    int s = 0;
    if (amax > 0.0f) {
        s = 141 - static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu);
        s = s > 126 ? 126 : s;
    }
    inv = __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
    return __uint_as_float(static_cast<uint32_t>(s + 127) << 23);
}

__device__ __forceinline__ float abs_max4(float m, float4 v) {
    return fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
}

// Unpacked fragments (5..8 rows of x): the lane's row of x is row g (zeros
// when !live), groups 0 .. ng - 1 from src = &x[g, 32 G + 4t]; the lane makes
// hi and lo of its 8 values a group. inv receives 2^-s of the slice's scale.
// Q4_K / Q5_K (SUMS): the lane's partial group sums (times 1/8, hi then lo)
// go to its 32 bytes of shared memory at sums.
template <bool SUMS>
__device__ __forceinline__ void tc_load_x_pair(const float* src, bool live, int ng, uint32_t sums, XFrag& xf,
                                               float& inv) {
    // all 64 values first (one round of loads), then the slice maximum
    float4 u[2 * TC_GROUPS_PER_SLICE];
#pragma unroll
    for (int j = 0; j < TC_GROUPS_PER_SLICE; j++) {
        u[2 * j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        u[2 * j + 1] = u[2 * j];
        if (live && j < ng) {
            u[2 * j] = __ldg(reinterpret_cast<const float4*>(src + 32 * j));
            u[2 * j + 1] = __ldg(reinterpret_cast<const float4*>(src + 32 * j + 16));
        }
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 2 * TC_GROUPS_PER_SLICE; i++) amax = abs_max4(amax, u[i]);
    const float p2 = tc_scale(amax, false, inv);
    if (SUMS) {
        // group sums of the lane's eight values (scaled: the power of two
        // commutes with the rounding), before the conversion frees u
        uint32_t sh[4], sl[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float4 a0 = u[4 * i], a1 = u[4 * i + 1], b0 = u[4 * i + 2], b1 = u[4 * i + 3];
            const float a = ((((a0.x + a0.y) + (a0.z + a0.w)) + ((a1.x + a1.y) + (a1.z + a1.w))) * p2) * 0.125f;
            const float b = ((((b0.x + b0.y) + (b0.z + b0.w)) + ((b1.x + b1.y) + (b1.z + b1.w))) * p2) * 0.125f;
            sh[i] = pack_h2(a, b);
            const float2 f = unpack_h2(sh[i]);
            sl[i] = pack_h2(a - f.x, b - f.y);
        }
        sts128(sums, make_uint4(sh[0], sh[1], sh[2], sh[3]));
        sts128(sums + 16u, make_uint4(sl[0], sl[1], sl[2], sl[3]));
    }
#pragma unroll
    for (int j = 0; j < TC_GROUPS_PER_SLICE; j++) {
        const float v[8] = {u[2 * j].x * p2,     u[2 * j].y * p2,     u[2 * j].z * p2,     u[2 * j].w * p2,
                            u[2 * j + 1].x * p2, u[2 * j + 1].y * p2, u[2 * j + 1].z * p2, u[2 * j + 1].w * p2};
        // MMA-k order of a half: (4t, 4t+2) then (4t+1, 4t+3)
        const uint32_t h0 = pack_h2(v[0], v[2]), h1 = pack_h2(v[1], v[3]);
        const uint32_t h2 = pack_h2(v[4], v[6]), h3 = pack_h2(v[5], v[7]);
        const float2 f0 = unpack_h2(h0), f1 = unpack_h2(h1), f2 = unpack_h2(h2), f3 = unpack_h2(h3);
        xf.h[j][0] = h0; xf.h[j][1] = h1; xf.h[j][2] = h2; xf.h[j][3] = h3;
        xf.l[j][0] = pack_h2(v[0] - f0.x, v[2] - f0.y);
        xf.l[j][1] = pack_h2(v[1] - f1.x, v[3] - f1.y);
        xf.l[j][2] = pack_h2(v[4] - f2.x, v[6] - f2.y);
        xf.l[j][3] = pack_h2(v[5] - f3.x, v[7] - f3.y);
    }
}

// Packed fragments (2..4 rows of x): lanes g and g + 4 (lane ^ 16) share row
// g & 3 of x; lane g holds hi (MMA columns 0-3), its partner lo (4-7). Each
// of the two converts half of the row's values, the first 16-column half of
// every group (positions 4t..) in lane g and the second (16 + 4t..) in the
// partner, and they trade the parts the other needs: lane g sends the lo of
// its half and receives the hi of the other. inv receives 2^-s; Q4_K / Q5_K
// (SUMS): xf.sh holds the pair's partial group sums (times 1/8), hi in lane
// g, lo in the partner.
template <bool SUMS>
__device__ __forceinline__ void tc_load_x_split(const float* src, bool live, int ng, bool lo_lane, XFrag& xf,
                                                float& inv) {
    const int off = lo_lane ? 16 : 0;
    float4 u[TC_GROUPS_PER_SLICE];
#pragma unroll
    for (int j = 0; j < TC_GROUPS_PER_SLICE; j++) {
        u[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (live && j < ng) u[j] = __ldg(reinterpret_cast<const float4*>(src + 32 * j + off));
    }
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < TC_GROUPS_PER_SLICE; j++) amax = abs_max4(amax, u[j]);
    const float p2 = tc_scale(amax, true, inv);
    const float neg = lo_lane ? -1.0f : 0.0f;
    if (SUMS) {
        float ps[TC_GROUPS_PER_SLICE];
#pragma unroll
        for (int j = 0; j < TC_GROUPS_PER_SLICE; j++) {
            ps[j] = ((u[j].x + u[j].y) + (u[j].z + u[j].w)) * p2;
            ps[j] += __shfl_xor_sync(FULL, ps[j], 16);   // both halves of the lane pair's positions
        }
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float a = ps[2 * i] * 0.125f, b = ps[2 * i + 1] * 0.125f;
            const float2 f = unpack_h2(pack_h2(a, b));
            xf.sh[i] = pack_h2(__fmaf_rn(f.x, neg, a), __fmaf_rn(f.y, neg, b));
        }
    }
#pragma unroll
    for (int j = 0; j < TC_GROUPS_PER_SLICE; j++) {
        const float4 v = make_float4(u[j].x * p2, u[j].y * p2, u[j].z * p2, u[j].w * p2);
        // MMA-k order of a half: (4t, 4t+2) then (4t+1, 4t+3)
        const uint32_t h0 = pack_h2(v.x, v.z), h1 = pack_h2(v.y, v.w);
        const float2 f0 = unpack_h2(h0), f1 = unpack_h2(h1);
        const uint32_t l0 = pack_h2(v.x - f0.x, v.z - f0.y), l1 = pack_h2(v.y - f1.x, v.w - f1.y);
        const uint32_t r0 = __shfl_xor_sync(FULL, lo_lane ? h0 : l0, 16);
        const uint32_t r1 = __shfl_xor_sync(FULL, lo_lane ? h1 : l1, 16);
        xf.h[j][0] = lo_lane ? r0 : h0;
        xf.h[j][1] = lo_lane ? r1 : h1;
        xf.h[j][2] = lo_lane ? l0 : r0;
        xf.h[j][3] = lo_lane ? l1 : r1;
    }
}

// ------------------------------------------------------- format bodies
//
// slice(): one 16-row tile against the warp's slice of groups. ra / rb:
// shared addresses of rows g and g + 8 of the tile (the first byte of their
// k-chunk); ks: the slice within the chunk; ng: its groups (Q8_0's last slice
// may hold fewer than 8); xf: the lane's fragments; sums (Q4_K unpacked): the
// shared address of the lane's min-term fragments; y4: the row sums of (g,
// 2t), (g, 2t + 1), (g + 8, 2t), (g + 8, 2t + 1) in the slice's scaled units.

// Shared by Q4_K and Q5_K, whose 16-byte block headers are alike: d, dmin
// (f16) and the twelve bytes of six-bit scales and mins.
struct KHead {
    uint32_t s_lo, s_hi, m_lo, m_hi;   // sc / m of sub-blocks 0-3 (lo) and 4-7 (hi), one a byte
    float d, dmin;
    __device__ __forceinline__ explicit KHead(uint4 h)
        : s_lo(h.y & 0x3f3f3f3fu),
          s_hi((h.w & 0x0f0f0f0fu) | ((h.y >> 2) & 0x30303030u)),
          m_lo(h.z & 0x3f3f3f3fu),
          m_hi(((h.w >> 4) & 0x0f0f0f0fu) | ((h.z >> 2) & 0x30303030u)),
          d(f16_lo(h.x)),
          dmin(f16_hi(h.x)) {}
    // D * sc_j exactly (sc_j as the float 2^23 + sc_j), D a scaled d.
    __device__ __forceinline__ float dsc(float D, int j) const {
        const uint32_t sel = 0x7440u | static_cast<uint32_t>(j & 3);
        return __fmaf_rn(D, __uint_as_float(prmt(j < 4 ? s_lo : s_hi, 0x4B000000u, sel)), -D * TWO23);
    }
};

// The min term, y4 -= dmin * sum_j m_j S_j for rows g and g + 8, as one more
// product: A' = the m_j as f16 pairs (groups 0,1 | 2,3 | 4,5 | 6,7), B' = the
// lane's partial group sums (times 1/8; packed in xf.sh, else hi and lo at
// the shared address sums).
template <bool P>
__device__ __forceinline__ void k_min_term(const KHead& a, const KHead& b, const XFrag& xf, uint32_t sums,
                                           float (&y4)[4]) {
    const uint32_t one = 0x64006400u;
    const uint32_t m01a = hsub2(prmt(a.m_lo, 0x64646464u, 0x4140u), one);
    const uint32_t m23a = hsub2(prmt(a.m_lo, 0x64646464u, 0x4342u), one);
    const uint32_t m45a = hsub2(prmt(a.m_hi, 0x64646464u, 0x4140u), one);
    const uint32_t m67a = hsub2(prmt(a.m_hi, 0x64646464u, 0x4342u), one);
    const uint32_t m01b = hsub2(prmt(b.m_lo, 0x64646464u, 0x4140u), one);
    const uint32_t m23b = hsub2(prmt(b.m_lo, 0x64646464u, 0x4342u), one);
    const uint32_t m45b = hsub2(prmt(b.m_hi, 0x64646464u, 0x4140u), one);
    const uint32_t m67b = hsub2(prmt(b.m_hi, 0x64646464u, 0x4342u), one);
    float Dm[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (P) {
        mma16816(Dm, m01a, m01b, m23a, m23b, xf.sh[0], xf.sh[1]);
        mma16816(Dm, m45a, m45b, m67a, m67b, xf.sh[2], xf.sh[3]);
    } else {
        const uint4 sh = lds128<0>(sums), sl = lds128<16>(sums);
        mma16816(Dm, m01a, m01b, m23a, m23b, sh.x, sh.y);
        mma16816(Dm, m01a, m01b, m23a, m23b, sl.x, sl.y);
        mma16816(Dm, m45a, m45b, m67a, m67b, sh.z, sh.w);
        mma16816(Dm, m45a, m45b, m67a, m67b, sl.z, sl.w);
    }
    fold(y4, Dm, -8.0f * a.dmin, -8.0f * b.dmin);
}

// Q4_K: a slice is one 144-byte block; group j = sub-block j. The code bytes
// of a lane's positions in chunk c (sub-blocks 2c, 2c+1) are qs[32c + 4t ..]
// and qs[32c + 16 + 4t ..]: low nibbles sub-block 2c, high nibbles 2c + 1.
struct Q4KT {
    static constexpr int QK = 256;
    static constexpr int BLOCK_BYTES = 144;
    static constexpr int SLACK = 0;
    static constexpr bool SUMS = true;

    template <bool P>
    __device__ __forceinline__ static void slice(uint32_t ra, uint32_t rb, int ks, int, int t, const XFrag& xf,
                                                 uint32_t sums, float (&y4)[4]) {
        const uint32_t ba = ra + static_cast<uint32_t>(ks) * BLOCK_BYTES;
        const uint32_t bb = rb + static_cast<uint32_t>(ks) * BLOCK_BYTES;
        const KHead A(lds128<0>(ba)), B(lds128<0>(bb));
        k_min_term<P>(A, B, xf, sums, y4);   // first: its operands then die
        // d * 2^24 for the low nibbles (q * 2^-24), d * 2^20 for the high ones
        // (16 q * 2^-24), exactly
        const float da0 = A.d * TWO24, da1 = A.d * (TWO24 / 16.0f);
        const float db0 = B.d * TWO24, db1 = B.d * (TWO24 / 16.0f);
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
                mma_half_a<P>(D, wa0 & me, wb0 & me, (wa0 >> 8) & me, (wb0 >> 8) & me, xf.h[j][0], xf.h[j][1],
                              xf.l[j][0], xf.l[j][1]);
                mma_half_a<P>(D, wa1 & me, wb1 & me, (wa1 >> 8) & me, (wb1 >> 8) & me, xf.h[j][2], xf.h[j][3],
                              xf.l[j][2], xf.l[j][3]);
                fold(y4, D, A.dsc(h ? da1 : da0, j), B.dsc(h ? db1 : db0, j));
            }
        }
    }
};

// Q5_K: a slice is one 176-byte block: the Q4_K header, qh[32] at 16 and
// qs[128] at 48. Sub-block j's five-bit code at position l is nibble j % 2 of
// qs[32 (j / 2) + l] plus 16 times bit j of qh[l]; a lane's positions are l =
// 4t.. and 16 + 4t.. as for Q4_K.
struct Q5KT {
    static constexpr int QK = 256;
    static constexpr int BLOCK_BYTES = 176;
    static constexpr int SLACK = 0;
    static constexpr bool SUMS = true;

    // Four code bytes (q <= 31) of sub-block j: nibble j % 2 of w, bit j of
    // qh moved to bit 4 (j is a constant once the loops are unrolled).
    __device__ __forceinline__ static uint32_t codes(uint32_t w, uint32_t qh, int j) {
        const uint32_t nib = (j & 1) ? (w >> 4) & 0x0f0f0f0fu : w & 0x0f0f0f0fu;
        const uint32_t top = (j <= 4 ? qh << (4 - j) : qh >> (j - 4)) & 0x10101010u;
        return nib | top;
    }

    template <bool P>
    __device__ __forceinline__ static void slice(uint32_t ra, uint32_t rb, int ks, int, int t, const XFrag& xf,
                                                 uint32_t sums, float (&y4)[4]) {
        const uint32_t ba = ra + static_cast<uint32_t>(ks) * BLOCK_BYTES;
        const uint32_t bb = rb + static_cast<uint32_t>(ks) * BLOCK_BYTES;
        const KHead A(lds128<0>(ba)), B(lds128<0>(bb));
        k_min_term<P>(A, B, xf, sums, y4);
        const uint32_t lt = 4u * static_cast<uint32_t>(t);
        const uint32_t qha0 = lds32<16>(ba + lt), qha1 = lds32<32>(ba + lt);
        const uint32_t qhb0 = lds32<16>(bb + lt), qhb1 = lds32<32>(bb + lt);
        // d * 2^24: the codes enter as the f16 subnormals q * 2^-24
        const float da = A.d * TWO24, db = B.d * TWO24;
#pragma unroll
        for (int c = 0; c < 4; c++) {
            const uint32_t off = 48u + 32u * c + lt;
            const uint32_t wa0 = lds32<0>(ba + off), wa1 = lds32<16>(ba + off);
            const uint32_t wb0 = lds32<0>(bb + off), wb1 = lds32<16>(bb + off);
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int j = 2 * c + h;
                const uint32_t ca0 = codes(wa0, qha0, j), ca1 = codes(wa1, qha1, j);
                const uint32_t cb0 = codes(wb0, qhb0, j), cb1 = codes(wb1, qhb1, j);
                // bytes 0 and 2 (even columns) by a mask, 1 and 3 by a shift
                // and a mask: f16 subnormals q * 2^-24
                const uint32_t me = 0x00ff00ffu;
                float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                mma_half_a<P>(D, ca0 & me, cb0 & me, (ca0 >> 8) & me, (cb0 >> 8) & me, xf.h[j][0], xf.h[j][1],
                              xf.l[j][0], xf.l[j][1]);
                mma_half_a<P>(D, ca1 & me, cb1 & me, (ca1 >> 8) & me, (cb1 >> 8) & me, xf.h[j][2], xf.h[j][3],
                              xf.l[j][2], xf.l[j][3]);
                fold(y4, D, A.dsc(da, j), B.dsc(db, j));
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
    static constexpr bool SUMS = false;

    // Every field read sits a multiple of 4 bytes into the block, so all of a
    // block's loads share its phase ph (see lds32_ph).
    template <bool P>
    __device__ __forceinline__ static void slice(uint32_t ra, uint32_t rb, int ks, int, int t, const XFrag& xf,
                                                 uint32_t, float (&y4)[4]) {
        const uint32_t ba = ra + static_cast<uint32_t>(ks) * BLOCK_BYTES;
        const uint32_t bb = rb + static_cast<uint32_t>(ks) * BLOCK_BYTES;
        switch (warp_phase(ba, bb)) {
        case 0: body<P>(ba, bb, t, xf, y4, 0); break;
        case 2: body<P>(ba, bb, t, xf, y4, 2); break;
        default: body<P>(ba, bb, t, xf, y4, -1); break;
        }
    }

    template <bool P>
    __device__ __forceinline__ static void body(uint32_t ba, uint32_t bb, int t, const XFrag& xf, float (&y4)[4],
                                                int ph) {
        const uint32_t bias = 0x64206420u;   // 1024 + 32: the codes become q - 32
        const float da = ldh_ph(ba + 208u, ph), db = ldh_ph(bb + 208u, ph);
        const float nda = -da * THREE22, ndb = -db * THREE22;
        const uint32_t lt = 4u * static_cast<uint32_t>(t);
#pragma unroll
        for (int H = 0; H < 2; H++) {
            const uint32_t qha0 = lds32_ph(ba + 128u + 32u * H + lt, ph), qha1 = lds32_ph(ba + 144u + 32u * H + lt, ph);
            const uint32_t qhb0 = lds32_ph(bb + 128u + 32u * H + lt, ph), qhb1 = lds32_ph(bb + 144u + 32u * H + lt, ph);
            // scales 8H .. 8H + 7 of both rows
            const uint32_t sca0 = lds32_ph(ba + 192u + 8u * H, ph), sca1 = lds32_ph(ba + 196u + 8u * H, ph);
            const uint32_t scb0 = lds32_ph(bb + 192u + 8u * H, ph), scb1 = lds32_ph(bb + 196u + 8u * H, ph);
#pragma unroll
            for (int p = 0; p < 2; p++) {   // qd % 2
                const uint32_t o = 64u * H + 32u * p + lt;
                const uint32_t qla0 = lds32_ph(ba + o, ph), qla1 = lds32_ph(ba + o + 16u, ph);
                const uint32_t qlb0 = lds32_ph(bb + o, ph), qlb1 = lds32_ph(bb + o + 16u, ph);
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
                    mma_half<P>(D0, ka0, kb0, bias, xf.h[q][0], xf.h[q][1], xf.l[q][0], xf.l[q][1]);
                    mma_half<P>(D1, ka1, kb1, bias, xf.h[q][2], xf.h[q][3], xf.l[q][2], xf.l[q][3]);
                    // scale bytes 2qd and 2qd + 1 of this half's 8 (sign-extended),
                    // times d exactly: the int8 as the float 1.5 * 2^23 + sc
                    const uint32_t wa = qd < 2 ? sca0 : sca1, wb = qd < 2 ? scb0 : scb1;
                    const uint32_t b0 = static_cast<uint32_t>((2 * qd) & 3), b1 = b0 + 1u;
                    const uint32_t s0 = b0 | ((8u | b0) * 0x1110u), s1 = b1 | ((8u | b1) * 0x1110u);
                    const float ds0a = __fmaf_rn(da, __uint_as_float(prmt(wa, 0u, s0) + 0x4B400000u), nda);
                    const float ds1a = __fmaf_rn(da, __uint_as_float(prmt(wa, 0u, s1) + 0x4B400000u), nda);
                    const float ds0b = __fmaf_rn(db, __uint_as_float(prmt(wb, 0u, s0) + 0x4B400000u), ndb);
                    const float ds1b = __fmaf_rn(db, __uint_as_float(prmt(wb, 0u, s1) + 0x4B400000u), ndb);
                    fold(y4, D0, ds0a, ds0b);
                    fold(y4, D1, ds1a, ds1b);
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
    static constexpr bool SUMS = false;

    // Block j of the slice starts 34 (8 ks + j) bytes into the row: its phase
    // is the row's plus 2j (mod 4); d sits at that phase and the codes at the
    // other one (see lds32_ph).
    template <bool P>
    __device__ __forceinline__ static void slice(uint32_t ra, uint32_t rb, int ks, int ng, int t, const XFrag& xf,
                                                 uint32_t, float (&y4)[4]) {
        switch (warp_phase(ra, rb)) {
        case 0: body<P>(ra, rb, ks, ng, t, xf, y4, 0); break;
        case 2: body<P>(ra, rb, ks, ng, t, xf, y4, 2); break;
        default: body<P>(ra, rb, ks, ng, t, xf, y4, -1); break;
        }
    }

    template <bool P>
    __device__ __forceinline__ static void body(uint32_t ra, uint32_t rb, int ks, int ng, int t, const XFrag& xf,
                                                float (&y4)[4], int ph0) {
        const uint32_t bias = 0x64806480u;
        const uint32_t lt = 4u * static_cast<uint32_t>(t);
#pragma unroll
        for (int j = 0; j < TC_GROUPS_PER_SLICE; j++) {
            if (j < ng) {
                const int ph = ph0 < 0 ? -1 : ((ph0 + 2 * j) & 3), pc = ph0 < 0 ? -1 : ((ph + 2) & 3);
                const uint32_t off = static_cast<uint32_t>(ks * TC_GROUPS_PER_SLICE + j) * BLOCK_BYTES;
                const uint32_t ba = ra + off, bb = rb + off;
                const float da = ldh_ph(ba, ph), db = ldh_ph(bb, ph);
                const uint32_t ka0 = lds32_ph(ba + 2u + lt, pc) ^ 0x80808080u, ka1 = lds32_ph(ba + 18u + lt, pc) ^ 0x80808080u;
                const uint32_t kb0 = lds32_ph(bb + 2u + lt, pc) ^ 0x80808080u, kb1 = lds32_ph(bb + 18u + lt, pc) ^ 0x80808080u;
                float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                mma_half<P>(D, ka0, kb0, bias, xf.h[j][0], xf.h[j][1], xf.l[j][0], xf.l[j][1]);
                mma_half<P>(D, ka1, kb1, bias, xf.h[j][2], xf.h[j][3], xf.l[j][2], xf.l[j][3]);
                fold(y4, D, da, db);
            }
        }
    }
};

// Q4_0: a slice is 8 consecutive 18-byte blocks (2-byte aligned), one per
// group: d, then qs[16] whose byte l carries position l in its low nibble and
// position 16 + l in its high nibble; a lane's bytes are qs[4t .. 4t + 3]
// (bias 1024 + 8: the codes become q - 8).
struct Q40T {
    static constexpr int QK = 32;
    static constexpr int BLOCK_BYTES = 18;
    static constexpr int SLACK = 16;
    static constexpr bool SUMS = false;

    // Phases as for Q8_0: block j starts 18 (8 ks + j) bytes into the row.
    template <bool P>
    __device__ __forceinline__ static void slice(uint32_t ra, uint32_t rb, int ks, int ng, int t, const XFrag& xf,
                                                 uint32_t, float (&y4)[4]) {
        switch (warp_phase(ra, rb)) {
        case 0: body<P>(ra, rb, ks, ng, t, xf, y4, 0); break;
        case 2: body<P>(ra, rb, ks, ng, t, xf, y4, 2); break;
        default: body<P>(ra, rb, ks, ng, t, xf, y4, -1); break;
        }
    }

    template <bool P>
    __device__ __forceinline__ static void body(uint32_t ra, uint32_t rb, int ks, int ng, int t, const XFrag& xf,
                                                float (&y4)[4], int ph0) {
        const uint32_t bias = 0x64086408u;
        const uint32_t lt = 4u * static_cast<uint32_t>(t);
#pragma unroll
        for (int j = 0; j < TC_GROUPS_PER_SLICE; j++) {
            if (j < ng) {
                const int ph = ph0 < 0 ? -1 : ((ph0 + 2 * j) & 3), pc = ph0 < 0 ? -1 : ((ph + 2) & 3);
                const uint32_t off = static_cast<uint32_t>(ks * TC_GROUPS_PER_SLICE + j) * BLOCK_BYTES;
                const uint32_t ba = ra + off, bb = rb + off;
                const float da = ldh_ph(ba, ph), db = ldh_ph(bb, ph);
                const uint32_t wa = lds32_ph(ba + 2u + lt, pc), wb = lds32_ph(bb + 2u + lt, pc);
                float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                mma_half<P>(D, wa & 0x0f0f0f0fu, wb & 0x0f0f0f0fu, bias, xf.h[j][0], xf.h[j][1], xf.l[j][0],
                            xf.l[j][1]);
                mma_half<P>(D, (wa >> 4) & 0x0f0f0f0fu, (wb >> 4) & 0x0f0f0f0fu, bias, xf.h[j][2], xf.h[j][3],
                            xf.l[j][2], xf.l[j][3]);
                fold(y4, D, da, db);
            }
        }
    }
};

// ------------------------------------------------------------------ kernel

// Copy rows [r0, r0 + nr) of W, bytes [woff, woff + rowbytes) of each, into
// the slot at shared address dst (row i at dst + i * stride + (its address &
// 15)), one bulk copy per row, the rows spread over the lanes of the calling
// warp (all 32 lanes call it). The ragged bytes of a row whose 16-byte cover
// would run past the buffer are copied by hand before the barrier is armed.
__device__ __forceinline__ void tc_issue_warp(const TParams& p, uint8_t* dst_ptr, uint32_t dst, uint32_t bar, int r0,
                                              int nr, uint32_t woff, uint32_t rowbytes, int lane) {
    const uintptr_t lim = reinterpret_cast<uintptr_t>(p.w) + static_cast<uintptr_t>(p.wbytes);
    // The checking build: row i of the piece is a row of the matrix and of the
    // slot, its 16-byte cover fits the row stride, and it reads only weights.
    // (Both passes below take the same rows.)
    auto row_ok = [&](int i, uintptr_t a0, uintptr_t a1, uintptr_t ge) {
        return in_bounds(static_cast<uint32_t>(i + 1) * p.stride <= p.slot_stride && r0 + i < p.rows &&
                         a1 - a0 <= p.stride && a0 >= (reinterpret_cast<uintptr_t>(p.w) & ~uintptr_t(15)) && ge <= lim);
    };
    uint32_t total = 0;
    for (int i = lane; i < nr; i += 32) {
        const uintptr_t gs = reinterpret_cast<uintptr_t>(p.w) + static_cast<uintptr_t>(r0 + i) * p.wpitch + woff;
        const uintptr_t ge = gs + rowbytes;
        const uintptr_t a0 = gs & ~uintptr_t(15);
        uintptr_t a1 = (ge + 15) & ~uintptr_t(15);
        if (!row_ok(i, a0, a1, ge)) continue;
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
        const uintptr_t gs = reinterpret_cast<uintptr_t>(p.w) + static_cast<uintptr_t>(r0 + i) * p.wpitch + woff;
        const uintptr_t ge = gs + rowbytes;
        const uintptr_t a0 = gs & ~uintptr_t(15);
        uintptr_t a1 = (ge + 15) & ~uintptr_t(15);
        if (!row_ok(i, a0, a1, ge)) continue;
        if (a1 > lim) a1 = ge & ~uintptr_t(15);
        if (a1 > a0)
            tma_bulk_g2s(dst + static_cast<uint32_t>(i) * p.stride, reinterpret_cast<const void*>(a0),
                         static_cast<uint32_t>(a1 - a0), bar);
    }
}

template <class F, bool P>
__global__ void __launch_bounds__(512, 1) qmm_tc_kernel(const TParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int ks = tid >> 5;   // this warp's slice of every k-chunk
    const int g = lane >> 2, t = lane & 3;

    const int part = blockIdx.x;
    const int nrows = p.rq + (part < p.rrem ? 1 : 0);
    const int R0 = part * p.rq + min(part, p.rrem);

    pdl_launch_dependents();
    if (nrows <= 0) return;

    const int npc = (nrows + p.CR - 1) / p.CR;   // row pieces per k-chunk
    const int np = npc * p.nchunks;              // pieces, k-chunk major
    const int cgroups = p.KS * TC_GROUPS_PER_SLICE;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t ring = sbase + p.off_ring;
    const uint32_t bars = sbase + p.off_bars;
    int* cnt = reinterpret_cast<int*>(smem + p.off_cnt);
    int* done = cnt;
    int* issued = cnt + p.S;
    int* timeout = cnt + p.S + 1;

    // Request piece pi into slot s (a whole warp).
    auto issue = [&](int pi, int s) {
        const int c = pi / npc, pc = pi - (pi / npc) * npc;
        const int gc = min(cgroups, p.ngroups - c * cgroups);
        const uint32_t cb = static_cast<uint32_t>(gc * 32 / F::QK) * F::BLOCK_BYTES;
        tc_issue_warp(p, smem + p.off_ring + static_cast<uint32_t>(s) * p.slot_stride,
                      ring + static_cast<uint32_t>(s) * p.slot_stride, bars + 8u * s, R0 + pc * p.CR,
                      min(p.CR, nrows - pc * p.CR), static_cast<uint32_t>(c) * p.chunk_bytes, cb, lane);
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
    }
    __syncthreads();   // barriers initialized (each warp then starts its tiles as soon as its x is ready)
    if (ks == 0) {
        const int first = np < p.S ? np : p.S;
        for (int pi = 0; pi < first; pi++) issue(pi, pi);
        if (lane == 0) *issued = first;
    }
    if (!p.early_inputs) pdl_dependency_wait();

    // this lane's x fragments for k-chunk c: MMA column g of the warp's slice
    // (row xr of x; packed, hi for g < 4 and lo for g >= 4)
    const int xr = P ? (g & 3) : g;
    const uint32_t sums_l = sbase + p.off_sums + static_cast<uint32_t>(tid) * 32u;
    XFrag xf;
    int ng = 0;
    float inv0 = 1.0f, inv1 = 1.0f;   // scale of columns 2t, 2t + 1
    auto load_chunk = [&](int c) {
        const int G = c * cgroups + ks * TC_GROUPS_PER_SLICE;
        ng = max(0, min(TC_GROUPS_PER_SLICE, p.ngroups - G));
        const bool live = xr < p.m && ng > 0;
        float inv;
        const float* src = p.x + static_cast<long long>(xr) * p.k + 32 * G + 4 * t;
        if constexpr (P)
            tc_load_x_split<F::SUMS>(src, live, ng, g >= 4, xf, inv);
        else
            tc_load_x_pair<F::SUMS>(src, live, ng, sums_l, xf, inv);
        inv0 = __shfl_sync(FULL, inv, 8 * t);
        inv1 = __shfl_sync(FULL, inv, 8 * t + 4);
    };
    load_chunk(0);

    float* red = reinterpret_cast<float*>(smem + p.off_red);
    const uint32_t wbase32 = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(p.w));

    int s = 0;
    uint32_t par = 0;
    for (int pi = 0; pi < np; pi++) {
        const int c = pi / npc, pc = pi - (pi / npc) * npc;
        if (pc == 0 && c > 0) load_chunk(c);
        const bool landed = !p.force_timeout && __all_sync(FULL, mbar_wait_bounded(bars + 8u * s, par));
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
        // low bits of the global address of the piece's first row chunk
        const uint32_t pbase = wbase32 + static_cast<uint32_t>(c) * p.chunk_bytes +
                               static_cast<uint32_t>(R0 + rl0) * p.wpitch;
        if (ng > 0) {
            for (int r = 0; r < nr; r += TC_TILE_ROWS) {
                const int ia = r + g, ib = r + g + 8;
                // rows past the piece read the slot's spare rows (results dropped)
                const uint32_t pa = (pbase + static_cast<uint32_t>(ia) * p.wpitch) & 15u;
                const uint32_t pb = (pbase + static_cast<uint32_t>(ib) * p.wpitch) & 15u;
                uint32_t ra = slot + static_cast<uint32_t>(ia) * p.stride + pa;
                uint32_t rb = slot + static_cast<uint32_t>(ib) * p.stride + pb;
                // the checking build: both rows lie in the slot
                if (!in_bounds(static_cast<uint32_t>(ia + 1) * p.stride <= p.slot_stride)) ra = slot;
                if (!in_bounds(static_cast<uint32_t>(ib + 1) * p.stride <= p.slot_stride)) rb = slot;
                float y4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                F::template slice<P>(ra, rb, ks, ng, t, xf, sums_l, y4);
                // park this slice's sums of columns 2t, 2t + 1, unscaled
                float2 va = make_float2(y4[0] * inv0, y4[1] * inv1);
                float2 vb = make_float2(y4[2] * inv0, y4[3] * inv1);
                float2* qa = reinterpret_cast<float2*>(red + ((rl0 + ia) * p.KS + ks) * TC_COLS + 2 * t);
                float2* qb = reinterpret_cast<float2*>(red + ((rl0 + ib) * p.KS + ks) * TC_COLS + 2 * t);
                const uint32_t red_cap = p.off_sums / 4u;   // parked sums: floats before B' sums
                if (ia < nr && in_bounds(static_cast<uint32_t>(((rl0 + ia) * p.KS + ks) * TC_COLS + 2 * t + 2) <= red_cap)) {
                    if (c > 0) {
                        const float2 o = *qa;
                        va.x += o.x;
                        va.y += o.y;
                    }
                    *qa = va;
                }
                if (ib < nr && in_bounds(static_cast<uint32_t>(((rl0 + ib) * p.KS + ks) * TC_COLS + 2 * t + 2) <= red_cap)) {
                    if (c > 0) {
                        const float2 o = *qb;
                        vb.x += o.x;
                        vb.y += o.y;
                    }
                    *qb = vb;
                }
            }
        }
        __syncwarp();
        if (pi + p.S < np) {
            // the last warp done with slot s re-fills it with piece pi + S
            int last = 1;
            if (lane == 0 && p.KS > 1) {
                __threadfence_block();
                last = atomicAdd(&done[s], 1) == p.KS - 1;
                if (last) done[s] = 0;
            }
            last = __shfl_sync(FULL, last, 0);
            if (last) {
                fence_proxy_async();
                issue(pi + p.S, s);
                if (lane == 0) atomicMax(issued, pi + p.S + 1);
            }
        }
        if (++s == p.S) {
            s = 0;
            par ^= 1u;
        }
    }

    __syncthreads();
    if (*timeout) {
        // a copy did not land in time: let the copies in flight land (bounded),
        // then mark the CTA's outputs NaN so that no stale y reads as a result
        if (tid == 0) {
            const int n = *issued;
            for (int pi = n - p.S > 0 ? n - p.S : 0; pi < n; pi++)
                if (!mbar_wait_bounded(bars + 8u * (pi % p.S), static_cast<uint32_t>((pi / p.S) & 1))) break;
        }
        pdl_dependency_wait();
        for (int e = tid; e < nrows * p.m; e += blockDim.x) {
            const int r = e / p.m, i = e - (e / p.m) * p.m;
            if (in_bounds(R0 + r < p.rows && i < TC_COLS))
                p.y[static_cast<long long>(i) * p.rows + R0 + r] = __int_as_float(0x7fc00000);
        }
        return;
    }
    if (p.early_inputs) pdl_dependency_wait();
    for (int e = tid; e < nrows * p.m; e += blockDim.x) {
        const int r = e / p.m, i = e - (e / p.m) * p.m;
        if (!in_bounds(R0 + r < p.rows && i < TC_COLS &&
                       static_cast<uint32_t>((r * p.KS + p.KS - 1) * TC_COLS + (P ? i + 4 : i) + 1) <= p.off_sums / 4u))
            continue;
        float v = 0.0f;
        for (int q = 0; q < p.KS; q++) {
            v += red[(r * p.KS + q) * TC_COLS + i];
            if (P) v += red[(r * p.KS + q) * TC_COLS + i + 4];
        }
        p.y[static_cast<long long>(i) * p.rows + R0 + r] = v;
    }
}

// ------------------------------------------------------------------ plan

// Shared-memory stride of one staged row: its bytes plus the 16-byte cover
// (and the format's read slack), rounded to 16 bytes past a multiple of 128.
inline uint32_t tc_row_stride(uint32_t rowbytes, int slack) {
    uint32_t s = static_cast<uint32_t>(round_up(static_cast<long long>(rowbytes) + 16 + slack, 16));
    return s + ((16u + 128u - (s & 127u)) & 127u);
}

// Launch plan for m (1..8) rows of x on a device described by di, in at most
// smem_cap bytes of shared memory a CTA. The k-slices of a row (8 groups
// each) are dealt into the fewest k-chunks of at most MAX_WARPS slices
// (cfg->warps, when given, lowers that bound), balanced; a chunk's slices are
// the CTA's warps.
template <class F>
inline int make_tc_plan_core(const DevInfo& di, int rows, int k, int m, const qmv_opts* cfg, long long smem_cap,
                             TParams* tp, Plan* pl) {
    if (m < 1 || m > TC_COLS || rows <= 0 || k <= 0 || k % F::QK) return QMV_EINVAL;
    const int ngroups = k / 32;
    const int NS = (ngroups + TC_GROUPS_PER_SLICE - 1) / TC_GROUPS_PER_SLICE;
    const int kmax = (cfg && cfg->warps > 0) ? std::min(cfg->warps, MAX_WARPS) : MAX_WARPS;
    const int nchunks = (NS + kmax - 1) / kmax;
    const int KS = (NS + nchunks - 1) / nchunks;
    const long long rowbytes = static_cast<long long>(k / F::QK) * F::BLOCK_BYTES;
    const long long chunk_bytes = static_cast<long long>(KS * TC_GROUPS_PER_SLICE * 32 / F::QK) * F::BLOCK_BYTES;
    if (rowbytes > 0x7fffffffLL) return QMV_ETOOBIG;
    const uint32_t stride = tc_row_stride(static_cast<uint32_t>(std::min(chunk_bytes, rowbytes)), F::SLACK);
    const int mode = overlap_of(cfg);
    const long long full = std::min<long long>(smem_cap, di.smem_optin);

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
        const long long pieces = static_cast<long long>((rpc + CR - 1) / CR) * nchunks;
        const long long sums = F::SUMS ? 32LL * 32 * KS : 0;   // 32 bytes a thread
        const long long fixed = round_up(4LL * rpc * KS * TC_COLS, 128) + sums;
        long long S = (cfg && cfg->chunks > 0) ? std::min<long long>(cfg->chunks, pieces) : pieces;
        while (S > 0 && fixed + S * slot + 8LL * S + 4LL * (S + 2) > full) S--;
        if (S >= 1 && slot <= 0x7fffffffLL) {
            long long off = 0;
            tp->off_red = 0;
            off = round_up(4LL * rpc * KS * TC_COLS, 128);
            tp->off_sums = static_cast<uint32_t>(off);
            off += sums;
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
            tp->wpitch = static_cast<uint32_t>(rowbytes);
            tp->ngroups = ngroups;
            tp->KS = KS;
            tp->nchunks = nchunks;
            tp->chunk_bytes = static_cast<uint32_t>(std::min(chunk_bytes, rowbytes));
            tp->stride = stride;
            tp->CR = CR;
            tp->S = static_cast<int>(S);
            tp->rq = rows / parts;
            tp->rrem = rows % parts;
            tp->early_inputs = mode >= QMV_OVERLAP_INDEPENDENT ? 1 : 0;
            pl->overlap = mode;
            tp->slot_stride = static_cast<uint32_t>(slot);
#ifdef QMV_BOUNDS_CHECK_PLANT
            // A planted fault for the checking build's own test: slots holding
            // half the rows the plan needs (the checks skip the rows past it
            // and read the slot's first row in their place).
            tp->slot_stride = static_cast<uint32_t>(slot / 2) & ~15u;
#endif
            return QMV_OK;
        }
        if (cfg && cfg->ctas > 0) return QMV_ETOOBIG;
        if (parts >= rows) return QMV_ETOOBIG;
        parts = std::min(rows, parts * 2);   // fewer rows per CTA, smaller tables
    }
}

// Warps a CTA of independent calls takes at most: 256 threads of 128
// registers fill half an SM's register file.
constexpr int TC_WARPS_HALF_SM = 8;
// Rows of a ring piece in the streaming plan of independent calls.
constexpr int TC_RING_ROWS = 32;

// The plan used. Independent calls (QMV_OVERLAP_INDEPENDENT) take
// CTAs of at most TC_WARPS_HALF_SM warps in at most half an SM's shared
// memory, so that two calls' CTAs share an SM, one converting its x while
// the other runs its tiles (measured on GB300, us a call: Q4_K 4096 x 4096
// m = 8 6.84 -> 5.97, m = 4 6.47 -> 5.51; Q6_K 4096 x 14336 m = 4 25.1 ->
// 21.6; Q8_0 14336 x 4096 m = 8 19.1 -> 18.2). Other modes, forced warps, and
// shapes whose plan does not fit use whole CTAs.
template <class F>
inline int make_tc_plan_for(const DevInfo& di, int rows, int k, int m, const qmv_opts* cfg, TParams* tp, Plan* pl) {
    const bool forced = cfg && (cfg->ctas > 0 || cfg->chunk_rows > 0 || cfg->chunks > 0 || cfg->warps > 0);
    if (overlap_of(cfg) == QMV_OVERLAP_INDEPENDENT && !forced && rows >= 2 * TC_RING_ROWS * (di.nsm / 4)) {
        // Independent calls of rows that fill a quarter of the SM count with
        // at least two ring pieces each: that many CTAs of at most
        // TC_WARPS_HALF_SM warps, streaming 32-row pieces through two ring
        // slots in half an SM (the matvec's plan for independent calls).
        // Measured on GB300, Q4_K 4096 x 4096, us a call: m = 2 5.04 -> 3.43,
        // m = 8 5.89 -> 4.06 (Q6_K 4096 x 14336, m = 4, seven k-chunks of
        // 8 slices: no gain, so rows of more than two k-chunks keep the plan
        // below).
        qmv_opts c = *cfg;
        c.ctas = di.nsm / 4;
        c.warps = TC_WARPS_HALF_SM;
        c.chunk_rows = TC_RING_ROWS;
        c.chunks = 2;
        const long long half = (di.smem_sm - 2LL * di.smem_reserved) / 2;
        TParams t2 = *tp;
        Plan p2;
        if (!make_tc_plan_core<F>(di, rows, k, m, &c, half, &t2, &p2) && t2.nchunks <= 2 && t2.S == 2 &&
            static_cast<long long>(p2.smem) <= half) {
            *tp = t2;
            *pl = p2;
            return QMV_OK;
        }
    }
    if (overlap_of(cfg) == QMV_OVERLAP_INDEPENDENT && !(cfg && cfg->warps > 0)) {
        qmv_opts c = *cfg;
        c.warps = TC_WARPS_HALF_SM;
        const long long half = (di.smem_sm - 2LL * di.smem_reserved) / 2;
        TParams t2 = *tp;
        Plan p2;
        if (!make_tc_plan_core<F>(di, rows, k, m, &c, half, &t2, &p2)) {
            *tp = t2;
            *pl = p2;
            return QMV_OK;
        }
    }
    return make_tc_plan_core<F>(di, rows, k, m, cfg, di.smem_optin, tp, pl);
}

template <class F, bool P>
inline int launch_tc_kernel(const TParams& tp, const Plan& pl, cudaStream_t stream) {
    auto kern = qmm_tc_kernel<F, P>;
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
    if (pl.overlap != QMV_OVERLAP_NONE) {
        at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[na].val.programmaticStreamSerializationAllowed = 1;
        na++;
    }
    lc.attrs = at;
    lc.numAttrs = na;
    return cuda_rc(cudaLaunchKernelEx(&lc, kern, tp));
}

// Up to 4 rows of x take the packed kernel (hi and lo in the two halves of
// the MMA's 8 columns: half the MMAs).
template <class F>
inline int launch_tc(const TParams& tp, const Plan& pl, cudaStream_t stream) {
    return tp.m <= TC_COLS / 2 ? launch_tc_kernel<F, true>(tp, pl, stream) : launch_tc_kernel<F, false>(tp, pl, stream);
}

// y[m, rows] = x[m, k] W^T on the tensor cores, m >= 1: ceil(m / 8) balanced
// tiles of rows of x, one launch each (each launch reads W once).
template <class F>
inline int qmm_tc_run(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg,
                      cudaStream_t s, int force_timeout = 0) {
    const int tiles = (m + TC_COLS - 1) / TC_COLS;
    DevInfo di;
    int rc = dev_info(&di, nullptr);
    if (rc) return rc;
    for (int t0 = 0, m0 = 0; t0 < tiles; t0++) {
        const int mt = m / tiles + (t0 < m % tiles ? 1 : 0);
        TParams tp{};
        Plan pl;
        rc = make_tc_plan_for<F>(di, rows, k, mt, cfg, &tp, &pl);
        if (rc) return rc;
        tp.w = static_cast<const uint8_t*>(w);
        tp.x = x + static_cast<long long>(m0) * k;
        tp.y = y + static_cast<long long>(m0) * rows;
        tp.wbytes = static_cast<unsigned long long>(rows) * tp.wpitch;
        tp.force_timeout = force_timeout;
        rc = launch_tc<F>(tp, pl, s);
        if (rc) return rc;
        m0 += mt;
    }
    return QMV_OK;
}

}  // namespace qmv
