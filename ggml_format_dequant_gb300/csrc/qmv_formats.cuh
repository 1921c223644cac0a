// qmv_formats.cuh -- in-register decode of one "unit" of a packed GGML block
// against the activation, for Q4_K, Q5_K, Q6_K, Q8_0 and Q4_0.
//
// A unit is the part of a row one lane owns for every row it processes:
//   Q4_K, Q5_K: one 64-weight chunk of a 256-weight super-block (4 per block)
//   Q6_K: one (half, 16-position) slice of a block, 64 weights (4 per block)
//   Q8_0, f32 x: one 32-weight block;  Q8_0, q8 x (dp4a): four blocks
//   Q4_0: one 32-weight block
// The lane keeps the activation for its unit in registers (as integer limbs or
// int8 codes) and, per row, reads the unit's packed bytes from the staged
// rows in shared memory (by 32-bit address), unpacks the codes into byte lanes
// and forms integer dot products with dp4a, then applies the block's scales
// once per scale group.
//
// Block layouts (hanzo-ml src/vulkan_backend.rs): Q4_K = d, dmin (f16), 12 bytes
// of packed 6-bit scales/mins, 128 bytes of 4-bit codes (quantize_q4k,
// quantize_q4k_split); Q6_K = ql[128], qh[64], int8 scales[16], d (f16)
// (quantize_q6k); Q8_0 = d (f16) + 32 int8 (quantize_q8_blocks); Q5_K = d,
// dmin (f16), 12 scale bytes, qh[32], qs[128] (quantize_q5k); Q4_0 = d (f16)
// + 16 bytes of 4-bit codes (matvec_q4_0_gpu). The bit mapping inside the
// blocks is GGML's layout.
//
// Every format states SLICE_BLOCKS (blocks of a row covered by one warp's 32
// units) and SLACK (bytes its loads may read past the end of a row).
#pragma once

#include <type_traits>

#include "qmv_device.cuh"

namespace qmv {

// Signed byte `sel` (selector with sign replication) of w, as an int.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// ====================================================================== Q4_K
//
// Chunk c (0..3) of a super-block covers weights 64c .. 64c+63: qs bytes
// 32c .. 32c+31, whose low nibbles are sub-block 2c (weights 64c + l) and high
// nibbles sub-block 2c+1 (weights 64c + 32 + l). Weight i of sub-block j is
// d*sc_j*q_i - dmin*m_j, so the chunk contributes
//     d*sc_2c * sum(q*x) - dmin*m_2c * sum(x)  +  (same for 2c+1).
struct Q4K {
    static constexpr int QK = 256;
    static constexpr int BLOCK_BYTES = 144;
    static constexpr int SLICE_BLOCKS = 8;    // 32 units (1152 bytes)
    static constexpr int SLACK = 0;
    static constexpr bool LIMBS = true;
    static constexpr int DEFAULT_UNROLL = 2;

    __host__ __device__ static int units(int nb) { return 4 * nb; }
    // Unit u of a slice: byte offset of its block in the slice, first weight.
    __device__ __forceinline__ static uint32_t unit_byte(int u) { return static_cast<uint32_t>(u >> 2) * BLOCK_BYTES; }
    __device__ __forceinline__ static int unit_elem(int u) { return (u >> 2) * QK + 64 * (u & 3); }

    struct X {
        uint32_t a[16], b[16], c[16];   // limbs of the chunk's 64 activations
        float xs0, xs1;                 // 2^-s of the two 32-groups
        float nxsum0, nxsum1;           // minus the activation sums of the two sub-blocks
    };
    struct L {
        uint32_t qoff;   // byte offset of the chunk's codes in the block: 16 + 32c
        uint32_t sel;    // prmt selector giving 0x4B0000vv for scale byte 2(c & 1)
        bool hic;        // c >= 2: scales and mins of sub-blocks 4..7
    };

    __device__ __forceinline__ static L lane_consts(int u, int /*nb*/, int /*ug*/) {
        const int c = u & 3;
        L l;
        l.qoff = 16u + 32u * static_cast<uint32_t>(c);
        l.sel = 0x7440u | static_cast<uint32_t>(2 * (c & 1));
        l.hic = c >= 2;
        return l;
    }

    // e0 = index of the chunk's first weight in the row.
    __device__ __forceinline__ static void load_x(X& x, const uint8_t* smem, const LimbTables& T, int e0) {
#pragma unroll
        for (int v = 0; v < 4; v++) {
            const uint32_t o = limb_chunk(static_cast<uint32_t>(e0 >> 4) + v) << 4;
            const uint4 a = *reinterpret_cast<const uint4*>(smem + T.la + o);
            const uint4 b = *reinterpret_cast<const uint4*>(smem + T.lb + o);
            const uint4 c = *reinterpret_cast<const uint4*>(smem + T.lc + o);
            x.a[4 * v] = a.x; x.a[4 * v + 1] = a.y; x.a[4 * v + 2] = a.z; x.a[4 * v + 3] = a.w;
            x.b[4 * v] = b.x; x.b[4 * v + 1] = b.y; x.b[4 * v + 2] = b.z; x.b[4 * v + 3] = b.w;
            x.c[4 * v] = c.x; x.c[4 * v + 1] = c.y; x.c[4 * v + 2] = c.z; x.c[4 * v + 3] = c.w;
        }
        const float* xs = reinterpret_cast<const float*>(smem + T.xs);
        const float* xsum16 = reinterpret_cast<const float*>(smem + T.xsum16);
        x.xs0 = xs[e0 >> 5];
        x.xs1 = xs[(e0 >> 5) + 1];
        x.nxsum0 = -(xsum16[e0 >> 4] + xsum16[(e0 >> 4) + 1]);
        x.nxsum1 = -(xsum16[(e0 >> 4) + 2] + xsum16[(e0 >> 4) + 3]);
    }

    // a: shared address of the super-block (16-byte aligned).
    __device__ __forceinline__ static float dot(uint32_t a, const L& l, const X& x, float r) {
        const uint4 h = lds128<0>(a);
        const uint32_t aq = a + l.qoff;
        const uint4 qa = lds128<0>(aq);
        const uint4 qb = lds128<16>(aq);
        const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        int a0 = 0, b0 = 0, c0 = 0, a1 = 0, b1 = 0, c1 = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t lo = q[i] & 0x0f0f0f0fu;
            const uint32_t hi = q[i] & 0xf0f0f0f0u;   // 16 * the high nibbles
            a0 = dp4a_us(lo, x.a[i], a0);
            b0 = dp4a_us(lo, x.b[i], b0);
            c0 = dp4a_us(lo, x.c[i], c0);
            a1 = dp4a_us(hi, x.a[8 + i], a1);
            b1 = dp4a_us(hi, x.b[8 + i], b1);
            c1 = dp4a_us(hi, x.c[8 + i], c1);
        }
        // Exact sums q*X, |.| <= 32 * 15 * 2^21 < 2^31 per sub-block. The high
        // nibbles' limb sums carry a factor 16 (a multiple of 16 each, so the
        // shift of c1 is exact).
        const int s0 = a0 * 65536 + b0 * 256 + c0;
        const int s1 = a1 * 4096 + b1 * 16 + (c1 >> 4);
        // The 6-bit scales and mins of sub-blocks 0..3 and 4..7 as byte lanes.
        const uint32_t sc_lo = h.y & 0x3f3f3f3fu;
        const uint32_t m_lo = h.z & 0x3f3f3f3fu;
        const uint32_t sc_hi = (h.w & 0x0f0f0f0fu) | ((h.y >> 2) & 0x30303030u);
        const uint32_t m_hi = ((h.w >> 4) & 0x0f0f0f0fu) | ((h.z >> 2) & 0x30303030u);
        const uint32_t SC = l.hic ? sc_hi : sc_lo;
        const uint32_t M = l.hic ? m_hi : m_lo;
        return scale_pairs(h.x, SC, M, l.sel, __int2float_rn(s0) * x.xs0, __int2float_rn(s1) * x.xs1, x.nxsum0,
                           x.nxsum1, r);
    }

    // r + d*sc_0*t0 - dmin*m_0*S0 + d*sc_1*t1 - dmin*m_1*S1 for the chunk's two
    // sub-blocks, (d, dmin) the block's f16 pair in dd, the 6-bit scales and
    // mins as byte lanes of SC and M (byte sel & 3 and the next one), S_j the
    // activation sums (given negated). The scale and min of a sub-block form
    // one f32 pair: one packed fma gives (d*sc_j, dmin*m_j) exactly (through
    // the exponent field, see TWO23), and one more adds d*sc_j*t_j and
    // -dmin*m_j*S_j into the pair (r, 0).
    __device__ __forceinline__ static float scale_pairs(uint32_t dd, uint32_t SC, uint32_t M, uint32_t sel, float t0,
                                                        float t1, float ns0, float ns1, float r) {
        const float2 d2 = __half22float2(*reinterpret_cast<const __half2*>(&dd));   // (d, dmin)
        const float2 n2 = __fmul2_rn(d2, make_float2(-TWO23, -TWO23));
        const float2 g0 = __ffma2_rn(d2, make_float2(__uint_as_float(prmt(SC, 0x4B000000u, sel)),
                                                     __uint_as_float(prmt(M, 0x4B000000u, sel))), n2);
        const float2 g1 = __ffma2_rn(d2, make_float2(__uint_as_float(prmt(SC, 0x4B000000u, sel + 1)),
                                                     __uint_as_float(prmt(M, 0x4B000000u, sel + 1))), n2);
        float2 acc = __ffma2_rn(g0, make_float2(t0, ns0), make_float2(r, 0.0f));
        acc = __ffma2_rn(g1, make_float2(t1, ns1), acc);
        return acc.x + acc.y;
    }
};

// ============================================================ Q4_K, q8 activation
//
// The dp4a path of Q4_K (hanzo-ml src/vulkan_backend.rs, the dense
// `matvec_q4k_dp4a_blk` decode): the activation is int8 codes with one f32
// scale xs per 32 values (quantize_act_q8). A unit is one 64-weight chunk as in
// Q4K; its two sub-blocks' integer dots with the codes give
//     xs_j * (d*sc_j * dot_j - dmin*m_j * sumq_j)
// with sumq_j the sum of the sub-block's activation codes, which the lane forms
// once from its codes (no separate sum input is needed).
struct Q4D {
    static constexpr int QK = 256;
    static constexpr int BLOCK_BYTES = 144;
    static constexpr int SLICE_BLOCKS = 8;    // 32 units (1152 bytes)
    static constexpr int SLACK = 0;
    static constexpr bool LIMBS = false;
    static constexpr int DEFAULT_UNROLL = 2;
    static constexpr int DOTS_PER_UNIT = 2;   // 32-weight sub-blocks per unit
    static constexpr int DOT_WEIGHTS = 32;    // weights per exported dot
    __device__ __forceinline__ static int dot_base(int ug) { return DOTS_PER_UNIT * ug; }

    __host__ __device__ static int units(int nb) { return 4 * nb; }
    __device__ __forceinline__ static uint32_t unit_byte(int u) { return static_cast<uint32_t>(u >> 2) * BLOCK_BYTES; }
    __device__ __forceinline__ static int unit_elem(int u) { return (u >> 2) * QK + 64 * (u & 3); }

    struct X {
        uint32_t q[16];        // codes of the chunk's 64 activations (sub-block 2c, then 2c+1)
        float xs0, xs1;        // their scales
        float xm0, xm1;        // xs_j * (sum of the sub-block's codes)
    };
    using L = Q4K::L;
    __device__ __forceinline__ static L lane_consts(int u, int nb, int ug) { return Q4K::lane_consts(u, nb, ug); }

    // e0 = index of the chunk's first activation in the row.
    __device__ __forceinline__ static void load_xq(X& x, const L&, const int8_t* __restrict__ xq,
                                                   const float* __restrict__ xs, int e0) {
        const uint4* v = reinterpret_cast<const uint4*>(xq + e0);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint4 t = __ldg(v + i);
            x.q[4 * i] = t.x; x.q[4 * i + 1] = t.y; x.q[4 * i + 2] = t.z; x.q[4 * i + 3] = t.w;
        }
        x.xs0 = __ldg(xs + (e0 >> 5));
        x.xs1 = __ldg(xs + (e0 >> 5) + 1);
        int s0 = 0, s1 = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            s0 = dp4a_ss(0x01010101u, x.q[i], s0);
            s1 = dp4a_ss(0x01010101u, x.q[8 + i], s1);
        }
        x.xm0 = x.xs0 * __int2float_rn(s0);
        x.xm1 = x.xs1 * __int2float_rn(s1);
    }

    // The two sub-blocks' exact dots (the high nibbles enter as 16 q, so the
    // second sum is divided by 16, exactly).
    __device__ __forceinline__ static void subblock_dots(uint32_t a, const L& l, const X& x, int& dot0, int& dot1) {
        const uint32_t aq = a + l.qoff;
        const uint4 qa = lds128<0>(aq);
        const uint4 qb = lds128<16>(aq);
        const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        int s0 = 0, s1 = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            s0 = dp4a_us(q[i] & 0x0f0f0f0fu, x.q[i], s0);
            s1 = dp4a_us(q[i] & 0xf0f0f0f0u, x.q[8 + i], s1);
        }
        dot0 = s0;
        dot1 = s1 >> 4;
    }

    // a: shared address of the super-block (16-byte aligned).
    __device__ __forceinline__ static float dot(uint32_t a, const L& l, const X& x, float r, bool) {
        const uint4 h = lds128<0>(a);
        int dot0, dot1;
        subblock_dots(a, l, x, dot0, dot1);
        const uint32_t sc_lo = h.y & 0x3f3f3f3fu;
        const uint32_t m_lo = h.z & 0x3f3f3f3fu;
        const uint32_t sc_hi = (h.w & 0x0f0f0f0fu) | ((h.y >> 2) & 0x30303030u);
        const uint32_t m_hi = ((h.w >> 4) & 0x0f0f0f0fu) | ((h.z >> 2) & 0x30303030u);
        const uint32_t SC = l.hic ? sc_hi : sc_lo;
        const uint32_t M = l.hic ? m_hi : m_lo;
        const float d = f16_lo(h.x), dmin = f16_hi(h.x);
        const float nd = -d * TWO23, ndm = -dmin * TWO23;
        const float dsc0 = __fmaf_rn(d, __uint_as_float(prmt(SC, 0x4B000000u, l.sel)), nd);
        const float dsc1 = __fmaf_rn(d, __uint_as_float(prmt(SC, 0x4B000000u, l.sel + 1)), nd);
        const float dm0 = __fmaf_rn(dmin, __uint_as_float(prmt(M, 0x4B000000u, l.sel)), ndm);
        const float dm1 = __fmaf_rn(dmin, __uint_as_float(prmt(M, 0x4B000000u, l.sel + 1)), ndm);
        r = __fmaf_rn(dsc0, __int2float_rn(dot0) * x.xs0, r);
        r = __fmaf_rn(-dm0, x.xm0, r);
        r = __fmaf_rn(dsc1, __int2float_rn(dot1) * x.xs1, r);
        r = __fmaf_rn(-dm1, x.xm1, r);
        return r;
    }

    // The exact int32 dots of the unit's two sub-blocks (MODE_BLOCKDOTS).
    __device__ __forceinline__ static void block_dots(uint32_t a, const L& l, const X& x, bool, int32_t* out) {
        int dot0, dot1;
        subblock_dots(a, l, x, dot0, dot1);
        out[0] = dot0;
        out[1] = dot1;
    }
};

// ====================================================================== Q5_K
//
// Laid out as Q4_K with 32 bytes qh between the scales and the codes: chunk c
// covers weights 64c .. 64c+63, the low 4 bits of its codes are the nibbles of
// qs bytes 32c .. 32c+31 (low: sub-block 2c, high: 2c+1), and the fifth bit of
// the code at position l of sub-block j is bit j of qh[l]. So qs word i and
// qh word i (bytes 4i .. 4i+3) carry the same four positions, and rotating the
// qh word left by 4 - 2c brings, in every byte, bit 2c to bit 4 and bit 2c+1
// to bit 5. w = d*sc_j*q - dmin*m_j with q in [0, 31].
struct Q5K {
    static constexpr int QK = 256;
    static constexpr int BLOCK_BYTES = 176;
    static constexpr int SLICE_BLOCKS = 8;    // 32 units (1408 bytes)
    static constexpr int SLACK = 0;
    static constexpr bool LIMBS = true;
    static constexpr int DEFAULT_UNROLL = 2;

    __host__ __device__ static int units(int nb) { return 4 * nb; }
    __device__ __forceinline__ static uint32_t unit_byte(int u) { return static_cast<uint32_t>(u >> 2) * BLOCK_BYTES; }
    __device__ __forceinline__ static int unit_elem(int u) { return (u >> 2) * QK + 64 * (u & 3); }

    using X = Q4K::X;
    struct L {
        uint32_t qoff;   // byte offset of the chunk's codes in the block: 48 + 32c
        uint32_t sel;    // prmt selector of scale byte 2(c & 1), as in Q4K
        uint32_t rot;    // left rotation of the qh words: (4 - 2c) mod 32
        bool hic;        // c >= 2
    };

    __device__ __forceinline__ static L lane_consts(int u, int /*nb*/, int /*ug*/) {
        const int c = u & 3;
        L l;
        l.qoff = 48u + 32u * static_cast<uint32_t>(c);
        l.sel = 0x7440u | static_cast<uint32_t>(2 * (c & 1));
        l.rot = static_cast<uint32_t>(4 - 2 * c) & 31u;
        l.hic = c >= 2;
        return l;
    }

    __device__ __forceinline__ static void load_x(X& x, const uint8_t* smem, const LimbTables& T, int e0) {
        Q4K::load_x(x, smem, T, e0);
    }

    // a: shared address of the super-block (16-byte aligned).
    __device__ __forceinline__ static float dot(uint32_t a, const L& l, const X& x, float r) {
        const uint4 h = lds128<0>(a);
        const uint4 ha = lds128<16>(a);
        const uint4 hb = lds128<32>(a);
        const uint32_t aq = a + l.qoff;
        const uint4 qa = lds128<0>(aq);
        const uint4 qb = lds128<16>(aq);
        const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        const uint32_t qh[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
        int a0 = 0, b0 = 0, c0 = 0, a1 = 0, b1 = 0, c1 = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t t = __funnelshift_l(qh[i], qh[i], l.rot);
            const uint32_t lo = (q[i] & 0x0f0f0f0fu) | (t & 0x10101010u);         // codes of sub-block 2c
            const uint32_t hi = ((q[i] >> 3) & 0x1e1e1e1eu) | (t & 0x20202020u);  // 2 * codes of 2c+1
            a0 = dp4a_us(lo, x.a[i], a0);
            b0 = dp4a_us(lo, x.b[i], b0);
            c0 = dp4a_us(lo, x.c[i], c0);
            a1 = dp4a_us(hi, x.a[8 + i], a1);
            b1 = dp4a_us(hi, x.b[8 + i], b1);
            c1 = dp4a_us(hi, x.c[8 + i], c1);
        }
        // Exact sums q*X, |.| <= 32 * 31 * 2^21 < 2^31 per sub-block; the
        // second carries a factor 2 (even limb sums, so the shift is exact).
        const int s0 = a0 * 65536 + b0 * 256 + c0;
        const int s1 = a1 * 32768 + b1 * 128 + (c1 >> 1);
        const uint32_t sc_lo = h.y & 0x3f3f3f3fu;
        const uint32_t m_lo = h.z & 0x3f3f3f3fu;
        const uint32_t sc_hi = (h.w & 0x0f0f0f0fu) | ((h.y >> 2) & 0x30303030u);
        const uint32_t m_hi = ((h.w >> 4) & 0x0f0f0f0fu) | ((h.z >> 2) & 0x30303030u);
        const uint32_t SC = l.hic ? sc_hi : sc_lo;
        const uint32_t M = l.hic ? m_hi : m_lo;
        return Q4K::scale_pairs(h.x, SC, M, l.sel, __int2float_rn(s0) * x.xs0, __int2float_rn(s1) * x.xs1, x.nxsum0,
                                x.nxsum1, r);
    }
};

// ====================================================================== Q6_K
//
// Unit v = 2*H + hh of a block covers, in half H (weights 128H..128H+127), the
// 16 positions l = 16*hh .. 16*hh+15 of each quarter qd = 0..3: weights
// 128H + 32qd + l. Their low 4 bits are the low (qd = 0, 1) or high (qd = 2, 3)
// nibbles of ql[64H + 32*(qd%2) + l], their top 2 bits are bits 2qd, 2qd+1 of
// qh[32H + l], and all 16 share scale 8H + 2qd + hh. w = d*scale*(q - 32), so
// each quarter contributes d*scale*(sum(q*x) - 32*sum(x)).
struct Q6K {
    static constexpr int QK = 256;
    static constexpr int BLOCK_BYTES = 210;
    static constexpr int SLICE_BLOCKS = 8;    // 32 units (1680 bytes)
    static constexpr int SLACK = 16;
    static constexpr bool LIMBS = true;
    static constexpr int DEFAULT_UNROLL = 2;

    __host__ __device__ static int units(int nb) { return 4 * nb; }
    __device__ __forceinline__ static uint32_t unit_byte(int u) { return static_cast<uint32_t>(u >> 2) * BLOCK_BYTES; }
    __device__ __forceinline__ static int unit_elem(int u) {
        return (u >> 2) * QK + 128 * ((u & 3) >> 1) + 16 * (u & 1);
    }

    struct X {
        uint32_t a[16], b[16], c[16];   // [4*qd + i]: limbs of weights 128H+32qd+16hh+4i..
        float xs[4], xsum[4];
    };
    struct L {
        uint32_t ql_off, qh_off, sc_off;   // byte offsets in the block
        uint32_t sel0, sel1;               // sign-extending selectors of scale bytes hh, 2 + hh
    };

    __device__ __forceinline__ static L lane_consts(int u, int /*nb*/, int /*ug*/) {
        const uint32_t H = static_cast<uint32_t>((u & 3) >> 1), hh = static_cast<uint32_t>(u & 1);
        L l;
        l.ql_off = 64u * H + 16u * hh;
        l.qh_off = 128u + 32u * H + 16u * hh;
        l.sc_off = 192u + 8u * H;
        const uint32_t b0 = hh, b1 = 2u + hh;
        l.sel0 = b0 | ((8u | b0) * 0x1110u);
        l.sel1 = b1 | ((8u | b1) * 0x1110u);
        return l;
    }

    // e0 = index (in the row) of weight 128H + 16hh of the unit's block.
    __device__ __forceinline__ static void load_x(X& x, const uint8_t* smem, const LimbTables& T, int e0) {
        const float* xs = reinterpret_cast<const float*>(smem + T.xs);
        const float* xsum16 = reinterpret_cast<const float*>(smem + T.xsum16);
#pragma unroll
        for (int qd = 0; qd < 4; qd++) {
            const int e = e0 + 32 * qd;
            const uint32_t o = limb_chunk(static_cast<uint32_t>(e >> 4)) << 4;
            const uint4 a = *reinterpret_cast<const uint4*>(smem + T.la + o);
            const uint4 b = *reinterpret_cast<const uint4*>(smem + T.lb + o);
            const uint4 c = *reinterpret_cast<const uint4*>(smem + T.lc + o);
            x.a[4 * qd] = a.x; x.a[4 * qd + 1] = a.y; x.a[4 * qd + 2] = a.z; x.a[4 * qd + 3] = a.w;
            x.b[4 * qd] = b.x; x.b[4 * qd + 1] = b.y; x.b[4 * qd + 2] = b.z; x.b[4 * qd + 3] = b.w;
            x.c[4 * qd] = c.x; x.c[4 * qd + 1] = c.y; x.c[4 * qd + 2] = c.z; x.c[4 * qd + 3] = c.w;
            x.xs[qd] = xs[e >> 5];
            x.xsum[qd] = xsum16[e >> 4];
        }
    }

    // a: shared address of the block (2-byte aligned).
    __device__ __forceinline__ static float dot(uint32_t a, const L& l, const X& x, float r) {
        const uint32_t wa = a & ~3u;
        const uint32_t sh = (a & 3u) * 8u;   // every field offset is a multiple of 4
        const uint32_t w1 = wa + l.ql_off;
        const uint4 qla = lds16_sh<0>(w1, sh);
        const uint4 qlb = lds16_sh<32>(w1, sh);
        const uint4 qhv = lds16_sh<0>(wa + l.qh_off, sh);
        const uint2 scw = lds8_sh<0>(wa + l.sc_off, sh);
        const float d = f16_lo(lds32<208>(wa) >> sh);
        const uint32_t A[4] = {qla.x, qla.y, qla.z, qla.w};
        const uint32_t B[4] = {qlb.x, qlb.y, qlb.z, qlb.w};
        const uint32_t Hq[4] = {qhv.x, qhv.y, qhv.z, qhv.w};
        int sa[4] = {0, 0, 0, 0}, sb[4] = {0, 0, 0, 0}, sc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t w0 = (A[i] & 0x0f0f0f0fu) | ((Hq[i] << 4) & 0x30303030u);
            const uint32_t w1q = (B[i] & 0x0f0f0f0fu) | ((Hq[i] << 2) & 0x30303030u);
            const uint32_t w2 = ((A[i] >> 4) & 0x0f0f0f0fu) | (Hq[i] & 0x30303030u);
            const uint32_t w3 = ((B[i] >> 4) & 0x0f0f0f0fu) | ((Hq[i] >> 2) & 0x30303030u);
            sa[0] = dp4a_us(w0, x.a[i], sa[0]);
            sb[0] = dp4a_us(w0, x.b[i], sb[0]);
            sc[0] = dp4a_us(w0, x.c[i], sc[0]);
            sa[1] = dp4a_us(w1q, x.a[4 + i], sa[1]);
            sb[1] = dp4a_us(w1q, x.b[4 + i], sb[1]);
            sc[1] = dp4a_us(w1q, x.c[4 + i], sc[1]);
            sa[2] = dp4a_us(w2, x.a[8 + i], sa[2]);
            sb[2] = dp4a_us(w2, x.b[8 + i], sb[2]);
            sc[2] = dp4a_us(w2, x.c[8 + i], sc[2]);
            sa[3] = dp4a_us(w3, x.a[12 + i], sa[3]);
            sb[3] = dp4a_us(w3, x.b[12 + i], sb[3]);
            sc[3] = dp4a_us(w3, x.c[12 + i], sc[3]);
        }
        // Quarters (0, 1) and (2, 3) as f32 pairs: scales d*scale (exact,
        // through the exponent field, see THREE22), the scaled integer sums,
        // the -32 fold and the accumulation each one packed instruction a pair.
        const float2 dd = make_float2(d, d);
        const float2 nd = __fmul2_rn(dd, make_float2(-THREE22, -THREE22));
        float2 acc = make_float2(r, 0.0f);
#pragma unroll
        for (int pr = 0; pr < 2; pr++) {
            // |sum q*X| <= 16 * 63 * 2^21 < 2^31 per quarter.
            const int s0 = sa[2 * pr] * 65536 + sb[2 * pr] * 256 + sc[2 * pr];
            const int s1 = sa[2 * pr + 1] * 65536 + sb[2 * pr + 1] * 256 + sc[2 * pr + 1];
            const uint32_t sw = pr == 0 ? scw.x : scw.y;
            const uint32_t sx0 = prmt(sw, 0u, l.sel0);   // the int8 scales, sign-extended
            const uint32_t sx1 = prmt(sw, 0u, l.sel1);
            const float2 ds = __ffma2_rn(dd, make_float2(__uint_as_float(sx0 + 0x4B400000u),
                                                         __uint_as_float(sx1 + 0x4B400000u)), nd);
            const float2 t = __fmul2_rn(make_float2(__int2float_rn(s0), __int2float_rn(s1)),
                                        make_float2(x.xs[2 * pr], x.xs[2 * pr + 1]));
            const float2 u = __ffma2_rn(make_float2(-32.0f, -32.0f), make_float2(x.xsum[2 * pr], x.xsum[2 * pr + 1]), t);
            acc = __ffma2_rn(ds, u, acc);
        }
        return acc.x + acc.y;
    }
};

// ============================================================ Q6_K, q8 activation
//
// The dp4a path of Q6_K (hanzo-ml src/vulkan_backend.rs, the
// `moe_matvec_q6k_dp4a_blk_dn` decode): units as in Q6K, the activation as
// int8 codes with one f32 scale per 32. The 6-bit codes q (unsigned bytes) are
// dotted with the codes exactly, and the -32 is folded against the sum of the
// 16 activation codes of each quarter, formed once at load:
//     d * scale * xs * (sum(q * xq) - 32 * sum(xq))   per 16-weight group.
struct Q6D {
    static constexpr int QK = 256;
    static constexpr int BLOCK_BYTES = 210;
    static constexpr int SLICE_BLOCKS = 8;    // 32 units (1680 bytes)
    static constexpr int SLACK = 16;
    static constexpr bool LIMBS = false;
    static constexpr int DEFAULT_UNROLL = 2;
    static constexpr int DOTS_PER_UNIT = 4;   // 16-weight scale groups per unit
    static constexpr int DOT_WEIGHTS = 16;    // weights per exported dot
    // The unit's groups are 8H + 2qd + hh of its block: the first at
    // 16 * block + 8H + hh, the others every 2.
    __device__ __forceinline__ static int dot_base(int ug) { return 16 * (ug >> 2) + 8 * ((ug & 3) >> 1) + (ug & 1); }

    __host__ __device__ static int units(int nb) { return 4 * nb; }
    __device__ __forceinline__ static uint32_t unit_byte(int u) { return Q6K::unit_byte(u); }
    __device__ __forceinline__ static int unit_elem(int u) { return Q6K::unit_elem(u); }

    struct X {
        uint32_t q[16];   // [4*qd + i]: codes of weights 128H + 32qd + 16hh + 4i ..
        float xs[4];      // scale of quarter qd's 32-group
        int xsum[4];      // sum of quarter qd's 16 codes
    };
    using L = Q6K::L;
    __device__ __forceinline__ static L lane_consts(int u, int nb, int ug) { return Q6K::lane_consts(u, nb, ug); }

    // e0 = index of weight 128H + 16hh of the unit's block, in the row.
    __device__ __forceinline__ static void load_xq(X& x, const L&, const int8_t* __restrict__ xq,
                                                   const float* __restrict__ xs, int e0) {
#pragma unroll
        for (int qd = 0; qd < 4; qd++) {
            const int e = e0 + 32 * qd;
            const uint4 t = __ldg(reinterpret_cast<const uint4*>(xq + e));
            x.q[4 * qd] = t.x; x.q[4 * qd + 1] = t.y; x.q[4 * qd + 2] = t.z; x.q[4 * qd + 3] = t.w;
            x.xs[qd] = __ldg(xs + (e >> 5));
            int sm = 0;
#pragma unroll
            for (int i = 0; i < 4; i++) sm = dp4a_ss(0x01010101u, x.q[4 * qd + i], sm);
            x.xsum[qd] = sm;
        }
    }

    // The four groups' exact dots sum((q - 32) * xq) (|.| <= 16 * 32 * 127).
    __device__ __forceinline__ static void group_dots(uint32_t a, const L& l, const X& x, int (&dot)[4], uint2& scw,
                                                      float& d) {
        const uint32_t wa = a & ~3u;
        const uint32_t sh = (a & 3u) * 8u;
        const uint32_t w1 = wa + l.ql_off;
        const uint4 qla = lds16_sh<0>(w1, sh);
        const uint4 qlb = lds16_sh<32>(w1, sh);
        const uint4 qhv = lds16_sh<0>(wa + l.qh_off, sh);
        scw = lds8_sh<0>(wa + l.sc_off, sh);
        d = f16_lo(lds32<208>(wa) >> sh);
        const uint32_t A[4] = {qla.x, qla.y, qla.z, qla.w};
        const uint32_t B[4] = {qlb.x, qlb.y, qlb.z, qlb.w};
        const uint32_t Hq[4] = {qhv.x, qhv.y, qhv.z, qhv.w};
        int s[4] = {0, 0, 0, 0};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            s[0] = dp4a_us((A[i] & 0x0f0f0f0fu) | ((Hq[i] << 4) & 0x30303030u), x.q[i], s[0]);
            s[1] = dp4a_us((B[i] & 0x0f0f0f0fu) | ((Hq[i] << 2) & 0x30303030u), x.q[4 + i], s[1]);
            s[2] = dp4a_us(((A[i] >> 4) & 0x0f0f0f0fu) | (Hq[i] & 0x30303030u), x.q[8 + i], s[2]);
            s[3] = dp4a_us(((B[i] >> 4) & 0x0f0f0f0fu) | ((Hq[i] >> 2) & 0x30303030u), x.q[12 + i], s[3]);
        }
#pragma unroll
        for (int qd = 0; qd < 4; qd++) dot[qd] = s[qd] - 32 * x.xsum[qd];
    }

    // a: shared address of the block (2-byte aligned).
    __device__ __forceinline__ static float dot(uint32_t a, const L& l, const X& x, float r, bool) {
        int dt[4];
        uint2 scw;
        float d;
        group_dots(a, l, x, dt, scw, d);
        const float nd = -d * THREE22;
#pragma unroll
        for (int qd = 0; qd < 4; qd++) {
            const uint32_t sw = (qd < 2) ? scw.x : scw.y;
            const uint32_t sx = prmt(sw, 0u, (qd & 1) ? l.sel1 : l.sel0);   // the int8 scale, sign-extended
            const float ds = __fmaf_rn(d, __uint_as_float(sx + 0x4B400000u), nd);
            r = __fmaf_rn(ds * x.xs[qd], __int2float_rn(dt[qd]), r);
        }
        return r;
    }

    // The exact int32 dots of the unit's four groups (MODE_BLOCKDOTS), at
    // out[0], out[2], out[4], out[6].
    __device__ __forceinline__ static void block_dots(uint32_t a, const L& l, const X& x, bool, int32_t* out) {
        int dt[4];
        uint2 scw;
        float d;
        group_dots(a, l, x, dt, scw, d);
#pragma unroll
        for (int qd = 0; qd < 4; qd++) out[2 * qd] = dt[qd];
    }
};

// ============================================================ Q8_0, f32 x
struct Q8F {
    static constexpr int QK = 32;
    static constexpr int BLOCK_BYTES = 34;
    static constexpr int SLICE_BLOCKS = 32;   // 32 one-block units (1088 bytes)
    static constexpr int SLACK = 16;
    static constexpr bool LIMBS = true;
    static constexpr int DEFAULT_UNROLL = 2;

    __host__ __device__ static int units(int nb) { return nb; }
    __device__ __forceinline__ static uint32_t unit_byte(int u) { return static_cast<uint32_t>(u) * BLOCK_BYTES; }
    __device__ __forceinline__ static int unit_elem(int u) { return u * QK; }

    struct X {
        uint32_t a[8], b[8], c[8];
        float xs;
    };
    struct L {
        int unused;
    };
    __device__ __forceinline__ static L lane_consts(int, int, int) { return L{0}; }

    __device__ __forceinline__ static void load_x(X& x, const uint8_t* smem, const LimbTables& T, int e0) {
#pragma unroll
        for (int v = 0; v < 2; v++) {
            const uint32_t o = limb_chunk(static_cast<uint32_t>(e0 >> 4) + v) << 4;
            const uint4 a = *reinterpret_cast<const uint4*>(smem + T.la + o);
            const uint4 b = *reinterpret_cast<const uint4*>(smem + T.lb + o);
            const uint4 c = *reinterpret_cast<const uint4*>(smem + T.lc + o);
            x.a[4 * v] = a.x; x.a[4 * v + 1] = a.y; x.a[4 * v + 2] = a.z; x.a[4 * v + 3] = a.w;
            x.b[4 * v] = b.x; x.b[4 * v + 1] = b.y; x.b[4 * v + 2] = b.z; x.b[4 * v + 3] = b.w;
            x.c[4 * v] = c.x; x.c[4 * v + 1] = c.y; x.c[4 * v + 2] = c.z; x.c[4 * v + 3] = c.w;
        }
        x.xs = reinterpret_cast<const float*>(smem + T.xs)[e0 >> 5];
    }

    // a: shared address of the 34-byte block (2-byte aligned).
    __device__ __forceinline__ static float dot(uint32_t a, const L&, const X& x, float r) {
        const uint32_t wa = a & ~3u;
        const uint32_t sh = (a & 3u) * 8u;
        const float d = f16_lo(lds32<0>(wa) >> sh);
        // the codes start at a + 2: word-aligned when sh == 16
        const uint32_t wq = wa + (sh >> 2);
        const uint32_t qsh = 16u - sh;
        const uint4 q0 = lds16_sh<0>(wq, qsh);
        const uint4 q1 = lds16_sh<16>(wq, qsh);
        const uint32_t q[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        int sa = 0, sb = 0, sc = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            sa = dp4a_ss(q[i], x.a[i], sa);
            sb = dp4a_ss(q[i], x.b[i], sb);
            sc = dp4a_ss(q[i], x.c[i], sc);
        }
        // |sa| <= 32*128*32 and |sb*256 + sc| < 2^28: the combination is done
        // in f32 (the full integer could exceed 2^31 here).
        const float t = __fmaf_rn(__int2float_rn(sa), 65536.0f, __int2float_rn(sb * 256 + sc)) * x.xs;
        return __fmaf_rn(d, t, r);
    }
};

// ============================================================ Q4_0, f32 x
//
// The native 18-byte block: d (f16), then 16 bytes whose low nibbles are the
// codes of weights 0..15 and high nibbles those of weights 16..31;
// w = d*(q - 8), so the block contributes d*(sum(q*x) - 8*sum(x)). Blocks sit
// at 2-byte alignment; five 32-bit loads from the word below the block hold
// all of it.
struct Q40 {
    static constexpr int QK = 32;
    static constexpr int BLOCK_BYTES = 18;
    static constexpr int SLICE_BLOCKS = 32;   // 32 one-block units (576 bytes)
    static constexpr int SLACK = 16;
    static constexpr bool LIMBS = true;
    static constexpr int DEFAULT_UNROLL = 2;

    __host__ __device__ static int units(int nb) { return nb; }
    __device__ __forceinline__ static uint32_t unit_byte(int u) { return static_cast<uint32_t>(u) * BLOCK_BYTES; }
    __device__ __forceinline__ static int unit_elem(int u) { return u * QK; }

    struct X {
        uint32_t a[8], b[8], c[8];   // limbs of the block's 32 activations
        float xs;                    // 2^-s of the 32-group
        float xsum;                  // its activation sum
    };
    struct L {
        int unused;
    };
    __device__ __forceinline__ static L lane_consts(int, int, int) { return L{0}; }

    __device__ __forceinline__ static void load_x(X& x, const uint8_t* smem, const LimbTables& T, int e0) {
#pragma unroll
        for (int v = 0; v < 2; v++) {
            const uint32_t o = limb_chunk(static_cast<uint32_t>(e0 >> 4) + v) << 4;
            const uint4 a = *reinterpret_cast<const uint4*>(smem + T.la + o);
            const uint4 b = *reinterpret_cast<const uint4*>(smem + T.lb + o);
            const uint4 c = *reinterpret_cast<const uint4*>(smem + T.lc + o);
            x.a[4 * v] = a.x; x.a[4 * v + 1] = a.y; x.a[4 * v + 2] = a.z; x.a[4 * v + 3] = a.w;
            x.b[4 * v] = b.x; x.b[4 * v + 1] = b.y; x.b[4 * v + 2] = b.z; x.b[4 * v + 3] = b.w;
            x.c[4 * v] = c.x; x.c[4 * v + 1] = c.y; x.c[4 * v + 2] = c.z; x.c[4 * v + 3] = c.w;
        }
        const float* xsum16 = reinterpret_cast<const float*>(smem + T.xsum16);
        x.xs = reinterpret_cast<const float*>(smem + T.xs)[e0 >> 5];
        x.xsum = xsum16[e0 >> 4] + xsum16[(e0 >> 4) + 1];
    }

    // a: shared address of the 18-byte block (2-byte aligned).
    __device__ __forceinline__ static float dot(uint32_t a, const L&, const X& x, float r) {
        const uint32_t wa = a & ~3u;
        const uint32_t sh = (a & 3u) * 8u;   // 0 or 16
        const uint32_t w[5] = {lds32<0>(wa), lds32<4>(wa), lds32<8>(wa), lds32<12>(wa), lds32<16>(wa)};
        const float d = f16_lo(__funnelshift_r(w[0], w[1], sh));
        int a0 = 0, b0 = 0, c0 = 0, a1 = 0, b1 = 0, c1 = 0;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            // code bytes 4j .. 4j+3 start 2 + 4j bytes past the block; the
            // clamped shift (16 or 32) takes them from words j, j+1
            const uint32_t q = __funnelshift_rc(w[j], w[j + 1], 16u + sh);
            const uint32_t lo = q & 0x0f0f0f0fu;   // weights 4j .. 4j+3
            const uint32_t hi = q & 0xf0f0f0f0u;   // 16 * weights 16+4j ..
            a0 = dp4a_us(lo, x.a[j], a0);
            b0 = dp4a_us(lo, x.b[j], b0);
            c0 = dp4a_us(lo, x.c[j], c0);
            a1 = dp4a_us(hi, x.a[4 + j], a1);
            b1 = dp4a_us(hi, x.b[4 + j], b1);
            c1 = dp4a_us(hi, x.c[4 + j], c1);
        }
        // |sum q*X| <= 16 * 15 * 2^21 per half; the high half carries a factor
        // 16 (multiples of 16, so the shift of c1 is exact).
        const int s = (a0 * 65536 + b0 * 256 + c0) + (a1 * 4096 + b1 * 16 + (c1 >> 4));
        const float t = __int2float_rn(s) * x.xs;
        return __fmaf_rn(d, __fmaf_rn(-8.0f, x.xsum, t), r);
    }
};

// ======================================================= Q8_0, q8 activation
//
// The dp4a path: the activation is already int8 codes with one f32 scale per
// 32-block (quantize_act_q8). A unit is 4 consecutive blocks (128 weights), so
// one warp's 32 units cover 4096 weights. Per block, dot = sum of 32
// int8*int8 products (exact int32), and the row sums d_w * d_x * dot in f32.
struct Q8D {
    static constexpr int QK = 32;
    static constexpr int BLOCK_BYTES = 34;
    static constexpr int SLICE_BLOCKS = 128;  // 32 four-block units (4352 bytes)
    static constexpr int SLACK = 144;         // a ragged last unit still loads 136 bytes
    static constexpr bool LIMBS = false;
    static constexpr int DEFAULT_UNROLL = 2;
    static constexpr int DOTS_PER_UNIT = 4;   // 32-weight blocks per unit
    static constexpr int DOT_WEIGHTS = 32;    // weights per exported dot
    __device__ __forceinline__ static int dot_base(int ug) { return DOTS_PER_UNIT * ug; }

    __host__ __device__ static int units(int nb) { return (nb + 3) / 4; }
    __device__ __forceinline__ static uint32_t unit_byte(int u) { return static_cast<uint32_t>(u) * 4u * BLOCK_BYTES; }
    __device__ __forceinline__ static int unit_elem(int u) { return u * 4 * QK; }

    struct X {
        uint32_t q[4][8];
        float xs[4];
    };
    struct L {
        int nblk;   // blocks in this unit (4 except at a row's ragged end)
    };
    // ug: the unit's index within the row; nb: blocks per row.
    __device__ __forceinline__ static L lane_consts(int, int nb, int ug) {
        const int left = nb - 4 * ug;
        return L{left < 4 ? left : 4};
    }

    __device__ __forceinline__ static void load_xq(X& x, const L& l, const int8_t* __restrict__ xq,
                                                   const float* __restrict__ xs, int e0) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            if (j < l.nblk) {
                const uint4 a = __ldg(reinterpret_cast<const uint4*>(xq + e0 + 32 * j));
                const uint4 b = __ldg(reinterpret_cast<const uint4*>(xq + e0 + 32 * j + 16));
                x.q[j][0] = a.x; x.q[j][1] = a.y; x.q[j][2] = a.z; x.q[j][3] = a.w;
                x.q[j][4] = b.x; x.q[j][5] = b.y; x.q[j][6] = b.z; x.q[j][7] = b.w;
                x.xs[j] = __ldg(xs + (e0 >> 5) + j);
            } else {
#pragma unroll
                for (int i = 0; i < 8; i++) x.q[j][i] = 0;
                x.xs[j] = 0.0f;
            }
        }
    }

    __device__ __forceinline__ static int block_dot8(const uint32_t* q, const uint32_t* xq) {
        int s = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) s = dp4a_ss(q[i], xq[i], s);
        return s;
    }

    // The four blocks of a unit that starts 8-byte aligned: 17 64-bit loads;
    // the codes of blocks 0 and 2 sit 2 bytes off a word boundary.
    // Outputs: d bit patterns (in the low 16 bits) and the code words.
    __device__ __forceinline__ static void load_unit8(uint32_t a, uint32_t (&dh)[4], uint32_t (&q)[4][8]) {
        uint32_t W[34];
#define QMV_LD(m) { const uint2 v = lds64<8 * (m)>(a); W[2 * (m)] = v.x; W[2 * (m) + 1] = v.y; }
        QMV_LD(0) QMV_LD(1) QMV_LD(2) QMV_LD(3) QMV_LD(4) QMV_LD(5) QMV_LD(6) QMV_LD(7) QMV_LD(8)
        QMV_LD(9) QMV_LD(10) QMV_LD(11) QMV_LD(12) QMV_LD(13) QMV_LD(14) QMV_LD(15) QMV_LD(16)
#undef QMV_LD
        dh[0] = W[0];
        dh[1] = W[8] >> 16;
        dh[2] = W[17];
        dh[3] = W[25] >> 16;
#pragma unroll
        for (int m = 0; m < 8; m++) {
            q[0][m] = __funnelshift_r(W[m], W[m + 1], 16);
            q[1][m] = W[9 + m];
            q[2][m] = __funnelshift_r(W[17 + m], W[18 + m], 16);
            q[3][m] = W[26 + m];
        }
    }

    // The same from any 2-byte aligned address, block by block.
    __device__ __forceinline__ static void load_block_a2(uint32_t a, uint32_t& dh, uint32_t (&q)[8]) {
        const uint32_t wa = a & ~3u;
        const uint32_t sh = (a & 3u) * 8u;
        dh = lds32<0>(wa) >> sh;
        const uint32_t wq = wa + (sh >> 2);
        const uint32_t qsh = 16u - sh;
        const uint4 q0 = lds16_sh<0>(wq, qsh);
        const uint4 q1 = lds16_sh<16>(wq, qsh);
        q[0] = q0.x; q[1] = q0.y; q[2] = q0.z; q[3] = q0.w;
        q[4] = q1.x; q[5] = q1.y; q[6] = q1.z; q[7] = q1.w;
    }

    __device__ __forceinline__ static void load_unit(uint32_t a, bool aligned8, uint32_t (&dh)[4],
                                                     uint32_t (&q)[4][8]) {
        if (aligned8) {
            load_unit8(a, dh, q);
        } else {
#pragma unroll
            for (int j = 0; j < 4; j++) load_block_a2(a + 34u * j, dh[j], q[j]);
        }
    }

    // a: shared address of the unit's first block.
    __device__ __forceinline__ static float dot(uint32_t a, const L& l, const X& x, float r, bool aligned8) {
        uint32_t dh[4], q[4][8];
        load_unit(a, aligned8, dh, q);
#pragma unroll
        for (int j = 0; j < 4; j++) {
            if (j < l.nblk) {
                const int s = block_dot8(q[j], x.q[j]);
                r = __fmaf_rn(f16_lo(dh[j]) * x.xs[j], __int2float_rn(s), r);
            }
        }
        return r;
    }

    // The exact int32 dots of the unit's blocks (MODE_BLOCKDOTS).
    __device__ __forceinline__ static void block_dots(uint32_t a, const L& l, const X& x, bool aligned8,
                                                      int32_t* out) {
        uint32_t dh[4], q[4][8];
        load_unit(a, aligned8, dh, q);
#pragma unroll
        for (int j = 0; j < 4; j++)
            if (j < l.nblk) out[j] = block_dot8(q[j], x.q[j]);
    }
};

// ============================================ Q8_0, f32 x quantized in the kernel
//
// The dp4a path of Q8_0 with the activation quantization folded into the
// launch (hanzo-ml src/vulkan_backend.rs: quantize_act_q8 once per decode step,
// then the dp4a matvec on its codes): every CTA quantizes the f32 x into its
// own shared memory exactly as quantize_act_q8 does (same IEEE steps, so the
// same codes and scales, bit for bit) while its first weight pieces are in
// flight, and the lanes read their codes from there. Decode as Q8D.
struct Q8DQ : Q8D {
    static constexpr bool QPREP = true;

    // Codes and scales from the CTA's shared tables (xq, xs point there).
    __device__ __forceinline__ static void load_xq(X& x, const L& l, const int8_t* xq, const float* xs, int e0) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            if (j < l.nblk) {
                const uint4 a = *reinterpret_cast<const uint4*>(xq + e0 + 32 * j);
                const uint4 b = *reinterpret_cast<const uint4*>(xq + e0 + 32 * j + 16);
                x.q[j][0] = a.x; x.q[j][1] = a.y; x.q[j][2] = a.z; x.q[j][3] = a.w;
                x.q[j][4] = b.x; x.q[j][5] = b.y; x.q[j][6] = b.z; x.q[j][7] = b.w;
                x.xs[j] = xs[(e0 >> 5) + j];
            } else {
#pragma unroll
                for (int i = 0; i < 8; i++) x.q[j][i] = 0;
                x.xs[j] = 0.0f;
            }
        }
    }
};

// Formats whose kernel quantizes the f32 activation itself (QPREP).
template <class F, class = void>
struct quantizes_x : std::false_type {};
template <class F>
struct quantizes_x<F, std::void_t<decltype(F::QPREP)>> : std::bool_constant<F::QPREP> {};

}  // namespace qmv
