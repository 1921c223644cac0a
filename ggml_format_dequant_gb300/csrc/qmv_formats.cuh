// qmv_formats.cuh -- in-register decode of one "unit" of a packed GGML block
// against the activation, for Q4_K, Q6_K and Q8_0.
//
// A unit is the slice of a block one lane owns for every row it processes:
//   Q4_K: one 64-weight chunk of a 256-weight super-block (4 per block)
//   Q6_K: one (half, 16-position) slice, 64 weights (4 per block)
//   Q8_0: one 32-weight block
// The lane keeps the activation for its unit in registers (as integer limbs or
// int8 codes) and, per row, reads the unit's packed bytes from the shared-memory
// stage, unpacks the codes into byte lanes and forms integer dot products with
// dp4a, then applies the block's scales once per scale group.
//
// Block layouts (hanzo-ml src/vulkan_backend.rs): Q4_K = d, dmin (f16), 12 bytes
// of packed 6-bit scales/mins, 128 bytes of 4-bit codes (quantize_q4k,
// quantize_q4k_split); Q6_K = ql[128], qh[64], int8 scales[16], d (f16)
// (quantize_q6k); Q8_0 = d (f16) + 32 int8 (quantize_q8_blocks). The bit
// mapping inside the blocks is GGML's k-quant layout.
#pragma once

#include "qmv_device.cuh"

namespace qmv {

// ====================================================================== Q4_K
//
// Chunk c (0..3) of a super-block covers weights 64c .. 64c+63: qs bytes
// 32c .. 32c+31, whose low nibbles are sub-block 2c (weights 64c + l) and high
// nibbles sub-block 2c+1 (weights 64c + 32 + l). Weight i of sub-block j is
// d*sc_j*q_i - dmin*m_j, so the chunk contributes
//     d*sc_2c * sum(q*x) - dmin*m_2c * sum(x)  +  (same for 2c+1).
struct Q4K {
    static constexpr int MAX_THREADS = 512;   // launch bound (registers: 65536 / MAX_THREADS)
    static constexpr int QK = 256;
    static constexpr int BLOCK_BYTES = 144;
    static constexpr int SLICE_BLOCKS = 8;    // 32 units = one warp's k-slice (1152 bytes)
    static constexpr bool LIMBS = true;

    __host__ __device__ static int units(int nb) { return 4 * nb; }
    // Unit u of a slice: byte offset of its block, index of its first weight.
    __device__ __forceinline__ static int unit_byte(int u) { return (u >> 2) * BLOCK_BYTES; }
    __device__ __forceinline__ static int unit_elem(int u) { return (u >> 2) * QK + 64 * (u & 3); }

    struct X {
        uint32_t a[16], b[16], c[16];   // limbs of the chunk's 64 activations
        float xs0, xs1;                 // 2^-s of the two 32-groups
        float xsum0, xsum1;             // activation sums of the two sub-blocks
    };
    // Lane-constant selectors for the scale/min bit fields of chunk c.
    struct L {
        int c, sh, shm;
        uint32_t mlo, mhi;
        bool hic;
    };

    __device__ __forceinline__ static L lane_consts(int u, int /*nb*/, int /*ug*/) {
        const int c = u & 3;
        L l;
        l.c = c;
        l.hic = c >= 2;
        l.sh = 16 * (c & 1);
        l.shm = l.hic ? l.sh + 4 : l.sh;
        l.mlo = l.hic ? 15u : 63u;
        l.mhi = l.hic ? 0x30u : 0u;
        return l;
    }

    // e0 = index of the chunk's first weight in the row.
    __device__ __forceinline__ static void load_x(X& x, const XPrepSmem& P, int e0) {
        const uint4* A = reinterpret_cast<const uint4*>(P.la + e0);
        const uint4* B = reinterpret_cast<const uint4*>(P.lb + e0);
        const uint4* C = reinterpret_cast<const uint4*>(P.lc + e0);
#pragma unroll
        for (int v = 0; v < 4; v++) {
            const uint4 a = A[v], b = B[v], c = C[v];
            x.a[4 * v] = a.x; x.a[4 * v + 1] = a.y; x.a[4 * v + 2] = a.z; x.a[4 * v + 3] = a.w;
            x.b[4 * v] = b.x; x.b[4 * v + 1] = b.y; x.b[4 * v + 2] = b.z; x.b[4 * v + 3] = b.w;
            x.c[4 * v] = c.x; x.c[4 * v + 1] = c.y; x.c[4 * v + 2] = c.z; x.c[4 * v + 3] = c.w;
        }
        x.xs0 = P.xs[e0 >> 5];
        x.xs1 = P.xs[(e0 >> 5) + 1];
        x.xsum0 = P.xsum16[e0 >> 4] + P.xsum16[(e0 >> 4) + 1];
        x.xsum1 = P.xsum16[(e0 >> 4) + 2] + P.xsum16[(e0 >> 4) + 3];
    }

    // blk: the super-block in shared memory (16-byte aligned).
    __device__ __forceinline__ static float dot(const uint8_t* blk, const L& l, const X& x, float r) {
        const uint4 h = *reinterpret_cast<const uint4*>(blk);
        const uint4 qa = *reinterpret_cast<const uint4*>(blk + 16 + 32 * l.c);
        const uint4 qb = *reinterpret_cast<const uint4*>(blk + 32 + 32 * l.c);
        const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        int a0 = 0, b0 = 0, c0 = 0, a1 = 0, b1 = 0, c1 = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t lo = q[i] & 0x0f0f0f0fu;
            const uint32_t hi = (q[i] >> 4) & 0x0f0f0f0fu;
            a0 = dp4a_us(lo, x.a[i], a0);
            b0 = dp4a_us(lo, x.b[i], b0);
            c0 = dp4a_us(lo, x.c[i], c0);
            a1 = dp4a_us(hi, x.a[8 + i], a1);
            b1 = dp4a_us(hi, x.b[8 + i], b1);
            c1 = dp4a_us(hi, x.c[8 + i], c1);
        }
        // |sum q*X| <= 32 * 15 * 2^21 < 2^31 per sub-block.
        const int s0 = limb_combine(a0, b0, c0);
        const int s1 = limb_combine(a1, b1, c1);
        const uint32_t srcS = l.hic ? h.w : h.y;
        const uint32_t srcM = l.hic ? h.w : h.z;
        const int sc0 = static_cast<int>(((srcS >> l.sh) & l.mlo) | ((h.y >> (l.sh + 2)) & l.mhi));
        const int m0 = static_cast<int>(((srcM >> l.shm) & l.mlo) | ((h.z >> (l.sh + 2)) & l.mhi));
        const int sc1 = static_cast<int>(((srcS >> (l.sh + 8)) & l.mlo) | ((h.y >> (l.sh + 10)) & l.mhi));
        const int m1 = static_cast<int>(((srcM >> (l.shm + 8)) & l.mlo) | ((h.z >> (l.sh + 10)) & l.mhi));
        const float d = f16_lo(h.x), dmin = f16_hi(h.x);
        const float t0 = __int2float_rn(s0) * x.xs0;
        const float t1 = __int2float_rn(s1) * x.xs1;
        r = __fmaf_rn(d * __int2float_rn(sc0), t0, r);
        r = __fmaf_rn(-(dmin * __int2float_rn(m0)), x.xsum0, r);
        r = __fmaf_rn(d * __int2float_rn(sc1), t1, r);
        r = __fmaf_rn(-(dmin * __int2float_rn(m1)), x.xsum1, r);
        return r;
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
    static constexpr int MAX_THREADS = 512;   // launch bound (registers: 65536 / MAX_THREADS)
    static constexpr int QK = 256;
    static constexpr int BLOCK_BYTES = 210;
    static constexpr int SLICE_BLOCKS = 8;    // 32 units = one warp's k-slice (1680 bytes)
    static constexpr bool LIMBS = true;

    __host__ __device__ static int units(int nb) { return 4 * nb; }
    __device__ __forceinline__ static int unit_byte(int u) { return (u >> 2) * BLOCK_BYTES; }
    __device__ __forceinline__ static int unit_elem(int u) {
        return (u >> 2) * QK + 128 * ((u & 3) >> 1) + 16 * (u & 1);
    }

    struct X {
        uint32_t a[16], b[16], c[16];   // [4*qd + i]: limbs of weights 128H+32qd+16hh+4i..
        float xs[4], xsum[4];
    };
    struct L {
        int H, hh;
    };

    __device__ __forceinline__ static L lane_consts(int u, int /*nb*/, int /*ug*/) {
        L l;
        l.H = (u & 3) >> 1;
        l.hh = u & 1;
        return l;
    }

    // e0 = index (in the row) of weight 128H + 16hh of the unit's block.
    __device__ __forceinline__ static void load_x(X& x, const XPrepSmem& P, int e0) {
#pragma unroll
        for (int qd = 0; qd < 4; qd++) {
            const int e = e0 + 32 * qd;
            const uint4 a = *reinterpret_cast<const uint4*>(P.la + e);
            const uint4 b = *reinterpret_cast<const uint4*>(P.lb + e);
            const uint4 c = *reinterpret_cast<const uint4*>(P.lc + e);
            x.a[4 * qd] = a.x; x.a[4 * qd + 1] = a.y; x.a[4 * qd + 2] = a.z; x.a[4 * qd + 3] = a.w;
            x.b[4 * qd] = b.x; x.b[4 * qd + 1] = b.y; x.b[4 * qd + 2] = b.z; x.b[4 * qd + 3] = b.w;
            x.c[4 * qd] = c.x; x.c[4 * qd + 1] = c.y; x.c[4 * qd + 2] = c.z; x.c[4 * qd + 3] = c.w;
            x.xs[qd] = P.xs[e >> 5];
            x.xsum[qd] = P.xsum16[e >> 4];
        }
    }

    // blk: the block in shared memory (2-byte aligned).
    __device__ __forceinline__ static float dot(const uint8_t* blk, const L& l, const X& x, float r) {
        const uint4 qla = lds16_a2(blk + 64 * l.H + 16 * l.hh);
        const uint4 qlb = lds16_a2(blk + 64 * l.H + 32 + 16 * l.hh);
        const uint4 qhv = lds16_a2(blk + 128 + 32 * l.H + 16 * l.hh);
        const uint2 scw = lds8_a2(blk + 192 + 8 * l.H);
        const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(lds_u16_a2(blk + 208))));
        const uint32_t A[4] = {qla.x, qla.y, qla.z, qla.w};
        const uint32_t B[4] = {qlb.x, qlb.y, qlb.z, qlb.w};
        const uint32_t Hq[4] = {qhv.x, qhv.y, qhv.z, qhv.w};
        int sa[4] = {0, 0, 0, 0}, sb[4] = {0, 0, 0, 0}, sc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t w0 = (A[i] & 0x0f0f0f0fu) | ((Hq[i] << 4) & 0x30303030u);
            const uint32_t w1 = (B[i] & 0x0f0f0f0fu) | ((Hq[i] << 2) & 0x30303030u);
            const uint32_t w2 = ((A[i] >> 4) & 0x0f0f0f0fu) | (Hq[i] & 0x30303030u);
            const uint32_t w3 = ((B[i] >> 4) & 0x0f0f0f0fu) | ((Hq[i] >> 2) & 0x30303030u);
            sa[0] = dp4a_us(w0, x.a[i], sa[0]);
            sb[0] = dp4a_us(w0, x.b[i], sb[0]);
            sc[0] = dp4a_us(w0, x.c[i], sc[0]);
            sa[1] = dp4a_us(w1, x.a[4 + i], sa[1]);
            sb[1] = dp4a_us(w1, x.b[4 + i], sb[1]);
            sc[1] = dp4a_us(w1, x.c[4 + i], sc[1]);
            sa[2] = dp4a_us(w2, x.a[8 + i], sa[2]);
            sb[2] = dp4a_us(w2, x.b[8 + i], sb[2]);
            sc[2] = dp4a_us(w2, x.c[8 + i], sc[2]);
            sa[3] = dp4a_us(w3, x.a[12 + i], sa[3]);
            sb[3] = dp4a_us(w3, x.b[12 + i], sb[3]);
            sc[3] = dp4a_us(w3, x.c[12 + i], sc[3]);
        }
#pragma unroll
        for (int qd = 0; qd < 4; qd++) {
            // |sum q*X| <= 16 * 63 * 2^21 < 2^31 per quarter.
            const int s = limb_combine(sa[qd], sb[qd], sc[qd]);
            const uint32_t sw = (qd < 2) ? scw.x : scw.y;
            const int scale = static_cast<int>(static_cast<int8_t>((sw >> (8 * (l.hh + 2 * (qd & 1)))) & 0xffu));
            const float t = __int2float_rn(s) * x.xs[qd];
            const float u = __fmaf_rn(-32.0f, x.xsum[qd], t);
            r = __fmaf_rn(d * __int2float_rn(scale), u, r);
        }
        return r;
    }
};

// ============================================================ Q8_0, f32 x
struct Q8F {
    static constexpr int MAX_THREADS = 512;   // launch bound (registers: 65536 / MAX_THREADS)
    static constexpr int QK = 32;
    static constexpr int BLOCK_BYTES = 34;
    static constexpr int SLICE_BLOCKS = 32;   // 32 one-block units (1088 bytes)
    static constexpr bool LIMBS = true;

    __host__ __device__ static int units(int nb) { return nb; }
    __device__ __forceinline__ static int unit_byte(int u) { return u * BLOCK_BYTES; }
    __device__ __forceinline__ static int unit_elem(int u) { return u * QK; }

    struct X {
        uint32_t a[8], b[8], c[8];
        float xs;
    };
    struct L {
        int unused;
    };
    __device__ __forceinline__ static L lane_consts(int, int, int) { return L{0}; }

    __device__ __forceinline__ static void load_x(X& x, const XPrepSmem& P, int e0) {
#pragma unroll
        for (int v = 0; v < 2; v++) {
            const uint4 a = *reinterpret_cast<const uint4*>(P.la + e0 + 16 * v);
            const uint4 b = *reinterpret_cast<const uint4*>(P.lb + e0 + 16 * v);
            const uint4 c = *reinterpret_cast<const uint4*>(P.lc + e0 + 16 * v);
            x.a[4 * v] = a.x; x.a[4 * v + 1] = a.y; x.a[4 * v + 2] = a.z; x.a[4 * v + 3] = a.w;
            x.b[4 * v] = b.x; x.b[4 * v + 1] = b.y; x.b[4 * v + 2] = b.z; x.b[4 * v + 3] = b.w;
            x.c[4 * v] = c.x; x.c[4 * v + 1] = c.y; x.c[4 * v + 2] = c.z; x.c[4 * v + 3] = c.w;
        }
        x.xs = P.xs[e0 >> 5];
    }

    // blk: the 34-byte block in shared memory (2-byte aligned).
    __device__ __forceinline__ static float dot(const uint8_t* blk, const L&, const X& x, float r) {
        const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(lds_u16_a2(blk))));
        const uint4 q0 = lds16_a2(blk + 2);
        const uint4 q1 = lds16_a2(blk + 18);
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

// ======================================================= Q8_0, q8 activation
//
// The dp4a path: the activation is already int8 codes with one f32 scale per
// 32-block (quantize_act_q8). A unit is 4 consecutive blocks (128 weights), so
// one warp's 32 units cover 4096 weights. Per block, dot = sum of 32
// int8*int8 products (exact int32), and the row sums d_w * d_x * dot in f32.
struct Q8D {
    static constexpr int MAX_THREADS = 512;   // launch bound (registers: 65536 / MAX_THREADS)
    static constexpr int QK = 32;
    static constexpr int BLOCK_BYTES = 34;
    static constexpr int SLICE_BLOCKS = 128;  // 32 four-block units (4352 bytes)
    static constexpr bool LIMBS = false;

    __host__ __device__ static int units(int nb) { return (nb + 3) / 4; }
    __device__ __forceinline__ static int unit_byte(int u) { return u * 4 * BLOCK_BYTES; }
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

    // blk: one 34-byte block in shared memory (2-byte aligned).
    __device__ __forceinline__ static int block_dot(const uint8_t* blk, const uint32_t* xq) {
        const uint4 q0 = lds16_a2(blk + 2);
        const uint4 q1 = lds16_a2(blk + 18);
        int s = 0;
        s = dp4a_ss(q0.x, xq[0], s);
        s = dp4a_ss(q0.y, xq[1], s);
        s = dp4a_ss(q0.z, xq[2], s);
        s = dp4a_ss(q0.w, xq[3], s);
        s = dp4a_ss(q1.x, xq[4], s);
        s = dp4a_ss(q1.y, xq[5], s);
        s = dp4a_ss(q1.z, xq[6], s);
        s = dp4a_ss(q1.w, xq[7], s);
        return s;
    }

    // ub: the unit's first block in shared memory.
    __device__ __forceinline__ static float dot(const uint8_t* ub, const L& l, const X& x, float r) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            if (j < l.nblk) {
                const uint8_t* blk = ub + j * BLOCK_BYTES;
                const float dw = __half2float(__ushort_as_half(static_cast<unsigned short>(lds_u16_a2(blk))));
                const int s = block_dot(blk, x.q[j]);
                r = __fmaf_rn(dw * x.xs[j], __int2float_rn(s), r);
            }
        }
        return r;
    }
};

}  // namespace qmv
