// qmm_formats.cuh -- the unit decoder of the register-activation batched
// product y[m, rows] = x[m, k] W^T over Q4_K rows (2 <= m <= 8 activation
// rows per launch; the entry point uses it for two rows, and Q6_K and Q8_0
// batches run on the tensor cores, qmm_tc.cuh).
//
// Each weight is decoded once per launch and used for all M rows of x. A lane
// owns UW consecutive weights of a row (a "unit": UW = 8 for M >= 5, 16 for
// M = 3, 4, and 32 for M = 2, so the lane's share of x, M * UW floats, stays at
// 64 registers or fewer) and keeps their activations of all M rows in
// registers while the rows of W stream past. Per row it decodes its UW weights
// into f32 -- each the round-to-nearest f32 of the exact value, the same value
// the dequantizers write -- and forms M dot products with packed f32 pair
// FMAs (fma.rn.f32x2).
//
// Byte layout and decode rule as in qmv_formats.cuh (hanzo-ml
// src/vulkan_backend.rs: quantize_q4k; the batched product is the
// matmul_q4k_gpu prefill GEMM, which decodes each weight once for up to eight
// rows of x).
#pragma once

#include "qmv_formats.cuh"

namespace qmv {

// ------------------------------------------------------- packed f32 pairs

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// 2^23 + byte b of w, as a float (exact for every byte value).
__device__ __forceinline__ float magic_byte(uint32_t w, uint32_t b) {
    return __uint_as_float(prmt(w, 0x4B000000u, 0x7440u | b));
}

// Weights per unit for a batch of M rows.
template <int M>
struct BatchUnit {
    static_assert(M >= 2 && M <= 8, "batch width");
    static constexpr int UW = M >= 5 ? 8 : (M >= 3 ? 16 : 32);
};

// UW/4 words of code bytes starting at shared address a (a % 8 == 0 for
// UW = 8, a % 16 == 0 otherwise).
template <int UW>
__device__ __forceinline__ void lds_words_aligned(uint32_t a, uint32_t (&q)[UW / 4]) {
    if constexpr (UW == 8) {
        const uint2 v = lds64<0>(a);
        q[0] = v.x; q[1] = v.y;
    } else {
#pragma unroll
        for (int i = 0; i < UW / 16; i++) {
            const uint4 v = lds128<0>(a + 16u * i);
            q[4 * i] = v.x; q[4 * i + 1] = v.y; q[4 * i + 2] = v.z; q[4 * i + 3] = v.w;
        }
    }
}

// The same from a 2-byte aligned address: word-aligned base wa, byte shift sh.
template <int UW>
__device__ __forceinline__ void lds_words_sh(uint32_t wa, uint32_t sh, uint32_t (&q)[UW / 4]) {
    if constexpr (UW == 8) {
        const uint2 v = lds8_sh<0>(wa, sh);
        q[0] = v.x; q[1] = v.y;
    } else {
#pragma unroll
        for (int i = 0; i < UW / 16; i++) {
            const uint4 v = lds16_sh<0>(wa + 16u * i, sh);
            q[4 * i] = v.x; q[4 * i + 1] = v.y; q[4 * i + 2] = v.z; q[4 * i + 3] = v.w;
        }
    }
}

// ============================================================== Q4_K batch
//
// Unit u of a block covers weights e0 = UW*u .. e0+UW-1, inside sub-block
// j = e0/32: the low (even j) or high (odd j) nibbles of qs bytes
// 32*(j/2) + e0%32 onwards. w = d*sc_j*q - dmin*m_j: t = fma(d*sc_j, 2^23 + q,
// -d*sc_j*2^23) is d*sc_j*q exactly, then w = t - dmin*m_j rounds once.
template <int M>
struct Q4KB {
    static constexpr int QK = 256;
    static constexpr int BLOCK_BYTES = 144;
    static constexpr int UW = BatchUnit<M>::UW;
    static constexpr int UPB = QK / UW;                // units per block
    static constexpr int SLICE_BLOCKS = 32 / UPB;      // blocks per warp slice
    static constexpr int SLACK = 0;
    static constexpr bool LIMBS = false;
    static constexpr int DEFAULT_UNROLL = 1;
    static constexpr int OUTS = M;

    __host__ __device__ static int units(int nb) { return UPB * nb; }
    __device__ __forceinline__ static uint32_t unit_byte(int u) { return static_cast<uint32_t>(u / UPB) * BLOCK_BYTES; }
    __device__ __forceinline__ static int unit_elem(int u) { return (u / UPB) * QK + (u % UPB) * UW; }

    struct L {
        uint32_t qoff;   // byte offset of the unit's codes in the block
        uint32_t sel;    // scale byte j & 3 within its word
        bool hinib;      // odd sub-block: high nibbles
        bool hic;        // j >= 4
    };
    __device__ __forceinline__ static L lane_consts(int u, int, int) {
        const int e0 = (u % UPB) * UW;
        const int j = e0 >> 5;
        L l;
        l.qoff = 16u + 32u * static_cast<uint32_t>(j >> 1) + static_cast<uint32_t>(e0 & 31);
        l.sel = 0x7440u | static_cast<uint32_t>(j & 3);
        l.hinib = (j & 1) != 0;
        l.hic = j >= 4;
        return l;
    }

    // a: shared address of the block (16-byte aligned).
    __device__ __forceinline__ static void decode(uint32_t a, const L& l, float2 (&w)[UW / 2]) {
        const uint4 h = lds128<0>(a);
        uint32_t q[UW / 4];
        lds_words_aligned<UW>(a + l.qoff, q);
        const uint32_t sc_lo = h.y & 0x3f3f3f3fu;
        const uint32_t m_lo = h.z & 0x3f3f3f3fu;
        const uint32_t sc_hi = (h.w & 0x0f0f0f0fu) | ((h.y >> 2) & 0x30303030u);
        const uint32_t m_hi = ((h.w >> 4) & 0x0f0f0f0fu) | ((h.z >> 2) & 0x30303030u);
        const uint32_t SC = l.hic ? sc_hi : sc_lo;
        const uint32_t MN = l.hic ? m_hi : m_lo;
        const float d = f16_lo(h.x), dmin = f16_hi(h.x);
        const float dsc = __fmaf_rn(d, __uint_as_float(prmt(SC, 0x4B000000u, l.sel)), -d * TWO23);
        const float dm = __fmaf_rn(dmin, __uint_as_float(prmt(MN, 0x4B000000u, l.sel)), -dmin * TWO23);
        const float2 s2 = make_float2(dsc, dsc);
        const float2 n2 = make_float2(-dsc * TWO23, -dsc * TWO23);
        const float2 m2 = make_float2(-dm, -dm);
#pragma unroll
        for (int i = 0; i < UW / 4; i++) {
            const uint32_t nib = l.hinib ? ((q[i] >> 4) & 0x0f0f0f0fu) : (q[i] & 0x0f0f0f0fu);
            const float2 f01 = make_float2(magic_byte(nib, 0), magic_byte(nib, 1));
            const float2 f23 = make_float2(magic_byte(nib, 2), magic_byte(nib, 3));
            w[2 * i] = add2(fma2(s2, f01, n2), m2);
            w[2 * i + 1] = add2(fma2(s2, f23, n2), m2);
        }
    }
};

}  // namespace qmv
