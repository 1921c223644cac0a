/*
 * qmv_oracle.c -- plain, slow, obviously-correct CPU oracle for the GGML-block
 * quantized matrix-vector product.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file; it exists so the CUDA kernels can be checked against an
 * independent restatement of what they compute. It shares no code, header,
 * table or constant with the CUDA library.
 *
 * Sources (docs.rs pages of hanzo-ml / hanzo-kernel):
 *  - hanzo-ml src/vulkan_backend.rs, `quantize_q4k`: the 144-byte Q4_K
 *    super-block is d (f16), dmin (f16), 12 bytes of packed 6-bit scales and
 *    mins, 128 bytes of 4-bit codes; decode is defined there as the CPU
 *    `BlockQ4K::to_float`, i.e. the GGML k-quant layout (the reading taken
 *    here: w = d*sc_j*q - dmin*m_j, sub-block j = i/32).
 *  - same file, `quantize_q6k` / `quantize_q6k_split`: the 210-byte Q6_K block
 *    is ql[128], qh[64], int8 scales[16], d (f16); w = d*scale*(q - 32).
 *  - same file, `quantize_q8_blocks` and `matvec_q8_0_gpu`: the 34-byte Q8_0
 *    block is d (f16, little endian) then 32 int8; w = d*q.
 *  - hanzo-ml tests/vulkan_quant_tests.rs, module doc and `run_case`: the
 *    reference is a host f64 matvec over the dequantized weights (not GGML's
 *    vec_dot, which quantizes the activation).
 *  - vulkan_backend.rs `quantize_q8` (amax, inv = 127/amax, round, clamp to
 *    +-127) and `quantize_act_q8` (per-32 block int8 codes, f32 scale and a
 *    per-block sum): the activation quantizer of the dp4a path, with the
 *    rounding taken as round-to-nearest-even on an IEEE f32 product.
 *  - same file, `matvec_q4_0_gpu`: the native 18-byte Q4_0 block, decode
 *    byte-exact with the CPU `BlockQ4_0::to_float` (the reading taken here: d
 *    (f16) then 16 bytes; weight i < 16 is the low nibble of qs[i], weight
 *    i >= 16 the high nibble of qs[i-16]; w = d*(q - 8)).
 *  - same file, `quantize_q5k` / `matvec_q5k`: the 176-byte GGUF Q5_K block is
 *    d, dmin, 12 scale bytes, 32 qh bytes, 128 qs bytes, decode matching the
 *    CPU `BlockQ5K::to_float` (the reading taken here: scales and mins packed
 *    as in Q4_K, the 4 low bits of each code laid out as Q4_K's, the fifth bit
 *    of weight i being bit (i/32) of qh[i%32]; w = d*sc_j*q - dmin*m_j).
 *  - vulkan_backend.rs `moe_matvec_gpu`: y[s, r] = sum_k W[ids[s], r, k] x[s, k]
 *    over one resident [E, n, k] bank, output in slot order.
 *
 * Floating point: decoded weights are formed exactly in f64 (every Q4_K/Q6_K/
 * Q8_0 weight has at most 50 significant bits from its f16 scale, small integer
 * scale and code, so f64 holds it exactly). Dot products accumulate in f64 in
 * index order. The activation quantizer works in IEEE binary32 exactly as
 * written (compile with -ffp-contract=off, no fast-math).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_QK_K 256
#define ORC_QK8_0 32
#define ORC_Q4K_BYTES 144
#define ORC_Q6K_BYTES 210
#define ORC_Q8_0_BYTES 34
#define ORC_Q4_0_BYTES 18
#define ORC_Q5K_BYTES 176

/* IEEE 754 binary16 -> binary64, exact for every encoding: normal numbers are
 * (1024 + mantissa) * 2^(exponent - 25), subnormals mantissa * 2^-24. */
double orc_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

static uint16_t rd_le16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* ---------------------------------------------------------------- Q4_K -- */

/* Six-bit scale and min of sub-block j (0..7) from the 12 packed bytes s[]:
 * sub-blocks 0..3 keep their 6 bits in the low bits of s[j] (scale) and
 * s[j+4] (min); sub-blocks 4..7 keep their low 4 bits in the nibbles of s[j+4]
 * and their top 2 bits in the top bits of s[j-4] (scale) and s[j] (min). */
static void q4k_scale_min(int j, const uint8_t *s, int *sc, int *m) {
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* Loop-structured decode of one super-block: four 64-weight chunks, each one
 * 32-byte run of qs whose low nibbles are sub-block 2c and high nibbles
 * sub-block 2c+1. */
void orc_q4k_block_decode(const uint8_t *b, double *out) {
    double d = orc_f16_to_f64(rd_le16(b));
    double dmin = orc_f16_to_f64(rd_le16(b + 2));
    const uint8_t *s = b + 4;
    const uint8_t *qs = b + 16;
    for (int c = 0; c < 4; c++) {
        int sc0, m0, sc1, m1;
        q4k_scale_min(2 * c, s, &sc0, &m0);
        q4k_scale_min(2 * c + 1, s, &sc1, &m1);
        for (int l = 0; l < 32; l++) {
            int lo = qs[32 * c + l] & 15;
            int hi = qs[32 * c + l] >> 4;
            out[64 * c + l] = d * sc0 * lo - dmin * m0;
            out[64 * c + 32 + l] = d * sc1 * hi - dmin * m1;
        }
    }
}

/* Bit field of the 12 packed scale bytes: nbits bits starting at bit `lo` of
 * byte `byte`. */
static int bits_of(const uint8_t *s, int byte, int lo, int nbits) {
    return (s[byte] >> lo) & ((1 << nbits) - 1);
}

/* Per-element closed form of the same decode, written independently of the
 * loop above: element i sits in sub-block j = i/32, in the qs byte
 * 32*(i/64) + i%32, low nibble when (i/32) is even, high nibble when odd. */
double orc_q4k_elem(const uint8_t *b, int i) {
    int j = i / 32;
    int byte = 16 + 32 * (i / 64) + (i % 32);
    int q = (j % 2 == 0) ? (b[byte] & 0x0F) : (b[byte] >> 4);
    const uint8_t *s = b + 4;
    int sc, m;
    if (j < 4) {
        sc = bits_of(s, j, 0, 6);
        m = bits_of(s, j + 4, 0, 6);
    } else {
        sc = bits_of(s, j + 4, 0, 4) + 16 * bits_of(s, j - 4, 6, 2);
        m = bits_of(s, j + 4, 4, 4) + 16 * bits_of(s, j, 6, 2);
    }
    double d = orc_f16_to_f64(rd_le16(b));
    double dmin = orc_f16_to_f64(rd_le16(b + 2));
    return d * sc * q - dmin * m;
}

/* ---------------------------------------------------------------- Q6_K -- */

/* Loop-structured decode: two 128-weight halves; in half H the 32 positions
 * l of ql[64H..], ql[64H+32..] and qh[32H..] give four weights each. */
void orc_q6k_block_decode(const uint8_t *b, double *out) {
    const uint8_t *ql = b;
    const uint8_t *qh = b + 128;
    const int8_t *sc = (const int8_t *)(b + 192);
    double d = orc_f16_to_f64(rd_le16(b + 208));
    for (int H = 0; H < 2; H++) {
        for (int l = 0; l < 32; l++) {
            int g = l / 16;
            int q0 = (ql[64 * H + l] & 15) | (((qh[32 * H + l] >> 0) & 3) << 4);
            int q1 = (ql[64 * H + l + 32] & 15) | (((qh[32 * H + l] >> 2) & 3) << 4);
            int q2 = (ql[64 * H + l] >> 4) | (((qh[32 * H + l] >> 4) & 3) << 4);
            int q3 = (ql[64 * H + l + 32] >> 4) | (((qh[32 * H + l] >> 6) & 3) << 4);
            out[128 * H + l] = d * sc[8 * H + g + 0] * (q0 - 32);
            out[128 * H + l + 32] = d * sc[8 * H + g + 2] * (q1 - 32);
            out[128 * H + l + 64] = d * sc[8 * H + g + 4] * (q2 - 32);
            out[128 * H + l + 96] = d * sc[8 * H + g + 6] * (q3 - 32);
        }
    }
}

/* Per-element closed form: element i -> half H = i/128, quarter qd = (i%128)/32,
 * position l = i%32; low 4 bits from the low (qd < 2) or high (qd >= 2) nibble
 * of ql[64H + 32*(qd%2) + l], high 2 bits from bits 2*qd..2*qd+1 of qh[32H + l],
 * scale index 8H + 2*qd + l/16. */
double orc_q6k_elem(const uint8_t *b, int i) {
    int H = i / 128, qd = (i % 128) / 32, l = i % 32;
    int qlb = b[64 * H + 32 * (qd % 2) + l];
    int lo4 = (qd < 2) ? (qlb & 0x0F) : ((qlb >> 4) & 0x0F);
    int hi2 = (b[128 + 32 * H + l] >> (2 * qd)) & 3;
    int q = lo4 + 16 * hi2;
    int scale = (int)(int8_t)b[192 + 8 * H + 2 * qd + l / 16];
    return orc_f16_to_f64(rd_le16(b + 208)) * scale * (q - 32);
}

/* ---------------------------------------------------------------- Q8_0 -- */

void orc_q8_0_block_decode(const uint8_t *b, double *out) {
    double d = orc_f16_to_f64(rd_le16(b));
    for (int i = 0; i < 32; i++) out[i] = d * (double)(int8_t)b[2 + i];
}

double orc_q8_0_elem(const uint8_t *b, int i) {
    return orc_f16_to_f64(rd_le16(b)) * (double)(int8_t)b[2 + i];
}

/* ---------------------------------------------------------------- Q4_0 -- */

/* Loop-structured decode: byte l of qs carries weight l in its low nibble and
 * weight l+16 in its high nibble. */
void orc_q4_0_block_decode(const uint8_t *b, double *out) {
    double d = orc_f16_to_f64(rd_le16(b));
    for (int l = 0; l < 16; l++) {
        out[l] = d * ((b[2 + l] & 15) - 8);
        out[l + 16] = d * ((b[2 + l] >> 4) - 8);
    }
}

/* Per-element closed form: code = bits 4*(i/16)..4*(i/16)+3 of byte i%16. */
double orc_q4_0_elem(const uint8_t *b, int i) {
    int q = (b[2 + i % 16] >> (4 * (i / 16))) & 0x0F;
    return orc_f16_to_f64(rd_le16(b)) * (q - 8);
}

/* ---------------------------------------------------------------- Q5_K -- */

/* Loop-structured decode: four 64-weight chunks as in Q4_K; in chunk c the 32
 * qh bytes give the fifth bit of the low-nibble weights in bit 2c and of the
 * high-nibble weights in bit 2c+1. Scales and mins use Q4_K's packing. */
void orc_q5k_block_decode(const uint8_t *b, double *out) {
    double d = orc_f16_to_f64(rd_le16(b));
    double dmin = orc_f16_to_f64(rd_le16(b + 2));
    const uint8_t *s = b + 4;
    const uint8_t *qh = b + 16;
    const uint8_t *qs = b + 48;
    for (int c = 0; c < 4; c++) {
        int sc0, m0, sc1, m1;
        q4k_scale_min(2 * c, s, &sc0, &m0);
        q4k_scale_min(2 * c + 1, s, &sc1, &m1);
        for (int l = 0; l < 32; l++) {
            int lo = (qs[32 * c + l] & 15) + (((qh[l] >> (2 * c)) & 1) ? 16 : 0);
            int hi = (qs[32 * c + l] >> 4) + (((qh[l] >> (2 * c + 1)) & 1) ? 16 : 0);
            out[64 * c + l] = d * sc0 * lo - dmin * m0;
            out[64 * c + 32 + l] = d * sc1 * hi - dmin * m1;
        }
    }
}

/* Per-element closed form, written apart from the loop above: sub-block
 * j = i/32; low 4 bits as Q4_K's element i (qs at byte 48 instead of 16); the
 * fifth bit is bit j of qh[i%32]; scale and min read with bits_of(). */
double orc_q5k_elem(const uint8_t *b, int i) {
    int j = i / 32;
    int byte = 48 + 32 * (i / 64) + (i % 32);
    int q = ((j % 2 == 0) ? (b[byte] & 0x0F) : (b[byte] >> 4)) + 16 * ((b[16 + i % 32] >> j) & 1);
    const uint8_t *s = b + 4;
    int sc, m;
    if (j < 4) {
        sc = bits_of(s, j, 0, 6);
        m = bits_of(s, j + 4, 0, 6);
    } else {
        sc = bits_of(s, j + 4, 0, 4) + 16 * bits_of(s, j - 4, 6, 2);
        m = bits_of(s, j + 4, 4, 4) + 16 * bits_of(s, j, 6, 2);
    }
    double d = orc_f16_to_f64(rd_le16(b));
    double dmin = orc_f16_to_f64(rd_le16(b + 2));
    return d * sc * q - dmin * m;
}

/* ----------------------------------------------------- row dequant + matvec */

/* fmt: 0 = Q4_K, 1 = Q6_K, 2 = Q8_0, 3 = Q4_0, 4 = Q5_K. Returns the block
 * geometry. */
static int fmt_geom(int fmt, int *qk, int *bb) {
    switch (fmt) {
    case 0: *qk = ORC_QK_K; *bb = ORC_Q4K_BYTES; return 0;
    case 1: *qk = ORC_QK_K; *bb = ORC_Q6K_BYTES; return 0;
    case 2: *qk = ORC_QK8_0; *bb = ORC_Q8_0_BYTES; return 0;
    case 3: *qk = ORC_QK8_0; *bb = ORC_Q4_0_BYTES; return 0;
    case 4: *qk = ORC_QK_K; *bb = ORC_Q5K_BYTES; return 0;
    default: return -1;
    }
}

static void decode_block(int fmt, const uint8_t *b, double *out) {
    switch (fmt) {
    case 0: orc_q4k_block_decode(b, out); break;
    case 1: orc_q6k_block_decode(b, out); break;
    case 2: orc_q8_0_block_decode(b, out); break;
    case 3: orc_q4_0_block_decode(b, out); break;
    default: orc_q5k_block_decode(b, out); break;
    }
}

/* Exact decoded weights of `rows` packed rows into out[rows*k] (f64). */
int orc_dequant(int fmt, const uint8_t *w, long rows, long k, double *out) {
    int qk, bb;
    if (fmt_geom(fmt, &qk, &bb) || k % qk) return -1;
    long nb = k / qk;
    for (long r = 0; r < rows; r++)
        for (long b = 0; b < nb; b++)
            decode_block(fmt, w + (r * nb + b) * bb, out + r * k + b * qk);
    return 0;
}

/* y[r] = sum_j W[r, j] * x[j]: every block decoded to its exact value, the dot
 * accumulated in f64 in index order. */
int orc_qmv(int fmt, const uint8_t *w, const float *x, long rows, long k, double *y) {
    int qk, bb;
    double blk[ORC_QK_K];
    if (fmt_geom(fmt, &qk, &bb) || k % qk) return -1;
    long nb = k / qk;
    for (long r = 0; r < rows; r++) {
        double acc = 0.0;
        for (long b = 0; b < nb; b++) {
            decode_block(fmt, w + (r * nb + b) * bb, blk);
            for (int i = 0; i < qk; i++) acc += blk[i] * (double)x[b * qk + i];
        }
        y[r] = acc;
    }
    return 0;
}

/* ----------------------------------------------- Q6_K x int8 activation */

/* Code minus 32 of element i of a Q6_K block (the layout of
 * orc_q6k_block_decode: half H = i/128, quarter qd = (i%128)/32, l = i%32). */
static int q6k_code(const uint8_t *b, int i) {
    int H = i / 128, qd = (i % 128) / 32, l = i % 32;
    int qlb = b[64 * H + 32 * (qd % 2) + l];
    int lo4 = (qd < 2) ? (qlb & 15) : (qlb >> 4);
    int hi2 = (b[128 + 32 * H + l] >> (2 * qd)) & 3;
    return lo4 + 16 * hi2 - 32;
}

/* dots[r, g] = sum over the 16 weights of scale group g of row r (elements
 * 16g .. 16g+15; the group of element i of a block is i/16, the index of its
 * scale) of (q - 32) * xq: the integer dots of the Q6_K dp4a decode
 * (hanzo-ml src/vulkan_backend.rs, `moe_matvec_q6k_dp4a_blk_dn`, which folds
 * the -32 against sums of the activation codes). */
int orc_q6k_dp4a_groupdots(const uint8_t *w, const int8_t *xq, long rows, long k, int32_t *dots) {
    if (k % ORC_QK_K) return -1;
    long nb = k / ORC_QK_K;
    for (long r = 0; r < rows; r++)
        for (long bi = 0; bi < nb; bi++) {
            const uint8_t *b = w + (r * nb + bi) * ORC_Q6K_BYTES;
            for (int g = 0; g < 16; g++) {
                long dot = 0;
                for (int t = 0; t < 16; t++)
                    dot += (long)q6k_code(b, 16 * g + t) * (long)xq[bi * 256 + 16 * g + t];
                dots[r * (k / 16) + bi * 16 + g] = (int32_t)dot;
            }
        }
    return 0;
}

/* y[r] = sum over 16-groups g of d * scale_g * xs[g/2] * dot_g in f64: the
 * Q6_K weights against the dequantized activation xs * xq. */
int orc_qmv_q6k_dp4a(const uint8_t *w, const int8_t *xq, const float *xs, long rows, long k, double *y) {
    if (k % ORC_QK_K) return -1;
    long nb = k / ORC_QK_K;
    for (long r = 0; r < rows; r++) {
        double acc = 0.0;
        for (long bi = 0; bi < nb; bi++) {
            const uint8_t *b = w + (r * nb + bi) * ORC_Q6K_BYTES;
            double d = orc_f16_to_f64(rd_le16(b + 208));
            for (int g = 0; g < 16; g++) {
                long dot = 0;
                for (int t = 0; t < 16; t++)
                    dot += (long)q6k_code(b, 16 * g + t) * (long)xq[bi * 256 + 16 * g + t];
                double scale = (double)(int8_t)b[192 + g];
                acc += d * scale * (double)xs[(bi * 256 + 16 * g) / 32] * (double)dot;
            }
        }
        y[r] = acc;
    }
    return 0;
}

/* MoE on the Q6_K dp4a path: slot s multiplies expert ids[s] of the
 * [E, rows, k] bank with its own codes xq[s, :] and scales xs[s, :]; NaN for
 * ids outside [0, n_experts). */
int orc_moe_qmv_q6k_dp4a(const uint8_t *bank, const int8_t *xq, const float *xs, const int32_t *ids,
                         long slots, long rows, long k, long n_experts, double *y) {
    if (k % ORC_QK_K) return -1;
    long rb = (k / ORC_QK_K) * ORC_Q6K_BYTES;
    for (long s = 0; s < slots; s++) {
        long e = ids[s];
        if (e < 0 || e >= n_experts) {
            for (long r = 0; r < rows; r++) y[s * rows + r] = NAN;
            continue;
        }
        orc_qmv_q6k_dp4a(bank + e * rows * rb, xq + s * k, xs + s * (k / 32), rows, k, y + s * rows);
    }
    return 0;
}

/* Small-M batch (hanzo-ml src/vulkan_backend.rs, the `matmul_q*_gpu`
 * prefill products): y[i, r] = sum_j W[r, j] * x[i, j] for the m rows of
 * x[m, k] (row-major), output y[m, rows] row-major. Each block is decoded to
 * its exact value once and used for every row of x; each dot accumulates in
 * f64 in index order. */
int orc_qmm(int fmt, const uint8_t *w, const float *x, long m, long rows, long k, double *y) {
    int qk, bb;
    double blk[ORC_QK_K];
    if (fmt_geom(fmt, &qk, &bb) || k % qk || m < 1) return -1;
    long nb = k / qk;
    for (long i = 0; i < m * rows; i++) y[i] = 0.0;
    for (long r = 0; r < rows; r++) {
        for (long b = 0; b < nb; b++) {
            decode_block(fmt, w + (r * nb + b) * bb, blk);
            for (long i = 0; i < m; i++) {
                double acc = y[i * rows + r];
                for (int t = 0; t < qk; t++) acc += blk[t] * (double)x[i * k + b * qk + t];
                y[i * rows + r] = acc;
            }
        }
    }
    return 0;
}

/* MoE: y[s, r] = dense matvec of expert ids[s] (rows r of bank slice
 * [ids[s]*rows, (ids[s]+1)*rows)) with x[s, :]. A slot whose id is outside
 * [0, n_experts) gets NaN in every output (the CUDA path's contract). */
int orc_moe_qmv(int fmt, const uint8_t *bank, const float *x, const int32_t *ids,
                long slots, long rows, long k, long n_experts, double *y) {
    int qk, bb;
    if (fmt_geom(fmt, &qk, &bb) || k % qk) return -1;
    long rb = (k / qk) * bb;
    for (long s = 0; s < slots; s++) {
        long e = ids[s];
        if (e < 0 || e >= n_experts) {
            for (long r = 0; r < rows; r++) y[s * rows + r] = NAN;
            continue;
        }
        orc_qmv(fmt, bank + e * rows * rb, x + s * k, rows, k, y + s * rows);
    }
    return 0;
}

/* ------------------------------------------------ activation quantization */

/* Per 32-block of x[m, k]: amax = max |x|; inv = 127/amax and d = amax/127 as
 * IEEE f32 divides; q = clamp(rne(x * inv), -127, 127) with one f32 multiply;
 * amax == 0 gives d = 0 and q = 0. xsum (optional) = d * (sum of q) as one f32
 * multiply of an exact integer sum. */
int orc_quantize_act_q8(const float *x, long m, long k, int8_t *xq, float *xs, float *xsum) {
    if (k % ORC_QK8_0) return -1;
    long nb = m * k / ORC_QK8_0;
    for (long b = 0; b < nb; b++) {
        const float *xb = x + b * ORC_QK8_0;
        float amax = 0.0f;
        for (int i = 0; i < ORC_QK8_0; i++) {
            float a = fabsf(xb[i]);
            if (a > amax) amax = a;
        }
        int sum = 0;
        if (amax == 0.0f) {
            for (int i = 0; i < ORC_QK8_0; i++) xq[b * ORC_QK8_0 + i] = 0;
            xs[b] = 0.0f;
        } else {
            volatile float inv = 127.0f / amax;
            for (int i = 0; i < ORC_QK8_0; i++) {
                volatile float v = xb[i] * inv;
                float r = rintf(v);
                if (r > 127.0f) r = 127.0f;
                if (r < -127.0f) r = -127.0f;
                xq[b * ORC_QK8_0 + i] = (int8_t)r;
                sum += (int)r;
            }
            volatile float d = amax / 127.0f;
            xs[b] = d;
        }
        if (xsum) {
            volatile float t = xs[b] * (float)sum;
            xsum[b] = t;
        }
    }
    return 0;
}

/* Exact int32 dot of every Q8_0 weight block with the matching 32 int8
 * activation codes: dots[r, b] = sum_t q_w[r, 32b + t] * xq[32b + t]. */
int orc_q8_blockdots(const uint8_t *w, const int8_t *xq, long rows, long k, int32_t *dots) {
    if (k % ORC_QK8_0) return -1;
    long nb = k / ORC_QK8_0;
    for (long r = 0; r < rows; r++)
        for (long b = 0; b < nb; b++) {
            const uint8_t *blk = w + (r * nb + b) * ORC_Q8_0_BYTES;
            int32_t acc = 0;
            for (int t = 0; t < ORC_QK8_0; t++)
                acc += (int32_t)(int8_t)blk[2 + t] * (int32_t)xq[b * ORC_QK8_0 + t];
            dots[r * nb + b] = acc;
        }
    return 0;
}

/* dp4a-path matvec: y[r] = sum_b d_w[r, b] * d_x[b] * dot[r, b], in f64. */
int orc_qmv_q8_dp4a(const uint8_t *w, const int8_t *xq, const float *xs, long rows, long k,
                    double *y) {
    if (k % ORC_QK8_0) return -1;
    long nb = k / ORC_QK8_0;
    for (long r = 0; r < rows; r++) {
        double acc = 0.0;
        for (long b = 0; b < nb; b++) {
            const uint8_t *blk = w + (r * nb + b) * ORC_Q8_0_BYTES;
            long dot = 0;
            for (int t = 0; t < ORC_QK8_0; t++)
                dot += (long)(int8_t)blk[2 + t] * (long)xq[b * ORC_QK8_0 + t];
            acc += orc_f16_to_f64(rd_le16(blk)) * (double)xs[b] * (double)dot;
        }
        y[r] = acc;
    }
    return 0;
}

/* ------------------------------------------- Q4_K x q8 activation (dp4a) -- */

/* The dense dp4a Q4_K matvec of hanzo-ml src/vulkan_backend.rs (the
 * `matvec_q4k_dp4a_blk` dispatch in the decode path): the activation is
 * quantized to int8 codes with one f32 scale per 32 values (quantize_act_q8),
 * and every 32-weight Q4_K sub-block is dotted, as integers, with the 32 codes
 * of the same positions. One sub-block's exact integer dot of its 4-bit codes
 * with the activation codes: */
static long q4k_subblock_dot(const uint8_t *b, int j, const int8_t *xq32) {
    const uint8_t *qs = b + 16 + 32 * (j / 2);
    long dot = 0;
    for (int l = 0; l < 32; l++) {
        int q = (j % 2 == 0) ? (qs[l] & 15) : (qs[l] >> 4);
        dot += (long)q * (long)xq32[l];
    }
    return dot;
}

/* dots[r, t] = integer dot of the 32-weight sub-block t of row r (t = 8 *
 * block + j) with xq[32t .. 32t + 31]. */
int orc_q4k_dp4a_blockdots(const uint8_t *w, const int8_t *xq, long rows, long k, int32_t *dots) {
    if (k % ORC_QK_K) return -1;
    long nb = k / ORC_QK_K;
    for (long r = 0; r < rows; r++)
        for (long bi = 0; bi < nb; bi++) {
            const uint8_t *b = w + (r * nb + bi) * ORC_Q4K_BYTES;
            for (int j = 0; j < 8; j++) {
                long t = bi * 8 + j;
                dots[r * (k / 32) + t] = (int32_t)q4k_subblock_dot(b, j, xq + 32 * t);
            }
        }
    return 0;
}

/* y[r] = sum over sub-blocks t of  xs[t] * (d*sc_j*dot_t - dmin*m_j*sumq_t),
 * with sumq_t the integer sum of the activation codes of sub-block t: the
 * weights w = d*sc*q - dmin*m against the dequantized activation xs*xq, in f64
 * with exact integer dots. */
int orc_qmv_q4k_dp4a(const uint8_t *w, const int8_t *xq, const float *xs, long rows, long k, double *y) {
    if (k % ORC_QK_K) return -1;
    long nb = k / ORC_QK_K;
    for (long r = 0; r < rows; r++) {
        double acc = 0.0;
        for (long bi = 0; bi < nb; bi++) {
            const uint8_t *b = w + (r * nb + bi) * ORC_Q4K_BYTES;
            double d = orc_f16_to_f64(rd_le16(b));
            double dmin = orc_f16_to_f64(rd_le16(b + 2));
            for (int j = 0; j < 8; j++) {
                long t = bi * 8 + j;
                int sc, m;
                q4k_scale_min(j, b + 4, &sc, &m);
                long dot = q4k_subblock_dot(b, j, xq + 32 * t);
                long sumq = 0;
                for (int l = 0; l < 32; l++) sumq += xq[32 * t + l];
                acc += (double)xs[t] * (d * sc * (double)dot - dmin * m * (double)sumq);
            }
        }
        y[r] = acc;
    }
    return 0;
}

/* MoE on the Q4_K dp4a path (hanzo-ml src/vulkan_backend.rs,
 * `moe_matvec_q4k_dp4a_blk_*`: the routed token's activation quantized once,
 * the experts' Q4_K codes dotted with it): slot s multiplies expert ids[s] of
 * the [E, rows, k] bank with its own codes xq[s, :] and scales xs[s, :]. A slot
 * whose id is outside [0, n_experts) gets NaN in every output. */
int orc_moe_qmv_q4k_dp4a(const uint8_t *bank, const int8_t *xq, const float *xs, const int32_t *ids,
                         long slots, long rows, long k, long n_experts, double *y) {
    if (k % ORC_QK_K) return -1;
    long rb = (k / ORC_QK_K) * ORC_Q4K_BYTES;
    for (long s = 0; s < slots; s++) {
        long e = ids[s];
        if (e < 0 || e >= n_experts) {
            for (long r = 0; r < rows; r++) y[s * rows + r] = NAN;
            continue;
        }
        orc_qmv_q4k_dp4a(bank + e * rows * rb, xq + s * k, xs + s * (k / 32), rows, k, y + s * rows);
    }
    return 0;
}
