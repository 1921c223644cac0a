// qmv_q4k.cu -- Q4_K dense and MoE matvec launches, and the Q4_K dequantizer
// used by the tests.
#include "qmv_internal.h"
#include "qmv_launch.cuh"

namespace {

using namespace qmv;

// One thread per (row, block, sub-block j): the 32 weights of sub-block j are
// d*sc_j*q - dmin*m_j, formed as one fma of exact operands (d*sc_j and
// dmin*m_j are exact in f32), i.e. the round-to-nearest f32 of the exact value.
__global__ void dequant_q4k_kernel(const uint8_t* __restrict__ w, float* __restrict__ out, long long nsub,
                                   int nb) {
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < nsub;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int j = static_cast<int>(idx & 7);
        const long long blk = idx >> 3;
        const uint8_t* p = w + blk * 144;
        const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(p[0] | (p[1] << 8))));
        const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(p[2] | (p[3] << 8))));
        const uint8_t* s = p + 4;
        int sc, m;
        if (j < 4) {
            sc = s[j] & 63;
            m = s[j + 4] & 63;
        } else {
            sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
            m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
        }
        const float a = d * static_cast<float>(sc);
        const float c = -(dmin * static_cast<float>(m));
        const uint8_t* qs = p + 16 + 32 * (j >> 1);
        float* o = out + blk * 256 + 32 * j;   // rows are contiguous: block blk of the matrix
        for (int l = 0; l < 32; l++) {
            const int q = (j & 1) ? (qs[l] >> 4) : (qs[l] & 15);
            o[l] = __fmaf_rn(a, static_cast<float>(q), c);
        }
    }
    (void)nb;
}

}  // namespace

namespace qmvi {

using namespace qmv;

int q4k(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg, cudaStream_t s,
        int force_timeout) {
    KParams kp{};
    kp.force_timeout = force_timeout;
    kp.w = static_cast<const uint8_t*>(w);
    kp.x = x;
    kp.y = y;
    kp.rows = rows;
    kp.k = k;
    kp.nb = k / 256;
    kp.rowbytes = static_cast<uint32_t>(kp.nb) * 144u;
    kp.matbytes = static_cast<unsigned long long>(rows) * kp.rowbytes;
    kp.wbytes = kp.matbytes;
    Plan pl;
    int rc = make_plan<Q4K>(rows, k, 1, cfg, &kp, &pl);
    if (rc) return rc;
    return launch<Q4K, false, MODE_MATVEC>(kp, pl, 1, s);
}

int moe_q4k(const void* bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
            int n_experts, const qmv_opts* cfg, cudaStream_t s) {
    KParams kp{};
    kp.w = static_cast<const uint8_t*>(bank);
    kp.x = x;
    kp.y = y;
    kp.ids = ids;
    kp.n_experts = n_experts;
    kp.rows = rows;
    kp.k = k;
    kp.nb = k / 256;
    kp.rowbytes = static_cast<uint32_t>(kp.nb) * 144u;
    kp.matbytes = static_cast<unsigned long long>(rows) * kp.rowbytes;
    kp.wbytes = static_cast<unsigned long long>(n_experts) * kp.matbytes;
    Plan pl;
    int rc = make_plan<Q4K>(rows, k, slots, cfg, &kp, &pl);
    if (rc) return rc;
    return launch<Q4K, true, MODE_MATVEC>(kp, pl, slots, s);
}

int q4k_dp4a(const void* w, const int8_t* xq, const float* xs, float* y, int rows, int k, const qmv_opts* cfg,
             cudaStream_t s) {
    KParams kp{};
    kp.w = static_cast<const uint8_t*>(w);
    kp.xq = xq;
    kp.xqs = xs;
    kp.y = y;
    kp.rows = rows;
    kp.k = k;
    kp.nb = k / 256;
    kp.rowbytes = static_cast<uint32_t>(kp.nb) * 144u;
    kp.matbytes = static_cast<unsigned long long>(rows) * kp.rowbytes;
    kp.wbytes = kp.matbytes;
    Plan pl;
    int rc = make_plan<Q4D>(rows, k, 1, cfg, &kp, &pl);
    if (rc) return rc;
    return launch<Q4D, false, MODE_MATVEC>(kp, pl, 1, s);
}

int q4k_dp4a_blockdots(const void* w, const int8_t* xq, int32_t* dots, int rows, int k, cudaStream_t s) {
    KParams kp{};
    kp.w = static_cast<const uint8_t*>(w);
    kp.xq = xq;
    kp.dots = dots;
    kp.rows = rows;
    kp.k = k;
    kp.nb = k / 256;
    kp.rowbytes = static_cast<uint32_t>(kp.nb) * 144u;
    kp.matbytes = static_cast<unsigned long long>(rows) * kp.rowbytes;
    kp.wbytes = kp.matbytes;
    Plan pl;
    int rc = make_plan<Q4D>(rows, k, 1, nullptr, &kp, &pl);
    if (rc) return rc;
    return launch<Q4D, false, MODE_BLOCKDOTS>(kp, pl, 1, s);
}

int moe_q4k_dp4a(const void* bank, const int8_t* xq, const float* xs, float* y, int rows, int k, const int32_t* ids,
                 int slots, int n_experts, const qmv_opts* cfg, cudaStream_t s) {
    KParams kp{};
    kp.w = static_cast<const uint8_t*>(bank);
    kp.xq = xq;
    kp.xqs = xs;
    kp.y = y;
    kp.ids = ids;
    kp.n_experts = n_experts;
    kp.rows = rows;
    kp.k = k;
    kp.nb = k / 256;
    kp.rowbytes = static_cast<uint32_t>(kp.nb) * 144u;
    kp.matbytes = static_cast<unsigned long long>(rows) * kp.rowbytes;
    kp.wbytes = static_cast<unsigned long long>(n_experts) * kp.matbytes;
    Plan pl;
    int rc = make_plan<Q4D>(rows, k, slots, cfg, &kp, &pl);
    if (rc) return rc;
    return launch<Q4D, true, MODE_MATVEC>(kp, pl, slots, s);
}

int dequant_q4k(const void* w, float* out, int rows, int k, cudaStream_t s) {
    const long long nsub = static_cast<long long>(rows) * (k / 256) * 8;
    const int threads = 256;
    const long long want = (nsub + threads - 1) / threads;
    const int blocks = static_cast<int>(want < 65536 ? want : 65536);
    dequant_q4k_kernel<<<blocks, threads, 0, s>>>(static_cast<const uint8_t*>(w), out, nsub, k / 256);
    return cuda_rc(cudaGetLastError());
}

int status_q4k(unsigned int* out, int clear) { return status_rw(out, clear); }

}  // namespace qmvi
