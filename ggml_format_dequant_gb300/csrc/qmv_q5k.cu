// qmv_q5k.cu -- Q5_K dense and MoE matvec launches, the small-M batched
// product, and the Q5_K dequantizer used by the tests.
#include "qmv_internal.h"
#include "qmv_launch.cuh"
#include "qmm_tc.cuh"

namespace {

using namespace qmv;

// One thread per (row, block, sub-block j): weight l of sub-block j is
// d*sc_j*q - dmin*m_j with q = nibble + 16 * (bit j of qh[l]), formed as one
// fma of exact operands (d*sc_j and dmin*m_j are exact in f32), i.e. the
// round-to-nearest f32 of the exact value.
__global__ void dequant_q5k_kernel(const uint8_t* __restrict__ w, float* __restrict__ out, long long nsub) {
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < nsub;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int j = static_cast<int>(idx & 7);
        const long long blk = idx >> 3;
        const uint8_t* p = w + blk * 176;
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
        const uint8_t* qh = p + 16;
        const uint8_t* qs = p + 48 + 32 * (j >> 1);
        float* o = out + blk * 256 + 32 * j;
        for (int l = 0; l < 32; l++) {
            const int q = ((j & 1) ? (qs[l] >> 4) : (qs[l] & 15)) | (((qh[l] >> j) & 1) << 4);
            o[l] = __fmaf_rn(a, static_cast<float>(q), c);
        }
    }
}

KParams q5k_params(const void* w, int rows, int k) {
    KParams kp{};
    kp.w = static_cast<const uint8_t*>(w);
    kp.rows = rows;
    kp.k = k;
    kp.nb = k / 256;
    kp.rowbytes = static_cast<uint32_t>(kp.nb) * 176u;
    kp.matbytes = static_cast<unsigned long long>(rows) * kp.rowbytes;
    kp.wbytes = kp.matbytes;
    return kp;
}

}  // namespace

namespace qmvi {

using namespace qmv;

int q5k(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg, cudaStream_t s) {
    KParams kp = q5k_params(w, rows, k);
    kp.x = x;
    kp.y = y;
    Plan pl;
    int rc = make_plan<Q5K>(rows, k, 1, cfg, &kp, &pl);
    if (rc) return rc;
    return launch<Q5K, false, MODE_MATVEC>(kp, pl, 1, s);
}

int moe_q5k(const void* bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
            int n_experts, const qmv_opts* cfg, cudaStream_t s) {
    KParams kp = q5k_params(bank, rows, k);
    kp.x = x;
    kp.y = y;
    kp.ids = ids;
    kp.n_experts = n_experts;
    kp.wbytes = static_cast<unsigned long long>(n_experts) * kp.matbytes;
    Plan pl;
    int rc = make_plan<Q5K>(rows, k, slots, cfg, &kp, &pl);
    if (rc) return rc;
    return launch<Q5K, true, MODE_MATVEC>(kp, pl, slots, s);
}

int dequant_q5k(const void* w, float* out, int rows, int k, cudaStream_t s) {
    const long long nsub = static_cast<long long>(rows) * (k / 256) * 8;
    const int threads = 256;
    const long long want = (nsub + threads - 1) / threads;
    const int blocks = static_cast<int>(want < 65536 ? want : 65536);
    dequant_q5k_kernel<<<blocks, threads, 0, s>>>(static_cast<const uint8_t*>(w), out, nsub);
    return cuda_rc(cudaGetLastError());
}

// Small-M batched product y[m, rows] = x[m, k] W^T, m >= 2: the
// tensor-core kernel of qmm_tc.cuh, one launch per tile of up to 8 rows of x.
int qmm_q5k(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg, cudaStream_t s) {
    return qmm_tc_run<Q5KT>(w, x, y, rows, k, m, cfg, s);
}

int status_q5k(unsigned int* out, int clear) { return status_rw(out, clear); }

}  // namespace qmvi
