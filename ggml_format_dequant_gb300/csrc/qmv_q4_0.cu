// qmv_q4_0.cu -- Q4_0 dense and MoE matvec launches, the small-M batched
// product, and the Q4_0 dequantizer used by the tests.
#include "qmv_internal.h"
#include "qmv_launch.cuh"
#include "qmm_tc.cuh"

namespace {

using namespace qmv;

// One thread per (row, block): weight i is d*(q - 8), exact in f32, with q
// the low nibble of byte i (i < 16) or the high nibble of byte i - 16.
__global__ void dequant_q4_0_kernel(const uint8_t* __restrict__ w, float* __restrict__ out, long long nblk) {
    for (long long blk = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; blk < nblk;
         blk += static_cast<long long>(gridDim.x) * blockDim.x) {
        const uint8_t* p = w + blk * 18;
        const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(p[0] | (p[1] << 8))));
        for (int l = 0; l < 16; l++) {
            out[blk * 32 + l] = __fmul_rn(d, static_cast<float>((p[2 + l] & 15) - 8));
            out[blk * 32 + 16 + l] = __fmul_rn(d, static_cast<float>((p[2 + l] >> 4) - 8));
        }
    }
}

KParams q4_0_params(const void* w, int rows, int k) {
    KParams kp{};
    kp.w = static_cast<const uint8_t*>(w);
    kp.rows = rows;
    kp.k = k;
    kp.nb = k / 32;
    kp.rowbytes = static_cast<uint32_t>(kp.nb) * 18u;
    kp.matbytes = static_cast<unsigned long long>(rows) * kp.rowbytes;
    kp.wbytes = kp.matbytes;
    return kp;
}

}  // namespace

namespace qmvi {

using namespace qmv;

int q4_0(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg, cudaStream_t s) {
    KParams kp = q4_0_params(w, rows, k);
    kp.x = x;
    kp.y = y;
    Plan pl;
    int rc = make_plan<Q40>(rows, k, 1, cfg, &kp, &pl);
    if (rc) return rc;
    return launch<Q40, false, MODE_MATVEC>(kp, pl, 1, s);
}

int moe_q4_0(const void* bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
             int n_experts, const qmv_opts* cfg, cudaStream_t s) {
    KParams kp = q4_0_params(bank, rows, k);
    kp.x = x;
    kp.y = y;
    kp.ids = ids;
    kp.n_experts = n_experts;
    kp.wbytes = static_cast<unsigned long long>(n_experts) * kp.matbytes;
    Plan pl;
    int rc = make_plan<Q40>(rows, k, slots, cfg, &kp, &pl);
    if (rc) return rc;
    return launch<Q40, true, MODE_MATVEC>(kp, pl, slots, s);
}

int dequant_q4_0(const void* w, float* out, int rows, int k, cudaStream_t s) {
    const long long nblk = static_cast<long long>(rows) * (k / 32);
    const int threads = 256;
    const long long want = (nblk + threads - 1) / threads;
    const int blocks = static_cast<int>(want < 65536 ? (want > 0 ? want : 1) : 65536);
    dequant_q4_0_kernel<<<blocks, threads, 0, s>>>(static_cast<const uint8_t*>(w), out, nblk);
    return cuda_rc(cudaGetLastError());
}

// Small-M batched product y[m, rows] = x[m, k] W^T, m >= 2: the
// tensor-core kernel of qmm_tc.cuh, one launch per tile of up to 8 rows of x.
int qmm_q4_0(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg, cudaStream_t s) {
    return qmm_tc_run<Q40T>(w, x, y, rows, k, m, cfg, s);
}

int status_q4_0(unsigned int* out, int clear) { return status_rw(out, clear); }

}  // namespace qmvi
