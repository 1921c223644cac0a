// qmv_q6k.cu -- Q6_K dense and MoE matvec launches (f32 activation and the
// int8-activation dp4a path), the dp4a group dots and the Q6_K dequantizer
// used by the tests.
#include "qmv_internal.h"
#include "qmv_launch.cuh"

namespace {

using namespace qmv;

// One thread per (row, block, 16-weight scale group gi): weight i = 16*gi + t
// sits in half H = i/128, quarter qd = (i%128)/32, position l = i%32, and
// d*scale*(q - 32) is exact in f32 (d*scale has at most 18 significant bits).
__global__ void dequant_q6k_kernel(const uint8_t* __restrict__ w, float* __restrict__ out, long long ngroups) {
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < ngroups;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int gi = static_cast<int>(idx & 15);
        const long long blk = idx >> 4;
        const uint8_t* p = w + blk * 210;
        const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(p[208] | (p[209] << 8))));
        const float ds = d * static_cast<float>(static_cast<int8_t>(p[192 + gi]));
        float* o = out + blk * 256;
        for (int t = 0; t < 16; t++) {
            const int i = 16 * gi + t;
            const int H = i >> 7, qd = (i & 127) >> 5, l = i & 31;
            const int qlb = p[64 * H + 32 * (qd & 1) + l];
            const int lo4 = (qd < 2) ? (qlb & 15) : (qlb >> 4);
            const int hi2 = (p[128 + 32 * H + l] >> (2 * qd)) & 3;
            o[i] = __fmul_rn(ds, static_cast<float>((lo4 | (hi2 << 4)) - 32));
        }
    }
}

}  // namespace

namespace qmvi {

using namespace qmv;

int q6k(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg, cudaStream_t s) {
    KParams kp{};
    kp.w = static_cast<const uint8_t*>(w);
    kp.x = x;
    kp.y = y;
    kp.rows = rows;
    kp.k = k;
    kp.nb = k / 256;
    kp.rowbytes = static_cast<uint32_t>(kp.nb) * 210u;
    kp.matbytes = static_cast<unsigned long long>(rows) * kp.rowbytes;
    kp.wbytes = kp.matbytes;
    Plan pl;
    int rc = make_plan<Q6K>(rows, k, 1, cfg, &kp, &pl);
    if (rc) return rc;
    return launch<Q6K, false, MODE_MATVEC>(kp, pl, 1, s);
}

int moe_q6k(const void* bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
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
    kp.rowbytes = static_cast<uint32_t>(kp.nb) * 210u;
    kp.matbytes = static_cast<unsigned long long>(rows) * kp.rowbytes;
    kp.wbytes = static_cast<unsigned long long>(n_experts) * kp.matbytes;
    Plan pl;
    int rc = make_plan<Q6K>(rows, k, slots, cfg, &kp, &pl);
    if (rc) return rc;
    return launch<Q6K, true, MODE_MATVEC>(kp, pl, slots, s);
}

namespace {

KParams q6k_params(const void* w, int rows, int k) {
    KParams kp{};
    kp.w = static_cast<const uint8_t*>(w);
    kp.rows = rows;
    kp.k = k;
    kp.nb = k / 256;
    kp.rowbytes = static_cast<uint32_t>(kp.nb) * 210u;
    kp.matbytes = static_cast<unsigned long long>(rows) * kp.rowbytes;
    kp.wbytes = kp.matbytes;
    return kp;
}

}  // namespace

int q6k_dp4a(const void* w, const int8_t* xq, const float* xs, float* y, int rows, int k, const qmv_opts* cfg,
             cudaStream_t s) {
    KParams kp = q6k_params(w, rows, k);
    kp.xq = xq;
    kp.xqs = xs;
    kp.y = y;
    Plan pl;
    int rc = make_plan<Q6D>(rows, k, 1, cfg, &kp, &pl);
    if (rc) return rc;
    return launch<Q6D, false, MODE_MATVEC>(kp, pl, 1, s);
}

int q6k_dp4a_blockdots(const void* w, const int8_t* xq, int32_t* dots, int rows, int k, cudaStream_t s) {
    KParams kp = q6k_params(w, rows, k);
    kp.xq = xq;
    kp.dots = dots;
    Plan pl;
    int rc = make_plan<Q6D>(rows, k, 1, nullptr, &kp, &pl);
    if (rc) return rc;
    return launch<Q6D, false, MODE_BLOCKDOTS>(kp, pl, 1, s);
}

int moe_q6k_dp4a(const void* bank, const int8_t* xq, const float* xs, float* y, int rows, int k, const int32_t* ids,
                 int slots, int n_experts, const qmv_opts* cfg, cudaStream_t s) {
    KParams kp = q6k_params(bank, rows, k);
    kp.xq = xq;
    kp.xqs = xs;
    kp.y = y;
    kp.ids = ids;
    kp.n_experts = n_experts;
    kp.wbytes = static_cast<unsigned long long>(n_experts) * kp.matbytes;
    Plan pl;
    int rc = make_plan<Q6D>(rows, k, slots, cfg, &kp, &pl);
    if (rc) return rc;
    return launch<Q6D, true, MODE_MATVEC>(kp, pl, slots, s);
}

int dequant_q6k(const void* w, float* out, int rows, int k, cudaStream_t s) {
    const long long ng = static_cast<long long>(rows) * (k / 256) * 16;
    const int threads = 256;
    const long long want = (ng + threads - 1) / threads;
    const int blocks = static_cast<int>(want < 65536 ? want : 65536);
    dequant_q6k_kernel<<<blocks, threads, 0, s>>>(static_cast<const uint8_t*>(w), out, ng);
    return cuda_rc(cudaGetLastError());
}

int status_q6k(unsigned int* out, int clear) { return status_rw(out, clear); }

}  // namespace qmvi
