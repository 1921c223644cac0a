// qmv_q8.cu -- Q8_0 matvecs (f32 activation, dense and MoE, and dp4a), the dp4a block dots,
// the activation quantizer and the Q8_0 dequantizer.
#include "qmv_internal.h"
#include "qmv_launch.cuh"

namespace {

using namespace qmv;

// One thread per 32-element block of x (quantize_block_q8: the IEEE f32
// divide / multiply / round-half-even steps of the quantizer). With x and xq
// 16-byte aligned (VEC) a block's 128 bytes of x are read as eight 16-byte
// loads and its 32 codes written as two; otherwise element by element. xsum
// is d times the integer sum of the codes, one f32 multiply. The kernel lets
// a dependent launch after it start at once (that launch still waits for
// this kernel before it reads what this one wrote).
template <bool VEC>
__global__ void quantize_act_q8_kernel(const float* __restrict__ x, int8_t* __restrict__ xq,
                                       float* __restrict__ xs, float* __restrict__ xsum, long long nblocks) {
    pdl_launch_dependents();
    for (long long b = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; b < nblocks;
         b += static_cast<long long>(gridDim.x) * blockDim.x) {
        float4 v[8];
        if constexpr (VEC) {
            const float4* src = reinterpret_cast<const float4*>(x + 32 * b);
#pragma unroll
            for (int j = 0; j < 8; j++) v[j] = __ldg(src + j);
        } else {
            const float* src = x + 32 * b;
#pragma unroll
            for (int j = 0; j < 8; j++)
                v[j] = make_float4(__ldg(src + 4 * j), __ldg(src + 4 * j + 1), __ldg(src + 4 * j + 2),
                                   __ldg(src + 4 * j + 3));
        }
        uint32_t codes[8];
        int sum;
        const float d = quantize_block_q8(v, codes, sum);
        if constexpr (VEC) {
            uint4* dst = reinterpret_cast<uint4*>(xq + 32 * b);
            dst[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
            dst[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
        } else {
#pragma unroll
            for (int i = 0; i < 32; i++) xq[32 * b + i] = static_cast<int8_t>((codes[i >> 2] >> (8 * (i & 3))) & 0xffu);
        }
        xs[b] = d;
        if (xsum) xsum[b] = __fmul_rn(d, __int2float_rn(sum));
    }
}

// One thread per (row, block): d*q is exact in f32.
__global__ void dequant_q8_0_kernel(const uint8_t* __restrict__ w, float* __restrict__ out, long long nblk) {
    for (long long blk = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; blk < nblk;
         blk += static_cast<long long>(gridDim.x) * blockDim.x) {
        const uint8_t* p = w + blk * 34;
        const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(p[0] | (p[1] << 8))));
        for (int i = 0; i < 32; i++) out[blk * 32 + i] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(p[2 + i])));
    }
}

// Failure-path self-test: one thread waits, with the kernels' bounded wait,
// on a shared-memory barrier that nothing ever arrives on; when the limit runs
// out it raises STATUS_WAIT_TIMEOUT, exactly as a matvec whose staged copy
// never landed would, and the kernel returns.
__global__ void selftest_wait_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) unsigned long long bar_storage;
    const uint32_t bar = smem_u32(&bar_storage);
    mbar_init(bar, 1);
    fence_mbar_init();
    if (!mbar_wait_bounded_ns(bar, 0u, limit_ns)) atomicOr(&g_status, STATUS_WAIT_TIMEOUT);
}

KParams q8_params(const void* w, int rows, int k) {
    KParams kp{};
    kp.w = static_cast<const uint8_t*>(w);
    kp.rows = rows;
    kp.k = k;
    kp.nb = k / 32;
    kp.rowbytes = static_cast<uint32_t>(kp.nb) * 34u;
    kp.matbytes = static_cast<unsigned long long>(rows) * kp.rowbytes;
    kp.wbytes = kp.matbytes;
    return kp;
}

int grid_for(long long items, int threads) {
    const long long want = (items + threads - 1) / threads;
    return static_cast<int>(want < 65536 ? (want > 0 ? want : 1) : 65536);
}

}  // namespace

namespace qmvi {

using namespace qmv;

int q8_0(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg, cudaStream_t s) {
    KParams kp = q8_params(w, rows, k);
    kp.x = x;
    kp.y = y;
    Plan pl;
    int rc = make_plan<Q8F>(rows, k, 1, cfg, &kp, &pl);
    if (rc) return rc;
    return launch<Q8F, false, MODE_MATVEC>(kp, pl, 1, s);
}

int moe_q8_0(const void* bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
             int n_experts, const qmv_opts* cfg, cudaStream_t s) {
    KParams kp = q8_params(bank, rows, k);
    kp.x = x;
    kp.y = y;
    kp.ids = ids;
    kp.n_experts = n_experts;
    kp.wbytes = static_cast<unsigned long long>(n_experts) * kp.matbytes;
    Plan pl;
    int rc = make_plan<Q8F>(rows, k, slots, cfg, &kp, &pl);
    if (rc) return rc;
    return launch<Q8F, true, MODE_MATVEC>(kp, pl, slots, s);
}

int q8_dp4a(const void* w, const int8_t* xq, const float* xs, float* y, int rows, int k, const qmv_opts* cfg,
            cudaStream_t s) {
    KParams kp = q8_params(w, rows, k);
    kp.xq = xq;
    kp.xqs = xs;
    kp.y = y;
    Plan pl;
    int rc = make_plan<Q8D>(rows, k, 1, cfg, &kp, &pl);
    if (rc) return rc;
    return launch<Q8D, false, MODE_MATVEC>(kp, pl, 1, s);
}

int q8_dp4a_quant(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg, cudaStream_t s) {
    KParams kp = q8_params(w, rows, k);
    kp.x = x;
    kp.y = y;
    Plan pl;
    int rc = make_plan<Q8DQ>(rows, k, 1, cfg, &kp, &pl);
    if (rc) return rc;
    return launch<Q8DQ, false, MODE_MATVEC>(kp, pl, 1, s);
}

int q8_blockdots(const void* w, const int8_t* xq, int32_t* dots, int rows, int k, cudaStream_t s) {
    KParams kp = q8_params(w, rows, k);
    kp.xq = xq;
    kp.dots = dots;
    Plan pl;
    int rc = make_plan<Q8D>(rows, k, 1, nullptr, &kp, &pl);
    if (rc) return rc;
    return launch<Q8D, false, MODE_BLOCKDOTS>(kp, pl, 1, s);
}

int quantize_act(const float* x, int8_t* xq, float* xs, float* xsum, int m, int k, cudaStream_t s) {
    const long long nblocks = static_cast<long long>(m) * (k / 32);
    const bool vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(xq)) & 15u) == 0;
    if (vec)
        quantize_act_q8_kernel<true><<<grid_for(nblocks, 64), 64, 0, s>>>(x, xq, xs, xsum, nblocks);
    else
        quantize_act_q8_kernel<false><<<grid_for(nblocks, 64), 64, 0, s>>>(x, xq, xs, xsum, nblocks);
    return cuda_rc(cudaGetLastError());
}

int dequant_q8_0(const void* w, float* out, int rows, int k, cudaStream_t s) {
    const long long nblk = static_cast<long long>(rows) * (k / 32);
    dequant_q8_0_kernel<<<grid_for(nblk, 256), 256, 0, s>>>(static_cast<const uint8_t*>(w), out, nblk);
    return cuda_rc(cudaGetLastError());
}

int selftest_wait_timeout(unsigned long long limit_ns, cudaStream_t s) {
    selftest_wait_kernel<<<1, 1, 0, s>>>(limit_ns);
    return cuda_rc(cudaGetLastError());
}

int status_q8(unsigned int* out, int clear) { return status_rw(out, clear); }

}  // namespace qmvi
