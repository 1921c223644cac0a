// qmv_api.cu -- the extern "C" entry points of libqmv.so: argument validation
// on the host (nothing is enqueued for a bad call), then the launch in the
// format's translation unit.
#include <climits>
#include <cstdint>

#include "qmm_tc.cuh"
#include "qmv_internal.h"
#include "qmv_launch.cuh"

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Common checks of a dense matvec: non-null pointers, rows > 0, k a positive
// multiple of the block size, weight and activation 16-byte and the output
// 4-byte aligned, and a total weight size that fits the address arithmetic.
int check_dense(const void* w, const void* x, const void* y, int rows, int k, int qk, int block_bytes) {
    if (!w || !x || !y) return QMV_EINVAL;
    if (rows <= 0 || k <= 0 || k % qk) return QMV_EINVAL;
    if (!aligned(w, 16) || !aligned(x, 16) || !aligned(y, 4)) return QMV_EALIGN;
    const long long rb = static_cast<long long>(k / qk) * block_bytes;
    if (rb > INT_MAX || static_cast<long long>(rows) > LLONG_MAX / rb) return QMV_EINVAL;
    return QMV_OK;
}

// Checks shared by the MoE entry points beyond the dense ones: ids, slot and
// expert counts, and a bank size that fits the address arithmetic.
int check_moe(const int32_t* ids, int slots, int n_experts, int rows, int k, int qk, int block_bytes) {
    if (!ids) return QMV_EINVAL;
    if (slots <= 0 || slots > 65535 || n_experts <= 0) return QMV_EINVAL;
    if (!aligned(ids, 4)) return QMV_EALIGN;
    const long long rb = static_cast<long long>(k / qk) * block_bytes;
    if (static_cast<long long>(n_experts) > LLONG_MAX / rb / rows) return QMV_EINVAL;
    return QMV_OK;
}

// Launch options: the overlap mode must be one of QMV_OVERLAP_*; the forced
// plan fields may take any value (<= 0 keeps the automatic choice).
bool opts_ok(const qmv_opts* o) {
    return !o || (o->overlap >= QMV_OVERLAP_NONE && o->overlap <= QMV_OVERLAP_INDEPENDENT);
}

}  // namespace

extern "C" {

int qmv_q4k_ex(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg,
                cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w, x, y, rows, k, 256, 144);
    return rc ? rc : qmvi::q4k(w, x, y, rows, k, cfg, stream);
}

int qmv_q4k(const void* w, const float* x, float* y, int rows, int k, cudaStream_t stream) {
    return qmv_q4k_ex(w, x, y, rows, k, nullptr, stream);
}

int qmv_q6k_ex(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg,
                cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w, x, y, rows, k, 256, 210);
    return rc ? rc : qmvi::q6k(w, x, y, rows, k, cfg, stream);
}

int qmv_q6k(const void* w, const float* x, float* y, int rows, int k, cudaStream_t stream) {
    return qmv_q6k_ex(w, x, y, rows, k, nullptr, stream);
}

int qmv_q8_0_ex(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg,
                 cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w, x, y, rows, k, 32, 34);
    return rc ? rc : qmvi::q8_0(w, x, y, rows, k, cfg, stream);
}

int qmv_q8_0(const void* w, const float* x, float* y, int rows, int k, cudaStream_t stream) {
    return qmv_q8_0_ex(w, x, y, rows, k, nullptr, stream);
}

int qmv_q5k_ex(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg,
                cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w, x, y, rows, k, 256, 176);
    return rc ? rc : qmvi::q5k(w, x, y, rows, k, cfg, stream);
}

int qmv_q5k(const void* w, const float* x, float* y, int rows, int k, cudaStream_t stream) {
    return qmv_q5k_ex(w, x, y, rows, k, nullptr, stream);
}

int qmv_q4_0_ex(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg,
                 cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w, x, y, rows, k, 32, 18);
    return rc ? rc : qmvi::q4_0(w, x, y, rows, k, cfg, stream);
}

int qmv_q4_0(const void* w, const float* x, float* y, int rows, int k, cudaStream_t stream) {
    return qmv_q4_0_ex(w, x, y, rows, k, nullptr, stream);
}

// Small-M batch: m == 1 is the matvec itself; m >= 2 the batched kernels.
int qmm_q4k_ex(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg,
                cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w, x, y, rows, k, 256, 144);
    if (!rc && (m <= 0 || static_cast<long long>(m) * k > INT_MAX || static_cast<long long>(m) * rows > INT_MAX))
        rc = QMV_EINVAL;
    if (rc) return rc;
    return m == 1 ? qmvi::q4k(w, x, y, rows, k, cfg, stream) : qmvi::qmm_q4k(w, x, y, rows, k, m, cfg, stream);
}

int qmm_q4k(const void* w, const float* x, float* y, int rows, int k, int m, cudaStream_t stream) {
    return qmm_q4k_ex(w, x, y, rows, k, m, nullptr, stream);
}

int qmm_q4k_tc5_ex(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg,
                   cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w, x, y, rows, k, 256, 144);
    if (!rc && (m <= 0 || static_cast<long long>(m) * k > INT_MAX || static_cast<long long>(m) * rows > INT_MAX))
        rc = QMV_EINVAL;
    if (rc) return rc;
    return qmvi::qmm_q4k_tc5(w, x, y, rows, k, m, cfg, stream);
}

int qmm_q6k_ex(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg,
                cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w, x, y, rows, k, 256, 210);
    if (!rc && (m <= 0 || static_cast<long long>(m) * k > INT_MAX || static_cast<long long>(m) * rows > INT_MAX))
        rc = QMV_EINVAL;
    if (rc) return rc;
    return m == 1 ? qmvi::q6k(w, x, y, rows, k, cfg, stream) : qmvi::qmm_q6k(w, x, y, rows, k, m, cfg, stream);
}

int qmm_q6k(const void* w, const float* x, float* y, int rows, int k, int m, cudaStream_t stream) {
    return qmm_q6k_ex(w, x, y, rows, k, m, nullptr, stream);
}

int qmm_q8_0_ex(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg,
                 cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w, x, y, rows, k, 32, 34);
    if (!rc && (m <= 0 || static_cast<long long>(m) * k > INT_MAX || static_cast<long long>(m) * rows > INT_MAX))
        rc = QMV_EINVAL;
    if (rc) return rc;
    return m == 1 ? qmvi::q8_0(w, x, y, rows, k, cfg, stream) : qmvi::qmm_q8_0(w, x, y, rows, k, m, cfg, stream);
}

int qmm_q8_0(const void* w, const float* x, float* y, int rows, int k, int m, cudaStream_t stream) {
    return qmm_q8_0_ex(w, x, y, rows, k, m, nullptr, stream);
}

int qmm_q5k_ex(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg,
                 cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w, x, y, rows, k, 256, 176);
    if (!rc && (m <= 0 || static_cast<long long>(m) * k > INT_MAX || static_cast<long long>(m) * rows > INT_MAX))
        rc = QMV_EINVAL;
    if (rc) return rc;
    return m == 1 ? qmvi::q5k(w, x, y, rows, k, cfg, stream) : qmvi::qmm_q5k(w, x, y, rows, k, m, cfg, stream);
}

int qmm_q5k(const void* w, const float* x, float* y, int rows, int k, int m, cudaStream_t stream) {
    return qmm_q5k_ex(w, x, y, rows, k, m, nullptr, stream);
}

int qmm_q4_0_ex(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg,
                  cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w, x, y, rows, k, 32, 18);
    if (!rc && (m <= 0 || static_cast<long long>(m) * k > INT_MAX || static_cast<long long>(m) * rows > INT_MAX))
        rc = QMV_EINVAL;
    if (rc) return rc;
    return m == 1 ? qmvi::q4_0(w, x, y, rows, k, cfg, stream) : qmvi::qmm_q4_0(w, x, y, rows, k, m, cfg, stream);
}

int qmm_q4_0(const void* w, const float* x, float* y, int rows, int k, int m, cudaStream_t stream) {
    return qmm_q4_0_ex(w, x, y, rows, k, m, nullptr, stream);
}

int quantize_act_q8(const float* x, int8_t* xq, float* xs, float* xsum, int m, int k, cudaStream_t stream) {
    if (!x || !xq || !xs) return QMV_EINVAL;
    if (m <= 0 || k <= 0 || k % 32) return QMV_EINVAL;
    if (!aligned(x, 4) || !aligned(xs, 4) || (xsum && !aligned(xsum, 4))) return QMV_EALIGN;
    if (static_cast<long long>(m) * k > (LLONG_MAX >> 8)) return QMV_EINVAL;
    return qmvi::quantize_act(x, xq, xs, xsum, m, k, stream);
}

int qmv_q8_dp4a_ex(const void* w, const int8_t* xq, const float* xs, float* y, int rows, int k,
                    const qmv_opts* cfg, cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    if (!xs) return QMV_EINVAL;
    int rc = check_dense(w, xq, y, rows, k, 32, 34);
    if (rc) return rc;
    if (!aligned(xq, 16) || !aligned(xs, 4)) return QMV_EALIGN;
    return qmvi::q8_dp4a(w, xq, xs, y, rows, k, cfg, stream);
}

int qmv_q8_dp4a(const void* w, const int8_t* xq, const float* xs, float* y, int rows, int k,
                cudaStream_t stream) {
    return qmv_q8_dp4a_ex(w, xq, xs, y, rows, k, nullptr, stream);
}

int qmv_q8_dp4a_quant_ex(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg,
                         cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w, x, y, rows, k, 32, 34);
    return rc ? rc : qmvi::q8_dp4a_quant(w, x, y, rows, k, cfg, stream);
}

int qmv_q8_dp4a_quant(const void* w, const float* x, float* y, int rows, int k, cudaStream_t stream) {
    return qmv_q8_dp4a_quant_ex(w, x, y, rows, k, nullptr, stream);
}

int qmv_q4k_dp4a_ex(const void* w, const int8_t* xq, const float* xs, float* y, int rows, int k,
                     const qmv_opts* cfg, cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    if (!xs) return QMV_EINVAL;
    int rc = check_dense(w, xq, y, rows, k, 256, 144);
    if (rc) return rc;
    if (!aligned(xq, 16) || !aligned(xs, 4)) return QMV_EALIGN;
    return qmvi::q4k_dp4a(w, xq, xs, y, rows, k, cfg, stream);
}

int qmv_q4k_dp4a(const void* w, const int8_t* xq, const float* xs, float* y, int rows, int k,
                 cudaStream_t stream) {
    return qmv_q4k_dp4a_ex(w, xq, xs, y, rows, k, nullptr, stream);
}

int qmv_q6k_dp4a_ex(const void* w, const int8_t* xq, const float* xs, float* y, int rows, int k,
                     const qmv_opts* cfg, cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    if (!xs) return QMV_EINVAL;
    int rc = check_dense(w, xq, y, rows, k, 256, 210);
    if (rc) return rc;
    if (!aligned(xq, 16) || !aligned(xs, 4)) return QMV_EALIGN;
    return qmvi::q6k_dp4a(w, xq, xs, y, rows, k, cfg, stream);
}

int qmv_q6k_dp4a(const void* w, const int8_t* xq, const float* xs, float* y, int rows, int k,
                 cudaStream_t stream) {
    return qmv_q6k_dp4a_ex(w, xq, xs, y, rows, k, nullptr, stream);
}

int moe_qmv_q6k_dp4a_ex(const void* w_bank, const int8_t* xq, const float* xs, float* y, int rows, int k,
                         const int32_t* ids, int slots, int n_experts, const qmv_opts* cfg, cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    if (!xs) return QMV_EINVAL;
    int rc = check_dense(w_bank, xq, y, rows, k, 256, 210);
    if (!rc) rc = check_moe(ids, slots, n_experts, rows, k, 256, 210);
    if (rc) return rc;
    if (!aligned(xq, 16) || !aligned(xs, 4)) return QMV_EALIGN;
    return qmvi::moe_q6k_dp4a(w_bank, xq, xs, y, rows, k, ids, slots, n_experts, cfg, stream);
}

int moe_qmv_q6k_dp4a(const void* w_bank, const int8_t* xq, const float* xs, float* y, int rows, int k,
                     const int32_t* ids, int slots, int n_experts, cudaStream_t stream) {
    return moe_qmv_q6k_dp4a_ex(w_bank, xq, xs, y, rows, k, ids, slots, n_experts, nullptr, stream);
}

int qmv_q6k_dp4a_blockdots(const void* w, const int8_t* xq, int32_t* dots, int rows, int k, cudaStream_t stream) {
    int rc = check_dense(w, xq, dots, rows, k, 256, 210);
    if (rc) return rc;
    if (!aligned(xq, 16)) return QMV_EALIGN;
    return qmvi::q6k_dp4a_blockdots(w, xq, dots, rows, k, stream);
}

int moe_qmv_q4k_ex(const void* w_bank, const float* x, float* y, int rows, int k, const int32_t* ids,
                    int slots, int n_experts, const qmv_opts* cfg, cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w_bank, x, y, rows, k, 256, 144);
    if (!rc) rc = check_moe(ids, slots, n_experts, rows, k, 256, 144);
    return rc ? rc : qmvi::moe_q4k(w_bank, x, y, rows, k, ids, slots, n_experts, cfg, stream);
}

int moe_qmv_q4k(const void* w_bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
                int n_experts, cudaStream_t stream) {
    return moe_qmv_q4k_ex(w_bank, x, y, rows, k, ids, slots, n_experts, nullptr, stream);
}

int moe_qmv_q6k_ex(const void* w_bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
                    int n_experts, const qmv_opts* cfg, cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w_bank, x, y, rows, k, 256, 210);
    if (!rc) rc = check_moe(ids, slots, n_experts, rows, k, 256, 210);
    return rc ? rc : qmvi::moe_q6k(w_bank, x, y, rows, k, ids, slots, n_experts, cfg, stream);
}

int moe_qmv_q6k(const void* w_bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
                int n_experts, cudaStream_t stream) {
    return moe_qmv_q6k_ex(w_bank, x, y, rows, k, ids, slots, n_experts, nullptr, stream);
}

int moe_qmv_q8_0_ex(const void* w_bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
                     int n_experts, const qmv_opts* cfg, cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w_bank, x, y, rows, k, 32, 34);
    if (!rc) rc = check_moe(ids, slots, n_experts, rows, k, 32, 34);
    return rc ? rc : qmvi::moe_q8_0(w_bank, x, y, rows, k, ids, slots, n_experts, cfg, stream);
}

int moe_qmv_q8_0(const void* w_bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
                 int n_experts, cudaStream_t stream) {
    return moe_qmv_q8_0_ex(w_bank, x, y, rows, k, ids, slots, n_experts, nullptr, stream);
}

int moe_qmv_q4_0_ex(const void* w_bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
                     int n_experts, const qmv_opts* cfg, cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w_bank, x, y, rows, k, 32, 18);
    if (!rc) rc = check_moe(ids, slots, n_experts, rows, k, 32, 18);
    return rc ? rc : qmvi::moe_q4_0(w_bank, x, y, rows, k, ids, slots, n_experts, cfg, stream);
}

int moe_qmv_q4_0(const void* w_bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
                 int n_experts, cudaStream_t stream) {
    return moe_qmv_q4_0_ex(w_bank, x, y, rows, k, ids, slots, n_experts, nullptr, stream);
}

int moe_qmv_q5k_ex(const void* w_bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
                    int n_experts, const qmv_opts* cfg, cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    int rc = check_dense(w_bank, x, y, rows, k, 256, 176);
    if (!rc) rc = check_moe(ids, slots, n_experts, rows, k, 256, 176);
    return rc ? rc : qmvi::moe_q5k(w_bank, x, y, rows, k, ids, slots, n_experts, cfg, stream);
}

int moe_qmv_q5k(const void* w_bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
                int n_experts, cudaStream_t stream) {
    return moe_qmv_q5k_ex(w_bank, x, y, rows, k, ids, slots, n_experts, nullptr, stream);
}

int moe_qmv_q4k_dp4a_ex(const void* w_bank, const int8_t* xq, const float* xs, float* y, int rows, int k,
                         const int32_t* ids, int slots, int n_experts, const qmv_opts* cfg, cudaStream_t stream) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    if (!xs) return QMV_EINVAL;
    int rc = check_dense(w_bank, xq, y, rows, k, 256, 144);
    if (!rc) rc = check_moe(ids, slots, n_experts, rows, k, 256, 144);
    if (rc) return rc;
    if (!aligned(xq, 16) || !aligned(xs, 4)) return QMV_EALIGN;
    return qmvi::moe_q4k_dp4a(w_bank, xq, xs, y, rows, k, ids, slots, n_experts, cfg, stream);
}

int moe_qmv_q4k_dp4a(const void* w_bank, const int8_t* xq, const float* xs, float* y, int rows, int k,
                     const int32_t* ids, int slots, int n_experts, cudaStream_t stream) {
    return moe_qmv_q4k_dp4a_ex(w_bank, xq, xs, y, rows, k, ids, slots, n_experts, nullptr, stream);
}

int qmv_dequant_q4k(const void* w, float* out, int rows, int k, cudaStream_t stream) {
    int rc = check_dense(w, w, out, rows, k, 256, 144);
    return rc ? rc : qmvi::dequant_q4k(w, out, rows, k, stream);
}

int qmv_dequant_q6k(const void* w, float* out, int rows, int k, cudaStream_t stream) {
    int rc = check_dense(w, w, out, rows, k, 256, 210);
    return rc ? rc : qmvi::dequant_q6k(w, out, rows, k, stream);
}

int qmv_dequant_q8_0(const void* w, float* out, int rows, int k, cudaStream_t stream) {
    int rc = check_dense(w, w, out, rows, k, 32, 34);
    return rc ? rc : qmvi::dequant_q8_0(w, out, rows, k, stream);
}

int qmv_dequant_q5k(const void* w, float* out, int rows, int k, cudaStream_t stream) {
    int rc = check_dense(w, w, out, rows, k, 256, 176);
    return rc ? rc : qmvi::dequant_q5k(w, out, rows, k, stream);
}

int qmv_dequant_q4_0(const void* w, float* out, int rows, int k, cudaStream_t stream) {
    int rc = check_dense(w, w, out, rows, k, 32, 18);
    return rc ? rc : qmvi::dequant_q4_0(w, out, rows, k, stream);
}

int qmv_q8_dp4a_blockdots(const void* w, const int8_t* xq, int32_t* dots, int rows, int k, cudaStream_t stream) {
    int rc = check_dense(w, xq, dots, rows, k, 32, 34);
    if (rc) return rc;
    if (!aligned(xq, 16)) return QMV_EALIGN;
    return qmvi::q8_blockdots(w, xq, dots, rows, k, stream);
}

int qmv_q4k_dp4a_blockdots(const void* w, const int8_t* xq, int32_t* dots, int rows, int k, cudaStream_t stream) {
    int rc = check_dense(w, xq, dots, rows, k, 256, 144);
    if (rc) return rc;
    if (!aligned(xq, 16)) return QMV_EALIGN;
    return qmvi::q4k_dp4a_blockdots(w, xq, dots, rows, k, stream);
}

const char* qmv_strerror(int code) {
    switch (code) {
    case QMV_OK: return "ok";
    case QMV_EINVAL: return "invalid argument (null pointer or shape not a positive block multiple)";
    case QMV_EALIGN: return "misaligned pointer (weights and int8 activations need 16 bytes, f32 buffers 4)";
    case QMV_ECUDA: return "CUDA runtime error or kernel launch failure";
    case QMV_ETOOBIG: return "shape too large for the shared-memory plan of this build";
    default: return "unknown qmv error code";
    }
}

int qmv_selftest_timeout_path(const void* w, const float* x, float* y, int rows, int k, int m,
                              cudaStream_t stream) {
    int rc = check_dense(w, x, y, rows, k, 256, 144);
    if (!rc && (m <= 0 || m > 8)) rc = QMV_EINVAL;
    if (rc) return rc;
    return m == 1 ? qmvi::q4k(w, x, y, rows, k, nullptr, stream, 1)
                  : qmvi::qmm_q4k(w, x, y, rows, k, m, nullptr, stream, 1);
}

int qmm_q4k_tc5_plan_detail(int rows, int k, int m, const qmv_opts* cfg, const int* device, int* out) {
    if (!device || !out || !opts_ok(cfg) || rows <= 0 || k <= 0 || k % 256 || m <= 0 || m > 8) return QMV_EINVAL;
    return qmvi::qmm_q4k_tc5_plan(device, rows, k, m, cfg, out);
}

int qmm_q4k_tc5_selftest_timeout_path(const void* w, const float* x, float* y, int rows, int k, int m,
                                      const qmv_opts* opts, cudaStream_t stream) {
    int rc = check_dense(w, x, y, rows, k, 256, 144);
    if (!rc && (m <= 0 || m > 8)) rc = QMV_EINVAL;
    if (!rc && !opts_ok(opts)) rc = QMV_EINVAL;
    if (rc) return rc;
    return qmvi::qmm_q4k_tc5(w, x, y, rows, k, m, opts, stream, 1);
}

int qmv_selftest_wait_timeout(unsigned long long limit_ns, cudaStream_t stream) {
    if (limit_ns == 0 || limit_ns > 100000000ull) return QMV_EINVAL;
    return qmvi::selftest_wait_timeout(limit_ns, stream);
}

const char* qmv_last_cuda_error(void) {
    return cudaGetErrorString(qmv::last_cuda_error());
}

int qmv_device_status(unsigned int* status, int clear) {
    if (!status) return QMV_EINVAL;
    int (*const readers[])(unsigned int*, int) = {qmvi::status_q4k,     qmvi::status_q6k,     qmvi::status_q8,
                                                  qmvi::status_q5k,     qmvi::status_q4_0,    qmvi::status_qmm_q4k,
                                                  qmvi::status_qmm_q6k, qmvi::status_qmm_q8_0,
                                                  qmvi::status_qmm_q4k_tc5};
    unsigned int all = 0;
    for (auto rd : readers) {
        unsigned int v = 0;
        const int rc = rd(&v, clear);
        if (rc) return rc;
        all |= v;
    }
    *status = all;
    return QMV_OK;
}

namespace {

// Plan ids that describe an MoE launch (grid.y = slots).
bool plan_is_moe(int fmt) { return fmt == 4 || fmt == 6 || fmt == 7 || (fmt >= 10 && fmt <= 12) || fmt == 17; }

// Plan of format fmt on device `di`.
int plan_of(const qmv::DevInfo& di, int fmt, int rows, int k, int slots, const qmv_opts* cfg, qmv::KParams* kp,
            qmv::Plan* pl) {
    static const int qk[19] = {256, 256, 32, 32, 256, 256, 256, 256, 256, 32, 32, 32, 256, 256, 256, 32, 256, 256, 32};
    if (fmt < 0 || fmt > 18 || rows <= 0 || k <= 0 || k % qk[fmt]) return QMV_EINVAL;
    const bool moe = plan_is_moe(fmt);
    if (moe && slots <= 0) return QMV_EINVAL;
    if (fmt == 16) return qmv::make_plan_for<qmv::Q6D>(di, rows, k, 1, cfg, kp, pl);
    if (fmt == 17) return qmv::make_plan_for<qmv::Q6D>(di, rows, k, slots, cfg, kp, pl);
    if (fmt == 18) return qmv::make_plan_for<qmv::Q8DQ>(di, rows, k, 1, cfg, kp, pl);
    if (fmt >= 13 && fmt <= 15) return QMV_EINVAL;   // batches of two or more rows run on the tensor cores
    if (!moe) slots = 1;
    switch (fmt) {
    case 0: return qmv::make_plan_for<qmv::Q4K>(di, rows, k, 1, cfg, kp, pl);
    case 1: return qmv::make_plan_for<qmv::Q6K>(di, rows, k, 1, cfg, kp, pl);
    case 2: return qmv::make_plan_for<qmv::Q8F>(di, rows, k, 1, cfg, kp, pl);
    case 3: return qmv::make_plan_for<qmv::Q8D>(di, rows, k, 1, cfg, kp, pl);
    case 5: return qmv::make_plan_for<qmv::Q4D>(di, rows, k, 1, cfg, kp, pl);
    case 6: return qmv::make_plan_for<qmv::Q6K>(di, rows, k, slots, cfg, kp, pl);
    case 7: return qmv::make_plan_for<qmv::Q4D>(di, rows, k, slots, cfg, kp, pl);
    case 8: return qmv::make_plan_for<qmv::Q5K>(di, rows, k, 1, cfg, kp, pl);
    case 9: return qmv::make_plan_for<qmv::Q40>(di, rows, k, 1, cfg, kp, pl);
    case 10: return qmv::make_plan_for<qmv::Q8F>(di, rows, k, slots, cfg, kp, pl);
    case 11: return qmv::make_plan_for<qmv::Q40>(di, rows, k, slots, cfg, kp, pl);
    case 12: return qmv::make_plan_for<qmv::Q5K>(di, rows, k, slots, cfg, kp, pl);
    default: return qmv::make_plan_for<qmv::Q4K>(di, rows, k, slots, cfg, kp, pl);
    }
}

}  // namespace

int qmv_plan_info(int fmt, int rows, int k, int slots, const qmv_opts* cfg, int* threads, int* ctas,
                  int* chunk_rows, int* chunks, int* smem_bytes) {
    if (!opts_ok(cfg)) return QMV_EINVAL;
    qmv::DevInfo di;
    int rc = qmv::dev_info(&di, nullptr);
    if (rc) return rc;
    qmv::KParams kp{};
    qmv::Plan pl;
    rc = plan_of(di, fmt, rows, k, slots, cfg, &kp, &pl);
    if (rc) return rc;
    if (threads) *threads = pl.T;
    if (ctas) *ctas = pl.parts * (plan_is_moe(fmt) ? slots : 1);
    if (chunk_rows) *chunk_rows = kp.CR;
    if (chunks) *chunks = kp.S;
    if (smem_bytes) *smem_bytes = static_cast<int>(pl.smem);
    return QMV_OK;
}

int qmv_plan_detail(int fmt, int rows, int k, int slots, const qmv_opts* cfg, const int* device, int* out) {
    if (!device || !out || !opts_ok(cfg)) return QMV_EINVAL;
    qmv::DevInfo di;
    di.nsm = device[0];
    di.smem_optin = device[1];
    di.smem_sm = device[2];
    di.smem_reserved = device[3];
    if (di.nsm <= 0 || di.smem_optin <= 0 || di.smem_sm <= 0 || di.smem_reserved < 0) return QMV_EINVAL;
    qmv::KParams kp{};
    qmv::Plan pl;
    const int rc = plan_of(di, fmt, rows, k, slots, cfg, &kp, &pl);
    if (rc) return rc;
    const int v[QMV_PLAN_DETAIL_FIELDS] = {
        pl.T, pl.parts, pl.R, static_cast<int>(pl.smem), kp.U, kp.KS, kp.GS, kp.NG, kp.CR, kp.S,
        static_cast<int>(kp.rowbytes), kp.W, static_cast<int>(kp.slot_stride), kp.aligned8, kp.rq, kp.rrem,
        kp.gq[0], kp.grem[0], kp.gq[1], kp.grem[1], static_cast<int>(kp.lt.la), static_cast<int>(kp.lt.lb),
        static_cast<int>(kp.lt.lc), static_cast<int>(kp.lt.xs), static_cast<int>(kp.lt.xsum16),
        static_cast<int>(kp.off_red), static_cast<int>(kp.off_ring), static_cast<int>(kp.off_bars),
        static_cast<int>(kp.off_cnt), pl.CL};
    for (int i = 0; i < QMV_PLAN_DETAIL_FIELDS; i++) out[i] = v[i];
    return QMV_OK;
}

int qmm_tc_plan_detail(int fmt, int rows, int k, int m, const qmv_opts* cfg, const int* device, int* out) {
    if (!device || !out || !opts_ok(cfg)) return QMV_EINVAL;
    qmv::DevInfo di;
    di.nsm = device[0];
    di.smem_optin = device[1];
    di.smem_sm = device[2];
    di.smem_reserved = device[3];
    if (di.nsm <= 0 || di.smem_optin <= 0 || di.smem_sm <= 0 || di.smem_reserved < 0) return QMV_EINVAL;
    qmv::TParams tp{};
    qmv::Plan pl;
    int rc;
    switch (fmt) {
    case 0: rc = qmv::make_tc_plan_for<qmv::Q4KT>(di, rows, k, m, cfg, &tp, &pl); break;
    case 1: rc = qmv::make_tc_plan_for<qmv::Q6KT>(di, rows, k, m, cfg, &tp, &pl); break;
    case 2: rc = qmv::make_tc_plan_for<qmv::Q8T>(di, rows, k, m, cfg, &tp, &pl); break;
    case 3: rc = qmv::make_tc_plan_for<qmv::Q5KT>(di, rows, k, m, cfg, &tp, &pl); break;
    case 4: rc = qmv::make_tc_plan_for<qmv::Q40T>(di, rows, k, m, cfg, &tp, &pl); break;
    default: rc = QMV_EINVAL;
    }
    if (rc) return rc;
    const int v[QMM_TC_PLAN_FIELDS] = {pl.T,
                                      pl.parts,
                                      static_cast<int>(pl.smem),
                                      tp.KS,
                                      tp.CR,
                                      tp.S,
                                      static_cast<int>(tp.chunk_bytes),
                                      static_cast<int>(tp.stride),
                                      static_cast<int>(tp.slot_stride),
                                      tp.rq,
                                      tp.rrem,
                                      tp.ngroups,
                                      tp.nchunks,
                                      static_cast<int>(tp.off_red),
                                      static_cast<int>(tp.off_sums),
                                      static_cast<int>(tp.off_ring),
                                      static_cast<int>(tp.off_bars),
                                      static_cast<int>(tp.off_cnt)};
    for (int i = 0; i < QMM_TC_PLAN_FIELDS; i++) out[i] = v[i];
    return QMV_OK;
}

}  // extern "C"
