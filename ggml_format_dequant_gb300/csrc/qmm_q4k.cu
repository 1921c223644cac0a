// qmm_q4k.cu -- small-M batched product y[m, rows] = x[m, k] W^T over packed
// Q4_K rows (m >= 2). Two rows of x: the register-activation kernel of
// qmm_kernel.cuh (one launch, or two of one row each when k is too large for
// one); from three rows on, the tensor-core kernel of qmm_tc.cuh, one launch
// per tile of up to 8 rows.
#include "qmv_internal.h"
#include "qmm_kernel.cuh"
#include "qmm_tc.cuh"

namespace qmvi {

using namespace qmv;

int qmm_q4k(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_cfg* cfg, cudaStream_t s) {
    // Three or more rows of x: the tensor-core kernel (its cost hardly
    // depends on m; measured faster from m = 3 on); two: the register-activation
    // kernel.
    if (m >= 3) return qmm_tc_run<Q4KT>(w, x, y, rows, k, m, cfg, s);
    KParams kp{};
    kp.w = static_cast<const uint8_t*>(w);
    kp.rows = rows;
    kp.k = k;
    kp.nb = k / 256;
    kp.rowbytes = static_cast<uint32_t>(kp.nb) * 144u;
    kp.matbytes = static_cast<unsigned long long>(rows) * kp.rowbytes;
    kp.wbytes = kp.matbytes;
    return qmm_run<Q4KB>(kp, x, y, m, cfg, s, q4k);
}

int status_qmm_q4k(unsigned int* out, int clear) { return status_rw(out, clear); }

}  // namespace qmvi
