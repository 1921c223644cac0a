// qmm_q8_0.cu -- small-M batched product y[m, rows] = x[m, k] W^T over packed
// Q8_0 rows (m >= 2; tiles of up to 8 rows of x per launch, fewer when k
// is large; tiles of one row run the matvec). From three rows of x on, the
// tensor-core kernel of qmm_tc.cuh takes over.
#include "qmv_internal.h"
#include "qmm_kernel.cuh"
#include "qmm_tc.cuh"

namespace qmvi {

using namespace qmv;

int qmm_q8_0(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_cfg* cfg, cudaStream_t s) {
    // Three or more rows of x: the tensor-core kernel (its cost hardly
    // depends on m; measured faster from m = 3 on); two: the register-activation
    // kernel.
    if (m >= 3) return qmm_tc_run<Q8T>(w, x, y, rows, k, m, cfg, s);
    KParams kp{};
    kp.w = static_cast<const uint8_t*>(w);
    kp.rows = rows;
    kp.k = k;
    kp.nb = k / 32;
    kp.rowbytes = static_cast<uint32_t>(kp.nb) * 34u;
    kp.matbytes = static_cast<unsigned long long>(rows) * kp.rowbytes;
    kp.wbytes = kp.matbytes;
    return qmm_run<Q8B>(kp, x, y, m, cfg, s, q8_0);
}

int status_qmm_q8_0(unsigned int* out, int clear) { return status_rw(out, clear); }

}  // namespace qmvi
