// qmm_q6k.cu -- small-M batched product y[m, rows] = x[m, k] W^T over packed
// Q6_K rows (m >= 2): the tensor-core kernel of qmm_tc.cuh, one launch per
// tile of up to 8 rows of x.
#include "qmv_internal.h"
#include "qmm_tc.cuh"

namespace qmvi {

using namespace qmv;

int qmm_q6k(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg, cudaStream_t s) {
    return qmm_tc_run<Q6KT>(w, x, y, rows, k, m, cfg, s);
}

int status_qmm_q6k(unsigned int* out, int clear) { return status_rw(out, clear); }

}  // namespace qmvi
