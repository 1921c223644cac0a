// qmm_q4k.cu -- small-M batched product y[m, rows] = x[m, k] W^T over packed
// Q4_K rows (m >= 2): the tensor-core kernel of qmm_tc.cuh, one launch per
// tile of up to 8 rows of x.
#include "qmv_internal.h"
#include "qmm_tc.cuh"

namespace qmvi {

using namespace qmv;

int qmm_q4k(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg, cudaStream_t s,
            int force_timeout) {
    return qmm_tc_run<Q4KT>(w, x, y, rows, k, m, cfg, s, force_timeout);
}

int status_qmm_q4k(unsigned int* out, int clear) { return status_rw(out, clear); }

}  // namespace qmvi
