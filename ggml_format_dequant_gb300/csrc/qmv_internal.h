// qmv_internal.h -- host functions each kernel translation unit exports to the
// C ABI layer (qmv_api.cu). Arguments are already validated by the caller.
#pragma once

#include <cstdint>
#include <cuda_runtime_api.h>

#include "../../include/qmv.h"

namespace qmvi {

// qmv_q4k.cu
// force_timeout (failure-path tests only): every CTA takes the path of a
// staged copy that did not land in time.
int q4k(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg, cudaStream_t s,
        int force_timeout = 0);
int moe_q4k(const void* bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
            int n_experts, const qmv_opts* cfg, cudaStream_t s);
int q4k_dp4a(const void* w, const int8_t* xq, const float* xs, float* y, int rows, int k, const qmv_opts* cfg,
             cudaStream_t s);
int q4k_dp4a_blockdots(const void* w, const int8_t* xq, int32_t* dots, int rows, int k, cudaStream_t s);
int moe_q4k_dp4a(const void* bank, const int8_t* xq, const float* xs, float* y, int rows, int k, const int32_t* ids,
                 int slots, int n_experts, const qmv_opts* cfg, cudaStream_t s);
int dequant_q4k(const void* w, float* out, int rows, int k, cudaStream_t s);
int status_q4k(unsigned int* out, int clear);

// qmv_q6k.cu
int q6k(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg, cudaStream_t s);
int moe_q6k(const void* bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
            int n_experts, const qmv_opts* cfg, cudaStream_t s);
int q6k_dp4a(const void* w, const int8_t* xq, const float* xs, float* y, int rows, int k, const qmv_opts* cfg,
             cudaStream_t s);
int q6k_dp4a_blockdots(const void* w, const int8_t* xq, int32_t* dots, int rows, int k, cudaStream_t s);
int moe_q6k_dp4a(const void* bank, const int8_t* xq, const float* xs, float* y, int rows, int k, const int32_t* ids,
                 int slots, int n_experts, const qmv_opts* cfg, cudaStream_t s);
int dequant_q6k(const void* w, float* out, int rows, int k, cudaStream_t s);
int status_q6k(unsigned int* out, int clear);

// qmv_q5k.cu
int q5k(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg, cudaStream_t s);
int moe_q5k(const void* bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
            int n_experts, const qmv_opts* cfg, cudaStream_t s);
int dequant_q5k(const void* w, float* out, int rows, int k, cudaStream_t s);
int qmm_q5k(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg, cudaStream_t s);
int status_q5k(unsigned int* out, int clear);

// qmv_q4_0.cu
int q4_0(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg, cudaStream_t s);
int moe_q4_0(const void* bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
             int n_experts, const qmv_opts* cfg, cudaStream_t s);
int dequant_q4_0(const void* w, float* out, int rows, int k, cudaStream_t s);
int qmm_q4_0(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg, cudaStream_t s);
int status_q4_0(unsigned int* out, int clear);

// qmv_q8.cu
int q8_0(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg, cudaStream_t s);
int moe_q8_0(const void* bank, const float* x, float* y, int rows, int k, const int32_t* ids, int slots,
             int n_experts, const qmv_opts* cfg, cudaStream_t s);
int q8_dp4a(const void* w, const int8_t* xq, const float* xs, float* y, int rows, int k, const qmv_opts* cfg,
            cudaStream_t s);
int q8_blockdots(const void* w, const int8_t* xq, int32_t* dots, int rows, int k, cudaStream_t s);
int q8_dp4a_quant(const void* w, const float* x, float* y, int rows, int k, const qmv_opts* cfg, cudaStream_t s);
int quantize_act(const float* x, int8_t* xq, float* xs, float* xsum, int m, int k, cudaStream_t s);
int dequant_q8_0(const void* w, float* out, int rows, int k, cudaStream_t s);
int selftest_wait_timeout(unsigned long long limit_ns, cudaStream_t s);
int status_q8(unsigned int* out, int clear);

// qmm_q4k.cu, qmm_q6k.cu, qmm_q8_0.cu: the small-M batched product (m >= 2)
int qmm_q4k(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg, cudaStream_t s,
            int force_timeout = 0);
int qmm_q6k(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg, cudaStream_t s);
int qmm_q8_0(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg, cudaStream_t s);
int status_qmm_q4k(unsigned int* out, int clear);
int status_qmm_q6k(unsigned int* out, int clear);
int status_qmm_q8_0(unsigned int* out, int clear);

// qmm_q4k_tc5.cu: the small-M batched product on the fifth-generation tensor
// cores (Q4_K rows)
int qmm_q4k_tc5(const void* w, const float* x, float* y, int rows, int k, int m, const qmv_opts* cfg,
                cudaStream_t s, int force_timeout = 0);
int status_qmm_q4k_tc5(unsigned int* out, int clear);
int qmm_q4k_tc5_plan(const int* device, int rows, int k, int m, const qmv_opts* cfg, int* out);

}  // namespace qmvi
