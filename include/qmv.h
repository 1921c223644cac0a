/*
 * qmv.h -- C ABI of the GB300 (sm_103a) GGML-block quantized matrix-vector
 * product library (libqmv.so).
 *
 * Operation (hanzo-ml src/vulkan_backend.rs, matvec_q4k_gpu / matvec_q6k_gpu /
 * matvec_q8_0_gpu and moe_matvec_gpu): y = W x for a weight matrix W[rows, k]
 * whose rows are stored verbatim in GGML block formats and decoded inside the
 * kernel, never materialized:
 *   Q4_K: 144-byte super-blocks of 256 weights (d, dmin f16; 12 bytes of packed
 *         6-bit scales and mins; 128 bytes of 4-bit codes),
 *         w = d*sc_j*q - dmin*m_j for sub-block j = i/32 (quantize_q4k);
 *   Q6_K: 210-byte blocks of 256 weights (ql[128], qh[64], int8 scales[16],
 *         d f16), w = d*scale*(q - 32) (quantize_q6k);
 *   Q8_0: 34-byte blocks of 32 weights (d f16 then 32 int8), w = d*q
 *         (quantize_q8_blocks);
 *   Q5_K: 176-byte super-blocks of 256 weights (d, dmin f16; 12 scale bytes
 *         packed as Q4_K's; qh[32]; qs[128]), 5-bit codes whose fifth bit for
 *         weight i is bit i/32 of qh[i%32], w = d*sc_j*q - dmin*m_j
 *         (quantize_q5k, matvec_q5k_gpu);
 *   Q4_0: 18-byte blocks of 32 weights (d f16, then 16 bytes: low nibbles are
 *         weights 0..15, high nibbles 16..31), w = d*(q - 8) (matvec_q4_0_gpu).
 *
 * Conventions shared by every entry point:
 *  - All data pointers are DEVICE pointers owned by the caller. The library
 *    allocates no memory, keeps no per-call state and never synchronizes.
 *  - Work is enqueued on `stream` (0 = the legacy default stream) and runs
 *    asynchronously; outputs are valid once the stream reaches that point.
 *  - Packed weights are rows of whole blocks, row-major and contiguous (row r
 *    starts at byte r * (k / block_weights) * block_bytes). The weight pointer
 *    and the activation pointer (f32 x, or int8 xq) must be 16-byte aligned;
 *    f32 outputs and scales 4-byte aligned. Only the bytes of the rows read
 *    are accessed.
 *  - Outputs are overwritten, never accumulated into.
 *  - Return value: QMV_OK (0) or a negative QMV_E* code; qmv_strerror() names
 *    it. Argument errors are detected on the host before anything is enqueued.
 *  - Numerics: decoded weights are exact (each is the round-to-nearest f32 of
 *    its exact value). The f32-activation entry points carry x into integer
 *    dp4a dot products as three signed-byte limbs per element, with one
 *    power-of-two scale per 32 activations (21 bits kept below the block's
 *    largest |x|), and sum scaled group results in f32; results agree with an
 *    f64 dequantize-then-dot reference to a scale-relative error
 *    max|a-b|/max|a| far below 1e-4. Non-finite inputs give unspecified
 *    (possibly non-finite) outputs.
 *  - Threading: every entry point is reentrant; calls on different streams may
 *    run concurrently.
 */
#ifndef QMV_H
#define QMV_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QMV_OK 0
#define QMV_EINVAL (-1)  /* bad shape or null pointer (k not a block multiple, rows/m/slots/n_experts <= 0) */
#define QMV_EALIGN (-2)  /* a pointer that must be 16-byte (or 4-byte) aligned is not */
#define QMV_ECUDA (-3)   /* a CUDA runtime call or the kernel launch failed */
#define QMV_ETOOBIG (-4) /* valid shape too large for this build's shared-memory plan */

/* ----------------------------------------------------------------------
 * Launch options. Every entry point that launches a matvec, an MoE matvec or
 * a batch has an `_ex` twin with the same arguments plus `const qmv_opts
 * *opts` (before the stream); opts == NULL, or the entry point without `_ex`,
 * is a plain launch with the automatic plan. The options belong to the one
 * call: nothing is remembered between calls, and calls with different options
 * may run concurrently from any threads.
 *
 * overlap (the pages' decode engine records one whole decode step and replays
 * it, hanzo-ml src/vulkan_backend.rs, VkGraph; on a CUDA stream the same
 * back-to-back launches overlap through programmatic dependent launch):
 *   QMV_OVERLAP_NONE: plain launch; the kernel starts after the previous
 *     work on the stream has finished.
 *   QMV_OVERLAP_CHAIN: the call may be scheduled while the kernel launched
 *     just before it on the same stream still runs; it starts streaming its
 *     packed weights at once and waits for that kernel to finish before it
 *     reads x (MoE: ids) and before it writes y. Only valid if that kernel
 *     writes none of this call's packed weights (inference: weights are
 *     constant). Use it for a dependent decode chain, where each call reads
 *     the output of the one before.
 *   QMV_OVERLAP_INDEPENDENT: as CHAIN, and x and ids are read (and the whole
 *     product computed) before that wait; only the writes of y wait. Only
 *     valid if the kernel launched just before writes none of this call's
 *     inputs, e.g. consecutive projections of one activation (Q, K and V;
 *     gate and up). The plan then takes fewer CTAs so that several calls are
 *     in flight at once.
 *   Any other value is QMV_EINVAL.
 * Forced plan (tests and tuning sweeps; any field <= 0 keeps the automatic
 * choice): ctas: CTAs per weight matrix (per MoE slot); chunk_rows: rows per
 * ring slot (one bulk copy); chunks: ring slots per row group; unroll: rows
 * each warp decodes per step (1 or 2); warps: at most this many warps per CTA
 * (at least the k-slices of one row); cluster: CTAs (a power of two up to 8)
 * that share the conversion of the f32 activation (the CTA count is rounded
 * down to a multiple of it). */
#define QMV_OVERLAP_NONE 0
#define QMV_OVERLAP_CHAIN 1
#define QMV_OVERLAP_INDEPENDENT 2

typedef struct qmv_opts {
    int overlap;
    int ctas;
    int chunk_rows;
    int chunks;
    int unroll;
    int warps;
    int cluster;
} qmv_opts;

/* Q4_K matvec: y[r] = sum_j W[r, j] * x[j].
 * w: rows * (k/256) * 144 bytes; x: f32 [k]; y: f32 [rows].
 * k must be a positive multiple of 256, rows > 0.
 * Cites hanzo-ml src/vulkan_backend.rs, matvec_q4k_gpu_off and quantize_q4k. */
int qmv_q4k(const void *w, const float *x, float *y, int rows, int k, cudaStream_t stream);

/* Q6_K matvec: y = W x. w: rows * (k/256) * 210 bytes (the 210-byte blocks are
 * read unpadded); x: f32 [k]; y: f32 [rows]; k % 256 == 0.
 * Cites hanzo-ml src/vulkan_backend.rs, matvec_q6k_gpu and quantize_q6k. */
int qmv_q6k(const void *w, const float *x, float *y, int rows, int k, cudaStream_t stream);

/* Q8_0 matvec with an f32 activation: y = W x. w: rows * (k/32) * 34 bytes,
 * x: f32 [k]; y: f32 [rows]; k % 32 == 0.
 * Cites hanzo-ml src/vulkan_backend.rs, matvec_q8_0_gpu (raw 34-byte blocks). */
int qmv_q8_0(const void *w, const float *x, float *y, int rows, int k, cudaStream_t stream);

/* Q5_K matvec: y = W x. w: rows * (k/256) * 176 bytes (verbatim GGUF
 * super-blocks); x: f32 [k]; y: f32 [rows]; k % 256 == 0.
 * Cites hanzo-ml src/vulkan_backend.rs, matvec_q5k_gpu and quantize_q5k. */
int qmv_q5k(const void *w, const float *x, float *y, int rows, int k, cudaStream_t stream);

/* Q4_0 matvec: y = W x. w: rows * (k/32) * 18 bytes (native 18-byte blocks,
 * read unpadded); x: f32 [k]; y: f32 [rows]; k % 32 == 0.
 * Cites hanzo-ml src/vulkan_backend.rs, matvec_q4_0_gpu. */
int qmv_q4_0(const void *w, const float *x, float *y, int rows, int k, cudaStream_t stream);

/* Small-M batched product (several decode rows sharing one weight read):
 * y[i, r] = sum_j W[r, j] * x[i, j] for the m rows of x.
 * x: f32 [m, k] row-major, 16-byte aligned; y: f32 [m, rows] row-major;
 * w and k as for the matvec of the same format; m >= 1. m == 1 runs the
 * matvec; otherwise the tensor-core kernel, one launch per tile of 2..8 rows
 * of x (ceil(m/8) balanced tiles, each reading W once; rows of any length, in
 * k-chunks inside the launch), decoding every weight once per tile and
 * accumulating the m dot products in f32. Numerics: each decoded weight is
 * the round-to-nearest f32 of its exact value; results agree with an f64
 * reference to a scale-relative error far below 1e-4 per row of y. Each plan
 * is deterministic; independent calls (QMV_OVERLAP_INDEPENDENT) use
 * smaller k-chunks, so rows longer than 2048 weights may round differently
 * there than in plain or chained calls, within the same bound.
 * Cites hanzo-ml src/vulkan_backend.rs, matmul_q4k_gpu / matmul_q6k_gpu /
 * matmul_q8_gpu (decode once, reuse across up to MATMUL_Q_MAX_M = 8 rows). */
int qmm_q4k(const void *w, const float *x, float *y, int rows, int k, int m, cudaStream_t stream);
int qmm_q6k(const void *w, const float *x, float *y, int rows, int k, int m, cudaStream_t stream);
int qmm_q8_0(const void *w, const float *x, float *y, int rows, int k, int m, cudaStream_t stream);
/* The same product over Q5_K and Q4_0 rows (w and k as for qmv_q5k /
 * qmv_q4_0): m == 1 runs the matvec, m >= 2 the tensor-core kernel.
 * Cites hanzo-ml src/vulkan_backend.rs, matmul_q5k_gpu / matmul_q4_0_gpu. */
int qmm_q5k(const void *w, const float *x, float *y, int rows, int k, int m, cudaStream_t stream);
int qmm_q4_0(const void *w, const float *x, float *y, int rows, int k, int m, cudaStream_t stream);

/* Activation quantization for the dp4a path, per 32-element block of x[m, k]:
 * amax = max|x|; inv = 127/amax and d = amax/127 (IEEE f32 divides);
 * q = clamp(round_half_even(x * inv), -127, 127) (one f32 multiply); amax == 0
 * gives d = 0 and q = 0. Outputs: xq int8 [m, k]; xs f32 [m, k/32] = d;
 * xsum (may be NULL) f32 [m, k/32] = d * (integer sum of the block's q).
 * m > 0, k % 32 == 0; x, xs, xsum 4-byte aligned.
 * Cites hanzo-ml src/vulkan_backend.rs, quantize_act_q8 and quantize_q8. */
int quantize_act_q8(const float *x, int8_t *xq, float *xs, float *xsum, int m, int k,
                    cudaStream_t stream);

/* dp4a matvec of Q8_0 weights with a quantized activation:
 * y[r] = sum_b (d_w[r, b] * d_x[b]) * dot[r, b] in f32, where dot[r, b] is the
 * exact int32 sum of the block's 32 int8*int8 products.
 * w: Q8_0 rows as for qmv_q8_0; xq: int8 [k], 16-byte aligned; xs: f32 [k/32];
 * y: f32 [rows]. Cites hanzo-kernel src/main.rs, check_dp4a (matvec_q8_dp4a_*). */
int qmv_q8_dp4a(const void *w, const int8_t *xq, const float *xs, float *y, int rows, int k,
                cudaStream_t stream);

/* quantize_act_q8 and qmv_q8_dp4a in one launch: y = the Q8_0 dp4a matvec of
 * x quantized exactly as quantize_act_q8 quantizes it (the same codes and
 * scales, bit for bit; every CTA quantizes x into its own shared memory while
 * its first weight pieces are in flight, so the quantization costs no
 * separate launch and no trip of the codes through global memory). w as for
 * qmv_q8_0; x: f32 [k], 16-byte aligned; y: f32 [rows]; k % 32 == 0.
 * Numerics and results as quantize_act_q8 followed by qmv_q8_dp4a.
 * Cites hanzo-ml src/vulkan_backend.rs, quantize_act_q8 (quantize once per
 * decode step) and hanzo-kernel src/main.rs, check_dp4a. */
int qmv_q8_dp4a_quant(const void *w, const float *x, float *y, int rows, int k, cudaStream_t stream);

/* dp4a matvec of Q4_K weights with a quantized activation (the pages' dense
 * dp4a Q4_K decode): y[r] = sum_t xs[t] * (d*sc_t * dot[r, t] - dmin*m_t *
 * sumq[t]) in f32, over the 32-weight sub-blocks t of row r, where dot[r, t]
 * is the exact int32 dot of the sub-block's 4-bit codes with the 32 int8 codes
 * xq of the same positions and sumq[t] the sum of those codes (formed in the
 * kernel from xq; no separate sum input). w: Q4_K rows as for qmv_q4k;
 * xq: int8 [k], 16-byte aligned; xs: f32 [k/32]; y: f32 [rows]; k % 256 == 0.
 * Cites hanzo-ml src/vulkan_backend.rs, the `matvec_q4k_dp4a_blk` dispatch of
 * the decode matvec (quantize the activation once, dp4a the Q4_K codes). */
int qmv_q4k_dp4a(const void *w, const int8_t *xq, const float *xs, float *y, int rows, int k,
                 cudaStream_t stream);

/* dp4a matvec of Q6_K weights with a quantized activation (the pages' Q6_K
 * dp4a decode): y[r] = sum_g d*scale_g * xs[g/2] * dot[r, g] in f32 over the
 * 16-weight scale groups g of row r, where dot[r, g] is the exact int32
 * sum of (q - 32) * xq over the group (formed as sum(q * xq) - 32 * sum(xq)).
 * w: Q6_K rows as for qmv_q6k; xq: int8 [k], 16-byte aligned; xs: f32 [k/32];
 * y: f32 [rows]; k % 256 == 0. Cites hanzo-ml src/vulkan_backend.rs,
 * `moe_matvec_q6k_dp4a_blk_dn` (the -32 folded against activation sums). */
int qmv_q6k_dp4a(const void *w, const int8_t *xq, const float *xs, float *y, int rows, int k,
                 cudaStream_t stream);

/* MoE indexed Q4_K matvec: y[s, r] = sum_j W[ids[s], r, j] * x[s, j].
 * w_bank: one resident bank [n_experts, rows, k] of Q4_K rows (expert e's
 * matrix starts at byte e * rows * (k/256) * 144);
 * x: f32 [slots, k] (one activation row per slot); y: f32 [slots, rows];
 * ids: DEVICE int32 [slots], read on the GPU (duplicates allowed). Only the
 * rows of the routed experts are read. A slot whose id lies outside
 * [0, n_experts) gets NaN in all its outputs and raises QMV_STATUS_BAD_EXPERT_ID
 * in the device status word (see qmv_device_status); nothing traps.
 * Cites hanzo-ml src/vulkan_backend.rs, moe_matvec_gpu. */
int moe_qmv_q4k(const void *w_bank, const float *x, float *y, int rows, int k,
                const int32_t *ids, int slots, int n_experts, cudaStream_t stream);

/* MoE indexed Q6_K matvec (the pages' Q6_K down-projection experts):
 * y[s, r] = sum_j W[ids[s], r, j] * x[s, j] over one resident bank
 * [n_experts, rows, k] of Q6_K rows (expert e's matrix starts at byte
 * e * rows * (k/256) * 210); x f32 [slots, k]; y f32 [slots, rows]; ids as for
 * moe_qmv_q4k (out-of-range ids: NaN rows and QMV_STATUS_BAD_EXPERT_ID).
 * Cites hanzo-ml src/vulkan_backend.rs, the `moe_matvec_q6k*` kernels. */
int moe_qmv_q6k(const void *w_bank, const float *x, float *y, int rows, int k,
                const int32_t *ids, int slots, int n_experts, cudaStream_t stream);

/* MoE indexed matvecs over banks of the other formats, f32 activation; bank
 * layout [n_experts, rows, k] of verbatim rows (expert e's matrix starts at
 * byte e * rows * (k / block_weights) * block_bytes), x, y, ids and errors as
 * for moe_qmv_q4k.
 *   moe_qmv_q8_0: 34-byte Q8_0 blocks, k % 32 == 0 (the pages' moe_matvec_q8_0
 *                 reads a repacked bank; here the blocks are read as stored);
 *   moe_qmv_q4_0: 18-byte Q4_0 blocks, k % 32 == 0 (moe_matvec_q4_0);
 *   moe_qmv_q5k:  176-byte Q5_K blocks, k % 256 == 0 (one expert's slice of a
 *                 bank, as matvec_q5k_gpu_off selects it, for every slot).
 * Cites hanzo-ml src/vulkan_backend.rs, moe_matvec_gpu and the
 * `moe_matvec_q8_0` / `moe_matvec_q4_0` kernels. */
int moe_qmv_q8_0(const void *w_bank, const float *x, float *y, int rows, int k,
                 const int32_t *ids, int slots, int n_experts, cudaStream_t stream);
int moe_qmv_q4_0(const void *w_bank, const float *x, float *y, int rows, int k,
                 const int32_t *ids, int slots, int n_experts, cudaStream_t stream);
int moe_qmv_q5k(const void *w_bank, const float *x, float *y, int rows, int k,
                const int32_t *ids, int slots, int n_experts, cudaStream_t stream);

/* MoE indexed Q4_K matvec on the dp4a path: slot s multiplies expert ids[s]
 * with its own quantized activation, xq int8 [slots, k] (16-byte aligned) and
 * xs f32 [slots, k/32] (quantize_act_q8 with m = slots), as qmv_q4k_dp4a does.
 * Bank, ids, y and errors as for moe_qmv_q4k.
 * Cites hanzo-ml src/vulkan_backend.rs, `moe_matvec_q4k_dp4a_blk_*`. */
int moe_qmv_q4k_dp4a(const void *w_bank, const int8_t *xq, const float *xs, float *y, int rows, int k,
                     const int32_t *ids, int slots, int n_experts, cudaStream_t stream);

/* MoE indexed Q6_K matvec on the dp4a path: slot s multiplies expert ids[s]
 * with its own quantized activation, xq int8 [slots, k] (16-byte aligned) and
 * xs f32 [slots, k/32], as qmv_q6k_dp4a does. Bank, ids, y and errors as for
 * moe_qmv_q6k. Cites hanzo-ml src/vulkan_backend.rs,
 * `moe_matvec_q6k_dp4a_blk_dn`. */
int moe_qmv_q6k_dp4a(const void *w_bank, const int8_t *xq, const float *xs, float *y, int rows, int k,
                     const int32_t *ids, int slots, int n_experts, cudaStream_t stream);

/* Name of a QMV_* return code. Never NULL. */
const char *qmv_strerror(int code);

/* Text of the last CUDA error behind a QMV_ECUDA return on the calling thread
 * ("no error" if there was none). Never NULL. */
const char *qmv_last_cuda_error(void);

/* ----------------------------------------------------------------------
 * Device status word: bits raised by kernels on conditions that cannot be
 * seen on the host without a synchronization.
 */
#define QMV_STATUS_BAD_EXPERT_ID 1u /* an MoE id was outside [0, n_experts) */
#define QMV_STATUS_WAIT_TIMEOUT 2u  /* a staged weight copy did not land in time (the
                                     * CTA's outputs are then NaN) */
#define QMV_STATUS_OUT_OF_BOUNDS 4u /* only in the checking build of the library (compiled
                                     * with QMV_BOUNDS_CHECK, a file of its own): the matvec
                                     * kernel met an access outside the region its plan
                                     * gives it, and skipped it (outputs then undefined) */

/* Failure-path self-test: launches one thread that waits, through the same
 * bounded wait every staged copy goes through, on a barrier nothing arrives
 * on, for limit_ns (1 ns .. 100 ms); when the limit runs out it raises
 * QMV_STATUS_WAIT_TIMEOUT and returns, as a matvec whose copy never landed
 * would. Nothing hangs or traps; the context stays usable. */
int qmv_selftest_wait_timeout(unsigned long long limit_ns, cudaStream_t stream);

/* Failure-path self-test of the product kernels: runs qmv_q4k (m == 1) or
 * qmm_q4k (m = 2..8) on real Q4_K rows with every CTA taking the path of a
 * staged weight copy that did not land in time: the CTA raises
 * QMV_STATUS_WAIT_TIMEOUT, lets the copies it issued land (bounded), writes
 * NaN to all of its outputs and returns. Arguments as for qmv_q4k / qmm_q4k.
 * Nothing hangs or traps; the context stays usable. */
int qmv_selftest_timeout_path(const void *w, const float *x, float *y, int rows, int k, int m,
                              cudaStream_t stream);

/* The same failure-path self-test for qmm_q4k_tc5_ex (m = 1..8), in the plan
 * `opts` selects (NULL: the cluster plan; QMV_OVERLAP_INDEPENDENT: the
 * streaming plan where it fits): every CTA's decoder warps take the path of a
 * staged copy that did not land; the CTA lets its copies land (bounded),
 * releases its tensor memory, raises QMV_STATUS_WAIT_TIMEOUT and its partial
 * sums are NaN, so every output of the product is NaN. Other arguments as for
 * qmm_q4k_tc5_ex. Nothing hangs or traps; the context stays usable. */
int qmm_q4k_tc5_selftest_timeout_path(const void *w, const float *x, float *y, int rows, int k, int m,
                                      const qmv_opts *opts, cudaStream_t stream);

/* OR of the status bits raised on the current device since the last clear;
 * clears them when `clear` is non-zero. Waits for all work on the current
 * device (cudaDeviceSynchronize), then reads the word and clears it in one
 * atomic exchange, so that a bit raised by a kernel launched concurrently
 * from another host thread is either returned or kept, never lost. */
int qmv_device_status(unsigned int *status, int clear);

/* ----------------------------------------------------------------------
 * The entry points above with launch options (qmv_opts: overlap mode and an
 * optional forced plan). Arguments, numerics and errors as for the entry
 * point of the same name without `_ex`; an overlap value outside
 * QMV_OVERLAP_* is QMV_EINVAL.
 */
int qmv_q4k_ex(const void *w, const float *x, float *y, int rows, int k, const qmv_opts *opts,
                cudaStream_t stream);
int qmv_q6k_ex(const void *w, const float *x, float *y, int rows, int k, const qmv_opts *opts,
                cudaStream_t stream);
int qmv_q8_0_ex(const void *w, const float *x, float *y, int rows, int k, const qmv_opts *opts,
                 cudaStream_t stream);
int qmv_q8_dp4a_ex(const void *w, const int8_t *xq, const float *xs, float *y, int rows, int k,
                    const qmv_opts *opts, cudaStream_t stream);
int qmv_q8_dp4a_quant_ex(const void *w, const float *x, float *y, int rows, int k, const qmv_opts *opts,
                         cudaStream_t stream);
int qmv_q4k_dp4a_ex(const void *w, const int8_t *xq, const float *xs, float *y, int rows, int k,
                     const qmv_opts *opts, cudaStream_t stream);
int moe_qmv_q6k_ex(const void *w_bank, const float *x, float *y, int rows, int k,
                    const int32_t *ids, int slots, int n_experts, const qmv_opts *opts,
                    cudaStream_t stream);
int moe_qmv_q4k_dp4a_ex(const void *w_bank, const int8_t *xq, const float *xs, float *y, int rows,
                         int k, const int32_t *ids, int slots, int n_experts, const qmv_opts *opts,
                         cudaStream_t stream);
int moe_qmv_q4k_ex(const void *w_bank, const float *x, float *y, int rows, int k,
                    const int32_t *ids, int slots, int n_experts, const qmv_opts *opts,
                    cudaStream_t stream);
int qmv_q6k_dp4a_ex(const void *w, const int8_t *xq, const float *xs, float *y, int rows, int k,
                     const qmv_opts *opts, cudaStream_t stream);
int moe_qmv_q6k_dp4a_ex(const void *w_bank, const int8_t *xq, const float *xs, float *y, int rows,
                         int k, const int32_t *ids, int slots, int n_experts, const qmv_opts *opts,
                         cudaStream_t stream);
int qmm_q4k_ex(const void *w, const float *x, float *y, int rows, int k, int m, const qmv_opts *opts,
                cudaStream_t stream);

/* The batched product of qmm_q4k_ex (hanzo-ml src/vulkan_backend.rs,
 * matmul_q4k_gpu) on the fifth-generation tensor cores: tcgen05.mma with the
 * decoded weights (sc * q, exact in f16) as the A operand in tensor memory, x
 * as hi + lo f16 parts in shared memory and f32 accumulators in tensor memory.
 * Two plans:
 *  - the cluster plan: each 128-row tile is split along k over the CTAs of one
 *    thread-block cluster, which add their partial sums in rank order;
 *  - the streaming plan, for independent calls (opts->overlap ==
 *    QMV_OVERLAP_INDEPENDENT and no forced cluster size): one CTA a tile for
 *    the whole of k, one role per warp. Its results are bit for bit those of
 *    the cluster plan with one k-chunk.
 * Same result contract as qmm_q4k_ex (unit rows of x give the weight columns
 * bit for bit; otherwise within 1e-4 scale-relative of the exact product);
 * arguments, layouts and errors as there, m >= 1 (tiles of 8 rows of x, one
 * launch each); w and x must be 16-byte aligned (QMV_EINVAL otherwise).
 * opts->cluster forces the number of k-chunks of a tile (1..8) and the
 * cluster plan; opts->chunks sets the ring depth; opts->overlap the launch
 * overlap.
 * On a GB300 this path measured slower than qmm_q4k_ex for m <= 8 on the
 * 4096 x 4096 matrix (the streaming plan by 5-15 %), so qmm_q4k_ex does not
 * use it. A thread issues one tcgen05.mma (M = 128, K = 16) in 50-100 cycles
 * whatever N, and with N = 16 (8 rows of x, hi and lo) each covers only
 * 128 x 16 weights; the streaming plan issues from two threads, and is then
 * bound by the decode's instruction issue. */
int qmm_q4k_tc5_ex(const void *w, const float *x, float *y, int rows, int k, int m, const qmv_opts *opts,
                   cudaStream_t stream);

/* The plan qmm_q4k_tc5_ex takes for one launch (m = 1..8 rows of x) on a
 * described device {SM count, opt-in shared memory per CTA, shared memory per
 * SM, reserved shared memory per CTA}, computed on the host (no GPU needed):
 * out[13] = {CTAs, threads, dynamic shared memory, cluster size (k-chunks of a
 * tile), ring slots, super-blocks per row, and the shared-memory offsets of
 * B, B', the scales, the staged x, the partial-sum inbox and the barriers,
 * and the plan's kind: 0 the cluster plan, 1 the streaming plan that
 * independent calls (QMV_OVERLAP_INDEPENDENT, no forced cluster size) take --
 * one CTA a 128-row tile for the whole of k, with rings of B, B' and scales
 * (4 super-blocks each) in place of B for a whole chunk; its staged-x field
 * holds the offset of the ring of the rows' d and dmin (8 super-blocks), and
 * it has no inbox (offset 0)}. Returns QMV_ETOOBIG for a cluster-plan shape
 * whose chunk does not fit one CTA. */
int qmm_q4k_tc5_plan_detail(int rows, int k, int m, const qmv_opts *opts, const int *device, int *out);
int qmm_q6k_ex(const void *w, const float *x, float *y, int rows, int k, int m, const qmv_opts *opts,
                cudaStream_t stream);
int qmm_q8_0_ex(const void *w, const float *x, float *y, int rows, int k, int m, const qmv_opts *opts,
                 cudaStream_t stream);
int qmm_q5k_ex(const void *w, const float *x, float *y, int rows, int k, int m, const qmv_opts *opts,
                cudaStream_t stream);
int qmm_q4_0_ex(const void *w, const float *x, float *y, int rows, int k, int m, const qmv_opts *opts,
                 cudaStream_t stream);
int qmv_q5k_ex(const void *w, const float *x, float *y, int rows, int k, const qmv_opts *opts,
                cudaStream_t stream);
int qmv_q4_0_ex(const void *w, const float *x, float *y, int rows, int k, const qmv_opts *opts,
                 cudaStream_t stream);
int moe_qmv_q8_0_ex(const void *w_bank, const float *x, float *y, int rows, int k,
                     const int32_t *ids, int slots, int n_experts, const qmv_opts *opts,
                     cudaStream_t stream);
int moe_qmv_q4_0_ex(const void *w_bank, const float *x, float *y, int rows, int k,
                     const int32_t *ids, int slots, int n_experts, const qmv_opts *opts,
                     cudaStream_t stream);
int moe_qmv_q5k_ex(const void *w_bank, const float *x, float *y, int rows, int k,
                    const int32_t *ids, int slots, int n_experts, const qmv_opts *opts,
                    cudaStream_t stream);

/* ----------------------------------------------------------------------
 * Test and benchmark exports (not needed for inference).
 */

/* Exact decoded weights: out f32 [rows, k] (each the round-to-nearest f32 of
 * the weight's exact value). Same argument rules as the matvecs. */
int qmv_dequant_q4k(const void *w, float *out, int rows, int k, cudaStream_t stream);
int qmv_dequant_q6k(const void *w, float *out, int rows, int k, cudaStream_t stream);
int qmv_dequant_q8_0(const void *w, float *out, int rows, int k, cudaStream_t stream);
int qmv_dequant_q5k(const void *w, float *out, int rows, int k, cudaStream_t stream);
int qmv_dequant_q4_0(const void *w, float *out, int rows, int k, cudaStream_t stream);

/* Per-block int32 dots of the dp4a path, dots[r, b] (int32 [rows, k/32]),
 * computed by the same code path qmv_q8_dp4a uses. */
int qmv_q8_dp4a_blockdots(const void *w, const int8_t *xq, int32_t *dots, int rows, int k,
                          cudaStream_t stream);
/* The same for Q4_K rows: dots[r, t] (int32 [rows, k/32]) of every 32-weight
 * sub-block t, computed by the code path qmv_q4k_dp4a uses. */
int qmv_q4k_dp4a_blockdots(const void *w, const int8_t *xq, int32_t *dots, int rows, int k,
                           cudaStream_t stream);
/* The same for Q6_K rows: dots[r, g] (int32 [rows, k/16]) of every 16-weight
 * scale group g, sum((q - 32) * xq), computed by the code path qmv_q6k_dp4a
 * uses. */
int qmv_q6k_dp4a_blockdots(const void *w, const int8_t *xq, int32_t *dots, int rows, int k,
                           cudaStream_t stream);

/* Launch plan the library would use (for benchmark reports): threads per CTA,
 * CTAs (all slots), rows per ring slot, ring slots per row group and dynamic
 * shared bytes per CTA.
 * fmt: 0 = Q4_K, 1 = Q6_K, 2 = Q8_0 (f32 x), 3 = Q8_0 dp4a, 4 = MoE Q4_K,
 * 5 = Q4_K dp4a, 6 = MoE Q6_K, 7 = MoE Q4_K dp4a, 8 = Q5_K, 9 = Q4_0,
 * 10 = MoE Q8_0, 11 = MoE Q4_0, 12 = MoE Q5_K, 16 = Q6_K dp4a, 17 = MoE Q6_K
 * dp4a, 18 = Q8_0 dp4a with the quantization in the kernel
 * (qmv_q8_dp4a_quant). 13, 14 and 15 are not plans (QMV_EINVAL): batches of two or more rows
 * of x run on the tensor cores (qmm_tc_plan_detail). */
int qmv_plan_info(int fmt, int rows, int k, int slots, const qmv_opts *opts, int *threads, int *ctas,
                  int *chunk_rows, int *chunks, int *smem_bytes);

/* The complete launch plan for a described device, computed on the host
 * without touching a GPU (for tests of the planner). device = {SM count,
 * opt-in shared bytes per CTA, shared bytes per SM, reserved shared bytes per
 * CTA}. out receives QMV_PLAN_DETAIL_FIELDS ints in this order: threads, ctas
 * (per matrix), rows per warp step, dynamic shared bytes, units per row,
 * k-slices per row, lanes per row, row groups, rows per ring slot, ring slots
 * per group, bytes per row, parked row width, slot stride, 8-byte unit
 * alignment flag, rows per CTA (q, rem), rows per group for the smaller CTAs
 * (q, rem) and the larger ones (q, rem), shared offsets of the limb tables
 * (a, b, c, scales, sums), of the parked partials, the ring, the barriers and
 * the counters, and the cluster size. */
#define QMV_PLAN_DETAIL_FIELDS 30
int qmv_plan_detail(int fmt, int rows, int k, int slots, const qmv_opts *opts, const int *device, int *out);

/* The tensor-core plan of the batched product for one tile of m (1..8) rows
 * of x on a described device (as for qmv_plan_detail). fmt: 0 = Q4_K,
 * 1 = Q6_K, 2 = Q8_0, 3 = Q5_K, 4 = Q4_0. out receives QMM_TC_PLAN_FIELDS ints: threads, ctas,
 * dynamic shared bytes, warps (k-slices of 256 weights per k-chunk), rows per
 * ring slot, ring slots, bytes of one row's k-chunk, shared row stride, slot
 * stride, rows per CTA (q, rem), 32-weight groups per row, k-chunks, shared
 * offsets of the parked partials, the min-term fragments (Q4_K and Q5_K, 32
 * bytes a thread; none for the other formats), the ring, the barriers and the
 * counters. */
#define QMM_TC_PLAN_FIELDS 18
int qmm_tc_plan_detail(int fmt, int rows, int k, int m, const qmv_opts *opts, const int *device, int *out);

#ifdef __cplusplus
}
#endif

#endif /* QMV_H */
