/*
 * qgemv.h -- C ABI of libqgemv.so: ggml block-quantized weights (Q4_0, Q4_1,
 * Q8_0) dequantized and contracted with activations on one NVIDIA GB300
 * (sm_103a) GPU.
 *
 * Sources for what each call computes ("llama_cpp 0.12.1 -> 0.12.2", the
 * my.diffend.io diff of the vendored ggml-cuda.cu):
 *   - hunk adding dequantize_block_q4_0 / dequantize_block_q4_1 and their
 *     dequantize_row_*_cuda launchers (to fp16 / fp32);
 *   - hunk adding dequantize_block_q8_0_f16 and its launcher;
 *   - the ggml_get_to_fp16_cuda / ggml_get_to_fp32_cuda dispatch hunk;
 *   - the dmmv ("dequantize_mul_mat_vec") and mul_mat_q names in the
 *     ggml_cuda_mul_mat / ggml_cuda_op_mul_mat hunks (batch-1 fused dequant
 *     + dot, and the quantized matmul used for prefill).
 *
 * Block formats (32 weights per block, fp16 little-endian scalars):
 *   Q4_0 (18 bytes) = [d : fp16][qs : 16 bytes]
 *        element j < 16 is the low nibble q of qs[j], element j+16 its high
 *        nibble; w = d * (q - 8).
 *   Q4_1 (20 bytes) = [d : fp16][m : fp16][qs : 16 bytes], same nibble order;
 *        w = d*q + m (the product and the sum each rounded to fp32).
 *   Q8_0 (34 bytes) = [d : fp16][qs : 32 x int8]; element j = qs[j]; w = d*q.
 * A weight matrix W of nrows x ncols is nrows consecutive rows, each row
 * ncols/32 consecutive blocks (ggml row order, ne0 = ncols fastest).
 *
 * Conventions for every call:
 *   - Pointers W, x, y, out, X, Y are DEVICE pointers owned by the caller;
 *     the library never frees or retains them.  They must be 16-byte
 *     aligned (QGEMV_ERR_ALIGN otherwise).  Outputs must not overlap inputs.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on that stream: a QGEMV_OK return
 *     means the work was validated and launched, not that it finished.
 *   - Arguments are validated on the host before any launch; a rejected call
 *     launches nothing and writes nothing.  After the launch the call checks
 *     cudaGetLastError() and returns QGEMV_ERR_LAUNCH (detail in
 *     qgemv_last_error_string()).
 *   - nrows == 0 (or m == 0, or ncols == 0) is a valid empty problem: OK, no
 *     launch.  ncols must be a multiple of 32; sizes are int64_t.
 *   - Kernels never trap.  A kernel whose bounded wait on an asynchronous
 *     copy expires records it in a per-device error word; qgemv_sync_check()
 *     reports it as QGEMV_ERR_TIMEOUT.
 *   - The device must be compute capability 10.3 (GB300); otherwise
 *     QGEMV_ERR_ARCH.
 *   - The dequantize and GEMV calls allocate no device memory.  The qgemm_*
 *     prefill calls keep the fp16 copy of the activations in a library-owned
 *     per-device workspace: the first call on a device, and any later call
 *     that needs a larger one, allocates it with cudaMalloc (make such a call
 *     before any stream capture); qgemv_shutdown() releases it.  Calls on one
 *     device share it, so prefill calls that overlap on the GPU race on it.
 *     qgemm_q4_0_noalloc uses a fixed array instead (below).
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QGEMV_OK = 0,
    QGEMV_ERR_NULL = 1,          /* a required pointer is NULL */
    QGEMV_ERR_SHAPE = 2,         /* negative size, or ncols % 32 != 0, or too large */
    QGEMV_ERR_BATCH = 3,         /* batch < 1 or batch > QGEMV_MAX_BATCH */
    QGEMV_ERR_ALIGN = 4,         /* a pointer is not 16-byte aligned */
    QGEMV_ERR_DTYPE = 5,         /* unknown output dtype */
    QGEMV_ERR_ARCH = 6,          /* current device is not sm_103 */
    QGEMV_ERR_LAUNCH = 7,        /* kernel launch failed */
    QGEMV_ERR_TIMEOUT = 8,       /* a kernel's bounded wait expired */
    QGEMV_ERR_UNIMPLEMENTED = 9, /* combination not built */
    QGEMV_ERR_CUDA = 10,         /* another CUDA runtime call failed */
    QGEMV_ERR_INDEX = 11         /* an expert id outside [0, n_expert) (device-detected) */
} qgemv_status;

typedef enum { QGEMV_F32 = 0, QGEMV_F16 = 1 } qgemv_out_dtype;

#define QGEMV_QK 32
#define QGEMV_MAX_BATCH 8
#define QGEMV_MAX_ID_BATCH 64

/* ------------------------------------------------------------ dequantize
 * Standalone dequantization (the to-fp16 / to-fp32 converters of the
 * dequantize_block_q4_0 / _q4_1 / _q8_0_f16 hunks).
 *   W    : nrows * (ncols/32) blocks, row-major, as above.
 *   out  : nrows x ncols row-major, fp32 (out_dtype = QGEMV_F32) or fp16
 *          (QGEMV_F16: round-to-nearest-even of the fp32 value).
 * Bit-exact: every output equals the IEEE evaluation of the formula above
 * (Q4_0 d*(q-8), Q4_1 fl(fl(d*q)+m), Q8_0 d*q), with no fused multiply-add.
 * NaN outputs (only possible for NaN/Inf scales) are NaN, payload unspecified.
 */
qgemv_status qdequant_q4_0(const void *W, void *out, int64_t nrows, int64_t ncols,
                           int out_dtype, void *stream);
qgemv_status qdequant_q4_1(const void *W, void *out, int64_t nrows, int64_t ncols,
                           int out_dtype, void *stream);
qgemv_status qdequant_q8_0(const void *W, void *out, int64_t nrows, int64_t ncols,
                           int out_dtype, void *stream);

/* ------------------------------------------------------------------ GEMV
 * Decode / small-batch matrix-vector product (the batch-1 "dmmv" path and
 * its small-batch extension):  y[b][r] = sum_k w[r][k] * x[b][k].
 *   x     : fp32 [batch][ncols] row-major.
 *   y     : fp32 [batch][nrows] row-major, overwritten (not accumulated).
 *   batch : 1 .. QGEMV_MAX_BATCH.
 * Accuracy: |y - exact| <= 1e-3 * sum_k |w[r][k] x[b][k]| + 1e-6 per
 * element for all finite W and x.  The default kernel for ncols a multiple
 * of 1024 (tensor cores, fp32 accumulation) multiplies the weights' exact
 * small integer codes (q - 8 for Q4_0; q - q0 for Q4_1, with q0 the code
 * nearest -m/d of the block, so that d * sum((q - q0) x) and (m + d q0) *
 * sum(x) cannot cancel; q for Q8_0) by x scaled per 128 values by a power of
 * two and rounded to fp16 (relative error <= 2^-11); a group of 128 values
 * whose magnitudes span more than fp16 keeps (a non-finite value, or a
 * nonzero value 2^23 or more below the group's largest) is computed exactly
 * in fp32 instead.  The other kernels compute each weight exactly in fp32.
 * Non-finite inputs give non-finite outputs in the rows they reach.
 * Activations are never quantized to integers below 11 significant bits: a
 * fixed-point kernel (24-bit per-block fixed point contracted with integer
 * dot products, small or non-finite elements exactly in fp32) exists as an
 * alternative path with the same bound.  Deterministic: the same inputs give
 * the same bits on every call.
 */
qgemv_status qgemv_q4_0(const void *W, const float *x, float *y, int64_t nrows,
                        int64_t ncols, int batch, void *stream);
qgemv_status qgemv_q4_1(const void *W, const float *x, float *y, int64_t nrows,
                        int64_t ncols, int batch, void *stream);
qgemv_status qgemv_q8_0(const void *W, const float *x, float *y, int64_t nrows,
                        int64_t ncols, int batch, void *stream);

/* ------------------------------------------- quantized-activation GEMV
 * The pages' second decode family, mul_mat_vec_q (ggml_cuda_op_mul_mat_vec_q
 * and the "MMVQ = mul_mat_vec_q" note): ggml_cuda_op_mul_mat first converts
 * the activations to int8 blocks (its convert_src1_to_q8_1 flag) so that they
 * meet the weights' integer codes in byte-wise integer dot products (the
 * __dp4a note beside MIN_CC_DP4A).  The pages print neither the activation
 * block layout nor its quantizer; this library's reading, for every 32
 * consecutive values x_i of one batch column:
 *     amax = max |x_i|,   d = amax / 127   (fp32 division, round to nearest),
 *     q_i  = x_i / d (fp32 division) rounded to nearest, ties to even, then
 *            clamped to [-127, 127];  q_i = 0 when d == 0,
 *     a block holding a NaN or an infinity gets d = NaN and q_i = 0,
 *     s    = sum_i q_i (exact).
 * Quantized activations of `batch` columns of ncols values form one device
 * buffer xq of qgemv_q8_1_size(ncols, batch) = batch*ncols*5/4 bytes:
 *     int8  q[batch][ncols]       at byte 0,
 *     fp32  d[batch][ncols/32]    at byte batch*ncols,
 *     int32 s[batch][ncols/32]    right after d.
 * xq must be 16-byte aligned; batch is 1 .. QGEMV_MAX_BATCH.
 *
 * qquantize_q8_1: x fp32 [batch][ncols] -> xq, bit-exact to the reading.
 * qgemv_mmvq_xq_*: with xhat[b][k] = d[b][k/32] * q[b][k],
 *     y[b][r] = sum_k w[r][k] * xhat[b][k],
 *   evaluated block by block as d_w*(sum c*q - 8*s)*d_x (Q4_0),
 *   (d_w*sum c*q + m_w*s)*d_x (Q4_1) or d_w*(sum c*q)*d_x (Q8_0), where c are
 *   the weights' integer codes: the integer sums are exact, the block terms
 *   are accumulated in fp32, and |y - exact| <= 1e-5 * sum_k |w xhat| + 1e-30.
 *   Deterministic.  Shapes with ncols % 64 == 0 and row bytes a multiple of
 *   16 (ncols % 256 == 0 for Q4_0 and Q8_0, % 128 for Q4_1) run the streaming
 *   kernel; all others a general one.
 * qgemv_mmvq_*: both steps in one call (two kernels on `stream`).  The
 *   quantized activations go to a fixed library-owned __device__ array of
 *   2^21 activations (2.5 MiB, held by every GPU that loads the library):
 *   batch * ncols must not exceed 2097152 (QGEMV_ERR_SHAPE otherwise), and
 *   calls that overlap on the GPU race on the array.  No allocation.
 * Against the plain product of x (what qgemv_* computes), the activation
 * rounding adds at most (amax_j / 254) * sum_{k in block j} |w[r][k]| per
 * block (times 1 + 2^-14): this family is NOT held to the qgemv_* bound.
 */
int64_t qgemv_q8_1_size(int64_t ncols, int batch);
qgemv_status qquantize_q8_1(const float *x, void *xq, int64_t ncols, int batch, void *stream);
qgemv_status qgemv_mmvq_xq_q4_0(const void *W, const void *xq, float *y, int64_t nrows,
                                int64_t ncols, int batch, void *stream);
qgemv_status qgemv_mmvq_xq_q4_1(const void *W, const void *xq, float *y, int64_t nrows,
                                int64_t ncols, int batch, void *stream);
qgemv_status qgemv_mmvq_xq_q8_0(const void *W, const void *xq, float *y, int64_t nrows,
                                int64_t ncols, int batch, void *stream);
qgemv_status qgemv_mmvq_q4_0(const void *W, const float *x, float *y, int64_t nrows,
                             int64_t ncols, int batch, void *stream);
qgemv_status qgemv_mmvq_q4_1(const void *W, const float *x, float *y, int64_t nrows,
                             int64_t ncols, int batch, void *stream);
qgemv_status qgemv_mmvq_q8_0(const void *W, const float *x, float *y, int64_t nrows,
                             int64_t ncols, int batch, void *stream);

/* ------------------------------------------------- expert-selected GEMV
 * The mixture-of-experts decode product (the ggml_cuda_mul_mat_id hunk and
 * the GGML_OP_MUL_MAT_ID cases of the "llama_cpp 0.12.1 -> 0.12.2" page; the
 * ffn_(up|gate|down)_exps expert tensors of the tensor-parallel split rules
 * on the "backend-agnostic tensor parallelism" page).  The pages name the
 * operation without printing it; the reading implemented here:
 *   W       : n_expert matrices of nrows x ncols, one after the other, each
 *             in the layout above (expert e starts at byte
 *             e * nrows * (ncols/32) * block bytes).
 *   ids     : int32 [batch], DEVICE memory (e.g. written by the router's
 *             top-k kernel just before): output column b uses expert ids[b].
 *   x       : fp32 [batch / x_group][ncols]; output column b reads row
 *             b / x_group.  x_group = experts per token for the up and gate
 *             projections (a token's experts share its activations), 1 for
 *             the down projection (one row per output column).
 *   y       : fp32 [batch][nrows]: y[b][r] = sum_k w_{ids[b]}[r][k] * x[b / x_group][k].
 *   batch   : 1 .. QGEMV_MAX_ID_BATCH (tokens x experts per token), a
 *             multiple of x_group (QGEMV_ERR_BATCH otherwise).
 * Accuracy as for qgemv_* (every element enters with relative error <=
 * 2^-11 or exactly), deterministic.  The columns that select the same expert
 * are grouped on the device into work units so that expert's weights stream
 * once for them; experts no column selects are not read.  Kernels: with
 * more than 2 columns and ncols a multiple of 1024, the tensor-core GEMV
 * (units of up to 8 columns in the MMA's N dimension); otherwise the
 * fixed-point streaming GEMV (units of up to 4 columns; ncols % 64 == 0, row
 * bytes a multiple of 16, a column's activations within shared memory); all
 * other shapes a general kernel with the same result bound.
 * An id outside [0, n_expert) is detected on the device: that column of y is
 * not written, the others are, and qgemv_sync_check() returns
 * QGEMV_ERR_INDEX.  ids, x, y and W must be 16-byte aligned.  ncols == 0:
 * y is zeroed and ids are not read.  No allocation.
 */
qgemv_status qgemv_id_q4_0(const void *W, int64_t n_expert, const int32_t *ids, const float *x,
                           int x_group, float *y, int64_t nrows, int64_t ncols, int batch,
                           void *stream);
qgemv_status qgemv_id_q4_1(const void *W, int64_t n_expert, const int32_t *ids, const float *x,
                           int x_group, float *y, int64_t nrows, int64_t ncols, int batch,
                           void *stream);
qgemv_status qgemv_id_q8_0(const void *W, int64_t n_expert, const int32_t *ids, const float *x,
                           int x_group, float *y, int64_t nrows, int64_t ncols, int batch,
                           void *stream);

/* ------------------------------------------------------------------ GEMM
 * Prefill matmul (the role of mul_mat_q for many tokens):
 *   Y[i][n] = sum_k X[i][k] * w[n][k]
 *   X : bfloat16 [m][ncols] row-major (bit patterns, 2 bytes each).
 *   Y : fp32 [m][nrows] row-major, overwritten.
 * Runs on the tensor cores (tcgen05, fp32 TMEM accumulators) with fp16
 * operands: each token row of X is scaled by the power of two that puts its
 * largest magnitude in [2^14, 2^15) and converted to fp16 (exact for every
 * value at least 2^-28 times the row's largest, and for any finite bf16
 * magnitude), w = d*(q-8) etc. is rounded to fp16 (relative error <= 2^-11),
 * and each output row is scaled back.  Accuracy as for GEMV for every finite
 * X whose rows keep their nonzero magnitudes within a factor 2^28 of the
 * row's largest; values further below it are lost (exactly as in an fp16
 * cast of the scaled row).  Requires ncols % 64 == 0 (QGEMV_ERR_SHAPE
 * otherwise).
 */
qgemv_status qgemm_q4_0(const void *W, const void *X_bf16, float *Y, int64_t nrows,
                        int64_t ncols, int64_t m, void *stream);
qgemv_status qgemm_q4_1(const void *W, const void *X_bf16, float *Y, int64_t nrows,
                        int64_t ncols, int64_t m, void *stream);
qgemv_status qgemm_q8_0(const void *W, const void *X_bf16, float *Y, int64_t nrows,
                        int64_t ncols, int64_t m, void *stream);

/* Allocation-free Q4_0 prefill.  The pages have no counterpart: this entry
 * point exists for callers that cannot let a library call cudaMalloc --
 * runtimes that reserve all their device memory up front and treat a later
 * allocation as a fault, and latency-critical callers that cannot accept the
 * device-wide synchronization cudaMalloc / cudaFree can imply.
 * Same arguments and result as qgemm_q4_0.  The fp16 copy of the activations
 * goes to a fixed 8 MiB __device__ array owned by the library, and its row
 * scales to a fixed 256 KiB one (every GPU that loads the library holds both
 * until exit), instead of the grown workspace:
 *   - m * ncols * 2 must not exceed 8 MiB (8388608); larger problems return
 *     QGEMV_ERR_SHAPE and launch nothing;
 *   - the first call on a device looks up the array's device address (with
 *     that device current) and configures the kernel; make that first call
 *     before any stream capture;
 *   - the call itself allocates no device memory and calls no allocating
 *     library routine;
 *   - all calls on a device share the array and each overwrites the part it
 *     uses, so calls that overlap on the GPU (e.g. on two streams) race. */
qgemv_status qgemm_q4_0_noalloc(const void *W, const void *X_bf16, float *Y, int64_t nrows,
                                int64_t ncols, int64_t m, void *stream);

/* ----------------------------------------------------------- launch option
 * QGEMV_OPT_WEIGHTS_STATIC (value 0 or 1, default 0).  The tensor-core GEMV
 * kernels are launched with programmatic dependent launch: a GEMV may begin
 * while the kernel launched just before it on the same stream is still
 * finishing, and waits for that kernel to complete before it reads x or
 * writes y.  With the option at 1 the GEMV also starts copying W before that
 * wait, which hides more of the previous kernel's tail.  Set it to 1 only if
 * no kernel that runs immediately before a qgemv_* call on the same stream
 * writes that call's W (weights uploaded with cudaMemcpy, or written by
 * kernels followed by any other call on the stream, qualify).  Process-wide,
 * all devices; takes effect on the next launch.  Unknown option or value:
 * QGEMV_ERR_DTYPE.
 */
#define QGEMV_OPT_WEIGHTS_STATIC 1
/* QGEMV_OPT_WAIT_PROBES (value >= 1, default 1048576).  How many times a GEMV
 * warp probes a weight copy that has not landed before it gives up; the warp
 * sleeps at most 256 ns between probes, so the default bounds a wait near a
 * quarter of a second.  A call whose wait gives up writes unspecified values
 * to y, sets the device error word (qgemv_sync_check() then returns
 * QGEMV_ERR_TIMEOUT and resets the GEMV's internal counters) and leaves the
 * device usable.  Process-wide; takes effect on the next launch. */
#define QGEMV_OPT_WAIT_PROBES 2
/* QGEMV_OPT_TEST_WITHHOLD_COPY (value 1; for testing the timeout path only).
 * The next qgemv_* call that runs on the default GEMV kernel (ncols a
 * multiple of 1024), or the next qgemv_mmvq_* or qgemv_id_* call that runs on
 * its streaming kernel, never issues its first weight copy, so the warps waiting
 * for it give up after QGEMV_OPT_WAIT_PROBES probes exactly as they would on a
 * copy that never lands.  One-shot: cleared by that call. */
#define QGEMV_OPT_TEST_WITHHOLD_COPY 3
qgemv_status qgemv_set_option(int option, int value);

/* ------------------------------------------------------------- utilities */

/* Static text for a status code ("QGEMV_OK", ...). */
const char *qgemv_status_string(int status);

/* Detail of the most recent failure in the calling thread (empty if none). */
const char *qgemv_last_error_string(void);

/* Synchronizes the current device, then reads and clears its kernel error
 * word: QGEMV_ERR_TIMEOUT if a kernel's bounded wait expired since the last
 * check, else QGEMV_ERR_INDEX if an expert-selected GEMV met an id out of
 * range, QGEMV_ERR_CUDA if synchronization failed, else QGEMV_OK. */
qgemv_status qgemv_sync_check(void);

/* Library version as 10000*major + 100*minor + patch. */
int qgemv_version(void);

/* Frees the library-owned per-device workspaces (safe to call repeatedly). */
void qgemv_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_H */
