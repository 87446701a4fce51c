// gemv.cu -- decode / small-batch GEMV on block-quantized weights:
//   y[b][r] = sum_k w[r][k] * x[b][k]
// (the batch-1 fused dequantize + dot product named dequantize_mul_mat_vec in
// the "llama_cpp 0.12.1 -> 0.12.2" ggml-cuda.cu diff, extended to batch <= 8).
//
// Baseline kernel: one warp per row, lane j takes blocks j, j+32, ...; the
// block is decoded in registers and multiplied with fp32 activations; per-lane
// fp32 partial sums are reduced with a butterfly shuffle (the warp_reduce_sum
// pattern of the same diff).
#include "qgemv_common.cuh"

namespace qg {
namespace {

constexpr int kRowWarps = 8;

template <int F>
__device__ __forceinline__ void decode_block(const uint8_t *b, float w[32]) {
    const uint16_t *h = reinterpret_cast<const uint16_t *>(b);   // blocks are 2-byte aligned
    if constexpr (F == FMT_Q8_0) {
        const float d = fp16_bits_to_f32(h[0]);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t two = h[1 + i];
            w[2 * i] = d * static_cast<float>(static_cast<int8_t>(two & 0xff));
            w[2 * i + 1] = d * static_cast<float>(static_cast<int8_t>(two >> 8));
        }
    } else {
        constexpr int Q0 = (F == FMT_Q4_1) ? 2 : 1;               // first qs half-word
        const float d = fp16_bits_to_f32(h[0]);
        const float m = (F == FMT_Q4_1) ? fp16_bits_to_f32(h[1]) : -8.0f * d;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t two = h[Q0 + i];
            w[2 * i] = fmaf(d, static_cast<float>(two & 15), m);
            w[2 * i + 1] = fmaf(d, static_cast<float>((two >> 8) & 15), m);
            w[2 * i + 16] = fmaf(d, static_cast<float>((two >> 4) & 15), m);
            w[2 * i + 17] = fmaf(d, static_cast<float>((two >> 12) & 15), m);
        }
    }
}

template <int F, int NB>
__global__ void __launch_bounds__(kRowWarps * 32)
gemv_rowwarp_kernel(const uint8_t *__restrict__ W, const float *__restrict__ x, float *__restrict__ y,
                    int64_t nrows, int ncols) {
    constexpr int BB = FmtInfo<F>::kBytes;
    const int lane = threadIdx.x & 31;
    const int nb = ncols / 32;
    const int64_t rowbytes = static_cast<int64_t>(nb) * BB;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kRowWarps;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5); r < nrows; r += nwarps) {
        float acc[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
        const uint8_t *row = W + r * rowbytes;
        for (int blk = lane; blk < nb; blk += 32) {
            float w[32];
            decode_block<F>(row + static_cast<int64_t>(blk) * BB, w);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float4 *xv = reinterpret_cast<const float4 *>(x + static_cast<int64_t>(b) * ncols + blk * 32);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 xx = __ldg(xv + i);
                    acc[b] = fmaf(w[4 * i], xx.x, acc[b]);
                    acc[b] = fmaf(w[4 * i + 1], xx.y, acc[b]);
                    acc[b] = fmaf(w[4 * i + 2], xx.z, acc[b]);
                    acc[b] = fmaf(w[4 * i + 3], xx.w, acc[b]);
                }
            }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const float s = warp_sum(acc[b]);
            if (lane == 0) y[static_cast<int64_t>(b) * nrows + r] = s;
        }
    }
}

template <int F, int NB>
qgemv_status launch_rowwarp(const void *W, const float *x, float *y, int64_t nrows, int64_t ncols,
                            cudaStream_t s, const DevInfo &di) {
    int64_t ctas = (nrows + kRowWarps - 1) / kRowWarps;
    const int64_t cap = static_cast<int64_t>(di.sm_count) * 8;
    if (ctas > cap) ctas = cap;
    gemv_rowwarp_kernel<F, NB><<<static_cast<unsigned>(ctas), kRowWarps * 32, 0, s>>>(
        static_cast<const uint8_t *>(W), x, y, nrows, static_cast<int>(ncols));
    return check_launch("qgemv");
}

template <int F>
qgemv_status launch_fmt(const void *W, const float *x, float *y, int64_t nrows, int64_t ncols, int batch,
                        cudaStream_t s, const DevInfo &di) {
    switch (batch) {
    case 1: return launch_rowwarp<F, 1>(W, x, y, nrows, ncols, s, di);
    case 2: return launch_rowwarp<F, 2>(W, x, y, nrows, ncols, s, di);
    case 3: return launch_rowwarp<F, 3>(W, x, y, nrows, ncols, s, di);
    case 4: return launch_rowwarp<F, 4>(W, x, y, nrows, ncols, s, di);
    case 5: return launch_rowwarp<F, 5>(W, x, y, nrows, ncols, s, di);
    case 6: return launch_rowwarp<F, 6>(W, x, y, nrows, ncols, s, di);
    case 7: return launch_rowwarp<F, 7>(W, x, y, nrows, ncols, s, di);
    default: return launch_rowwarp<F, 8>(W, x, y, nrows, ncols, s, di);
    }
}

}  // namespace

qgemv_status launch_gemv(int fmt, const void *W, const float *x, float *y, int64_t nrows,
                         int64_t ncols, int batch, cudaStream_t s, const DevInfo &di, unsigned *err) {
    (void)err;
    if (ncols == 0) {
        // empty contraction: y = 0
        cudaError_t e = cudaMemsetAsync(y, 0, sizeof(float) * static_cast<size_t>(nrows) * batch, s);
        if (e != cudaSuccess) {
            set_last_error("cudaMemsetAsync: %s", cudaGetErrorString(e));
            return QGEMV_ERR_CUDA;
        }
        return QGEMV_OK;
    }
    switch (fmt) {
    case FMT_Q4_0: return launch_fmt<FMT_Q4_0>(W, x, y, nrows, ncols, batch, s, di);
    case FMT_Q4_1: return launch_fmt<FMT_Q4_1>(W, x, y, nrows, ncols, batch, s, di);
    case FMT_Q8_0: return launch_fmt<FMT_Q8_0>(W, x, y, nrows, ncols, batch, s, di);
    default:
        set_last_error("unknown format %d", fmt);
        return QGEMV_ERR_DTYPE;
    }
}

}  // namespace qg
