// gemm.cu -- prefill matmul on block-quantized weights:
//   Y[i][n] = sum_k X[i][k] * w[n][k],  X bf16 [m][ncols], Y fp32 [m][nrows]
// (the role of mul_mat_q in the "llama_cpp 0.12.1 -> 0.12.2" ggml-cuda.cu diff).
//
// Dispatch to the tensor-core kernel (gemm_tc.cu), plus a simple CUDA-core
// kernel (64 x 64 output tiles, one 32-wide block column of W dequantized into
// shared memory per step, fp32 FMA) kept as an independent cross-check.
#include <cstdlib>
#include <cstring>

#include "qgemv_common.cuh"

namespace qg {
namespace {

constexpr int kTM = 64;     // tokens per tile
constexpr int kTN = 64;     // weight rows per tile

template <int F>
__device__ __forceinline__ float decode_one(const uint8_t *b, int j) {
    const uint16_t *h = reinterpret_cast<const uint16_t *>(b);
    const float d = fp16_bits_to_f32(h[0]);
    if constexpr (F == FMT_Q8_0) {
        return d * static_cast<float>(static_cast<int8_t>(b[2 + j]));
    } else if constexpr (F == FMT_Q4_0) {
        const uint32_t q = (b[2 + (j & 15)] >> ((j & 16) ? 4 : 0)) & 15;
        return d * static_cast<float>(static_cast<int>(q) - 8);
    } else {
        const float m = fp16_bits_to_f32(h[1]);
        const uint32_t q = (b[4 + (j & 15)] >> ((j & 16) ? 4 : 0)) & 15;
        return __fadd_rn(__fmul_rn(d, static_cast<float>(q)), m);
    }
}

template <int F>
__global__ void __launch_bounds__(256)
gemm_simple_kernel(const uint8_t *__restrict__ W, const uint16_t *__restrict__ X, float *__restrict__ Y,
                   int nrows, int ncols, int m) {
    constexpr int BB = FmtInfo<F>::kBytes;
    __shared__ float ws[32][kTN + 1];
    __shared__ float xs[32][kTM + 1];
    const int n0 = blockIdx.x * kTN;
    const int m0 = blockIdx.y * kTM;
    const int tx = threadIdx.x & 15;     // n direction
    const int ty = threadIdx.x >> 4;     // m direction
    const int nb = ncols / 32;
    float acc[4][4] = {};
    for (int blk = 0; blk < nb; ++blk) {
        for (int i = threadIdx.x; i < 32 * kTN; i += 256) {
            const int nn = i >> 5, j = i & 31;
            const int n = n0 + nn;
            ws[j][nn] = (n < nrows) ? decode_one<F>(W + (static_cast<int64_t>(n) * nb + blk) * BB, j) : 0.0f;
        }
        for (int i = threadIdx.x; i < 32 * kTM; i += 256) {
            const int mm = i >> 5, j = i & 31;
            const int r = m0 + mm;
            float v = 0.0f;
            if (r < m) v = __uint_as_float(static_cast<uint32_t>(X[static_cast<int64_t>(r) * ncols + blk * 32 + j]) << 16);
            xs[j][mm] = v;
        }
        __syncthreads();
#pragma unroll 8
        for (int j = 0; j < 32; ++j) {
            float a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) { a[u] = xs[j][ty * 4 + u]; b[u] = ws[j][tx * 4 + u]; }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(a[u], b[v], acc[u][v]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int r = m0 + ty * 4 + u;
        if (r >= m) continue;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int n = n0 + tx * 4 + v;
            if (n < nrows) Y[static_cast<int64_t>(r) * nrows + n] = acc[u][v];
        }
    }
}

template <int F>
qgemv_status launch_simple(const void *W, const void *X, float *Y, int64_t nrows, int64_t ncols, int64_t m,
                           cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((nrows + kTN - 1) / kTN), static_cast<unsigned>((m + kTM - 1) / kTM));
    if (grid.y > 65535u) {
        set_last_error("m=%lld too large for the baseline prefill kernel", (long long)m);
        return QGEMV_ERR_SHAPE;
    }
    gemm_simple_kernel<F><<<grid, 256, 0, s>>>(static_cast<const uint8_t *>(W), static_cast<const uint16_t *>(X), Y,
                                                static_cast<int>(nrows), static_cast<int>(ncols), static_cast<int>(m));
    return check_launch("qgemm");
}

}  // namespace

qgemv_status launch_gemm(int fmt, const void *W, const void *X, float *Y, int64_t nrows, int64_t ncols,
                         int64_t m, cudaStream_t s, const DevInfo &di, int dev) {
    if (ncols == 0) {
        cudaError_t e = cudaMemsetAsync(Y, 0, sizeof(float) * static_cast<size_t>(nrows) * m, s);
        if (e != cudaSuccess) {
            set_last_error("cudaMemsetAsync: %s", cudaGetErrorString(e));
            return QGEMV_ERR_CUDA;
        }
        return QGEMV_OK;
    }
    // QGEMV_GEMM_PATH=simple selects the CUDA-core kernel (a cross-check of
    // the tensor-core kernel); the default is the tensor-core kernel.
    const char *path = getenv("QGEMV_GEMM_PATH");
    if (!(path && !strcmp(path, "simple"))) {
        return launch_gemm_tc(fmt, W, X, Y, nrows, ncols, m, s, di, dev, device_error_word(dev));
    }
    switch (fmt) {
    case FMT_Q4_0: return launch_simple<FMT_Q4_0>(W, X, Y, nrows, ncols, m, s);
    case FMT_Q4_1: return launch_simple<FMT_Q4_1>(W, X, Y, nrows, ncols, m, s);
    case FMT_Q8_0: return launch_simple<FMT_Q8_0>(W, X, Y, nrows, ncols, m, s);
    default:
        set_last_error("unknown format %d", fmt);
        return QGEMV_ERR_DTYPE;
    }
}

}  // namespace qg
