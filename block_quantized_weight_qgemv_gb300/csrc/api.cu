// api.cu -- the extern "C" boundary of libqgemv: argument validation, device
// checks, error reporting and dispatch to the kernel launchers.
//
// Every entry point validates on the host before launching anything; no
// entry point aborts, traps or prints.  See include/qgemv.h for the contract.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "qgemv_common.cuh"

namespace qg {

// Kernel error word of each device (a separate instance per device context).
__device__ unsigned int g_qgemv_error_word = 0;

namespace {
thread_local char t_last_error[512] = {0};

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
bool g_dev_valid[kMaxDevices] = {false};
DevInfo g_dev_info[kMaxDevices];
unsigned *g_err_addr[kMaxDevices] = {nullptr};

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

void set_last_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
    va_end(ap);
}

qgemv_status check_launch(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_last_error("%s: launch failed: %s", what, cudaGetErrorString(e));
        if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction) {
            return QGEMV_ERR_ARCH;
        }
        return QGEMV_ERR_LAUNCH;
    }
    return QGEMV_OK;
}

qgemv_status current_device(DevInfo *info, int *dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_last_error("cudaGetDevice: %s", cudaGetErrorString(e));
        return QGEMV_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        set_last_error("device ordinal %d out of range", dev);
        return QGEMV_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_dev_mutex);
    if (!g_dev_valid[dev]) {
        DevInfo d{};
        int v = 0;
        if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
            set_last_error("cudaDeviceGetAttribute failed on device %d", dev);
            return QGEMV_ERR_CUDA;
        }
        d.smem_optin = static_cast<size_t>(v);
        void *addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_qgemv_error_word);
        if (e != cudaSuccess) {
            set_last_error("cudaGetSymbolAddress(error word): %s", cudaGetErrorString(e));
            return e == cudaErrorNoKernelImageForDevice ? QGEMV_ERR_ARCH : QGEMV_ERR_CUDA;
        }
        g_err_addr[dev] = static_cast<unsigned *>(addr);
        g_dev_info[dev] = d;
        g_dev_valid[dev] = true;
    }
    *info = g_dev_info[dev];
    *dev_out = dev;
    if (!(info->major == 10 && info->minor == 3)) {
        set_last_error("device %d has compute capability %d.%d; libqgemv is built for sm_103a only",
                       dev, info->major, info->minor);
        return QGEMV_ERR_ARCH;
    }
    return QGEMV_OK;
}

unsigned *device_error_word(int dev) { return g_err_addr[dev]; }

}  // namespace qg

using namespace qg;

namespace {

qgemv_status dequant_entry(int fmt, const void *W, void *out, int64_t nrows, int64_t ncols,
                           int out_dtype, void *stream) {
    t_last_error[0] = 0;
    if (out_dtype != QGEMV_F32 && out_dtype != QGEMV_F16) {
        set_last_error("out_dtype %d is neither QGEMV_F32 nor QGEMV_F16", out_dtype);
        return QGEMV_ERR_DTYPE;
    }
    if (nrows < 0 || ncols < 0 || ncols % QGEMV_QK != 0) {
        set_last_error("bad shape nrows=%lld ncols=%lld (ncols must be a non-negative multiple of 32)",
                       (long long)nrows, (long long)ncols);
        return QGEMV_ERR_SHAPE;
    }
    // element count must fit the kernels' 64-bit indexing with headroom
    if (ncols > 0 && nrows > (int64_t(1) << 40) / ncols) {
        set_last_error("problem too large: %lld x %lld", (long long)nrows, (long long)ncols);
        return QGEMV_ERR_SHAPE;
    }
    if (nrows == 0 || ncols == 0) return QGEMV_OK;
    if (!W || !out) {
        set_last_error("null pointer (W=%p out=%p)", W, out);
        return QGEMV_ERR_NULL;
    }
    if (!aligned16(W) || !aligned16(out)) {
        set_last_error("W and out must be 16-byte aligned (W=%p out=%p)", W, out);
        return QGEMV_ERR_ALIGN;
    }
    DevInfo di;
    int dev;
    qgemv_status st = current_device(&di, &dev);
    if (st != QGEMV_OK) return st;
    return launch_dequant(fmt, W, out, nrows, ncols, out_dtype == QGEMV_F16,
                          static_cast<cudaStream_t>(stream), di);
}

qgemv_status gemv_entry(int fmt, const void *W, const float *x, float *y, int64_t nrows,
                        int64_t ncols, int batch, void *stream) {
    t_last_error[0] = 0;
    if (nrows < 0 || ncols < 0 || ncols % QGEMV_QK != 0) {
        set_last_error("bad shape nrows=%lld ncols=%lld (ncols must be a non-negative multiple of 32)",
                       (long long)nrows, (long long)ncols);
        return QGEMV_ERR_SHAPE;
    }
    if (nrows > (int64_t(1) << 31) - 1 || ncols > (int64_t(1) << 24)) {
        set_last_error("problem too large: nrows=%lld (max 2^31-1) ncols=%lld (max 2^24)",
                       (long long)nrows, (long long)ncols);
        return QGEMV_ERR_SHAPE;
    }
    if (batch < 1 || batch > QGEMV_MAX_BATCH) {
        set_last_error("batch %d outside 1..%d", batch, QGEMV_MAX_BATCH);
        return QGEMV_ERR_BATCH;
    }
    if (nrows == 0) return QGEMV_OK;
    if (!W || !x || !y) {
        set_last_error("null pointer (W=%p x=%p y=%p)", W, (const void *)x, (void *)y);
        return QGEMV_ERR_NULL;
    }
    if (!aligned16(W) || !aligned16(x) || !aligned16(y)) {
        set_last_error("W, x and y must be 16-byte aligned");
        return QGEMV_ERR_ALIGN;
    }
    DevInfo di;
    int dev;
    qgemv_status st = current_device(&di, &dev);
    if (st != QGEMV_OK) return st;
    return launch_gemv(fmt, W, x, y, nrows, ncols, batch, static_cast<cudaStream_t>(stream), di, dev,
                       device_error_word(dev));
}

qgemv_status gemm_entry(int fmt, const void *W, const void *X, float *Y, int64_t nrows,
                        int64_t ncols, int64_t m, void *stream) {
    t_last_error[0] = 0;
    if (nrows < 0 || ncols < 0 || m < 0 || ncols % 64 != 0) {
        set_last_error("bad shape nrows=%lld ncols=%lld m=%lld (ncols must be a non-negative multiple of 64)",
                       (long long)nrows, (long long)ncols, (long long)m);
        return QGEMV_ERR_SHAPE;
    }
    if (nrows > (int64_t(1) << 31) - 1 || m > (int64_t(1) << 31) - 1 || ncols > (int64_t(1) << 24)) {
        set_last_error("problem too large");
        return QGEMV_ERR_SHAPE;
    }
    if (nrows == 0 || m == 0) return QGEMV_OK;
    if (!W || !X || !Y) {
        set_last_error("null pointer (W=%p X=%p Y=%p)", W, X, (void *)Y);
        return QGEMV_ERR_NULL;
    }
    if (!aligned16(W) || !aligned16(X) || !aligned16(Y)) {
        set_last_error("W, X and Y must be 16-byte aligned");
        return QGEMV_ERR_ALIGN;
    }
    DevInfo di;
    int dev;
    qgemv_status st = current_device(&di, &dev);
    if (st != QGEMV_OK) return st;
    return launch_gemm(fmt, W, X, Y, nrows, ncols, m, static_cast<cudaStream_t>(stream), di, dev);
}

// Shared checks of the quantized-activation calls: shape, batch, and
// whether the problem is empty (*empty = true: return OK, launch nothing).
qgemv_status mmvq_check_shape(const char *what, int64_t nrows, int64_t ncols, int batch, bool *empty) {
    t_last_error[0] = 0;
    *empty = false;
    if (nrows < 0 || ncols < 0 || ncols % QGEMV_QK != 0) {
        set_last_error("%s: bad shape nrows=%lld ncols=%lld (ncols must be a non-negative multiple of 32)", what,
                       (long long)nrows, (long long)ncols);
        return QGEMV_ERR_SHAPE;
    }
    if (nrows > (int64_t(1) << 31) - 1 || ncols > (int64_t(1) << 24)) {
        set_last_error("%s: problem too large: nrows=%lld (max 2^31-1) ncols=%lld (max 2^24)", what,
                       (long long)nrows, (long long)ncols);
        return QGEMV_ERR_SHAPE;
    }
    if (batch < 1 || batch > QGEMV_MAX_BATCH) {
        set_last_error("%s: batch %d outside 1..%d", what, batch, QGEMV_MAX_BATCH);
        return QGEMV_ERR_BATCH;
    }
    *empty = nrows == 0 || ncols == 0;
    return QGEMV_OK;
}

qgemv_status mmvq_xq_entry(int fmt, const void *W, const void *xq, float *y, int64_t nrows, int64_t ncols,
                           int batch, void *stream) {
    bool empty;
    qgemv_status st = mmvq_check_shape("qgemv_mmvq_xq", nrows, ncols, batch, &empty);
    if (st != QGEMV_OK) return st;
    if (nrows == 0) return QGEMV_OK;
    if (!W || !xq || !y) {
        set_last_error("null pointer (W=%p xq=%p y=%p)", W, xq, (void *)y);
        return QGEMV_ERR_NULL;
    }
    if (!aligned16(W) || !aligned16(xq) || !aligned16(y)) {
        set_last_error("W, xq and y must be 16-byte aligned");
        return QGEMV_ERR_ALIGN;
    }
    DevInfo di;
    int dev;
    st = current_device(&di, &dev);
    if (st != QGEMV_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (ncols == 0) {
        cudaError_t e = cudaMemsetAsync(y, 0, sizeof(float) * static_cast<size_t>(nrows) * batch, s);
        if (e != cudaSuccess) {
            set_last_error("cudaMemsetAsync: %s", cudaGetErrorString(e));
            return QGEMV_ERR_CUDA;
        }
        return QGEMV_OK;
    }
    return launch_gemv_mmvq(fmt, W, xq, y, nrows, ncols, batch, s, di, dev, device_error_word(dev));
}

qgemv_status mmvq_entry(int fmt, const void *W, const float *x, float *y, int64_t nrows, int64_t ncols, int batch,
                        void *stream) {
    bool empty;
    qgemv_status st = mmvq_check_shape("qgemv_mmvq", nrows, ncols, batch, &empty);
    if (st != QGEMV_OK) return st;
    if (static_cast<int64_t>(batch) * ncols > mmvq_scratch_values()) {
        set_last_error("qgemv_mmvq: batch * ncols = %lld exceeds the fixed scratch of %lld activations "
                       "(quantize into a buffer of your own with qquantize_q8_1 and call qgemv_mmvq_xq_*)",
                       (long long)(static_cast<int64_t>(batch) * ncols), (long long)mmvq_scratch_values());
        return QGEMV_ERR_SHAPE;
    }
    if (nrows == 0) return QGEMV_OK;
    if (!W || !x || !y) {
        set_last_error("null pointer (W=%p x=%p y=%p)", W, (const void *)x, (void *)y);
        return QGEMV_ERR_NULL;
    }
    if (!aligned16(W) || !aligned16(x) || !aligned16(y)) {
        set_last_error("W, x and y must be 16-byte aligned");
        return QGEMV_ERR_ALIGN;
    }
    DevInfo di;
    int dev;
    st = current_device(&di, &dev);
    if (st != QGEMV_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (ncols == 0) {
        cudaError_t e = cudaMemsetAsync(y, 0, sizeof(float) * static_cast<size_t>(nrows) * batch, s);
        if (e != cudaSuccess) {
            set_last_error("cudaMemsetAsync: %s", cudaGetErrorString(e));
            return QGEMV_ERR_CUDA;
        }
        return QGEMV_OK;
    }
    void *xq = nullptr;
    st = mmvq_scratch(&xq);
    if (st != QGEMV_OK) return st;
    st = launch_quantize_q8_1(x, xq, ncols, batch, s);
    if (st != QGEMV_OK) return st;
    return launch_gemv_mmvq(fmt, W, xq, y, nrows, ncols, batch, s, di, dev, device_error_word(dev));
}

qgemv_status id_entry(int fmt, const void *W, int64_t n_expert, const int32_t *ids, const float *x, int x_group,
                      float *y, int64_t nrows, int64_t ncols, int batch, void *stream) {
    t_last_error[0] = 0;
    if (nrows < 0 || ncols < 0 || ncols % QGEMV_QK != 0 || n_expert < 1) {
        set_last_error("qgemv_id: bad shape nrows=%lld ncols=%lld n_expert=%lld (ncols a non-negative multiple "
                       "of 32, n_expert >= 1)", (long long)nrows, (long long)ncols, (long long)n_expert);
        return QGEMV_ERR_SHAPE;
    }
    if (nrows > (int64_t(1) << 31) - 1 || ncols > (int64_t(1) << 24) || n_expert > (int64_t(1) << 31) - 1 ||
        (ncols > 0 && nrows > 0 && n_expert > (int64_t(1) << 56) / (nrows * (ncols / 32) * 34))) {
        set_last_error("qgemv_id: problem too large");
        return QGEMV_ERR_SHAPE;
    }
    if (batch < 1 || batch > QGEMV_MAX_ID_BATCH || x_group < 1 || batch % x_group != 0) {
        set_last_error("qgemv_id: batch %d outside 1..%d or not a multiple of x_group %d", batch,
                       QGEMV_MAX_ID_BATCH, x_group);
        return QGEMV_ERR_BATCH;
    }
    if (nrows == 0) return QGEMV_OK;
    if (!W || !ids || !x || !y) {
        set_last_error("null pointer (W=%p ids=%p x=%p y=%p)", W, (const void *)ids, (const void *)x, (void *)y);
        return QGEMV_ERR_NULL;
    }
    if (!aligned16(W) || !aligned16(ids) || !aligned16(x) || !aligned16(y)) {
        set_last_error("W, ids, x and y must be 16-byte aligned");
        return QGEMV_ERR_ALIGN;
    }
    DevInfo di;
    int dev;
    qgemv_status st = current_device(&di, &dev);
    if (st != QGEMV_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (ncols == 0) {
        cudaError_t e = cudaMemsetAsync(y, 0, sizeof(float) * static_cast<size_t>(nrows) * batch, s);
        if (e != cudaSuccess) {
            set_last_error("cudaMemsetAsync: %s", cudaGetErrorString(e));
            return QGEMV_ERR_CUDA;
        }
        return QGEMV_OK;
    }
    return launch_gemv_id(fmt, W, n_expert, ids, x, x_group, y, nrows, ncols, batch, s, di, dev,
                          device_error_word(dev));
}

}  // namespace

extern "C" {

qgemv_status qgemv_id_q4_0(const void *W, int64_t n_expert, const int32_t *ids, const float *x, int x_group,
                           float *y, int64_t nrows, int64_t ncols, int batch, void *stream) {
    return id_entry(FMT_Q4_0, W, n_expert, ids, x, x_group, y, nrows, ncols, batch, stream);
}
qgemv_status qgemv_id_q4_1(const void *W, int64_t n_expert, const int32_t *ids, const float *x, int x_group,
                           float *y, int64_t nrows, int64_t ncols, int batch, void *stream) {
    return id_entry(FMT_Q4_1, W, n_expert, ids, x, x_group, y, nrows, ncols, batch, stream);
}
qgemv_status qgemv_id_q8_0(const void *W, int64_t n_expert, const int32_t *ids, const float *x, int x_group,
                           float *y, int64_t nrows, int64_t ncols, int batch, void *stream) {
    return id_entry(FMT_Q8_0, W, n_expert, ids, x, x_group, y, nrows, ncols, batch, stream);
}

int64_t qgemv_q8_1_size(int64_t ncols, int batch) {
    if (ncols < 0 || ncols % QGEMV_QK != 0 || batch < 1) return -1;
    return q8_1_bytes(ncols, batch);
}

qgemv_status qquantize_q8_1(const float *x, void *xq, int64_t ncols, int batch, void *stream) {
    bool empty;
    qgemv_status st = mmvq_check_shape("qquantize_q8_1", 1, ncols, batch, &empty);
    if (st != QGEMV_OK) return st;
    if (empty) return QGEMV_OK;
    if (!x || !xq) {
        set_last_error("null pointer (x=%p xq=%p)", (const void *)x, xq);
        return QGEMV_ERR_NULL;
    }
    if (!aligned16(x) || !aligned16(xq)) {
        set_last_error("x and xq must be 16-byte aligned");
        return QGEMV_ERR_ALIGN;
    }
    DevInfo di;
    int dev;
    st = current_device(&di, &dev);
    if (st != QGEMV_OK) return st;
    return launch_quantize_q8_1(x, xq, ncols, batch, static_cast<cudaStream_t>(stream));
}

qgemv_status qgemv_mmvq_xq_q4_0(const void *W, const void *xq, float *y, int64_t nrows, int64_t ncols, int batch,
                                void *stream) {
    return mmvq_xq_entry(FMT_Q4_0, W, xq, y, nrows, ncols, batch, stream);
}
qgemv_status qgemv_mmvq_xq_q4_1(const void *W, const void *xq, float *y, int64_t nrows, int64_t ncols, int batch,
                                void *stream) {
    return mmvq_xq_entry(FMT_Q4_1, W, xq, y, nrows, ncols, batch, stream);
}
qgemv_status qgemv_mmvq_xq_q8_0(const void *W, const void *xq, float *y, int64_t nrows, int64_t ncols, int batch,
                                void *stream) {
    return mmvq_xq_entry(FMT_Q8_0, W, xq, y, nrows, ncols, batch, stream);
}
qgemv_status qgemv_mmvq_q4_0(const void *W, const float *x, float *y, int64_t nrows, int64_t ncols, int batch,
                             void *stream) {
    return mmvq_entry(FMT_Q4_0, W, x, y, nrows, ncols, batch, stream);
}
qgemv_status qgemv_mmvq_q4_1(const void *W, const float *x, float *y, int64_t nrows, int64_t ncols, int batch,
                             void *stream) {
    return mmvq_entry(FMT_Q4_1, W, x, y, nrows, ncols, batch, stream);
}
qgemv_status qgemv_mmvq_q8_0(const void *W, const float *x, float *y, int64_t nrows, int64_t ncols, int batch,
                             void *stream) {
    return mmvq_entry(FMT_Q8_0, W, x, y, nrows, ncols, batch, stream);
}

qgemv_status qdequant_q4_0(const void *W, void *out, int64_t nrows, int64_t ncols, int out_dtype, void *stream) {
    return dequant_entry(FMT_Q4_0, W, out, nrows, ncols, out_dtype, stream);
}
qgemv_status qdequant_q4_1(const void *W, void *out, int64_t nrows, int64_t ncols, int out_dtype, void *stream) {
    return dequant_entry(FMT_Q4_1, W, out, nrows, ncols, out_dtype, stream);
}
qgemv_status qdequant_q8_0(const void *W, void *out, int64_t nrows, int64_t ncols, int out_dtype, void *stream) {
    return dequant_entry(FMT_Q8_0, W, out, nrows, ncols, out_dtype, stream);
}

qgemv_status qgemv_q4_0(const void *W, const float *x, float *y, int64_t nrows, int64_t ncols, int batch, void *stream) {
    return gemv_entry(FMT_Q4_0, W, x, y, nrows, ncols, batch, stream);
}
qgemv_status qgemv_q4_1(const void *W, const float *x, float *y, int64_t nrows, int64_t ncols, int batch, void *stream) {
    return gemv_entry(FMT_Q4_1, W, x, y, nrows, ncols, batch, stream);
}
qgemv_status qgemv_q8_0(const void *W, const float *x, float *y, int64_t nrows, int64_t ncols, int batch, void *stream) {
    return gemv_entry(FMT_Q8_0, W, x, y, nrows, ncols, batch, stream);
}

qgemv_status qgemm_q4_0(const void *W, const void *X, float *Y, int64_t nrows, int64_t ncols, int64_t m, void *stream) {
    return gemm_entry(FMT_Q4_0, W, X, Y, nrows, ncols, m, stream);
}
qgemv_status qgemm_q4_1(const void *W, const void *X, float *Y, int64_t nrows, int64_t ncols, int64_t m, void *stream) {
    return gemm_entry(FMT_Q4_1, W, X, Y, nrows, ncols, m, stream);
}
qgemv_status qgemm_q8_0(const void *W, const void *X, float *Y, int64_t nrows, int64_t ncols, int64_t m, void *stream) {
    return gemm_entry(FMT_Q8_0, W, X, Y, nrows, ncols, m, stream);
}

qgemv_status qgemm_q4_0_noalloc(const void *W, const void *X, float *Y, int64_t nrows, int64_t ncols, int64_t m,
                                void *stream) {
    t_last_error[0] = 0;
    if (nrows < 0 || ncols < 0 || m < 0 || ncols % 64 != 0) {
        set_last_error("bad shape nrows=%lld ncols=%lld m=%lld (ncols must be a non-negative multiple of 64)",
                       (long long)nrows, (long long)ncols, (long long)m);
        return QGEMV_ERR_SHAPE;
    }
    if (nrows > (int64_t(1) << 31) - 1 || m > (int64_t(1) << 31) - 1 || ncols > (int64_t(1) << 24)) {
        set_last_error("problem too large");
        return QGEMV_ERR_SHAPE;
    }
    if (static_cast<uint64_t>(m) * static_cast<uint64_t>(ncols) * 2 > noalloc_scratch_bytes()) {
        set_last_error("qgemm_q4_0_noalloc: m * ncols * 2 = %llu bytes exceeds its fixed %zu-byte scratch",
                       (unsigned long long)(static_cast<uint64_t>(m) * static_cast<uint64_t>(ncols) * 2),
                       noalloc_scratch_bytes());
        return QGEMV_ERR_SHAPE;
    }
    if (nrows == 0 || m == 0) return QGEMV_OK;
    if (!W || !X || !Y) {
        set_last_error("null pointer (W=%p X=%p Y=%p)", W, X, (void *)Y);
        return QGEMV_ERR_NULL;
    }
    if (!aligned16(W) || !aligned16(X) || !aligned16(Y)) {
        set_last_error("W, X and Y must be 16-byte aligned");
        return QGEMV_ERR_ALIGN;
    }
    DevInfo di;
    int dev;
    qgemv_status st = current_device(&di, &dev);
    if (st != QGEMV_OK) return st;
    if (ncols == 0) {
        cudaError_t e = cudaMemsetAsync(Y, 0, sizeof(float) * static_cast<size_t>(nrows) * m,
                                        static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) {
            set_last_error("cudaMemsetAsync: %s", cudaGetErrorString(e));
            return QGEMV_ERR_CUDA;
        }
        return QGEMV_OK;
    }
    return launch_gemm_q4_0_noalloc(W, X, Y, nrows, ncols, m, static_cast<cudaStream_t>(stream), di, dev,
                                    device_error_word(dev));
}

const char *qgemv_status_string(int status) {
    switch (status) {
    case QGEMV_OK: return "QGEMV_OK";
    case QGEMV_ERR_NULL: return "QGEMV_ERR_NULL";
    case QGEMV_ERR_SHAPE: return "QGEMV_ERR_SHAPE";
    case QGEMV_ERR_BATCH: return "QGEMV_ERR_BATCH";
    case QGEMV_ERR_ALIGN: return "QGEMV_ERR_ALIGN";
    case QGEMV_ERR_DTYPE: return "QGEMV_ERR_DTYPE";
    case QGEMV_ERR_ARCH: return "QGEMV_ERR_ARCH";
    case QGEMV_ERR_LAUNCH: return "QGEMV_ERR_LAUNCH";
    case QGEMV_ERR_TIMEOUT: return "QGEMV_ERR_TIMEOUT";
    case QGEMV_ERR_UNIMPLEMENTED: return "QGEMV_ERR_UNIMPLEMENTED";
    case QGEMV_ERR_CUDA: return "QGEMV_ERR_CUDA";
    case QGEMV_ERR_INDEX: return "QGEMV_ERR_INDEX";
    default: return "QGEMV_ERR_UNKNOWN";
    }
}

const char *qgemv_last_error_string(void) { return t_last_error; }

qgemv_status qgemv_sync_check(void) {
    t_last_error[0] = 0;
    DevInfo di;
    int dev;
    qgemv_status st = current_device(&di, &dev);
    if (st != QGEMV_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        set_last_error("cudaDeviceSynchronize: %s", cudaGetErrorString(e));
        return QGEMV_ERR_CUDA;
    }
    unsigned word = 0;
    e = cudaMemcpyFromSymbol(&word, g_qgemv_error_word, sizeof(word));
    if (e == cudaSuccess && word != 0) {
        unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_qgemv_error_word, &zero, sizeof(zero));
    }
    if (e != cudaSuccess) {
        set_last_error("reading the kernel error word: %s", cudaGetErrorString(e));
        return QGEMV_ERR_CUDA;
    }
    if (word & ERRBIT_TIMEOUT) {
        // a GEMV that gave up may have left a split-tile counter mid-count
        gemv_sk_reset_scratch();
        set_last_error("a kernel's bounded wait on an asynchronous copy expired");
        return QGEMV_ERR_TIMEOUT;
    }
    if (word & ERRBIT_INDEX) {
        set_last_error("an expert-selected GEMV met an expert id outside [0, n_expert)");
        return QGEMV_ERR_INDEX;
    }
    return QGEMV_OK;
}

int qgemv_version(void) { return 100; }

qgemv_status qgemv_set_option(int option, int value) {
    if (option == QGEMV_OPT_WEIGHTS_STATIC && (value == 0 || value == 1)) {
        g_opt_weights_static = value;
        return QGEMV_OK;
    }
    if (option == QGEMV_OPT_WAIT_PROBES && value >= 1) {
        g_opt_wait_probes = static_cast<unsigned>(value);
        return QGEMV_OK;
    }
    if (option == QGEMV_OPT_TEST_WITHHOLD_COPY && (value == 0 || value == 1)) {
        g_opt_withhold_next = value;
        return QGEMV_OK;
    }
    set_last_error("unknown option %d or value %d", option, value);
    return QGEMV_ERR_DTYPE;
}

void qgemv_shutdown(void) { gemm_release_workspaces(); }

}  // extern "C"
