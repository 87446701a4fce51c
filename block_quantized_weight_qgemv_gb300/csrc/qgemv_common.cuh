// qgemv_common.cuh -- shared device/host helpers of libqgemv (sm_103a only).
//
// Inline-PTX wrappers for mbarriers and bulk asynchronous copies, the block
// format constants, and the per-device error word that kernels set instead of
// trapping when a bounded wait expires.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/qgemv.h"

namespace qg {

// ---------------------------------------------------------------- formats
enum Fmt { FMT_Q4_0 = 0, FMT_Q4_1 = 1, FMT_Q8_0 = 2 };

template <int F> struct FmtInfo;
template <> struct FmtInfo<FMT_Q4_0> { static constexpr int kBytes = 18; };
template <> struct FmtInfo<FMT_Q4_1> { static constexpr int kBytes = 20; };
template <> struct FmtInfo<FMT_Q8_0> { static constexpr int kBytes = 34; };

__host__ __device__ constexpr int block_bytes(int f) {
    return f == FMT_Q4_0 ? 18 : (f == FMT_Q4_1 ? 20 : 34);
}

// Bit flags stored in the per-device error word.
enum : unsigned { ERRBIT_TIMEOUT = 1u, ERRBIT_INDEX = 2u };   // INDEX: an expert id out of range

// Kernels receive the device address of the per-device error word (a
// __device__ variable of api.cu, looked up once per device with
// cudaGetSymbolAddress) and OR these flags into it.

// Spin limit for every mbarrier wait (each try_wait may itself suspend for
// a short, hardware-defined time).  Far above any legitimate wait.
constexpr uint32_t kSpinLimit = 1u << 22;

// ------------------------------------------------------------ mbarrier PTX
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}

// One probe of the barrier phase with the given parity; true once complete.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait: returns false (and flags the device error word) if the
// phase does not complete within kSpinLimit probes.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, unsigned *err) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
    }
    atomicOr(err, ERRBIT_TIMEOUT);
    return false;
}

// Same, but each probe may suspend the thread for up to `hint_ns` (it wakes
// as soon as the phase completes), so waiting warps stop competing for issue
// slots.  The total wait stays bounded by kSpinLimit probes.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns) : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity, unsigned *err) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
    }
    atomicOr(err, ERRBIT_TIMEOUT);
    return false;
}

// --------------------------------------------------- bulk async copy (TMA)
// 1-D bulk copy global -> shared, completion counted on an mbarrier in bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy / tensor core) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// CTA-wide barrier in its unaligned form, which counts arriving threads one
// by one.  The aligned form (bar.sync, __syncthreads) counts a whole warp
// each time any of its lanes executes it: a warp whose lanes reach it apart
// (lane 0 still initializing barriers or issuing copies) is counted twice and
// releases the barrier before every warp has arrived.
__device__ __forceinline__ void cta_sync() { asm volatile("barrier.sync 0;" ::: "memory"); }

// ------------------------------------------------------------ misc device
__device__ __forceinline__ float fp16_bits_to_f32(uint32_t h16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h16 & 0xffffu)));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace qg

// ------------------------------------------------------------- host side
namespace qg {

// Records a formatted detail string for qgemv_last_error_string().
void set_last_error(const char *fmt, ...);

// Checks cudaGetLastError() after a launch; returns QGEMV_ERR_LAUNCH (with
// detail) on failure.
qgemv_status check_launch(const char *what);

// Cached per-device properties.
struct DevInfo {
    int sm_count;
    int major, minor;
    size_t smem_optin;
};
// Fills *info for the current device; QGEMV_ERR_ARCH if not sm_103.
qgemv_status current_device(DevInfo *info, int *dev);

// Device address of the current device's kernel error word.
unsigned *device_error_word(int dev);

// qgemv_set_option(QGEMV_OPT_WEIGHTS_STATIC, v): the GEMV may copy W before
// waiting on the preceding kernel of its stream.
extern int g_opt_weights_static;

// Launchers (validated arguments, non-empty problems).
qgemv_status launch_dequant(int fmt, const void *W, void *out, int64_t nrows, int64_t ncols,
                            int out_f16, cudaStream_t s, const DevInfo &di);
qgemv_status launch_gemv(int fmt, const void *W, const float *x, float *y, int64_t nrows,
                         int64_t ncols, int batch, cudaStream_t s, const DevInfo &di, int dev,
                         unsigned *err);
// Stream-K tensor-core GEMV (all formats, ncols a multiple of 2048); *taken
// = false when the shape is not supported by it.
qgemv_status launch_gemv_sk(int fmt, const void *W, const float *x, float *y, int64_t nrows, int64_t ncols,
                            int batch, cudaStream_t s, const DevInfo &di, unsigned *err, bool *taken);
// Zeroes the split-tile counters of the current device (after a timeout).
void gemv_sk_reset_scratch();
// qgemv_set_option(QGEMV_OPT_WAIT_PROBES, v) and (QGEMV_OPT_TEST_WITHHOLD_COPY, 1).
extern unsigned g_opt_wait_probes;
extern int g_opt_withhold_next;
// Tensor-core prefill matmul (all formats; needs ncols % 64 == 0).
qgemv_status launch_gemm_tc(int fmt, const void *W, const void *X, float *Y, int64_t nrows, int64_t ncols,
                            int64_t m, cudaStream_t s, const DevInfo &di, int dev, unsigned *err);
qgemv_status launch_gemm(int fmt, const void *W, const void *X, float *Y, int64_t nrows,
                         int64_t ncols, int64_t m, cudaStream_t s, const DevInfo &di, int dev);
void gemm_release_workspaces();

// Quantized-activation GEMV family (gemv_int.cu).  q8_1_bytes: size of the
// quantized activations of `batch` columns of ncols values; the one-call
// entry points quantize into a library-lifetime scratch of
// mmvq_scratch_values() activations (mmvq_scratch gives its address).
int64_t q8_1_bytes(int64_t ncols, int batch);
int64_t mmvq_scratch_values();
qgemv_status mmvq_scratch(void **ptr);
qgemv_status launch_quantize_q8_1(const float *x, void *xq, int64_t ncols, int batch, cudaStream_t s);
qgemv_status launch_gemv_mmvq(int fmt, const void *W, const void *xq, float *y, int64_t nrows, int64_t ncols,
                              int batch, cudaStream_t s, const DevInfo &di, int dev, unsigned *err);
// fp32-activation GEMV on byte-wise integer dot products of fixed-point
// limbs (gemv_int.cu; up to 4 batch columns a launch, row bytes a multiple
// of 16, ncols a multiple of 64); *taken = false when the shape is not
// supported by it.
qgemv_status launch_gemv_fx(int fmt, const void *W, const float *x, float *y, int64_t nrows, int64_t ncols,
                            int batch, cudaStream_t s, const DevInfo &di, int dev, unsigned *err, bool *taken);
// Expert-selected GEMV on the same fixed-point contraction: output column b
// against matrix ids[b] of W (n_expert matrices of nrows x ncols) and
// activation row b / x_group; batch <= id_max_batch(), row bytes a multiple
// of 16, ncols a multiple of 64.
int id_max_batch();
// The same product on the tensor cores (gemv_sk.cu): ncols a multiple of
// 1024; *taken = false when the shape is not supported by it.
qgemv_status launch_gemv_sk_id(int fmt, const void *W, int64_t n_expert, const int *ids, const float *x,
                               int x_group, float *y, int64_t nrows, int64_t ncols, int batch, cudaStream_t s,
                               const DevInfo &di, unsigned *err, bool *taken);
qgemv_status launch_gemv_id(int fmt, const void *W, int64_t n_expert, const int *ids, const float *x, int x_group,
                            float *y, int64_t nrows, int64_t ncols, int batch, cudaStream_t s, const DevInfo &di,
                            int dev, unsigned *err);

// Q4_0 prefill whose activation copy lives in a fixed __device__ array
// (see qgemm_q4_0_noalloc in qgemv.h); noalloc_scratch_bytes() is its size.
qgemv_status launch_gemm_q4_0_noalloc(const void *W, const void *X, float *Y, int64_t nrows, int64_t ncols,
                                      int64_t m, cudaStream_t s, const DevInfo &di, int dev, unsigned *err);
size_t noalloc_scratch_bytes();

}  // namespace qg
