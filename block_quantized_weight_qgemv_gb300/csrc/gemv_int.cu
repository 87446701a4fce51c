// gemv_int.cu -- GEMV kernels whose inner products are byte-wise integer dot
// products (dp4a) of the weights' integer codes with integer forms of the
// activations, streamed through a shared-memory ring by 1-D bulk copies.
//
// Two activation forms share one streaming kernel:
//
// 1. Quantized activations (the pages' mul_mat_vec_q family: the
//    ggml_cuda_op_mul_mat_vec_q hunk, the "MMVQ = mul_mat_vec_q" note, the
//    convert_src1_to_q8_1 flag of ggml_cuda_op_mul_mat and the __dp4a note
//    beside MIN_CC_DP4A on the "llama_cpp 0.12.1 -> 0.12.2" page).  The pages
//    print neither the activation block layout nor its quantizer; the
//    reading implemented here is
//      amax = max |x_i| over 32 consecutive values of one batch column,
//      d = amax / 127 (IEEE fp32 division),
//      q_i = x_i / d (IEEE fp32 division) rounded to nearest, ties to even,
//            clamped to [-127, 127]; q_i = 0 when d == 0,
//      a block holding a NaN or an infinity: d = NaN and every q_i = 0,
//      s = sum_i q_i (exact int32),
//    stored as one buffer: q int8 [batch][ncols], then d fp32 [batch]
//    [ncols/32], then s int32 [batch][ncols/32].  Per weight block j the
//    GEMV adds
//      Q4_0: d_w * (sum_i c_i q_i - 8 s) * d_x     (c = the 4-bit codes)
//      Q4_1: (d_w * sum_i c_i q_i + m_w * s) * d_x
//      Q8_0: d_w * (sum_i c_i q_i) * d_x            (c = the int8 codes).
//
// 2. fp32 activations held to the GEMV's stated bound (the batch-1
//    "dequantize_mul_mat_vec" role).  Each CTA copies x into shared memory
//    and writes every 32-value block of it in fixed point: with E the
//    exponent of the block's largest magnitude, e = E - 21 and
//    X_i = rne(x_i / 2^e) (|X_i| < 2^22, an exact scaling then one
//    rounding), split into three int8 limbs X = 65536 hi + 256 mid + lo (hi
//    signed, mid and lo unsigned: the bytes of X in two's complement).
//    Elements that keep at least 11 significant bits (|X_i| >= 1024) are
//    contracted by dp4a, limb by limb, exactly in integers; each block's
//    three exact limb sums are combined in fp32.  Every other nonzero
//    element (small next to its block's largest, or any element of a block
//    that holds a NaN or an infinity, or of a block whose largest magnitude
//    is below 2^-105) is left out of the limbs and multiplied in fp32 with
//    its exactly decoded weight.  So every element enters either with a
//    relative error <= 2^-11 or exactly, for all finite inputs:
//    |y - exact| <= 2^-11 sum_k |w_k x_k| + fp32 accumulation error.  For
//    Q4_1 the block term d_w * sum c X + m_w * sum X can cancel; a block
//    whose two parts cancel by more than a factor 2048 is recomputed
//    element by element in fp32.
//
// Streaming: one CTA per SM owns a contiguous range of weight rows, i.e. one
// contiguous byte range.  Rows are taken in row groups (sr whole rows, or
// one row cut into h parts of spc 32-pair segments); row group q belongs to
// warp q % 16, which walks its chunks (row group, part) in order through m
// ring slots of its own (slots k, k + 16, ..., k + 16 (m - 1) of warp k).
// Each warp copies its own chunks with 1-D bulk copies (lane 0): the first
// m when the kernel starts (before the wait on the preceding kernel when
// the weights are declared static), then chunk j + m into the slot that
// chunk j has just left.  A slot has one reader and one writer, and every
// parity wait is for the phase after the one its warp consumed last.  The
// activations are staged once per CTA as records per pair of blocks whose
// strides (80 and 240 bytes) keep 16-byte shared loads free of bank
// conflicts, as are the 36-, 40- and 68-byte weight pairs.  A row is
// reduced by its own warp in a fixed order: results are deterministic.
//
// A general warp-per-row kernel takes the quantized-activation shapes the
// streaming kernel does not; fp32 shapes it does not take go to the other
// GEMV kernels.
//
// The expert-selected GEMV (MUL_MAT_ID: output column b on matrix ids[b] of
// a stack of experts) runs the fixed-point streaming body per work unit --
// up to 4 columns of one expert, grouped on the device from ids -- with the
// unit's x rows gathered into shared memory; a warp-per-(row, column) kernel
// with exact fp32 decode takes the shapes the streaming body does not.
#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "qgemv_common.cuh"

namespace qg {

namespace {

constexpr int kMvCW = 16;                    // warps of the streaming kernel
constexpr int kChunkTarget = 4096;           // bytes a ring chunk aims at
constexpr int kMaxPerWarp = 8;               // ring slots per consumer warp, at most
constexpr int kQuantWarps = 8;               // warps of a quantizer CTA
constexpr int kRowWarps = 8;                 // warps of a general-kernel CTA

enum Mode { MODE_Q8 = 0, MODE_FX = 1 };
template <int MODE> struct Rec;              // staged activation record of a block pair, per column
template <> struct Rec<MODE_Q8> { static constexpr int kBytes = 80; };    // 64 codes, d0 s0 d1 s1
template <> struct Rec<MODE_FX> { static constexpr int kBytes = 240; };   // hi[64] mid[64] lo[64], 2 x 20 meta
constexpr int kFxMaxBatch = 4;               // fp32 activations: batch columns the streaming kernel stages
constexpr int kIdMaxBatch = 64;              // output columns of an expert-selected GEMV, at most

// ------------------------------------------------------------ device helpers
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> shared with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                              uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol) : "memory");
}

// The same without a cache policy.
__device__ __forceinline__ void bulk_g2s_a(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_test_a(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ void mbar_arrive_a(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx_a(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
}
// Bounded wait: probes separated by 32 ns sleeps; gives up after `probes`
// sleeps, or once another warp of the CTA has given up.
__device__ __forceinline__ bool mbar_ready(uint32_t bar, uint32_t parity, unsigned probes,
                                           volatile int *abort_flag) {
    if (mbar_test_a(bar, parity)) return true;
    for (unsigned i = 0; i < probes; ++i) {
        __nanosleep(32);
        if (mbar_test_a(bar, parity)) return true;
        if (*abort_flag) return false;
    }
    return false;
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Byte-wise dot products: four unsigned bytes of a against four signed bytes
// of b, added to c (exact int32).
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ float half_lo(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
}
__device__ __forceinline__ float half_hi(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// The 4-bit codes of a 16-byte nibble group as two masked words per 4 bytes:
// lo = low nibbles (elements 4t..4t+3), hi16 = high nibbles times 16
// (elements 16+4t..16+4t+3).  hi16 against int8 codes sums to 16 times the
// high-nibble dot product, exactly.
struct Nib {
    uint32_t lo[4], hi[4];
};
__device__ __forceinline__ void split_nibbles(const uint32_t a[4], Nib &n) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        n.lo[t] = a[t] & 0x0f0f0f0fu;
        n.hi[t] = a[t] & 0xf0f0f0f0u;
    }
}
// sum_i c_i q_i of one 4-bit block against the 8 code words X[0..7] of its
// 32 activations (X[t] = codes 4t..4t+3).
__device__ __forceinline__ int dot_nib(const Nib &n, const uint32_t X[8]) {
    int lo = 0, hi = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        lo = dp4a_us(n.lo[t], X[t], lo);
        hi = dp4a_us(n.hi[t], X[4 + t], hi);
    }
    return lo + (hi >> 4);
}

// ------------------------------------------------------------- quantizer
__global__ void __launch_bounds__(kQuantWarps * 32)
quantize_q8_1_kernel(const float *__restrict__ x, int8_t *__restrict__ q, float *__restrict__ d,
                     int *__restrict__ s, int64_t nblocks) {
    griddep_launch_dependents();
    griddep_wait();                              // x: after the preceding kernel
    const int lane = threadIdx.x & 31;
    const int64_t blk = static_cast<int64_t>(blockIdx.x) * kQuantWarps + (threadIdx.x >> 5);
    if (blk >= nblocks) return;
    const float v = x[blk * 32 + lane];
    const float a = fabsf(v);
    const bool bad = __any_sync(0xffffffffu, !isfinite(a));
    float amax = bad ? 0.0f : a;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float dd = bad ? __int_as_float(0x7fc00000) : __fdiv_rn(amax, 127.0f);
    int c = 0;
    if (!bad && dd != 0.0f) c = min(max(__float2int_rn(__fdiv_rn(v, dd)), -127), 127);
    q[blk * 32 + lane] = static_cast<int8_t>(c);
    const int sum = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0) {
        d[blk] = dd;
        s[blk] = sum;
    }
}

// --------------------------------------------- quantized activations (q8_1)
// A weight pair decoded for the integer dot products.
template <int F> struct WQ;
template <> struct WQ<FMT_Q4_0> { Nib n0, n1; float d0, d1; };
template <> struct WQ<FMT_Q4_1> { Nib n0, n1; float d0, d1, m0, m1; };
template <> struct WQ<FMT_Q8_0> { uint32_t a0[8], a1[8]; float d0, d1; };

// wa: shared address of the pair.
template <int F>
__device__ __forceinline__ void wq_load(uint32_t wa, WQ<F> &q) {
    if constexpr (F == FMT_Q4_0) {
        // [d0 | c0 c1] [c2..c5] [c6..c9] [c10..c13] [c14 c15 | d1] [block 1 codes x4]
        uint32_t w[9];
#pragma unroll
        for (int t = 0; t < 9; ++t) w[t] = lds32(wa + 4 * t);
        uint32_t a0[4], a1[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            a0[t] = __byte_perm(w[t], w[t + 1], 0x5432);
            a1[t] = w[5 + t];
        }
        split_nibbles(a0, q.n0);
        split_nibbles(a1, q.n1);
        q.d0 = half_lo(w[0]);
        q.d1 = half_hi(w[4]);
    } else if constexpr (F == FMT_Q4_1) {
        // [d0 | m0] [codes x4] [d1 | m1] [codes x4]
        uint32_t w[10];
#pragma unroll
        for (int t = 0; t < 5; ++t) {
            const uint2 v = lds64(wa + 8 * t);
            w[2 * t] = v.x;
            w[2 * t + 1] = v.y;
        }
        const uint32_t a0[4] = {w[1], w[2], w[3], w[4]};
        const uint32_t a1[4] = {w[6], w[7], w[8], w[9]};
        split_nibbles(a0, q.n0);
        split_nibbles(a1, q.n1);
        q.d0 = half_lo(w[0]);
        q.m0 = half_hi(w[0]);
        q.d1 = half_lo(w[5]);
        q.m1 = half_hi(w[5]);
    } else {
        // [d0 | c0 c1] [c2..c5] ... [c30 c31 | d1] [block 1 codes x8]
        uint32_t w[17];
#pragma unroll
        for (int t = 0; t < 17; ++t) w[t] = lds32(wa + 4 * t);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            q.a0[t] = __byte_perm(w[t], w[t + 1], 0x5432);
            q.a1[t] = w[9 + t];
        }
        q.d0 = half_lo(w[0]);
        q.d1 = half_hi(w[8]);
    }
}

// One activation record (two blocks of one batch column): codes, then
// {d0, s0, d1, s1}.
struct RecQ {
    uint32_t X0[8], X1[8];
    uint4 ds;
};
__device__ __forceinline__ void recq_load(uint32_t r, RecQ &x) {
    const uint4 v0 = lds128(r), v1 = lds128(r + 16), v2 = lds128(r + 32), v3 = lds128(r + 48);
    x.ds = lds128(r + 64);
    x.X0[0] = v0.x; x.X0[1] = v0.y; x.X0[2] = v0.z; x.X0[3] = v0.w;
    x.X0[4] = v1.x; x.X0[5] = v1.y; x.X0[6] = v1.z; x.X0[7] = v1.w;
    x.X1[0] = v2.x; x.X1[1] = v2.y; x.X1[2] = v2.z; x.X1[3] = v2.w;
    x.X1[4] = v3.x; x.X1[5] = v3.y; x.X1[6] = v3.z; x.X1[7] = v3.w;
}

// acc + the pair's two block terms against one record.
template <int F>
__device__ __forceinline__ float wq_acc(const WQ<F> &q, const RecQ &x, float acc) {
    if constexpr (F == FMT_Q4_0) {
        const int s0 = dot_nib(q.n0, x.X0) - 8 * static_cast<int>(x.ds.y);
        const int s1 = dot_nib(q.n1, x.X1) - 8 * static_cast<int>(x.ds.w);
        acc = fmaf(q.d0 * static_cast<float>(s0), __uint_as_float(x.ds.x), acc);
        return fmaf(q.d1 * static_cast<float>(s1), __uint_as_float(x.ds.z), acc);
    } else if constexpr (F == FMT_Q4_1) {
        const float t0 = fmaf(q.d0, static_cast<float>(dot_nib(q.n0, x.X0)),
                              q.m0 * static_cast<float>(static_cast<int>(x.ds.y)));
        const float t1 = fmaf(q.d1, static_cast<float>(dot_nib(q.n1, x.X1)),
                              q.m1 * static_cast<float>(static_cast<int>(x.ds.w)));
        acc = fmaf(t0, __uint_as_float(x.ds.x), acc);
        return fmaf(t1, __uint_as_float(x.ds.z), acc);
    } else {
        int s0 = 0, s1 = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            s0 = dp4a_ss(q.a0[t], x.X0[t], s0);
            s1 = dp4a_ss(q.a1[t], x.X1[t], s1);
        }
        acc = fmaf(q.d0 * static_cast<float>(s0), __uint_as_float(x.ds.x), acc);
        return fmaf(q.d1 * static_cast<float>(s1), __uint_as_float(x.ds.z), acc);
    }
}

// The two blocks of a weight pair, decoded once and contracted with NB
// activation records.  wa: shared address of the pair; xa: shared address of
// batch column 0's record; xstride: bytes between the records of two columns.
template <int F, int NB>
__device__ __forceinline__ void pair_dot(uint32_t wa, uint32_t xa, uint32_t xstride, float acc[NB]) {
    WQ<F> q;
    wq_load<F>(wa, q);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        RecQ x;
        recq_load(xa + b * xstride, x);
        acc[b] = wq_acc<F>(q, x, acc[b]);
    }
}

// The same pair of up to RR rows (wa0: pair of the first row; wrs: bytes
// between rows in the slot) against NB records: each record is read from
// shared memory once for all rows (acc[ri][b]: row ri, column b).
template <int F, int NB, int RR>
__device__ __forceinline__ void pair_dot_rows(uint32_t wa0, uint32_t wrs, int rows, uint32_t xa, uint32_t xstride,
                                              float (&acc)[RR][NB]) {
    WQ<F> q[RR];
#pragma unroll
    for (int ri = 0; ri < RR; ++ri) {
        if (ri < rows) wq_load<F>(wa0 + ri * wrs, q[ri]);
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        RecQ x;
        recq_load(xa + b * xstride, x);
#pragma unroll
        for (int ri = 0; ri < RR; ++ri) {
            if (ri < rows) acc[ri][b] = wq_acc<F>(q[ri], x, acc[ri][b]);
        }
    }
}

// --------------------------------------------------- fixed-point activations
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" :: "r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ldsu8(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// Records of the fixed-point blocks of NB columns of fp32 activations x
// ([NB][ncols]): limbs at rec + 32 * half (+ 0, 64, 128 for hi, mid, lo) and
// meta {2^e, sparse mask, sum hi, sum mid, sum lo} at rec + 192 + 20 * half,
// rec = rec0 + 240 * (pair of the block).  Eight lanes per block: lane s of
// a group holds values 4s .. 4s+3 (so float4 t of x is task t, coalesced);
// the block's largest magnitude, sparse mask and limb sums are combined over
// the group with shuffles.  All threads of the CTA (512) take part.
template <int NB>
__device__ __forceinline__ void fx_build(bool xsm, uint32_t xs, const float *xg, int ncols, uint32_t rec0, int tid) {
    constexpr int kT = 4;                                  // tasks per thread per pass
    const int nb = ncols / 32;
    const int ntask = NB * nb * 8;
    const int npair = ncols / 64;
    const int sub = tid & 7;
    for (int t0 = tid; t0 - (tid & 31) < ntask; t0 += kT * kMvCW * 32) {     // warp-uniform bound
        float4 v[kT];
#pragma unroll
        for (int u = 0; u < kT; ++u) {
            const int t = t0 + u * kMvCW * 32;
            if (t < ntask && xsm) {
                const uint4 w = lds128(xs + 16u * t);
                v[u] = make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                                   __uint_as_float(w.w));
            } else if (t < ntask) {
                v[u] = reinterpret_cast<const float4 *>(xg)[t];
            } else {
                v[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
        }
#pragma unroll
        for (int u = 0; u < kT; ++u) {
            const int t = t0 + u * kMvCW * 32;
            if (t - (tid & 31) >= ntask) break;                                // warp-uniform
            const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            uint32_t mx = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) mx = max(mx, __float_as_uint(f[i]) & 0x7fffffffu);
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            const int e = static_cast<int>(mx >> 23) - 127 - 21;
            // limbs only for finite blocks whose scale 2^e is a normal float
            const bool limbs = mx < 0x7f800000u && mx != 0 && e >= -126;
            const float scale = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);   // 2^-e
            int X[4];
            uint32_t mask = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int xi = limbs ? __float2int_rn(f[i] * scale) : 0;
                const bool small = xi > -1024 && xi < 1024;
                X[i] = small ? 0 : xi;
                if (small && f[i] != 0.0f) mask |= 1u << (4 * sub + i);       // (NaN != 0 holds)
            }
            const uint32_t wl = __byte_perm(__byte_perm(X[0], X[1], 0x0040), __byte_perm(X[2], X[3], 0x0040), 0x5410);
            const uint32_t wm = __byte_perm(__byte_perm(X[0], X[1], 0x0051), __byte_perm(X[2], X[3], 0x0051), 0x5410);
            const uint32_t wh = __byte_perm(__byte_perm(X[0], X[1], 0x0062), __byte_perm(X[2], X[3], 0x0062), 0x5410);
            int slo = dp4a_uu(wl, 0x01010101u, 0), smid = dp4a_uu(wm, 0x01010101u, 0);
            int shi = dp4a_ss(wh, 0x01010101u, 0);
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                mask |= __shfl_xor_sync(0xffffffffu, mask, o);
                slo += __shfl_xor_sync(0xffffffffu, slo, o);
                smid += __shfl_xor_sync(0xffffffffu, smid, o);
                shi += __shfl_xor_sync(0xffffffffu, shi, o);
            }
            if (t < ntask) {
                int blk = t >> 3, b = 0;                                        // block over [NB][ncols/32]
#pragma unroll
                for (int c = 1; c < NB; ++c)
                    if (blk >= nb) {
                        blk -= nb;
                        ++b;
                    }
                const uint32_t rec = rec0 + static_cast<uint32_t>(b * npair + (blk >> 1)) * 240u;
                const uint32_t lb = rec + 32u * (blk & 1) + 4u * sub;
                sts32(lb, wh);
                sts32(lb + 64u, wm);
                sts32(lb + 128u, wl);
                if (sub == 0) {
                    const uint32_t mb = rec + 192u + 20u * (blk & 1);
                    sts32(mb, limbs ? __float_as_uint(__uint_as_float(static_cast<uint32_t>(127 + e) << 23)) : 0u);
                    sts32(mb + 4, mask);
                    sts32(mb + 8, static_cast<uint32_t>(shi));
                    sts32(mb + 12, static_cast<uint32_t>(smid));
                    sts32(mb + 16, static_cast<uint32_t>(slo));
                }
            }
        }
    }
}

// The fp32 activations of a weight pair: in shared memory (sa) when staged
// there, else in global memory (ga).
struct XSrc {
    uint32_t sa;
    const float *ga;
    bool smem;
    __device__ float at(int i) const { return smem ? __uint_as_float(lds32(sa + 4u * i)) : ga[i]; }
};

// Exact fp32 product of the sparse elements `mask` of one weight block with
// their activations (xb: the block's fp32 values).  qb: the block's code
// bytes in shared memory.
template <int F>
__device__ __forceinline__ float sparse_dot(uint32_t mask, uint32_t qb, float d, float m, const XSrc &xb, float acc) {
    while (mask) {
        const int i = __ffs(mask) - 1;
        mask &= mask - 1;
        float w;
        if constexpr (F == FMT_Q8_0) {
            w = d * static_cast<float>(static_cast<int8_t>(ldsu8(qb + i)));
        } else {
            const uint32_t byte = ldsu8(qb + (i & 15));
            const int q = i < 16 ? static_cast<int>(byte & 15u) : static_cast<int>(byte >> 4);
            w = F == FMT_Q4_0 ? d * static_cast<float>(q - 8) : __fadd_rn(__fmul_rn(d, static_cast<float>(q)), m);
        }
        acc = fmaf(w, xb.at(i), acc);
    }
    return acc;
}

// sum_i c_i X_i of a 4-bit block against one limb (X[0..7]), exact.
template <bool SIGNED>
__device__ __forceinline__ int dot_nib_limb(const Nib &n, const uint32_t *X) {
    int lo = 0, hi = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        if (SIGNED) {
            lo = dp4a_us(n.lo[t], X[t], lo);
            hi = dp4a_us(n.hi[t], X[4 + t], hi);
        } else {
            lo = dp4a_uu(n.lo[t], X[t], lo);
            hi = dp4a_uu(n.hi[t], X[4 + t], hi);
        }
    }
    return lo + (hi >> 4);
}
// ... of an 8-bit block (signed codes a[0..7]).
template <bool SIGNED>
__device__ __forceinline__ int dot_q8_limb(const uint32_t *a, const uint32_t *X) {
    int s = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) s = SIGNED ? dp4a_ss(a[t], X[t], s) : dp4a_su(a[t], X[t], s);
    return s;
}
__device__ __forceinline__ void load16(uint32_t a, uint32_t X[16]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 v = lds128(a + 16u * c);
        X[4 * c] = v.x; X[4 * c + 1] = v.y; X[4 * c + 2] = v.z; X[4 * c + 3] = v.w;
    }
}
// Exact integer limb sums -> fp32 (two roundings).
__device__ __forceinline__ float limbs_to_f(int hi, int mid, int lo) {
    return fmaf(static_cast<float>(hi), 65536.0f, fmaf(static_cast<float>(mid), 256.0f, static_cast<float>(lo)));
}

// A weight pair decoded for the fixed-point contraction: code words of the
// two blocks (4-bit: 4 words each; 8-bit: 8 words each), scales, and the
// shared addresses of the code bytes (for the exact elements).
template <int F> struct WPair {
    uint32_t a0[8], a1[8];
    float d0, d1, m0, m1;
    uint32_t q0, q1;
};
template <int F>
__device__ __forceinline__ void wpair_load(uint32_t wa, WPair<F> &w) {
    w.m0 = w.m1 = 0.0f;
    if constexpr (F == FMT_Q4_0) {
        uint32_t v[9];
#pragma unroll
        for (int t = 0; t < 9; ++t) v[t] = lds32(wa + 4 * t);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            w.a0[t] = __byte_perm(v[t], v[t + 1], 0x5432);
            w.a1[t] = v[5 + t];
        }
        w.d0 = half_lo(v[0]);
        w.d1 = half_hi(v[4]);
        w.q0 = wa + 2;
        w.q1 = wa + 20;
    } else if constexpr (F == FMT_Q4_1) {
        uint32_t v[10];
#pragma unroll
        for (int t = 0; t < 5; ++t) {
            const uint2 u = lds64(wa + 8 * t);
            v[2 * t] = u.x;
            v[2 * t + 1] = u.y;
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            w.a0[t] = v[1 + t];
            w.a1[t] = v[6 + t];
        }
        w.d0 = half_lo(v[0]);
        w.m0 = half_hi(v[0]);
        w.d1 = half_lo(v[5]);
        w.m1 = half_hi(v[5]);
        w.q0 = wa + 4;
        w.q1 = wa + 24;
    } else {
        uint32_t v[17];
#pragma unroll
        for (int t = 0; t < 17; ++t) v[t] = lds32(wa + 4 * t);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            w.a0[t] = __byte_perm(v[t], v[t + 1], 0x5432);
            w.a1[t] = v[9 + t];
        }
        w.d0 = half_lo(v[0]);
        w.d1 = half_hi(v[8]);
        w.q0 = wa + 2;
        w.q1 = wa + 36;
    }
}

// The fixed-point record of one column (limb words H, M, Lo of both blocks,
// meta mA mB mC) against a decoded weight pair; xb: the pair's fp32
// activations in shared memory (for the elements kept out of the limbs).
template <int F>
__device__ __forceinline__ float fx_col(const WPair<F> &w, const uint32_t *H, const uint32_t *M, const uint32_t *Lo,
                                        const uint4 mA, const uint4 mB, const uint4 mC, const XSrc &xb, float acc) {
    int s0[3], s1[3];
    const uint32_t *limb[3] = {H, M, Lo};
    if constexpr (F == FMT_Q8_0) {
#pragma unroll
        for (int l = 0; l < 3; ++l) {
            s0[l] = l == 0 ? dot_q8_limb<true>(w.a0, limb[l]) : dot_q8_limb<false>(w.a0, limb[l]);
            s1[l] = l == 0 ? dot_q8_limb<true>(w.a1, limb[l] + 8) : dot_q8_limb<false>(w.a1, limb[l] + 8);
        }
    } else {
        Nib n0, n1;
        split_nibbles(w.a0, n0);
        split_nibbles(w.a1, n1);
#pragma unroll
        for (int l = 0; l < 3; ++l) {
            s0[l] = l == 0 ? dot_nib_limb<true>(n0, limb[l]) : dot_nib_limb<false>(n0, limb[l]);
            s1[l] = l == 0 ? dot_nib_limb<true>(n1, limb[l] + 8) : dot_nib_limb<false>(n1, limb[l] + 8);
        }
    }
    // meta: block 0 {dx, mask, shi, smid, slo} = mA.x mA.y mA.z mA.w mB.x; block 1 = mB.y mB.z mB.w mC.x mC.y
    const int t0[3] = {static_cast<int>(mA.z), static_cast<int>(mA.w), static_cast<int>(mB.x)};
    const int t1[3] = {static_cast<int>(mB.w), static_cast<int>(mC.x), static_cast<int>(mC.y)};
    const float dx0 = __uint_as_float(mA.x), dx1 = __uint_as_float(mB.y);
    uint32_t sp0 = mA.y, sp1 = mB.z;
    if constexpr (F == FMT_Q4_0) {
        const float T0 = limbs_to_f(s0[0] - 8 * t0[0], s0[1] - 8 * t0[1], s0[2] - 8 * t0[2]);
        const float T1 = limbs_to_f(s1[0] - 8 * t1[0], s1[1] - 8 * t1[1], s1[2] - 8 * t1[2]);
        acc = fmaf(w.d0 * T0, dx0, acc);
        acc = fmaf(w.d1 * T1, dx1, acc);
    } else if constexpr (F == FMT_Q8_0) {
        acc = fmaf(w.d0 * limbs_to_f(s0[0], s0[1], s0[2]), dx0, acc);
        acc = fmaf(w.d1 * limbs_to_f(s1[0], s1[1], s1[2]), dx1, acc);
    } else {
        // d * sum c X + m * sum X, unless the two parts cancel by more than 2^11
        const float u0 = w.d0 * limbs_to_f(s0[0], s0[1], s0[2]), v0 = w.m0 * limbs_to_f(t0[0], t0[1], t0[2]);
        const float u1 = w.d1 * limbs_to_f(s1[0], s1[1], s1[2]), v1 = w.m1 * limbs_to_f(t1[0], t1[1], t1[2]);
        const float z0 = u0 + v0, z1 = u1 + v1;
        if (fabsf(u0) + fabsf(v0) > 2048.0f * fabsf(z0)) {
            sp0 = 0xffffffffu;                   // the whole block, exactly
        } else {
            acc = fmaf(z0, dx0, acc);
        }
        if (fabsf(u1) + fabsf(v1) > 2048.0f * fabsf(z1)) {
            sp1 = 0xffffffffu;
        } else {
            acc = fmaf(z1, dx1, acc);
        }
    }
    if ((sp0 | sp1) != 0u) {
        acc = sparse_dot<F>(sp0, w.q0, w.d0, w.m0, xb, acc);
        const XSrc x1 = {xb.sa + 128u, xb.ga + 32, xb.smem};
        acc = sparse_dot<F>(sp1, w.q1, w.d1, w.m1, x1, acc);
    }
    return acc;
}

// One weight pair against NB fixed-point records.  wa: shared address of the
// pair; ra: record of column 0; rstride: bytes between columns' records; xa:
// the pair's fp32 activations of column 0; ncols: values between columns.
template <int F, int NB>
__device__ __forceinline__ void pair_dot_fx(uint32_t wa, uint32_t ra, uint32_t rstride, const XSrc &xa, int ncols,
                                            float acc[NB]) {
    WPair<F> w;
    wpair_load<F>(wa, w);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const uint32_t r = ra + b * rstride;
        uint32_t H[16], M[16], Lo[16];
        load16(r, H);
        load16(r + 64u, M);
        load16(r + 128u, Lo);
        const uint4 mA = lds128(r + 192), mB = lds128(r + 208), mC = lds128(r + 224);
        const XSrc xb = {xa.sa + 4u * static_cast<uint32_t>(b * ncols), xa.ga + static_cast<size_t>(b) * ncols, xa.smem};
        acc[b] = fx_col<F>(w, H, M, Lo, mA, mB, mC, xb, acc[b]);
    }
}

// One fixed-point record (one column) against the same pair of up to RR
// rows (wa0: pair of the first row; wrs: bytes between rows in the slot):
// the record is read from shared memory once for all rows.
template <int F, int RR>
__device__ __forceinline__ void pair_dot_fx_rows(uint32_t wa0, uint32_t wrs, int rows, uint32_t ra, const XSrc &xa,
                                                 float acc[RR]) {
    uint32_t H[16], M[16], Lo[16];
    load16(ra, H);
    load16(ra + 64u, M);
    load16(ra + 128u, Lo);
    const uint4 mA = lds128(ra + 192), mB = lds128(ra + 208), mC = lds128(ra + 224);
#pragma unroll
    for (int ri = 0; ri < RR; ++ri) {
        if (ri < rows) {
            WPair<F> w;
            wpair_load<F>(wa0 + ri * wrs, w);
            acc[ri] = fx_col<F>(w, H, M, Lo, mA, mB, mC, xa, acc[ri]);
        }
    }
}

// --------------------------------------------------------- streaming GEMV
struct IntParams {
    const uint8_t *W;
    const int8_t *xq;       // quantized activations: codes [batch][ncols]
    const float *xd;        //   scales [batch][ncols/32]
    const int *xs;          //   code sums [batch][ncols/32]
    const float *x;         // fp32 activations [batch][ncols]
    float *y;               // [batch][nrows]
    unsigned *err;
    int nrows, ncols;
    int npair;              // ncols / 64
    int rb;                 // bytes of a weight row
    int spc;                // 32-pair segments of a row part
    int h;                  // parts of a row group (1: sr whole rows)
    int sr;                 // rows of a row group
    int pstride;            // bytes between the rows of a chunk in its slot
    int nst;                // ring slots, a multiple of kMvCW
    int slot;               // bytes of a ring slot
    int xsm;                // fixed point: fp32 x also staged in shared memory
    int early;              // weights static: copy them before the dependency wait
    unsigned probes;
    int withhold;           // testing: never copy the first chunk (its wait runs out)
};

template <int F> struct MvPairB;
template <> struct MvPairB<FMT_Q4_0> { static constexpr int kBytes = 36; };
template <> struct MvPairB<FMT_Q4_1> { static constexpr int kBytes = 40; };
template <> struct MvPairB<FMT_Q8_0> { static constexpr int kBytes = 68; };

// Shared memory: [fp32 x: NB * ncols * 4 (fixed point, when staged)][records: NB *
// npair * record bytes][ring: nst * slot][full: nst][x barrier][flag].
struct IntLayout {
    uint32_t xs, rec, ring, bars, flag, total;
};
__host__ __device__ inline IntLayout int_layout(int mode, int nb_cols, int npair, int slot, int nst, int xsm) {
    IntLayout L;
    L.xs = 0;
    L.rec = mode == MODE_FX && xsm ? static_cast<uint32_t>(nb_cols) * npair * 256u : 0u;
    L.ring = L.rec + static_cast<uint32_t>(nb_cols) * npair * (mode == MODE_FX ? 240u : 80u);
    L.bars = L.ring + static_cast<uint32_t>(nst) * slot;
    L.flag = (L.bars + 8u * nst + 8u + 15u) & ~15u;
    L.total = L.flag + 16u;
    return L;
}

// One warp's chunk stream: its row groups q = k, k + 16, ... in order, each
// cut into h parts; its chunks cycle through its m slots k, k + 16, ...,
// k + 16 (m - 1).  The warp copies its own chunks (lane 0), so a slot is
// refilled as soon as its only reader is done with it.
struct ChunkCursor {
    int q, part;             // row group and part of the next chunk to copy
    int slot_i;              // its slot index (0 .. m-1)
};

// Rows of a chunk contracted together (each activation record read from
// shared memory once for all of them): 4 for the fixed-point contraction at
// batch 1, 2 for the quantized activations at batches of 2 or more (whose
// records would otherwise be re-read for every row: 80 bytes per column).
__host__ __device__ constexpr int rows_together(int mode, int nb_cols) {
    return mode == MODE_FX ? (nb_cols == 1 ? 4 : 1) : (nb_cols >= 2 ? 2 : 1);
}

// Element offsets of the batch columns in x and y when they are gathered
// (the expert-selected GEMV); otherwise column b is at b * ncols and b * nrows.
template <int NB> struct ColMap {
    int64_t x[NB], y[NB];
};

// The streaming GEMV of one CTA over its rows of p.W (the kernel below, and
// the expert-selected kernel once it has picked its matrix and columns).
template <int F, int NB, int MODE, bool GATHER>
__device__ __forceinline__ void stream_body(const IntParams &p, const ColMap<NB> &cm, uint8_t *smem) {
    constexpr int RR = rows_together(MODE, NB);
    constexpr int PB = MvPairB<F>::kBytes;
    constexpr int RB = Rec<MODE>::kBytes;
    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    const int r0 = static_cast<int>(static_cast<int64_t>(cta) * p.nrows / G);
    const int r1 = static_cast<int>(static_cast<int64_t>(cta + 1) * p.nrows / G);
    const int nrow = r1 - r0;
    const int RG = (nrow + p.sr - 1) / p.sr;                       // row groups of this CTA
    const int m = p.nst / kMvCW;                                   // slots per warp
    const int nj = wid < RG ? ((RG - 1 - wid) / kMvCW + 1) * p.h : 0;   // chunks of this warp
    const IntLayout L = int_layout(MODE, NB, p.npair, p.slot, p.nst, p.xsm);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t full0 = sbase + L.bars;                         // full[s] at full0 + 8s
    const uint32_t xbar = full0 + 8u * p.nst;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.flag);
    const bool held = p.withhold && cta == 0 && blockIdx.y == 0 && wid == 0;   // first chunk withheld (testing)

    griddep_launch_dependents();
    if (tid == 0) {
        uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
        for (int s = 0; s <= p.nst; ++s) mbar_init(&bars[s], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    cta_sync();

    // copies of this warp's chunks, in order (lane 0)
    const uint64_t pol = l2_evict_first();
    ChunkCursor cur = {wid, 0, 0};
    int issued = 0;                                                // chunks copied (or withheld)
    auto issue = [&]() {
        const uint32_t s = static_cast<uint32_t>(wid + kMvCW * cur.slot_i);
        const int rows = min(p.sr, nrow - cur.q * p.sr);
        const size_t row0 = static_cast<size_t>(r0 + cur.q * p.sr);
        if (!(issued == 0 && held)) {
            if (p.h == 1) {
                // whole rows: one contiguous range
                const uint32_t bytes = static_cast<uint32_t>(rows) * p.rb;
                mbar_expect_tx_a(full0 + 8u * s, bytes);
                bulk_g2s_hint(sbase + L.ring + s * p.slot, p.W + row0 * p.rb, bytes, full0 + 8u * s, pol);
            } else {
                // one part of each row: a range per row
                const int j0 = cur.part * p.spc * 32, j1 = min(j0 + p.spc * 32, p.npair);
                const uint32_t bytes = static_cast<uint32_t>(j1 - j0) * PB;
                mbar_expect_tx_a(full0 + 8u * s, bytes * rows);
                for (int ri = 0; ri < rows; ++ri) {
                    bulk_g2s_hint(sbase + L.ring + s * p.slot + static_cast<uint32_t>(ri) * p.pstride,
                                  p.W + (row0 + ri) * p.rb + static_cast<size_t>(j0) * PB, bytes, full0 + 8u * s,
                                  pol);
                }
            }
        }
        ++issued;
        if (++cur.part == p.h) {
            cur.part = 0;
            cur.q += kMvCW;
        }
        if (++cur.slot_i == m) cur.slot_i = 0;
    };
    const int first = min(m, nj);
    if (lane == 0 && p.early)
        while (issued < first) issue();
    griddep_wait();                                                // W, x and y: after the preceding kernel
    if constexpr (MODE == MODE_FX) {
        if (tid == 0 && p.xsm) {
            const uint32_t xbytes = static_cast<uint32_t>(p.ncols) * 4u;
            mbar_expect_tx_a(xbar, NB * xbytes);
            if constexpr (GATHER) {
#pragma unroll
                for (int b = 0; b < NB; ++b) bulk_g2s_a(sbase + L.xs + b * xbytes, p.x + cm.x[b], xbytes, xbar);
            } else {
                bulk_g2s_a(sbase + L.xs, p.x, NB * xbytes, xbar);
            }
        }
    }
    if (lane == 0)
        while (issued < first) issue();

    // ------------------------------------------------ stage the activations
    if constexpr (MODE == MODE_Q8) {
        const int nb = p.ncols / 32;
        for (int i = tid; i < NB * p.npair; i += kMvCW * 32) {
            const int b = i / p.npair, j = i - b * p.npair;
            const uint4 *qs = reinterpret_cast<const uint4 *>(p.xq + static_cast<size_t>(b) * p.ncols + 64 * j);
            const uint4 v0 = qs[0], v1 = qs[1], v2 = qs[2], v3 = qs[3];
            const float2 dd = *reinterpret_cast<const float2 *>(p.xd + static_cast<size_t>(b) * nb + 2 * j);
            const int2 ss = *reinterpret_cast<const int2 *>(p.xs + static_cast<size_t>(b) * nb + 2 * j);
            const uint32_t r = sbase + L.rec + static_cast<uint32_t>(b * p.npair + j) * RB;
            sts128(r, v0);
            sts128(r + 16, v1);
            sts128(r + 32, v2);
            sts128(r + 48, v3);
            sts128(r + 64, make_uint4(__float_as_uint(dd.x), static_cast<uint32_t>(ss.x), __float_as_uint(dd.y),
                                      static_cast<uint32_t>(ss.y)));
        }
    } else {
        if (!p.xsm || mbar_ready(xbar, 0u, p.probes, abort_flag)) {
            fx_build<NB>(p.xsm != 0, sbase + L.xs, p.x, p.ncols, sbase + L.rec, tid);
        } else if (lane == 0 && !*abort_flag) {
            *abort_flag = 1;
            atomicOr(p.err, ERRBIT_TIMEOUT);
        }
    }
    cta_sync();

    // --------------------------------------------------------- contract
    const uint32_t rstride = static_cast<uint32_t>(p.npair) * RB;
    int consumed = 0;
    int slot_i = 0;
    uint32_t phase = 0;
    int q = wid, part = 0;
    float acc[RR > NB ? RR : NB];
    float accr[MODE == MODE_Q8 && RR > 1 ? RR : 1][NB];     // quantized activations, rows together
    for (; consumed < nj && !*abort_flag; ++consumed) {
        const uint32_t s = static_cast<uint32_t>(wid + kMvCW * slot_i);
        if (!mbar_ready(full0 + 8u * s, phase, p.probes, abort_flag)) {
            if (lane == 0 && !*abort_flag) {
                *abort_flag = 1;
                atomicOr(p.err, ERRBIT_TIMEOUT);
            }
            break;
        }
        const uint32_t sl = sbase + L.ring + s * p.slot;
        const int rows = min(p.sr, nrow - q * p.sr);
        const int j0 = p.h == 1 ? 0 : part * p.spc * 32;
        const int j1 = p.h == 1 ? p.npair : min(j0 + p.spc * 32, p.npair);
        if constexpr (MODE == MODE_Q8 && RR > 1) {
            // quantized activations, several columns: each record serves every row of the chunk
            if (p.h == 1 || part == 0) {
#pragma unroll
                for (int ri = 0; ri < RR; ++ri) {
#pragma unroll
                    for (int b = 0; b < NB; ++b) accr[ri][b] = 0.0f;
                }
            }
            for (int j = j0 + lane; j < j1; j += 32) {
                pair_dot_rows<F, NB, RR>(sl + static_cast<uint32_t>(j - j0) * PB, p.pstride, rows,
                                         sbase + L.rec + static_cast<uint32_t>(j) * RB, rstride, accr);
            }
            if (p.h == 1 || part == p.h - 1) {
#pragma unroll
                for (int ri = 0; ri < RR; ++ri) {
                    if (ri < rows) {
                        const int row = r0 + q * p.sr + ri;
#pragma unroll
                        for (int b = 0; b < NB; ++b) {
                            const float v = warp_sum(accr[ri][b]);
                            if (lane == 0)
                                p.y[(GATHER ? cm.y[b] : static_cast<int64_t>(b) * p.nrows) + row] = v;
                        }
                    }
                }
            }
        } else if constexpr (RR > 1) {
            // fixed point, batch 1: each lane's record serves every row of the chunk
            if (p.h == 1 || part == 0) {
#pragma unroll
                for (int ri = 0; ri < RR; ++ri) acc[ri] = 0.0f;
            }
            for (int j = j0 + lane; j < j1; j += 32) {
                const XSrc xa = {sbase + L.xs + static_cast<uint32_t>(j) * 256u, p.x + 64 * j, p.xsm != 0};
                pair_dot_fx_rows<F, RR>(sl + static_cast<uint32_t>(j - j0) * PB, p.pstride, rows,
                                        sbase + L.rec + static_cast<uint32_t>(j) * RB, xa, acc);
            }
            if (p.h == 1 || part == p.h - 1) {
#pragma unroll
                for (int ri = 0; ri < RR; ++ri) {
                    if (ri < rows) {
                        const float v = warp_sum(acc[ri]);
                        if (lane == 0) p.y[(GATHER ? cm.y[0] : 0) + r0 + q * p.sr + ri] = v;
                    }
                }
            }
        } else {
            for (int ri = 0; ri < rows; ++ri) {
                if (p.h == 1 || part == 0) {
#pragma unroll
                    for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
                }
                const uint32_t wrow = sl + static_cast<uint32_t>(ri) * p.pstride;
                for (int j = j0 + lane; j < j1; j += 32) {
                    const uint32_t wa = wrow + static_cast<uint32_t>(j - j0) * PB;
                    const uint32_t ra = sbase + L.rec + static_cast<uint32_t>(j) * RB;
                    if constexpr (MODE == MODE_Q8) {
                        pair_dot<F, NB>(wa, ra, rstride, acc);
                    } else {
                        const XSrc xa = {sbase + L.xs + static_cast<uint32_t>(j) * 256u, p.x + 64 * j, p.xsm != 0};
                        pair_dot_fx<F, NB>(wa, ra, rstride, xa, p.ncols, acc);
                    }
                }
                if (p.h == 1 || part == p.h - 1) {
                    const int row = r0 + q * p.sr + ri;
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        const float v = warp_sum(acc[b]);
                        if (lane == 0)
                            p.y[(GATHER ? cm.y[b] : static_cast<int64_t>(b) * p.nrows) + row] = v;
                    }
                }
            }
        }
        // the slot is free again: copy this warp's chunk m places ahead into it
        __syncwarp();
        if (lane == 0 && issued < nj) {
            fence_proxy_async_smem();
            issue();
        }
        if (++part == p.h) {
            part = 0;
            q += kMvCW;
        }
        if (++slot_i == m) {
            slot_i = 0;
            phase ^= 1u;
        }
    }
    if (lane == 0 && *abort_flag) {
        // a wait gave up: let this warp's copies still in flight land before exiting
        uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
        for (int jj = consumed; jj < issued; ++jj) {
            if (jj == 0 && held) continue;
            mbar_wait_bounded(&bars[wid + kMvCW * (jj % m)], static_cast<uint32_t>(jj / m) & 1u, p.err);
        }
        if (MODE == MODE_FX && tid == 0 && p.xsm) mbar_wait_bounded(&bars[p.nst], 0u, p.err);
    }
}

template <int F, int NB, int MODE>
__global__ void __launch_bounds__(kMvCW * 32, 1) int_stream_kernel(const IntParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    stream_body<F, NB, MODE, false>(p, ColMap<NB>{}, smem);
}

// ------------------------------------------------- expert-selected GEMV
// Ring geometry of the expert-selected kernel for a work unit of nb columns
// (entry nb - 1): each unit size has its own chunking, all on one grid.
struct IdPlan {
    int spc, h, sr, pstride, nst, slot;
};
struct IdParams {
    const int *ids;         // [batch] expert of each output column
    int batch;              // output columns, 1 .. kIdMaxBatch
    int n_expert;
    int x_group;            // column b reads activation row b / x_group
    int64_t ebytes;         // bytes of one expert matrix
    IdPlan pl[kFxMaxBatch];
};

// Work units: the distinct valid experts of ids in order of first
// appearance, each split into units of up to NBMAX of its columns (in
// column order).  Every CTA computes the same list from ids; CTA
// (blockIdx.x, u) runs rows blockIdx.x of unit u against that unit's expert,
// so each selected expert's weights stream once per NBMAX of its columns.
// Grid y spans the most units any ids can make; CTAs past the last unit
// return at once.  A column with an id outside [0, n_expert) is in no unit
// (its y is not written) and sets ERRBIT_INDEX.
template <int F, int NBMAX>
__global__ void __launch_bounds__(kMvCW * 32, 1) id_stream_kernel(const IntParams p, const IdParams q) {
    extern __shared__ __align__(128) uint8_t smem[];
    int *sid = reinterpret_cast<int *>(smem);                    // [kIdMaxBatch] ids
    int *snu = sid + kIdMaxBatch;                                // [kIdMaxBatch] units of a first column
    int *sinfo = snu + kIdMaxBatch;                              // expert, columns, column list
    const int tid = threadIdx.x;
    griddep_wait();                                              // ids, x and y: after the preceding kernel
    if (tid < 2 + NBMAX) sinfo[tid] = 0;
    if (tid < q.batch) sid[tid] = q.ids[tid];
    cta_sync();
    int id = -1, cnt = 0, rank = 0, first = tid;
    bool valid = false;
    if (tid < q.batch) {
        id = sid[tid];
        valid = id >= 0 && id < q.n_expert;
        for (int s = 0; s < q.batch; ++s) {
            if (sid[s] == id) {
                ++cnt;
                if (s < tid) {
                    ++rank;
                    first = min(first, s);
                }
            }
        }
        snu[tid] = valid && rank == 0 ? (cnt + NBMAX - 1) / NBMAX : 0;
        if (!valid && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(p.err, ERRBIT_INDEX);
    }
    cta_sync();
    if (valid) {
        int u = rank / NBMAX;
        for (int s = 0; s < first; ++s) u += snu[s];
        if (u == static_cast<int>(blockIdx.y)) {
            const int pos = rank % NBMAX;
            sinfo[2 + pos] = tid;
            if (pos == 0) {
                sinfo[0] = id;
                sinfo[1] = min(NBMAX, cnt - (rank / NBMAX) * NBMAX);
            }
        }
    }
    cta_sync();
    const int e = sinfo[0], nbu = sinfo[1];
    int col[NBMAX];
#pragma unroll
    for (int b = 0; b < NBMAX; ++b) col[b] = sinfo[2 + b];
    cta_sync();                                                  // the scratch is free for the ring
    if (nbu == 0) return;
    IntParams pp = p;
    pp.W = p.W + static_cast<int64_t>(e) * q.ebytes;
    const IdPlan &g = q.pl[nbu - 1];
    pp.spc = g.spc;
    pp.h = g.h;
    pp.sr = g.sr;
    pp.pstride = g.pstride;
    pp.nst = g.nst;
    pp.slot = g.slot;
    pp.xsm = 1;
    pp.early = 0;
    switch (nbu) {
#define QG_ID_UNIT(NBU)                                                                  \
    case NBU:                                                                            \
        if constexpr (NBU <= NBMAX) {                                                    \
            ColMap<NBU> cm;                                                              \
            _Pragma("unroll") for (int b = 0; b < NBU; ++b) {                            \
                cm.x[b] = static_cast<int64_t>(col[b] / q.x_group) * p.ncols;            \
                cm.y[b] = static_cast<int64_t>(col[b]) * p.nrows;                        \
            }                                                                            \
            stream_body<F, NBU, MODE_FX, true>(pp, cm, smem);                            \
        }                                                                                \
        break;
        QG_ID_UNIT(1)
        QG_ID_UNIT(2)
        QG_ID_UNIT(3)
        QG_ID_UNIT(4)
#undef QG_ID_UNIT
    default: break;
    }
}

// ----------------------------------------------------------- general GEMV
__device__ __forceinline__ uint32_t ldg_u16(const uint8_t *p) {
    return static_cast<uint32_t>(*reinterpret_cast<const unsigned short *>(p));
}
// Four bytes at a 2-byte aligned address.
__device__ __forceinline__ uint32_t ldg_w2(const uint8_t *p) { return ldg_u16(p) | (ldg_u16(p + 2) << 16); }

template <int F, int NB>
__global__ void __launch_bounds__(kRowWarps * 32)
mmvq_rowwarp_kernel(const IntParams p) {
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
    if (row >= p.nrows) return;
    const int nb = p.ncols / 32;
    const uint8_t *wr = p.W + row * p.rb;
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
    for (int j = lane; j < nb; j += 32) {
        const uint8_t *blk = wr + static_cast<int64_t>(j) * block_bytes(F);
        float dw, mw = 0.0f;
        uint32_t a[8];
        if constexpr (F == FMT_Q4_1) {
            const uint32_t dm = ldg_w2(blk);
            dw = half_lo(dm);
            mw = half_hi(dm);
#pragma unroll
            for (int t = 0; t < 4; ++t) a[t] = ldg_w2(blk + 4 + 4 * t);
        } else {
            dw = half_lo(ldg_u16(blk));
#pragma unroll
            for (int t = 0; t < (F == FMT_Q8_0 ? 8 : 4); ++t) a[t] = ldg_w2(blk + 2 + 4 * t);
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const uint4 *xp = reinterpret_cast<const uint4 *>(p.xq + static_cast<size_t>(b) * p.ncols + 32 * j);
            const uint4 v0 = xp[0], v1 = xp[1];
            const uint32_t X[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            const float dx = p.xd[static_cast<size_t>(b) * nb + j];
            const int sx = p.xs[static_cast<size_t>(b) * nb + j];
            if constexpr (F == FMT_Q8_0) {
                int s0 = 0;
#pragma unroll
                for (int t = 0; t < 8; ++t) s0 = dp4a_ss(a[t], X[t], s0);
                acc[b] = fmaf(dw * static_cast<float>(s0), dx, acc[b]);
            } else {
                Nib n;
                split_nibbles(a, n);
                const int c = dot_nib(n, X);
                if constexpr (F == FMT_Q4_0) {
                    acc[b] = fmaf(dw * static_cast<float>(c - 8 * sx), dx, acc[b]);
                } else {
                    acc[b] = fmaf(fmaf(dw, static_cast<float>(c), mw * static_cast<float>(sx)), dx, acc[b]);
                }
            }
        }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const float v = warp_sum(acc[b]);
        if (lane == 0) p.y[static_cast<int64_t>(b) * p.nrows + row] = v;
    }
}

// ------------------------------------------------------------------- host
constexpr int kMaxDev = 64;

// QGEMV_MMVQ_PATH=stream|rowwarp forces one quantized-activation kernel
// (read once; the path tests use it).
// Expert-selected GEMV for shapes the streaming kernel does not take: one
// warp per (row, output column), the weights decoded exactly in fp32 as the
// dequantizer does (no fused multiply-add in the decode) and multiplied by x
// with fmaf, lane-strided over the blocks, then a fixed-order warp sum.
template <int F>
__global__ void __launch_bounds__(kRowWarps * 32)
id_rowwarp_kernel(const IntParams p, const IdParams q) {
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int e = q.ids[b];
    if (e < 0 || e >= q.n_expert) {
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.err, ERRBIT_INDEX);
        return;
    }
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
    if (row >= p.nrows) return;
    const int nb = p.ncols / 32;
    const uint8_t *wr = p.W + static_cast<int64_t>(e) * q.ebytes + row * p.rb;
    const float *xr = p.x + static_cast<int64_t>(b / q.x_group) * p.ncols;
    float acc = 0.0f;
    for (int j = lane; j < nb; j += 32) {
        const uint8_t *blk = wr + static_cast<int64_t>(j) * block_bytes(F);
        const float4 *xp = reinterpret_cast<const float4 *>(xr + 32 * j);
        float w[32];
        if constexpr (F == FMT_Q8_0) {
            const float d = half_lo(ldg_u16(blk));
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const uint32_t v = ldg_u16(blk + 2 + 2 * t);
                w[2 * t] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(v & 0xffu)));
                w[2 * t + 1] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(v >> 8)));
            }
        } else {
            const int off = F == FMT_Q4_1 ? 4 : 2;
            const float d = half_lo(ldg_u16(blk));
            const float m = F == FMT_Q4_1 ? half_lo(ldg_u16(blk + 2)) : 0.0f;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const uint32_t v = ldg_u16(blk + off + 2 * t);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c = static_cast<int>((v >> (8 * h)) & 0xffu);
                    const int lo = c & 15, hi = c >> 4, i = 2 * t + h;
                    if constexpr (F == FMT_Q4_0) {
                        w[i] = __fmul_rn(d, static_cast<float>(lo - 8));
                        w[i + 16] = __fmul_rn(d, static_cast<float>(hi - 8));
                    } else {
                        w[i] = __fadd_rn(__fmul_rn(d, static_cast<float>(lo)), m);
                        w[i + 16] = __fadd_rn(__fmul_rn(d, static_cast<float>(hi)), m);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const float4 v = xp[t];
            acc = fmaf(w[4 * t], v.x, acc);
            acc = fmaf(w[4 * t + 1], v.y, acc);
            acc = fmaf(w[4 * t + 2], v.z, acc);
            acc = fmaf(w[4 * t + 3], v.w, acc);
        }
    }
    const float v = warp_sum(acc);
    if (lane == 0) p.y[static_cast<int64_t>(b) * p.nrows + row] = v;
}

// QGEMV_ID_PATH forces one kernel of the expert-selected GEMV (for testing
// each on shapes another would take): "tc" the tensor-core kernel, "fx" the
// fixed-point streaming kernel, "rowwarp" the general one.
enum { ID_AUTO = 0, ID_FX = 1, ID_ROWWARP = 2, ID_TC = 3 };
int id_path_override() {
    static int cached = -1;
    if (cached < 0) {
        const char *e = getenv("QGEMV_ID_PATH");
        int v = ID_AUTO;
        if (e && !strcmp(e, "fx")) v = ID_FX;
        if (e && !strcmp(e, "rowwarp")) v = ID_ROWWARP;
        if (e && !strcmp(e, "tc")) v = ID_TC;
        cached = v;
    }
    return cached;
}

int mmvq_path_override() {
    static int cached = -1;
    if (cached < 0) {
        const char *e = getenv("QGEMV_MMVQ_PATH");
        int v = 0;
        if (e && !strcmp(e, "stream")) v = 1;
        if (e && !strcmp(e, "rowwarp")) v = 2;
        cached = v;
    }
    return cached;
}

template <int F, int NB, int MODE>
bool set_smem_attr(int dev, size_t optin) {
    static bool done[kMaxDev] = {false};
    if (done[dev]) return true;
    if (cudaFuncSetAttribute(int_stream_kernel<F, NB, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(optin)) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    done[dev] = true;
    return true;
}

cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// Grid and ring of the streaming kernel; ok = false when the shape does not
// fit it (row bytes not a multiple of 16, ncols not a multiple of 64, or the
// staged activations leave no room for a ring slot per warp).
struct IntPlan {
    bool ok = false;
    int G = 0, spc = 0, h = 0, sr = 0, pstride = 0, nst = 0, slot = 0, xsm = 0;
    size_t smem = 0;
};
IntPlan int_plan_x(int fmt, int mode, int nb_cols, int64_t nrows, int64_t ncols, const DevInfo &di, int xsm,
                   int gmax = 0) {
    IntPlan P;
    P.xsm = xsm;
    const int64_t rb = ncols / 32 * block_bytes(fmt);
    if (rb % 16 != 0 || ncols % 64 != 0 || nrows < 1 || ncols < 64) return P;
    const int PB = 2 * block_bytes(fmt);
    const int npair = static_cast<int>(ncols / 64), nseg = (npair + 31) / 32;
    P.G = static_cast<int>(std::min<int64_t>(nrows, gmax > 0 ? gmax : di.sm_count));
    const int64_t rows_max = (nrows + P.G - 1) / P.G;
    const IntLayout L0 = int_layout(mode, nb_cols, npair, 0, 0, xsm);
    const int64_t room = static_cast<int64_t>(di.smem_optin) - L0.total;
    if (room <= 0) return P;
    const int64_t seg = 32 * PB;
    const int RR = rows_together(mode, nb_cols);
    // Candidate chunks, preferred first: rows of a group (sr), then the
    // largest part of a row (spc segments) up to kChunkTarget bytes per row;
    // the first that leaves each warp two ring slots wins, else the smallest
    // with one slot.
    const int64_t sr_top = rb >= kChunkTarget ? std::min<int64_t>(RR, 2)
                           : RR > 1           ? RR
                                              : std::max<int64_t>(1, kChunkTarget / rb);
    const int64_t spc_top = rb >= kChunkTarget ? std::min<int64_t>(nseg, std::max<int64_t>(1, kChunkTarget / seg)) : nseg;
    for (int pass = 0; pass < 2; ++pass) {
        for (int64_t sr = std::min(sr_top, rows_max); sr >= 1; --sr) {
            for (int64_t c = spc_top; c >= (rb >= kChunkTarget ? 1 : nseg); --c) {
                const int h = static_cast<int>((nseg + c - 1) / c);
                const int64_t pstride = h == 1 ? rb : c * seg;
                const int64_t slot = sr * pstride;
                if (slot >= (1 << 20)) continue;
                const int64_t groups = (rows_max + sr - 1) / sr;
                const int64_t chunks_per_warp = (groups + kMvCW - 1) / kMvCW * h;
                int64_t per_warp = std::min<int64_t>(kMaxPerWarp, room / (kMvCW * (slot + 8)));
                per_warp = std::min<int64_t>(per_warp, std::max<int64_t>(1, chunks_per_warp));
                if (per_warp < 1) continue;
                if (pass == 0 && per_warp < 2 && chunks_per_warp >= 2) continue;
                const IntLayout L = int_layout(mode, nb_cols, npair, static_cast<int>(slot),
                                               static_cast<int>(kMvCW * per_warp), xsm);
                if (L.total > di.smem_optin) continue;
                P.sr = static_cast<int>(sr);
                P.spc = static_cast<int>(c);
                P.h = h;
                P.pstride = static_cast<int>(pstride);
                P.slot = static_cast<int>(slot);
                P.nst = static_cast<int>(kMvCW * per_warp);
                P.smem = L.total;
                P.ok = true;
                return P;
            }
        }
    }
    return P;
}

// Fixed point: fp32 x staged in shared memory when it fits beside a ring of
// two slots per warp, else read from global memory by the exact elements.
IntPlan int_plan(int fmt, int mode, int nb_cols, int64_t nrows, int64_t ncols, const DevInfo &di) {
    if (mode == MODE_FX) {
        IntPlan P = int_plan_x(fmt, mode, nb_cols, nrows, ncols, di, 1);
        if (P.ok && P.nst >= 2 * kMvCW) return P;
        const IntPlan Q = int_plan_x(fmt, mode, nb_cols, nrows, ncols, di, 0);
        return Q.ok ? Q : P;
    }
    return int_plan_x(fmt, mode, nb_cols, nrows, ncols, di, 0);
}

template <int F, int NBMAX>
bool set_id_smem_attr(int dev, size_t optin) {
    static bool done[kMaxDev] = {false};
    if (done[dev]) return true;
    if (cudaFuncSetAttribute(id_stream_kernel<F, NBMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(optin)) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    done[dev] = true;
    return true;
}

template <int F, int NB, int MODE>
qgemv_status launch_stream(IntParams p, const IntPlan &P, int64_t ncols, cudaStream_t s, int dev,
                           const DevInfo &di, const char *what) {
    if (!set_smem_attr<F, NB, MODE>(dev, di.smem_optin)) {
        set_last_error("%s: cannot raise the shared-memory limit", what);
        return QGEMV_ERR_LAUNCH;
    }
    p.rb = static_cast<int>(ncols / 32 * block_bytes(F));
    p.npair = static_cast<int>(ncols / 64);
    p.spc = P.spc;
    p.h = P.h;
    p.sr = P.sr;
    p.pstride = P.pstride;
    p.xsm = P.xsm;
    p.nst = P.nst;
    p.slot = P.slot;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(static_cast<unsigned>(P.G)), dim3(kMvCW * 32), P.smem, s, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, int_stream_kernel<F, NB, MODE>, p);
    if (e != cudaSuccess) {
        set_last_error("%s launch: %s", what, cudaGetErrorString(e));
        return QGEMV_ERR_LAUNCH;
    }
    return check_launch(what);
}

template <int F, int NB>
qgemv_status launch_mmvq_nb(const IntParams &p, int64_t nrows, int64_t ncols, cudaStream_t s, const DevInfo &di,
                            int dev) {
    const int forced = mmvq_path_override();
    if (forced != 2) {
        const IntPlan P = int_plan(F, MODE_Q8, NB, nrows, ncols, di);
        if (P.ok) return launch_stream<F, NB, MODE_Q8>(p, P, ncols, s, dev, di, "qgemv_mmvq(stream)");
        if (forced == 1) {
            set_last_error("qgemv_mmvq: the streaming kernel does not take this shape");
            return QGEMV_ERR_UNIMPLEMENTED;
        }
    }
    IntParams q = p;
    q.rb = static_cast<int>(ncols / 32 * block_bytes(F));
    q.npair = static_cast<int>(ncols / 64);
    cudaLaunchAttribute attr[1];
    const unsigned grid = static_cast<unsigned>((nrows + kRowWarps - 1) / kRowWarps);
    cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(kRowWarps * 32), 0, s, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, mmvq_rowwarp_kernel<F, NB>, q);
    if (e != cudaSuccess) {
        set_last_error("qgemv_mmvq(rowwarp) launch: %s", cudaGetErrorString(e));
        return QGEMV_ERR_LAUNCH;
    }
    return check_launch("qgemv_mmvq(rowwarp)");
}

template <int F>
qgemv_status launch_mmvq_fmt(const IntParams &p, int64_t nrows, int64_t ncols, int batch, cudaStream_t s,
                             const DevInfo &di, int dev) {
    switch (batch) {
    case 1: return launch_mmvq_nb<F, 1>(p, nrows, ncols, s, di, dev);
    case 2: return launch_mmvq_nb<F, 2>(p, nrows, ncols, s, di, dev);
    case 3: return launch_mmvq_nb<F, 3>(p, nrows, ncols, s, di, dev);
    case 4: return launch_mmvq_nb<F, 4>(p, nrows, ncols, s, di, dev);
    case 5: return launch_mmvq_nb<F, 5>(p, nrows, ncols, s, di, dev);
    case 6: return launch_mmvq_nb<F, 6>(p, nrows, ncols, s, di, dev);
    case 7: return launch_mmvq_nb<F, 7>(p, nrows, ncols, s, di, dev);
    case 8: return launch_mmvq_nb<F, 8>(p, nrows, ncols, s, di, dev);
    default:
        set_last_error("qgemv_mmvq: batch %d outside 1..8", batch);
        return QGEMV_ERR_BATCH;
    }
}

template <int F>
qgemv_status launch_fx_fmt(const IntParams &p, const IntPlan &P, int64_t ncols, int batch, cudaStream_t s,
                           const DevInfo &di, int dev) {
    switch (batch) {
    case 1: return launch_stream<F, 1, MODE_FX>(p, P, ncols, s, dev, di, "qgemv(fixed-point)");
    case 2: return launch_stream<F, 2, MODE_FX>(p, P, ncols, s, dev, di, "qgemv(fixed-point)");
    case 3: return launch_stream<F, 3, MODE_FX>(p, P, ncols, s, dev, di, "qgemv(fixed-point)");
    default: return launch_stream<F, 4, MODE_FX>(p, P, ncols, s, dev, di, "qgemv(fixed-point)");
    }
}

IntParams base_params(const void *W, float *y, int64_t nrows, int64_t ncols, unsigned *err) {
    IntParams p = {};
    p.W = static_cast<const uint8_t *>(W);
    p.y = y;
    p.err = err;
    p.nrows = static_cast<int>(nrows);
    p.ncols = static_cast<int>(ncols);
    p.early = g_opt_weights_static;
    p.probes = g_opt_wait_probes;
    p.withhold = g_opt_withhold_next;
    return p;
}

}  // namespace

// Library-lifetime scratch of the one-call quantized-activation entry points
// (activations quantized inside the call): q8_1 of up to kMvqScratchValues
// activations.
constexpr int64_t kMvqScratchValues = int64_t(1) << 21;
__device__ __align__(16) uint8_t g_mvq_scratch[kMvqScratchValues + kMvqScratchValues / 4];

int64_t q8_1_bytes(int64_t ncols, int batch) { return static_cast<int64_t>(batch) * (ncols + ncols / 4); }
int64_t mmvq_scratch_values() { return kMvqScratchValues; }

qgemv_status launch_quantize_q8_1(const float *x, void *xq, int64_t ncols, int batch, cudaStream_t s) {
    const int64_t nblocks = static_cast<int64_t>(batch) * (ncols / 32);
    uint8_t *base = static_cast<uint8_t *>(xq);
    int8_t *q = reinterpret_cast<int8_t *>(base);
    float *d = reinterpret_cast<float *>(base + static_cast<int64_t>(batch) * ncols);
    int *sm = reinterpret_cast<int *>(base + static_cast<int64_t>(batch) * ncols + 4 * nblocks);
    cudaLaunchAttribute attr[1];
    const unsigned grid = static_cast<unsigned>((nblocks + kQuantWarps - 1) / kQuantWarps);
    cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(kQuantWarps * 32), 0, s, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel, x, q, d, sm, nblocks);
    if (e != cudaSuccess) {
        set_last_error("qquantize_q8_1 launch: %s", cudaGetErrorString(e));
        return QGEMV_ERR_LAUNCH;
    }
    return check_launch("qquantize_q8_1");
}

qgemv_status launch_gemv_mmvq(int fmt, const void *W, const void *xq, float *y, int64_t nrows, int64_t ncols,
                              int batch, cudaStream_t s, const DevInfo &di, int dev, unsigned *err) {
    const uint8_t *base = static_cast<const uint8_t *>(xq);
    const int64_t nblocks = static_cast<int64_t>(batch) * (ncols / 32);
    IntParams p = base_params(W, y, nrows, ncols, err);
    g_opt_withhold_next = 0;
    p.xq = reinterpret_cast<const int8_t *>(base);
    p.xd = reinterpret_cast<const float *>(base + static_cast<int64_t>(batch) * ncols);
    p.xs = reinterpret_cast<const int *>(base + static_cast<int64_t>(batch) * ncols + 4 * nblocks);
    switch (fmt) {
    case FMT_Q4_0: return launch_mmvq_fmt<FMT_Q4_0>(p, nrows, ncols, batch, s, di, dev);
    case FMT_Q4_1: return launch_mmvq_fmt<FMT_Q4_1>(p, nrows, ncols, batch, s, di, dev);
    case FMT_Q8_0: return launch_mmvq_fmt<FMT_Q8_0>(p, nrows, ncols, batch, s, di, dev);
    default: return QGEMV_ERR_DTYPE;
    }
}

qgemv_status launch_gemv_fx(int fmt, const void *W, const float *x, float *y, int64_t nrows, int64_t ncols,
                            int batch, cudaStream_t s, const DevInfo &di, int dev, unsigned *err, bool *taken) {
    *taken = false;
    if (batch < 1 || nrows > (int64_t(1) << 30) || ncols > (int64_t(1) << 20)) return QGEMV_OK;
    // the widest group of batch columns (up to kFxMaxBatch) whose records fit one CTA
    int cols = std::min(batch, kFxMaxBatch);
    IntPlan P;
    for (; cols >= 1; --cols) {
        P = int_plan(fmt, MODE_FX, cols, nrows, ncols, di);
        if (P.ok) break;
    }
    if (cols < 1) return QGEMV_OK;
    // Wider batches take one launch per group of columns only for Q4_1, whose
    // tensor-core path adds m * sum(x) without the cancellation check; the
    // other formats keep them on the tensor-core kernel.
    if (cols < batch && fmt != FMT_Q4_1) return QGEMV_OK;
    *taken = true;
    IntParams p = base_params(W, y, nrows, ncols, err);
    g_opt_withhold_next = 0;
    for (int b0 = 0; b0 < batch; b0 += cols) {
        const int n = std::min(cols, batch - b0);
        const IntPlan Pn = n == cols ? P : int_plan(fmt, MODE_FX, n, nrows, ncols, di);
        p.x = x + static_cast<int64_t>(b0) * ncols;
        p.y = y + static_cast<int64_t>(b0) * nrows;
        qgemv_status st = QGEMV_ERR_DTYPE;
        switch (fmt) {
        case FMT_Q4_0: st = launch_fx_fmt<FMT_Q4_0>(p, Pn, ncols, n, s, di, dev); break;
        case FMT_Q4_1: st = launch_fx_fmt<FMT_Q4_1>(p, Pn, ncols, n, s, di, dev); break;
        case FMT_Q8_0: st = launch_fx_fmt<FMT_Q8_0>(p, Pn, ncols, n, s, di, dev); break;
        default: break;
        }
        if (st != QGEMV_OK) return st;
        p.withhold = 0;
    }
    return QGEMV_OK;
}

namespace {

// Most work units any ids of `batch` columns over n_expert experts can make
// with up to nb columns a unit: D distinct experts give D units plus one for
// every further nb columns of an expert, at most D + (batch - D) / nb, which
// grows with D.
int id_max_units(int batch, int64_t n_expert, int nb) {
    const int D = static_cast<int>(std::min<int64_t>(batch, n_expert));
    return D + (batch - D) / nb;
}

template <int F, int NBMAX>
qgemv_status launch_id_nb(const IntParams &p, const IdParams &q, int G, int units, size_t smem, cudaStream_t s,
                          int dev, const DevInfo &di) {
    if (!set_id_smem_attr<F, NBMAX>(dev, di.smem_optin)) {
        set_last_error("qgemv_id: cannot raise the shared-memory limit");
        return QGEMV_ERR_LAUNCH;
    }
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(static_cast<unsigned>(G), static_cast<unsigned>(units)),
                                        dim3(kMvCW * 32), smem, s, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, id_stream_kernel<F, NBMAX>, p, q);
    if (e != cudaSuccess) {
        set_last_error("qgemv_id launch: %s", cudaGetErrorString(e));
        return QGEMV_ERR_LAUNCH;
    }
    return check_launch("qgemv_id");
}

template <int F>
qgemv_status launch_id_fmt(const IntParams &p, const IdParams &q, int nbmax, int G, int units, size_t smem,
                           cudaStream_t s, int dev, const DevInfo &di) {
    switch (nbmax) {
    case 1: return launch_id_nb<F, 1>(p, q, G, units, smem, s, dev, di);
    case 2: return launch_id_nb<F, 2>(p, q, G, units, smem, s, dev, di);
    case 3: return launch_id_nb<F, 3>(p, q, G, units, smem, s, dev, di);
    default: return launch_id_nb<F, 4>(p, q, G, units, smem, s, dev, di);
    }
}

}  // namespace

int id_max_batch() { return kIdMaxBatch; }

qgemv_status launch_gemv_id(int fmt, const void *W, int64_t n_expert, const int *ids, const float *x, int x_group,
                            float *y, int64_t nrows, int64_t ncols, int batch, cudaStream_t s, const DevInfo &di,
                            int dev, unsigned *err) {
    const int forced = id_path_override();
    // Up to two columns (one token's top-1 or top-2 experts): units of one
    // column, where the fixed-point kernel on half the SMs per expert is as
    // fast as the tensor cores or faster (Q4_1, Q8_0).  More columns -- more
    // experts per token, or several tokens whose experts repeat -- go to the
    // tensor cores, which take a unit's columns in one MMA and start faster
    // on the shorter row ranges of many experts.
    if (forced == ID_TC || (forced == ID_AUTO && batch > 2)) {
        bool taken = false;
        const qgemv_status st =
            launch_gemv_sk_id(fmt, W, n_expert, ids, x, x_group, y, nrows, ncols, batch, s, di, err, &taken);
        if (taken || st != QGEMV_OK) return st;
        if (forced == ID_TC) {
            set_last_error("qgemv_id: the tensor-core kernel does not take this shape");
            return QGEMV_ERR_UNIMPLEMENTED;
        }
    }
    // the widest unit (columns of one expert) whose activations and records
    // fit a CTA beside a ring
    int nbmax = std::min(batch, kFxMaxBatch);
    for (; nbmax >= 1; --nbmax) {
        const IntPlan P = int_plan_x(fmt, MODE_FX, nbmax, nrows, ncols, di, 1);
        if (P.ok) break;
    }
    IdParams q = {};
    q.ids = ids;
    q.batch = batch;
    q.n_expert = static_cast<int>(std::min<int64_t>(n_expert, INT32_MAX));
    q.x_group = x_group;
    q.ebytes = nrows * (ncols / 32) * block_bytes(fmt);
    if (nbmax < 1 || forced == ID_ROWWARP) {
        // no streaming plan (row bytes not a multiple of 16, ncols not a
        // multiple of 64, or a column's activations too large): the general kernel
        IntParams p = base_params(W, y, nrows, ncols, err);
        p.x = x;
        p.rb = static_cast<int>(ncols / 32 * block_bytes(fmt));
        cudaLaunchAttribute attr[1];
        const dim3 grid(static_cast<unsigned>((nrows + kRowWarps - 1) / kRowWarps), static_cast<unsigned>(batch));
        cudaLaunchConfig_t cfg = pdl_config(grid, dim3(kRowWarps * 32), 0, s, attr);
        cudaError_t e = cudaErrorInvalidValue;
        switch (fmt) {
        case FMT_Q4_0: e = cudaLaunchKernelEx(&cfg, id_rowwarp_kernel<FMT_Q4_0>, p, q); break;
        case FMT_Q4_1: e = cudaLaunchKernelEx(&cfg, id_rowwarp_kernel<FMT_Q4_1>, p, q); break;
        case FMT_Q8_0: e = cudaLaunchKernelEx(&cfg, id_rowwarp_kernel<FMT_Q8_0>, p, q); break;
        default: return QGEMV_ERR_DTYPE;
        }
        if (e != cudaSuccess) {
            set_last_error("qgemv_id(rowwarp) launch: %s", cudaGetErrorString(e));
            return QGEMV_ERR_LAUNCH;
        }
        return check_launch("qgemv_id(rowwarp)");
    }
    const int units = id_max_units(batch, n_expert, nbmax);
    const int G = std::max(1, di.sm_count / units);
    size_t smem = 0;
    int Gp = 0;
    for (int nb = 1; nb <= nbmax; ++nb) {
        const IntPlan P = int_plan_x(fmt, MODE_FX, nb, nrows, ncols, di, 1, G);
        if (!P.ok) {
            set_last_error("qgemv_id: no ring for units of %d columns", nb);
            return QGEMV_ERR_UNIMPLEMENTED;
        }
        q.pl[nb - 1] = {P.spc, P.h, P.sr, P.pstride, P.nst, P.slot};
        smem = std::max(smem, P.smem);
        Gp = P.G;
    }
    // the unit scratch (ids, unit counts, the chosen unit) sits at the start of the ring's shared memory
    smem = std::max(smem, static_cast<size_t>((2 * kIdMaxBatch + 2 + kFxMaxBatch) * 4));
    IntParams p = base_params(W, y, nrows, ncols, err);
    g_opt_withhold_next = 0;
    p.x = x;
    p.rb = static_cast<int>(ncols / 32 * block_bytes(fmt));
    p.npair = static_cast<int>(ncols / 64);
    switch (fmt) {
    case FMT_Q4_0: return launch_id_fmt<FMT_Q4_0>(p, q, nbmax, Gp, units, smem, s, dev, di);
    case FMT_Q4_1: return launch_id_fmt<FMT_Q4_1>(p, q, nbmax, Gp, units, smem, s, dev, di);
    case FMT_Q8_0: return launch_id_fmt<FMT_Q8_0>(p, q, nbmax, Gp, units, smem, s, dev, di);
    default: return QGEMV_ERR_DTYPE;
    }
}

qgemv_status mmvq_scratch(void **ptr) {
    cudaError_t e = cudaGetSymbolAddress(ptr, g_mvq_scratch);
    if (e != cudaSuccess) {
        set_last_error("cudaGetSymbolAddress(q8_1 scratch): %s", cudaGetErrorString(e));
        return QGEMV_ERR_CUDA;
    }
    return QGEMV_OK;
}

}  // namespace qg
