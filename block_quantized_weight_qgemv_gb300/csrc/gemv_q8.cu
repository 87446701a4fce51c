// gemv_q8.cu -- the quantized-activation GEMV family (mul_mat_vec_q):
// activations are converted to int8 blocks of 32 values and contracted with
// the weights' integer codes by byte-wise integer dot products.
//
// Source: "llama_cpp 0.12.1 -> 0.12.2" (the vendored ggml-cuda.cu diff):
// ggml_cuda_op_mul_mat_vec_q, the convert_src1_to_q8_1 flag of
// ggml_cuda_op_mul_mat, the "MMVQ = mul_mat_vec_q" note and the __dp4a note
// beside MIN_CC_DP4A.  The pages print neither the activation block layout
// nor its quantizer; the reading implemented here is
//   amax = max |x_i| over 32 consecutive values of one batch column,
//   d = amax / 127 (IEEE fp32 division),
//   q_i = x_i / d (IEEE fp32 division) rounded to nearest, ties to even,
//         clamped to [-127, 127]; q_i = 0 when d == 0,
//   a block holding a NaN or an infinity: d = NaN and every q_i = 0,
//   s = sum_i q_i (exact int32).
// Quantized activations live in one buffer: q int8 [batch][ncols], then d
// fp32 [batch][ncols/32], then s int32 [batch][ncols/32].
//
// The GEMV computes, for each weight block j of row r and batch column b,
//   Q4_0: d_w * (sum_i c_i q_i - 8 s) * d_x     (c = the 4-bit codes)
//   Q4_1: (d_w * sum_i c_i q_i + m_w * s) * d_x
//   Q8_0: d_w * (sum_i c_i q_i) * d_x            (c = the int8 codes)
// with the integer sums exact (dp4a) and the block terms accumulated in fp32.
//
// Kernels:
//  * quantize_q8_1_kernel -- one warp per block of 32 activations.
//  * mmvq_stream_kernel<F, NB> -- one CTA per SM owns a contiguous range of
//    weight rows.  Because the rows of a row-major block matrix are
//    consecutive, the range is one contiguous byte range: a producer lane
//    streams it through a ring of shared-memory stages with 1-D bulk copies
//    (whole rows per stage).  Slot k of the ring belongs to consumer warp k,
//    which takes the stages k, k + nst, k + 2 nst, ... in order, one lane per
//    pair of blocks: every wait on a slot's barrier is then for the phase
//    that follows the one its own warp consumed last, so a parity wait can
//    never match an older phase.  The activations of the call are staged once
//    per CTA as 80-byte records per pair of blocks (64 codes plus the two
//    blocks' d and s), a stride that keeps the 16-byte shared loads of 32
//    lanes free of bank conflicts, as is the 36-, 40- or 68-byte stride of
//    the weight pairs.  Each row is reduced by its own warp: no partial sums
//    leave the warp, and the order of every sum is fixed.
//  * mmvq_rowwarp_kernel<F, NB> -- any shape: one warp per row, blocks read
//    from global memory.
#include <cstdlib>
#include <cstring>
#include <algorithm>

#include "qgemv_common.cuh"

namespace qg {

namespace {

constexpr int kMvCW = 16;                    // consumer warps of the streaming kernel
constexpr int kMvProd = kMvCW;               // warp index of the producer
constexpr int kMvThreads = (kMvCW + 1) * 32;
constexpr int kRecBytes = 80;                // staged activation record of a block pair
constexpr int kMaxStages = kMvCW;            // ring slots: one per consumer warp
constexpr int kQuantWarps = 8;               // warps of a quantizer CTA
constexpr int kRowWarps = 8;                 // warps of a general-kernel CTA

// ------------------------------------------------------------ device helpers
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Barrier 1 over the consumer warps only (unaligned form).
__device__ __forceinline__ void consumers_sync() {
    asm volatile("barrier.sync 1, %0;" :: "n"(kMvCW * 32) : "memory");
}

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

// --------------------------------------------------------- streaming GEMV
struct MvqParams {
    const uint8_t *W;
    const int8_t *xq;       // codes [batch][ncols]
    const float *xd;        // scales [batch][ncols/32]
    const int *xs;          // code sums [batch][ncols/32]
    float *y;               // [batch][nrows]
    unsigned *err;
    int nrows, ncols;
    int npair;              // ncols / 64
    int rb;                 // bytes of a weight row
    int sr;                 // rows of a ring stage
    int nst;                // ring stages
    int early;              // weights static: copy them before the dependency wait
    unsigned probes;
    int withhold;           // testing: never copy the first stage (its wait runs out)
};

template <int F> struct MvPair;
template <> struct MvPair<FMT_Q4_0> { static constexpr int kBytes = 36; };
template <> struct MvPair<FMT_Q4_1> { static constexpr int kBytes = 40; };
template <> struct MvPair<FMT_Q8_0> { static constexpr int kBytes = 68; };

// The two blocks of a weight pair, decoded once and contracted with NB
// activation records.  wa: shared address of the pair; xa: shared address of
// batch column 0's record; xstride: bytes between the records of two columns.
template <int F, int NB>
__device__ __forceinline__ void pair_dot(uint32_t wa, uint32_t xa, uint32_t xstride, float acc[NB]) {
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
        Nib n0, n1;
        split_nibbles(a0, n0);
        split_nibbles(a1, n1);
        const float d0 = half_lo(w[0]), d1 = half_hi(w[4]);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const uint32_t r = xa + b * xstride;
            uint32_t X0[8], X1[8];
            const uint4 v0 = lds128(r), v1 = lds128(r + 16), v2 = lds128(r + 32), v3 = lds128(r + 48);
            const uint4 ds = lds128(r + 64);
            X0[0] = v0.x; X0[1] = v0.y; X0[2] = v0.z; X0[3] = v0.w;
            X0[4] = v1.x; X0[5] = v1.y; X0[6] = v1.z; X0[7] = v1.w;
            X1[0] = v2.x; X1[1] = v2.y; X1[2] = v2.z; X1[3] = v2.w;
            X1[4] = v3.x; X1[5] = v3.y; X1[6] = v3.z; X1[7] = v3.w;
            const int s0 = dot_nib(n0, X0) - 8 * static_cast<int>(ds.y);
            const int s1 = dot_nib(n1, X1) - 8 * static_cast<int>(ds.w);
            acc[b] = fmaf(d0 * static_cast<float>(s0), __uint_as_float(ds.x), acc[b]);
            acc[b] = fmaf(d1 * static_cast<float>(s1), __uint_as_float(ds.z), acc[b]);
        }
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
        Nib n0, n1;
        split_nibbles(a0, n0);
        split_nibbles(a1, n1);
        const float d0 = half_lo(w[0]), m0 = half_hi(w[0]);
        const float d1 = half_lo(w[5]), m1 = half_hi(w[5]);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const uint32_t r = xa + b * xstride;
            uint32_t X0[8], X1[8];
            const uint4 v0 = lds128(r), v1 = lds128(r + 16), v2 = lds128(r + 32), v3 = lds128(r + 48);
            const uint4 ds = lds128(r + 64);
            X0[0] = v0.x; X0[1] = v0.y; X0[2] = v0.z; X0[3] = v0.w;
            X0[4] = v1.x; X0[5] = v1.y; X0[6] = v1.z; X0[7] = v1.w;
            X1[0] = v2.x; X1[1] = v2.y; X1[2] = v2.z; X1[3] = v2.w;
            X1[4] = v3.x; X1[5] = v3.y; X1[6] = v3.z; X1[7] = v3.w;
            const float t0 = fmaf(d0, static_cast<float>(dot_nib(n0, X0)),
                                  m0 * static_cast<float>(static_cast<int>(ds.y)));
            const float t1 = fmaf(d1, static_cast<float>(dot_nib(n1, X1)),
                                  m1 * static_cast<float>(static_cast<int>(ds.w)));
            acc[b] = fmaf(t0, __uint_as_float(ds.x), acc[b]);
            acc[b] = fmaf(t1, __uint_as_float(ds.z), acc[b]);
        }
    } else {
        // [d0 | c0 c1] [c2..c5] ... [c30 c31 | d1] [block 1 codes x8]
        uint32_t w[17];
#pragma unroll
        for (int t = 0; t < 17; ++t) w[t] = lds32(wa + 4 * t);
        uint32_t a0[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) a0[t] = __byte_perm(w[t], w[t + 1], 0x5432);
        const float d0 = half_lo(w[0]), d1 = half_hi(w[8]);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const uint32_t r = xa + b * xstride;
            const uint4 v0 = lds128(r), v1 = lds128(r + 16), v2 = lds128(r + 32), v3 = lds128(r + 48);
            const uint4 ds = lds128(r + 64);
            const uint32_t X0[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            const uint32_t X1[8] = {v2.x, v2.y, v2.z, v2.w, v3.x, v3.y, v3.z, v3.w};
            int s0 = 0, s1 = 0;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                s0 = dp4a_ss(a0[t], X0[t], s0);
                s1 = dp4a_ss(w[9 + t], X1[t], s1);
            }
            acc[b] = fmaf(d0 * static_cast<float>(s0), __uint_as_float(ds.x), acc[b]);
            acc[b] = fmaf(d1 * static_cast<float>(s1), __uint_as_float(ds.z), acc[b]);
        }
    }
}

// Shared-memory layout: [records: NB * npair * 80][ring: nst * sr * rb]
// [full: nst][empty: nst][abort flag].
struct MvLayout {
    uint32_t rec, ring, stage, bars, flag, total;
};
__host__ __device__ inline MvLayout mv_layout(int nb_cols, int npair, int sr, int rb, int nst) {
    MvLayout L;
    L.rec = 0;
    L.ring = static_cast<uint32_t>(nb_cols) * npair * kRecBytes;
    L.stage = static_cast<uint32_t>(sr) * rb;
    L.bars = L.ring + static_cast<uint32_t>(nst) * L.stage;
    L.flag = L.bars + 16u * nst;
    L.total = L.flag + 16;
    return L;
}

template <int F, int NB>
__global__ void __launch_bounds__(kMvThreads, 1) mmvq_stream_kernel(const MvqParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    const int r0 = static_cast<int>(static_cast<int64_t>(cta) * p.nrows / G);
    const int r1 = static_cast<int>(static_cast<int64_t>(cta + 1) * p.nrows / G);
    const int nrow = r1 - r0;
    const int nstage = (nrow + p.sr - 1) / p.sr;
    const MvLayout L = mv_layout(NB, p.npair, p.sr, p.rb, p.nst);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t full0 = sbase + L.bars;               // full[k] at full0 + 8k
    const uint32_t empty0 = full0 + 8u * p.nst;          // empty[k] at empty0 + 8k
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.flag);

    griddep_launch_dependents();
    if (wid == kMvProd && lane == 0) {
        uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
        for (int k = 0; k < p.nst; ++k) {
            mbar_init(&bars[k], 1);
            mbar_init(&bars[p.nst + k], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    cta_sync();

    if (wid == kMvProd) {
        // ------------------------------------------------ producer warp
        // Lane 0 copies stage t (rows r0 + t*sr ...) into slot t % nst.  A
        // slot is reused once its consumer warp has released the stage before.
        int last = -1;                                   // last stage issued
        const bool held = p.withhold && cta == 0;        // stage 0 withheld (testing)
        if (lane == 0) {
            const uint64_t pol = l2_evict_first();
            auto issue = [&](int t) {
                const int k = t % p.nst;
                const int rows = min(p.sr, nrow - t * p.sr);
                const uint32_t bytes = static_cast<uint32_t>(rows) * p.rb;
                if (!(t == 0 && held)) {
                    mbar_expect_tx_a(full0 + 8u * k, bytes);
                    bulk_g2s_hint(sbase + L.ring + static_cast<uint32_t>(k) * L.stage,
                                  p.W + static_cast<size_t>(r0 + t * p.sr) * p.rb, bytes, full0 + 8u * k, pol);
                }
                last = t;
            };
            const int first = min(p.nst, nstage);
            int t = 0;
            if (p.early)
                for (; t < first; ++t) issue(t);
            griddep_wait();                              // W may come from the preceding kernel
            for (; t < first; ++t) issue(t);
            for (; t < nstage; ++t) {
                const int k = t % p.nst;
                if (!mbar_ready(empty0 + 8u * k, static_cast<uint32_t>(t / p.nst - 1) & 1u, p.probes, abort_flag)) {
                    if (!*abort_flag) {
                        *abort_flag = 1;
                        atomicOr(p.err, ERRBIT_TIMEOUT);
                    }
                    break;
                }
                issue(t);
            }
        }
        cta_sync();
        if (lane == 0 && *abort_flag) {
            // a wait gave up: let every copy still in flight land before exiting
            for (int t = max(0, last - p.nst + 1); t <= last; ++t) {
                if (t == 0 && held) continue;
                mbar_wait_bounded(reinterpret_cast<uint64_t *>(smem + L.bars) + (t % p.nst),
                                  static_cast<uint32_t>(t / p.nst) & 1u, p.err);
            }
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    griddep_wait();                                      // x and y: after the preceding kernel
    const int nb = p.ncols / 32;
    for (int i = tid; i < NB * p.npair; i += kMvCW * 32) {
        const int b = i / p.npair, j = i - b * p.npair;
        const uint4 *qs = reinterpret_cast<const uint4 *>(p.xq + static_cast<size_t>(b) * p.ncols + 64 * j);
        const uint4 v0 = qs[0], v1 = qs[1], v2 = qs[2], v3 = qs[3];
        const float2 dd = *reinterpret_cast<const float2 *>(p.xd + static_cast<size_t>(b) * nb + 2 * j);
        const int2 ss = *reinterpret_cast<const int2 *>(p.xs + static_cast<size_t>(b) * nb + 2 * j);
        const uint32_t r = sbase + L.rec + static_cast<uint32_t>(b * p.npair + j) * kRecBytes;
        sts128(r, v0);
        sts128(r + 16, v1);
        sts128(r + 32, v2);
        sts128(r + 48, v3);
        sts128(r + 64, make_uint4(__float_as_uint(dd.x), static_cast<uint32_t>(ss.x), __float_as_uint(dd.y),
                                  static_cast<uint32_t>(ss.y)));
    }
    consumers_sync();

    const uint32_t xstride = static_cast<uint32_t>(p.npair) * kRecBytes;
    const int nseg = (p.npair + 31) / 32;
    const int k = wid;                                   // this warp's slot (warps >= nst have none)
    uint32_t phase = 0;
    for (int t = k; k < p.nst && t < nstage; t += p.nst, phase ^= 1u) {
        if (!mbar_ready(full0 + 8u * k, phase, p.probes, abort_flag)) {
            if (lane == 0 && !*abort_flag) {
                *abort_flag = 1;
                atomicOr(p.err, ERRBIT_TIMEOUT);
            }
            break;
        }
        const int i0 = t * p.sr, rows = min(p.sr, nrow - i0);
        for (int ri = 0; ri < rows; ++ri) {
            const uint32_t wrow = sbase + L.ring + static_cast<uint32_t>(k) * L.stage +
                                  static_cast<uint32_t>(ri) * p.rb;
            float acc[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
            for (int g = 0; g < nseg; ++g) {
                const int j = g * 32 + lane;
                if (j < p.npair) {
                    pair_dot<F, NB>(wrow + static_cast<uint32_t>(j) * MvPair<F>::kBytes,
                                    sbase + L.rec + static_cast<uint32_t>(j) * kRecBytes, xstride, acc);
                }
            }
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float v = warp_sum(acc[b]);
                if (lane == 0) p.y[static_cast<int64_t>(b) * p.nrows + r0 + i0 + ri] = v;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_a(empty0 + 8u * k);
    }
    cta_sync();
}

// ----------------------------------------------------------- general GEMV
__device__ __forceinline__ uint32_t ldg_u16(const uint8_t *p) {
    return static_cast<uint32_t>(*reinterpret_cast<const unsigned short *>(p));
}
// Four bytes at a 2-byte aligned address.
__device__ __forceinline__ uint32_t ldg_w2(const uint8_t *p) { return ldg_u16(p) | (ldg_u16(p + 2) << 16); }

template <int F, int NB>
__global__ void __launch_bounds__(kRowWarps * 32)
mmvq_rowwarp_kernel(const MvqParams p) {
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

// QGEMV_MMVQ_PATH=stream|rowwarp forces one kernel (read once; the path
// tests use it).
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

template <int F, int NB>
bool set_smem_attr(int dev, size_t optin) {
    static bool done[kMaxDev] = {false};
    if (done[dev]) return true;
    if (cudaFuncSetAttribute(mmvq_stream_kernel<F, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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

template <int F, int NB>
qgemv_status launch_mmvq_nb(const MvqParams &base, int64_t nrows, int64_t ncols, cudaStream_t s,
                            const DevInfo &di, int dev) {
    MvqParams p = base;
    const int forced = mmvq_path_override();
    const int64_t rb = ncols / 32 * block_bytes(F);
    if (forced != 2 && rb % 16 == 0 && ncols % 64 == 0) {
        // Ring: as many whole rows as fit beside the staged activations, in
        // up to kMvCW slots (one per consumer warp) of sr rows each; no more
        // slots or rows than a CTA owns.
        const int G = static_cast<int>(std::min<int64_t>(nrows, di.sm_count));
        const int64_t rows_max = (nrows + G - 1) / G;
        const int npair = static_cast<int>(ncols / 64);
        const MvLayout L0 = mv_layout(NB, npair, 1, static_cast<int>(rb), 0);
        const int64_t room = static_cast<int64_t>(di.smem_optin) - L0.total - 16 * kMaxStages;
        const int64_t rows_fit = room > 0 ? room / rb : 0;
        const int nst = static_cast<int>(std::min<int64_t>(std::min<int64_t>(kMaxStages, rows_fit), rows_max));
        const int sr = nst > 0 ? static_cast<int>(std::max<int64_t>(
                                     1, std::min<int64_t>(rows_fit / nst, (rows_max + nst - 1) / nst)))
                               : 0;
        if ((nst >= 2 || (nst == 1 && rows_max == 1)) && static_cast<int64_t>(sr) * rb < (int64_t(1) << 20) &&
            set_smem_attr<F, NB>(dev, di.smem_optin)) {
            p.rb = static_cast<int>(rb);
            p.npair = npair;
            p.sr = sr;
            p.nst = nst;
            const MvLayout L = mv_layout(NB, npair, sr, p.rb, nst);
            cudaLaunchAttribute attr[1];
            cudaLaunchConfig_t cfg = pdl_config(dim3(static_cast<unsigned>(G)), dim3(kMvThreads), L.total, s, attr);
            cudaError_t e = cudaLaunchKernelEx(&cfg, mmvq_stream_kernel<F, NB>, p);
            if (e != cudaSuccess) {
                set_last_error("qgemv_mmvq(stream) launch: %s", cudaGetErrorString(e));
                return QGEMV_ERR_LAUNCH;
            }
            return check_launch("qgemv_mmvq(stream)");
        }
        if (forced == 1) {
            set_last_error("qgemv_mmvq: the streaming kernel does not take this shape");
            return QGEMV_ERR_UNIMPLEMENTED;
        }
    } else if (forced == 1) {
        set_last_error("qgemv_mmvq: the streaming kernel needs row bytes a multiple of 16 and ncols of 64");
        return QGEMV_ERR_UNIMPLEMENTED;
    }
    p.rb = static_cast<int>(rb);
    p.npair = static_cast<int>(ncols / 64);
    cudaLaunchAttribute attr[1];
    const unsigned grid = static_cast<unsigned>((nrows + kRowWarps - 1) / kRowWarps);
    cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(kRowWarps * 32), 0, s, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, mmvq_rowwarp_kernel<F, NB>, p);
    if (e != cudaSuccess) {
        set_last_error("qgemv_mmvq(rowwarp) launch: %s", cudaGetErrorString(e));
        return QGEMV_ERR_LAUNCH;
    }
    return check_launch("qgemv_mmvq(rowwarp)");
}

template <int F>
qgemv_status launch_mmvq_fmt(const MvqParams &p, int64_t nrows, int64_t ncols, int batch, cudaStream_t s,
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

}  // namespace

// Library-lifetime scratch of the one-call entry points (activations
// quantized inside the call): q8_1 of up to kMvqScratchValues activations.
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
    MvqParams p = {};
    p.W = static_cast<const uint8_t *>(W);
    p.xq = reinterpret_cast<const int8_t *>(base);
    p.xd = reinterpret_cast<const float *>(base + static_cast<int64_t>(batch) * ncols);
    p.xs = reinterpret_cast<const int *>(base + static_cast<int64_t>(batch) * ncols + 4 * nblocks);
    p.y = y;
    p.err = err;
    p.nrows = static_cast<int>(nrows);
    p.ncols = static_cast<int>(ncols);
    p.early = g_opt_weights_static;
    p.probes = g_opt_wait_probes;
    p.withhold = g_opt_withhold_next;
    g_opt_withhold_next = 0;
    switch (fmt) {
    case FMT_Q4_0: return launch_mmvq_fmt<FMT_Q4_0>(p, nrows, ncols, batch, s, di, dev);
    case FMT_Q4_1: return launch_mmvq_fmt<FMT_Q4_1>(p, nrows, ncols, batch, s, di, dev);
    case FMT_Q8_0: return launch_mmvq_fmt<FMT_Q8_0>(p, nrows, ncols, batch, s, di, dev);
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
