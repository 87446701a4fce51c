// gemv_tc.cu -- Q4_0 / Q4_1 GEMV on the tensor cores (mma.sync m16n8k16,
// bf16 operands, fp32 accumulation):  y[b][r] = sum_k w[r][k] * x[b][k],
// batch 1..8 (the batch-1 dequantize_mul_mat_vec path of the "llama_cpp
// 0.12.1 -> 0.12.2" ggml-cuda.cu diff, extended to small batches).
//
// Why tensor cores for a bandwidth-bound product: decoding 4-bit weights and
// multiplying them on the CUDA cores costs >= 2.5 instructions per weight,
// about what the SMs can issue while HBM delivers 6+ TB/s.  Here a lane turns
// two nibbles into two exact bf16 values with ONE logic instruction and the
// products and sums go to the tensor pipe; the batch (<= 8) rides along in
// the MMA's N dimension for free.
//
// Exactness of the operands:
//  - A (weights): (word >> s) & 0x000f000f | 0x43004300 is the bf16 pair
//    (128 + q_lo, 128 + q_hi), exact.  The 128 (and Q4_0's 8) are removed by
//    one extra "correction" MMA per block: A_corr = -(128 + OFF) on three
//    k-slots, B_corr = the block's sum of x split into three bf16 parts.
//  - B (activations): x = hi + lo with hi = bf16(x), lo = bf16(x - hi), so
//    |x - hi - lo| <= 2^-17 |x|, with fp32's exponent range.
//  - Each block's fp32 partial is scaled by its fp16 d (and, for Q4_1, m times
//    the block's sum of x is added) in fp32 on the CUDA cores.
//
// Work split: a thread-block cluster of CS CTAs owns a balanced range of rows;
// CTA j of the cluster takes the j-th 1/CS of the columns (so its slice of x
// fits in shared memory for any batch).  Rows are processed in tiles of 16
// (the MMA's M); a unit of work is (tile, 8 blocks); each warp owns a
// contiguous run of units and streams them with one 2-D TMA copy per unit
// (16 rows x 8 blocks) into a private ring of mbarrier-completed slots.  Per-warp tile
// partials are summed in a fixed order, then the CS partial vectors of the
// cluster are summed in rank order through distributed shared memory: the
// result is deterministic.
//
// mma.sync fragment layout (m16n8k16, g = lane/4, c = lane%4):
//   A: a0 = (row g,   k 2c..2c+1)  a1 = (row g+8, k 2c..2c+1)
//      a2 = (row g,   k 2c+8..+9)  a3 = (row g+8, k 2c+8..+9)
//   B: b0 = (k 2c..2c+1, n g)      b1 = (k 2c+8..+9, n g)
//   C: c0 = (g, 2c) c1 = (g, 2c+1) c2 = (g+8, 2c) c3 = (g+8, 2c+1)
// The k order inside a block is free as long as A and B agree: lane c holds
// one 4-byte qs word per row (bytes b0..b3, columns bc0..bc3 given below),
//   k-step 0: a0/a1 = (lo b0, lo b2)   a2/a3 = (lo b1, lo b3)
//   k-step 1: a0/a1 = (hi b0, hi b2)   a2/a3 = (hi b1, hi b3)
// and B is staged in exactly that order.
#include <cuda.h>

#include <mutex>

#include "qgemv_common.cuh"
#include "tc_ptx.cuh"

namespace qg {
namespace {

__device__ __forceinline__ void tma_load_2d_u8(void *dst, const CUtensorMap *tmap, int x_bytes, int row, uint64_t *bar) {
    tc::tma_load_2d(dst, tmap, x_bytes, row, bar);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Tensor maps of weight matrices, cached by (address, rows, row bytes, box
// bytes): the map is host data passed by value to the kernel.
struct WMapEntry {
    const void *ptr = nullptr;
    int64_t nrows = 0, rowbytes = 0;
    int box = 0;
    CUtensorMap map;
};
constexpr int kWMapCache = 32;
std::mutex g_wmap_mutex;
WMapEntry g_wmap[kWMapCache];
int g_wmap_next = 0;
EncodeTiledFn g_encode_w = nullptr;

qgemv_status weight_map(const void *W, int64_t nrows, int64_t rowbytes, int box_bytes, CUtensorMap *out) {
    std::lock_guard<std::mutex> lk(g_wmap_mutex);
    for (int i = 0; i < kWMapCache; ++i) {
        const WMapEntry &e = g_wmap[i];
        if (e.ptr == W && e.nrows == nrows && e.rowbytes == rowbytes && e.box == box_bytes) {
            *out = e.map;
            return QGEMV_OK;
        }
    }
    if (!g_encode_w) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
            set_last_error("cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(e));
            return QGEMV_ERR_CUDA;
        }
        g_encode_w = reinterpret_cast<EncodeTiledFn>(fn);
    }
    WMapEntry &e = g_wmap[g_wmap_next];
    g_wmap_next = (g_wmap_next + 1) % kWMapCache;
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(rowbytes), static_cast<cuuint64_t>(nrows)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(rowbytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_bytes), 16u};
    const cuuint32_t estride[2] = {1, 1};
    CUresult r = g_encode_w(&e.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(W), gdim, gstride, box,
                            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        e.ptr = nullptr;
        set_last_error("cuTensorMapEncodeTiled(weights) failed (%d)", static_cast<int>(r));
        return QGEMV_ERR_CUDA;
    }
    e.ptr = W;
    e.nrows = nrows;
    e.rowbytes = rowbytes;
    e.box = box_bytes;
    *out = e.map;
    return QGEMV_OK;
}

constexpr int kTcWarps = 16;
constexpr int kCB = 8;                 // blocks per unit (per row copy)
constexpr int kTile = 16;              // rows per MMA tile
constexpr int kMaxTcStages = 8;

struct TcParams {
    const uint8_t *W;
    const float *x;
    float *y;
    unsigned *err;
    int nrows, ncols, nb, batch;
    int cs;              // cluster size (CTAs splitting the columns)
    int nclusters;
    int rows_lo, extra;  // balanced rows per cluster
    int nbs;             // blocks per CTA column slice
    int stages;
    int max_tiles;       // tiles of the largest cluster row range
};

template <int F> struct TcFmt;
template <> struct TcFmt<FMT_Q4_0> { static constexpr int BB = 18; static constexpr float kOff = 136.0f; };  // 128 + 8
template <> struct TcFmt<FMT_Q4_1> { static constexpr int BB = 20; static constexpr float kOff = 128.0f; };

// Shared-memory layout of one CTA.
struct TcLayout {
    size_t xfh, xfl, xcorr, xsum, xmax, part, ypart, bars, ring, total;
};

__host__ __device__ inline TcLayout tc_layout(int F, int nbs, int batch, int stages, int max_tiles) {
    const int BB = block_bytes(F);
    TcLayout L;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o += (bytes + 127) & ~size_t(127); return at; };
    L.xfh = take(size_t(nbs) * batch * 4 * 16);        // hi fragments: [block][n][c] x 16 B
    // lo fragments (bf16 mode only: Q4_0 runs the fp16 mode with one part of x)
    L.xfl = take(F == FMT_Q4_0 ? 0 : size_t(nbs) * batch * 4 * 16);
    L.xcorr = take(size_t(nbs) * batch * 16);          // correction B fragments (lanes c == 0, 1)
    L.xsum = take(size_t(nbs) * batch * 4);            // fp32 block sums of x (Q4_1)
    L.xmax = take(8 * 4);                              // max |x| per batch column (fp16 mode)
    L.part = take(size_t(kTcWarps + max_tiles) * kTile * 8 * 4);
    L.ypart = take(size_t(max_tiles) * kTile * batch * 4);
    L.bars = take(size_t(kTcWarps) * stages * 8);
    L.ring = take(size_t(kTcWarps) * stages * kTile * kCB * BB);
    L.total = o;
    return L;
}

// (a & MASK) | c, one three-input logic instruction.
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
    return d;
}

__device__ __forceinline__ void mma_f16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float f16lo(uint32_t u) { return __half2float(__ushort_as_half(static_cast<unsigned short>(u & 0xffffu))); }
__device__ __forceinline__ float f16hi(uint32_t u) { return __half2float(__ushort_as_half(static_cast<unsigned short>(u >> 16))); }

// 2^e, with e the power of two that brings the largest |x| of a column into
// (2^9, 2^10] (0 if the column is zero or not finite).
__device__ __forceinline__ int x_exponent(float m) {
    if (!(m > 0.0f) || !isfinite(m)) return 0;
    int E;
    frexpf(m, &E);
    return 10 - E;
}

__device__ __forceinline__ void mma_bf16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint16_t bf16_bits_rn(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// Columns (within the 32-column block) of the 4 qs bytes lane c holds.
// Aligned blocks (Q4_1, odd Q4_0 blocks): qs[4c .. 4c+3].  Even Q4_0 blocks
// (realigned from 4-byte words): c = 0 holds qs[0, 1, 14, 15], c = 1..3 hold
// qs[4c-2 .. 4c+1].
__host__ __device__ inline int byte_col(int parity_odd, int c, int j) {
    if (parity_odd) return 4 * c + j;
    if (c == 0) return j < 2 ? j : 12 + j;
    return 4 * c - 2 + j;
}

// Stage the B fragments of this CTA's column slice: for block b, batch n and
// lane-column c, eight x values in MMA order, as bf16 hi and lo parts; plus
// the correction fragment (3-part split of the block's sum of x) and, for
// Q4_1, the fp32 block sum.  Split in two so the x loads can be issued
// before the weight copies: XItem::load issues the 8 global loads of one
// (block, batch) item, XItem::store converts and writes its fragments.
template <int ODD>
__device__ __forceinline__ void make_frags(const float v[32], int c, uint4 &hi, uint4 &lo, float &sum) {
    // MMA order: (lo b0, lo b2), (lo b1, lo b3), (hi b0, hi b2), (hi b1, hi b3)
    const int col[8] = {byte_col(ODD, c, 0), byte_col(ODD, c, 2), byte_col(ODD, c, 1), byte_col(ODD, c, 3),
                        16 + byte_col(ODD, c, 0), 16 + byte_col(ODD, c, 2), 16 + byte_col(ODD, c, 1),
                        16 + byte_col(ODD, c, 3)};
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float a = v[col[2 * k]], b = v[col[2 * k + 1]];
        const uint16_t ah = bf16_bits_rn(a), bh = bf16_bits_rn(b);
        const uint16_t al = bf16_bits_rn(a - bf16_bits_to_f32(ah));
        const uint16_t bl2 = bf16_bits_rn(b - bf16_bits_to_f32(bh));
        hw[k] = uint32_t(ah) | (uint32_t(bh) << 16);
        lw[k] = uint32_t(al) | (uint32_t(bl2) << 16);
        sum += bf16_bits_to_f32(ah) + bf16_bits_to_f32(al);
        sum += bf16_bits_to_f32(bh) + bf16_bits_to_f32(bl2);
    }
    hi = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    lo = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

struct XItem {
    float4 q[8];
    int bl, n;
    bool valid;

    __device__ __forceinline__ void load(const TcParams &p, int kb0, int t) {
        valid = t < p.nbs * p.batch;
        if (!valid) return;
        bl = t / p.batch;
        n = t - bl * p.batch;
        const float4 *xr = reinterpret_cast<const float4 *>(p.x + size_t(n) * p.ncols + size_t(kb0 + bl) * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = __ldg(xr + i);
    }

    template <int F>
    __device__ __forceinline__ void store(const TcParams &p, int kb0, uint8_t *smem, const TcLayout &L) const {
        if (!valid) return;
        uint4 *xfh = reinterpret_cast<uint4 *>(smem + L.xfh);
        uint4 *xfl = reinterpret_cast<uint4 *>(smem + L.xfl);
        uint4 *xcorr = reinterpret_cast<uint4 *>(smem + L.xcorr);
        float *xsum = reinterpret_cast<float *>(smem + L.xsum);
        float v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[4 * i] = q[i].x; v[4 * i + 1] = q[i].y; v[4 * i + 2] = q[i].z; v[4 * i + 3] = q[i].w;
        }
        // Q4_0 pairs realign the even block's words; Q4_1 blocks are all aligned
        const bool odd = (F == FMT_Q4_1) || ((kb0 + bl) & 1);
        float sum = 0.0f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint4 hi, lo;
            if (odd) make_frags<1>(v, c, hi, lo, sum);
            else make_frags<0>(v, c, hi, lo, sum);
            xfh[(bl * p.batch + n) * 4 + c] = hi;
            xfl[(bl * p.batch + n) * 4 + c] = lo;
        }
        // correction operand: sum = s0 + s1 + s2 (three bf16 parts)
        const uint16_t s0 = bf16_bits_rn(sum);
        const float r1 = sum - bf16_bits_to_f32(s0);
        const uint16_t s1 = bf16_bits_rn(r1);
        const uint16_t s2 = bf16_bits_rn(r1 - bf16_bits_to_f32(s1));
        xcorr[bl * p.batch + n] = make_uint4(uint32_t(s0) | (uint32_t(s1) << 16), uint32_t(s2), 0u, 0u);
        if constexpr (F == FMT_Q4_1) {
            float s = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) s += v[i];
            xsum[bl * p.batch + n] = s;
        }
    }

    __device__ __forceinline__ float absmax() const {
        float m = 0.0f;
        if (!valid) return m;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            m = fmaxf(m, fmaxf(fmaxf(fabsf(q[i].x), fabsf(q[i].y)), fmaxf(fabsf(q[i].z), fabsf(q[i].w))));
        }
        return m;
    }

    // fp16 mode (Q4_0): one fp16 part of x * 2^e (x * 2^e / 16 in the
    // high-nibble k-slots), and the correction operand: the sums of the
    // low-slot and of the high-slot values just rounded, each as three fp16
    // parts (lanes c == 0 and c == 1 of the correction MMA).
    __device__ __forceinline__ void store16(const TcParams &p, int kb0, uint8_t *smem, const TcLayout &L,
                                            int e) const {
        if (!valid) return;
        uint4 *xfh = reinterpret_cast<uint4 *>(smem + L.xfh);
        uint4 *xcorr = reinterpret_cast<uint4 *>(smem + L.xcorr);
        float v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[4 * i] = ldexpf(q[i].x, e); v[4 * i + 1] = ldexpf(q[i].y, e);
            v[4 * i + 2] = ldexpf(q[i].z, e); v[4 * i + 3] = ldexpf(q[i].w, e);
        }
        const bool odd = (kb0 + bl) & 1;
        float slo = 0.0f, shi = 0.0f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t w4[4];
            if (odd) frag16<1>(v, c, w4);
            else frag16<0>(v, c, w4);
            slo += f16lo(w4[0]) + f16hi(w4[0]) + f16lo(w4[1]) + f16hi(w4[1]);
            shi += f16lo(w4[2]) + f16hi(w4[2]) + f16lo(w4[3]) + f16hi(w4[3]);
            xfh[(bl * p.batch + n) * 4 + c] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        uint32_t cl[2], ch[2];
        split3_f16(slo, cl);
        split3_f16(shi, ch);
        xcorr[bl * p.batch + n] = make_uint4(cl[0], cl[1], ch[0], ch[1]);
    }

    template <int ODD>
    __device__ __forceinline__ static void frag16(const float v[32], int c, uint32_t w4[4]) {
        const int b0 = byte_col(ODD, c, 0), b1 = byte_col(ODD, c, 1);
        const int b2 = byte_col(ODD, c, 2), b3 = byte_col(ODD, c, 3);
        w4[0] = f16x2_rn(v[b0], v[b2]);                                    // k-step 0: (lo b0, lo b2)
        w4[1] = f16x2_rn(v[b1], v[b3]);                                    //           (lo b1, lo b3)
        w4[2] = f16x2_rn(v[16 + b0] * 0.0625f, v[16 + b2] * 0.0625f);     // k-step 1: high nibbles / 16
        w4[3] = f16x2_rn(v[16 + b1] * 0.0625f, v[16 + b3] * 0.0625f);
    }

    // s = a + b + c in three fp16 parts, packed as {a, b} and {c, 0}.
    __device__ __forceinline__ static void split3_f16(float s, uint32_t out[2]) {
        const float a = __half2float(__float2half_rn(s));
        const float r = s - a;
        const float b = __half2float(__float2half_rn(r));
        const float c = r - b;
        out[0] = f16x2_rn(a, b);
        out[1] = f16x2_rn(c, 0.0f);
    }
};

// H16 = true: fp16 operands with one part of x (Q4_0 only; see above).
template <int F, bool H16>
__global__ void __launch_bounds__(kTcWarps * 32, 1)
gemv_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const TcParams p) {
    constexpr int BB = TcFmt<F>::BB;
    constexpr int kRowBytes = kCB * BB;                 // bytes of one row in a unit
    constexpr int kSlotBytes = kTile * kRowBytes;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;

    uint32_t rank = 0;
    if (p.cs > 1) asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const int cl = blockIdx.x / p.cs;
    const int rc0 = cl * p.rows_lo + min(cl, p.extra);
    const int nrc = p.rows_lo + (cl < p.extra ? 1 : 0);
    const int ntiles = (nrc + kTile - 1) / kTile;
    const int kb0 = static_cast<int>(rank) * p.nbs;     // first block of this CTA's column slice
    const int nch = p.nbs / kCB;                        // units per tile
    const int S = p.stages;

    const TcLayout L = tc_layout(F, p.nbs, p.batch, S, p.max_tiles);
    uint64_t *wbar = reinterpret_cast<uint64_t *>(smem + L.bars) + wid * S;
    uint8_t *wring = smem + L.ring + size_t(wid) * S * kSlotBytes;
    float *part = reinterpret_cast<float *>(smem + L.part);
    float *ypart = reinterpret_cast<float *>(smem + L.ypart);

    const int units = ntiles * nch;
    const int u_begin = (units * wid) / kTcWarps;
    const int u_end = (units * (wid + 1)) / kTcWarps;
    const int my_units = u_end - u_begin;

    // copy cursor (tile, chunk) of the next unit: one 2-D TMA of 16 rows x
    // kRowBytes (rows past the matrix read as zeros)
    int f_t = u_begin / nch;
    int f_k = u_begin - f_t * nch;
    auto issue_next = [&](int slot) {
        if (lane == 0) {
            mbar_arrive_expect_tx(&wbar[slot], static_cast<uint32_t>(kSlotBytes));
            tma_load_2d_u8(wring + size_t(slot) * kSlotBytes, &tmap_w, (kb0 + f_k * kCB) * BB,
                           rc0 + f_t * kTile, &wbar[slot]);
        }
        if (++f_k == nch) { f_k = 0; ++f_t; }
    };

    // x loads of the first round go out before the weight copies
    int *xmax = reinterpret_cast<int *>(smem + L.xmax);
    if (H16 && threadIdx.x < 8) xmax[threadIdx.x] = 0;
    XItem xi;
    xi.load(p, kb0, threadIdx.x);
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&wbar[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    {
        const int n0 = min(S, my_units);
        for (int i = 0; i < n0; ++i) issue_next(i);
    }
    if constexpr (H16) {
        // per batch column, the largest |x| of this CTA's slice (non-negative
        // floats order like their bit patterns)
        __syncthreads();
        // one shared atomic per (warp, column): reduce over the lanes first
        // (for batch b the lanes of a warp cover columns t % b)
        {
            float m = xi.absmax();
            const int rounds = (p.nbs * p.batch + blockDim.x - 1) / blockDim.x;
            for (int r = 1; r < rounds; ++r) {
                XItem xr;
                xr.load(p, kb0, threadIdx.x + r * blockDim.x);
                if (xr.valid && xr.n == xi.n) m = fmaxf(m, xr.absmax());
                else if (xr.valid) atomicMax(&xmax[xr.n], __float_as_int(xr.absmax()));
            }
            // lanes with equal t % batch share a column; batch <= 8 divides 32 only
            // for 1, 2, 4, 8, so reduce per column with a masked max
            for (int n = 0; n < p.batch; ++n) {
                const float v = (xi.valid && xi.n == n) ? m : 0.0f;
                const unsigned wm = __reduce_max_sync(0xffffffffu, __float_as_uint(v));
                if (lane == 0 && wm != 0u) atomicMax(&xmax[n], static_cast<int>(wm));
            }
        }
        __syncthreads();
        if (xi.valid) xi.store16(p, kb0, smem, L, x_exponent(__int_as_float(xmax[xi.n])));
        for (int t0 = threadIdx.x + blockDim.x; t0 < p.nbs * p.batch; t0 += blockDim.x) {
            XItem xr;
            xr.load(p, kb0, t0);
            xr.store16(p, kb0, smem, L, x_exponent(__int_as_float(xmax[xr.n])));
        }
    } else {
        xi.store<F>(p, kb0, smem, L);
        for (int t0 = threadIdx.x + blockDim.x; t0 < p.nbs * p.batch; t0 += blockDim.x) {
            XItem xr;
            xr.load(p, kb0, t0);
            xr.store<F>(p, kb0, smem, L);
        }
    }
    {
        const int np = (kTcWarps + p.max_tiles) * kTile * 8;
        for (int i = threadIdx.x; i < np; i += blockDim.x) part[i] = 0.0f;
    }
    __syncthreads();

    const uint4 *xfh = reinterpret_cast<const uint4 *>(smem + L.xfh) + g * 4 + c;   // this lane's fragments
    const uint4 *xfl = reinterpret_cast<const uint4 *>(smem + L.xfl) + g * 4 + c;
    const uint4 *xcorr = reinterpret_cast<const uint4 *>(smem + L.xcorr) + g;
    const float *xsum = reinterpret_cast<const float *>(smem + L.xsum);
    const int bstride = p.batch * 4;                    // uint4 per block in xfh / xfl

    uint32_t magic = H16 ? 0x64006400u : 0x43004300u;   // fp16 (1024, 1024) / bf16 (128, 128)
    asm volatile("" : "+r"(magic));
    uint32_t acorr[4] = {0u, 0u, 0u, 0u};               // correction A fragment
    if constexpr (H16) {
        // lane c = 0: -(1024 + 8) on the low-slot sums; c = 1: -(1024 + 128) on
        // the high-slot sums (which hold x / 16)
        if (c < 2) {
            const uint32_t m = __half_as_ushort(__float2half_rn(c == 0 ? -1032.0f : -1152.0f));
            acorr[0] = m | (m << 16);
            acorr[1] = acorr[0];
            acorr[2] = m;
            acorr[3] = m;
        }
    } else if (c == 0) {
        const uint32_t m = bf16_bits_rn(-TcFmt<F>::kOff);
        acorr[0] = m | (m << 16);
        acorr[1] = acorr[0];
        acorr[2] = m;
        acorr[3] = m;
    }
    const bool nvalid = g < p.batch;                    // this lane's B column is a real batch entry

    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    bool ok = true;
    int i = 0, slot = 0;
    uint32_t phase = 0;
    int t = u_begin / nch;
    int kc = u_begin - t * nch;
    for (; i < my_units; ++i) {
        const bool got = mbar_wait_bounded(&wbar[slot], phase, p.err);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        const uint8_t *sl = wring + size_t(slot) * kSlotBytes;
        const uint32_t *r0w = reinterpret_cast<const uint32_t *>(sl + g * kRowBytes);        // row g
        const uint32_t *r1w = reinterpret_cast<const uint32_t *>(sl + (g + 8) * kRowBytes);  // row g + 8
        const int blk0 = kc * kCB;
#pragma unroll
        for (int pr = 0; pr < kCB / 2; ++pr) {
            // ---- qs words of the pair for rows g, g+8 and their scales
            uint32_t we[2], wo[2];
            float de[2], dd[2], me[2], md[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t *s = (h ? r1w : r0w) + pr * (2 * BB / 4);
                if constexpr (F == FMT_Q4_0) {
                    const uint32_t W0 = s[0], W4 = s[4];
                    we[h] = __byte_perm(s[c], W4, c == 0 ? 0x5432 : 0x3210);
                    wo[h] = s[5 + c];
                    de[h] = fp16_bits_to_f32(W0);
                    dd[h] = fp16_bits_to_f32(W4 >> 16);
                } else {
                    const uint32_t W0 = s[0], W5 = s[5];
                    we[h] = s[1 + c];
                    wo[h] = s[6 + c];
                    de[h] = fp16_bits_to_f32(W0);
                    me[h] = fp16_bits_to_f32(W0 >> 16);
                    dd[h] = fp16_bits_to_f32(W5);
                    md[h] = fp16_bits_to_f32(W5 >> 16);
                }
            }
            // ---- B fragments of the two blocks
            const int be = blk0 + 2 * pr;
            float ce[4] = {0.0f, 0.0f, 0.0f, 0.0f}, co[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if constexpr (H16) {
                uint4 bhe = make_uint4(0, 0, 0, 0), bho = bhe, bce = bhe, bco = bhe;
                if (nvalid) {
                    bhe = xfh[be * bstride];
                    bho = xfh[(be + 1) * bstride];
                    if (c < 2) {
                        bce = xcorr[be * p.batch];
                        bco = xcorr[(be + 1) * p.batch];
                    }
                }
                const uint32_t bc0e = c ? bce.z : bce.x, bc1e = c ? bce.w : bce.y;
                const uint32_t bc0o = c ? bco.z : bco.x, bc1o = c ? bco.w : bco.y;
                uint32_t ae[4], ao[4];
                const uint32_t we8 = we[0] >> 8, we8b = we[1] >> 8, wo8 = wo[0] >> 8, wo8b = wo[1] >> 8;
                ae[0] = and_or<0x000f000fu>(we[0], magic);      // k-step 0: low nibbles, 1024 + q
                ae[1] = and_or<0x000f000fu>(we[1], magic);
                ae[2] = and_or<0x000f000fu>(we8, magic);
                ae[3] = and_or<0x000f000fu>(we8b, magic);
                ao[0] = and_or<0x000f000fu>(wo[0], magic);
                ao[1] = and_or<0x000f000fu>(wo[1], magic);
                ao[2] = and_or<0x000f000fu>(wo8, magic);
                ao[3] = and_or<0x000f000fu>(wo8b, magic);
                mma_f16(ce, ae, bhe.x, bhe.y);
                mma_f16(co, ao, bho.x, bho.y);
                ae[0] = and_or<0x00f000f0u>(we[0], magic);      // k-step 1: high nibbles, 1024 + 16 q
                ae[1] = and_or<0x00f000f0u>(we[1], magic);
                ae[2] = and_or<0x00f000f0u>(we8, magic);
                ae[3] = and_or<0x00f000f0u>(we8b, magic);
                ao[0] = and_or<0x00f000f0u>(wo[0], magic);
                ao[1] = and_or<0x00f000f0u>(wo[1], magic);
                ao[2] = and_or<0x00f000f0u>(wo8, magic);
                ao[3] = and_or<0x00f000f0u>(wo8b, magic);
                mma_f16(ce, ae, bhe.z, bhe.w);
                mma_f16(co, ao, bho.z, bho.w);
                mma_f16(ce, acorr, bc0e, bc1e);                  // offset correction
                mma_f16(co, acorr, bc0o, bc1o);
            } else {
            uint4 bhe = make_uint4(0, 0, 0, 0), ble = bhe, bho = bhe, blo = bhe;
            uint4 bce = make_uint4(0, 0, 0, 0), bco = bce;
            if (nvalid) {
                bhe = xfh[be * bstride];
                ble = xfl[be * bstride];
                bho = xfh[(be + 1) * bstride];
                blo = xfl[(be + 1) * bstride];
                if (c == 0) {
                    bce = xcorr[be * p.batch];
                    bco = xcorr[(be + 1) * p.batch];
                }
            }
            // ---- two independent MMA chains (even block, odd block)
            uint32_t ae[4], ao[4];
            ae[0] = and_or<0x000f000fu>(we[0], magic);          // k-step 0: low nibbles
            ae[1] = and_or<0x000f000fu>(we[1], magic);
            ae[2] = and_or<0x000f000fu>(we[0] >> 8, magic);
            ae[3] = and_or<0x000f000fu>(we[1] >> 8, magic);
            ao[0] = and_or<0x000f000fu>(wo[0], magic);
            ao[1] = and_or<0x000f000fu>(wo[1], magic);
            ao[2] = and_or<0x000f000fu>(wo[0] >> 8, magic);
            ao[3] = and_or<0x000f000fu>(wo[1] >> 8, magic);
            mma_bf16(ce, ae, bhe.x, bhe.y);
            mma_bf16(co, ao, bho.x, bho.y);
            mma_bf16(ce, ae, ble.x, ble.y);
            mma_bf16(co, ao, blo.x, blo.y);
            ae[0] = and_or<0x000f000fu>(we[0] >> 4, magic);     // k-step 1: high nibbles
            ae[1] = and_or<0x000f000fu>(we[1] >> 4, magic);
            ae[2] = and_or<0x000f000fu>(we[0] >> 12, magic);
            ae[3] = and_or<0x000f000fu>(we[1] >> 12, magic);
            ao[0] = and_or<0x000f000fu>(wo[0] >> 4, magic);
            ao[1] = and_or<0x000f000fu>(wo[1] >> 4, magic);
            ao[2] = and_or<0x000f000fu>(wo[0] >> 12, magic);
            ao[3] = and_or<0x000f000fu>(wo[1] >> 12, magic);
            mma_bf16(ce, ae, bhe.z, bhe.w);
            mma_bf16(co, ao, bho.z, bho.w);
            mma_bf16(ce, ae, ble.z, ble.w);
            mma_bf16(co, ao, blo.z, blo.w);
            mma_bf16(ce, acorr, bce.x, bce.y);                  // offset correction
            mma_bf16(co, acorr, bco.x, bco.y);
            }
            acc[0] = fmaf(de[0], ce[0], acc[0]);
            acc[1] = fmaf(de[0], ce[1], acc[1]);
            acc[2] = fmaf(de[1], ce[2], acc[2]);
            acc[3] = fmaf(de[1], ce[3], acc[3]);
            acc[0] = fmaf(dd[0], co[0], acc[0]);
            acc[1] = fmaf(dd[0], co[1], acc[1]);
            acc[2] = fmaf(dd[1], co[2], acc[2]);
            acc[3] = fmaf(dd[1], co[3], acc[3]);
            if constexpr (F == FMT_Q4_1) {
                const int n0 = 2 * c, n1 = 2 * c + 1;
                const float se0 = n0 < p.batch ? xsum[be * p.batch + n0] : 0.0f;
                const float se1 = n1 < p.batch ? xsum[be * p.batch + n1] : 0.0f;
                const float so0 = n0 < p.batch ? xsum[(be + 1) * p.batch + n0] : 0.0f;
                const float so1 = n1 < p.batch ? xsum[(be + 1) * p.batch + n1] : 0.0f;
                acc[0] = fmaf(me[0], se0, fmaf(md[0], so0, acc[0]));
                acc[1] = fmaf(me[0], se1, fmaf(md[0], so1, acc[1]));
                acc[2] = fmaf(me[1], se0, fmaf(md[1], so0, acc[2]));
                acc[3] = fmaf(me[1], se1, fmaf(md[1], so1, acc[3]));
            }
        }
        __syncwarp();
        if (i + S < my_units) {
            if (lane == 0) fence_proxy_async_smem();
            issue_next(slot);
        }
        // end of a tile (or of this warp's run): park the partial C fragment
        if (kc == nch - 1 || i == my_units - 1) {
            float *pp = part + size_t(wid + t) * kTile * 8;
            pp[g * 8 + 2 * c] = acc[0];
            pp[g * 8 + 2 * c + 1] = acc[1];
            pp[(g + 8) * 8 + 2 * c] = acc[2];
            pp[(g + 8) * 8 + 2 * c + 1] = acc[3];
            acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
        }
        if (++slot == S) { slot = 0; phase ^= 1u; }
        if (++kc == nch) { kc = 0; ++t; }
    }
    if (!ok) {
        for (int j = i; j < my_units && j < i + S; ++j) {
            mbar_wait_bounded(&wbar[slot], phase, p.err);
            if (++slot == S) { slot = 0; phase ^= 1u; }
        }
    }
    __syncthreads();

    // ---- per tile, fixed-order sum over the warps whose unit range touches it
    for (int e = threadIdx.x; e < ntiles * kTile * p.batch; e += blockDim.x) {
        const int tt = e / (kTile * p.batch);
        const int rr = (e / p.batch) % kTile;
        const int n = e % p.batch;
        float s = 0.0f;
        // warps whose unit range [units*w/16, units*(w+1)/16) touches tile tt
        // (units < 2^26, so 32-bit products suffice)
        for (int w = 0; w < kTcWarps; ++w) {
            const int ub = (units * w) / kTcWarps;
            const int ue = (units * (w + 1)) / kTcWarps;
            if (ue > ub && ub < (tt + 1) * nch && ue > tt * nch) {
                s += part[(size_t(w + tt) * kTile + rr) * 8 + n];
            }
        }
        if constexpr (H16) s = ldexpf(s, -x_exponent(__int_as_float(xmax[n])));   // undo the x scaling (exact)
        ypart[(tt * kTile + rr) * p.batch + n] = s;
    }

    if (p.cs == 1) {
        __syncthreads();
        for (int e = threadIdx.x; e < nrc * p.batch; e += blockDim.x) {
            const int r = e / p.batch, n = e - r * p.batch;
            p.y[static_cast<int64_t>(n) * p.nrows + rc0 + r] = ypart[r * p.batch + n];
        }
        return;
    }
    // ---- cluster: CTA j sums its share of the rows over all ranks, in rank order
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    const int rpc = (nrc + p.cs - 1) / p.cs;
    const int rb = static_cast<int>(rank) * rpc;
    const int re = min(nrc, rb + rpc);
    const uint32_t ypart_s = smem_u32(ypart);
    for (int e = threadIdx.x; e < (re - rb) * p.batch; e += blockDim.x) {
        const int r = rb + e / p.batch, n = e % p.batch;
        const uint32_t off = static_cast<uint32_t>((r * p.batch + n) * 4);
        float s = 0.0f;
        for (int q = 0; q < p.cs; ++q) {
            uint32_t remote;
            float v;
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(ypart_s + off), "r"(q));
            asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
            s += v;
        }
        p.y[static_cast<int64_t>(n) * p.nrows + rc0 + r] = s;
    }
    // nobody leaves while a peer may still read its shared memory
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int F>
qgemv_status launch_tc_fmt(const void *W, const float *x, float *y, int64_t nrows, int64_t ncols, int batch,
                           cudaStream_t s, const DevInfo &di, unsigned *err, bool *taken) {
    *taken = false;
    const int nb = static_cast<int>(ncols / 32);
    if (nb % kCB != 0 || nrows < kTile) return QGEMV_OK;
    const size_t budget = di.smem_optin;
    // smallest cluster size whose column slice leaves room for >= 2 ring slots per warp
    for (int cs : {1, 2, 4, 8}) {
        if (nb % (cs * kCB) != 0) continue;
        if (di.sm_count % cs != 0) continue;
        const int nclusters = di.sm_count / cs;
        if (nrows < static_cast<int64_t>(nclusters)) continue;
        const int rows_hi = static_cast<int>((nrows + nclusters - 1) / nclusters);
        const int max_tiles = (rows_hi + kTile - 1) / kTile;
        const int nbs = nb / cs;
        const TcLayout L0 = tc_layout(F, nbs, batch, 0, max_tiles);
        if (L0.total >= budget) continue;
        const size_t per_stage = size_t(kTcWarps) * (kTile * kCB * block_bytes(F) + 8);
        int stages = static_cast<int>((budget - L0.total - 256) / per_stage);
        if (stages > kMaxTcStages) stages = kMaxTcStages;
        if (stages < 2) continue;
        const TcLayout L = tc_layout(F, nbs, batch, stages, max_tiles);
        if (L.total > budget) continue;

        static bool attr_set[64] = {false};
        int dev = 0;
        cudaGetDevice(&dev);
        if (dev >= 0 && dev < 64 && !attr_set[dev]) {
            cudaError_t e = cudaFuncSetAttribute(gemv_tc_kernel<F, (F == FMT_Q4_0)>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(budget));
            if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_tc_kernel<F, (F == FMT_Q4_0)>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) {
                set_last_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
                return QGEMV_ERR_CUDA;
            }
            attr_set[dev] = true;
        }
        // clusters that can be resident at once (a cluster must fit in one GPC)
        cudaLaunchConfig_t qcfg = {};
        qcfg.gridDim = dim3(static_cast<unsigned>(di.sm_count / cs * cs));
        qcfg.blockDim = dim3(kTcWarps * 32);
        qcfg.dynamicSmemBytes = L.total;
        cudaLaunchAttribute qattr[1];
        qattr[0].id = cudaLaunchAttributeClusterDimension;
        qattr[0].val.clusterDim.x = static_cast<unsigned>(cs);
        qattr[0].val.clusterDim.y = 1;
        qattr[0].val.clusterDim.z = 1;
        qcfg.attrs = qattr;
        qcfg.numAttrs = 1;
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, gemv_tc_kernel<F, (F == FMT_Q4_0)>, &qcfg) != cudaSuccess || active < 1) {
            cudaGetLastError();
            continue;
        }
        const int ncl = min(active, di.sm_count / cs);
        if (nrows < static_cast<int64_t>(ncl) * 1) continue;
        const int rows_hi2 = static_cast<int>((nrows + ncl - 1) / ncl);
        const int max_tiles2 = (rows_hi2 + kTile - 1) / kTile;
        const TcLayout L2 = tc_layout(F, nbs, batch, stages, max_tiles2);
        if (L2.total > budget) continue;

        TcParams p;
        p.W = static_cast<const uint8_t *>(W);
        p.x = x;
        p.y = y;
        p.err = err;
        p.nrows = static_cast<int>(nrows);
        p.ncols = static_cast<int>(ncols);
        p.nb = nb;
        p.batch = batch;
        p.cs = cs;
        p.nclusters = ncl;
        p.rows_lo = static_cast<int>(nrows / ncl);
        p.extra = static_cast<int>(nrows % ncl);
        p.nbs = nbs;
        p.stages = stages;
        p.max_tiles = max_tiles2;

        CUtensorMap wmap;
        qgemv_status ms = weight_map(W, nrows, static_cast<int64_t>(nb) * block_bytes(F), kCB * block_bytes(F), &wmap);
        if (ms != QGEMV_OK) return ms;

        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(ncl * cs));
        cfg.blockDim = dim3(kTcWarps * 32);
        cfg.dynamicSmemBytes = L2.total;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        *taken = true;
        cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_tc_kernel<F, (F == FMT_Q4_0)>, wmap, p);
        if (e != cudaSuccess) {
            set_last_error("qgemv(tensor core) launch: %s", cudaGetErrorString(e));
            return QGEMV_ERR_LAUNCH;
        }
        return check_launch("qgemv(tensor core)");
    }
    return QGEMV_OK;
}

}  // namespace

qgemv_status launch_gemv_tc(int fmt, const void *W, const float *x, float *y, int64_t nrows, int64_t ncols,
                            int batch, cudaStream_t s, const DevInfo &di, unsigned *err, bool *taken) {
    switch (fmt) {
    case FMT_Q4_0: return launch_tc_fmt<FMT_Q4_0>(W, x, y, nrows, ncols, batch, s, di, err, taken);
    case FMT_Q4_1: return launch_tc_fmt<FMT_Q4_1>(W, x, y, nrows, ncols, batch, s, di, err, taken);
    default:
        *taken = false;
        return QGEMV_OK;
    }
}

}  // namespace qg
