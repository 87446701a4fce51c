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
// contiguous run of units and streams them with 1-D bulk async copies (one
// per row) into a private ring of mbarrier-completed slots.  Per-warp tile
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
#include "qgemv_common.cuh"

namespace qg {
namespace {

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
    size_t xfh, xfl, xcorr, xsum, part, ypart, bars, ring, total;
};

__host__ __device__ inline TcLayout tc_layout(int F, int nbs, int batch, int stages, int max_tiles) {
    const int BB = block_bytes(F);
    TcLayout L;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o += (bytes + 127) & ~size_t(127); return at; };
    L.xfh = take(size_t(nbs) * batch * 4 * 16);        // hi fragments: [block][n][c] x 16 B
    L.xfl = take(size_t(nbs) * batch * 4 * 16);        // lo fragments
    L.xcorr = take(size_t(nbs) * batch * 8);           // correction B fragment (lane c == 0)
    L.xsum = take(size_t(nbs) * batch * 4);            // fp32 block sums of x (Q4_1)
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
// Q4_1, the fp32 block sum.
template <int F>
__device__ void stage_x_frags(const TcParams &p, int kb0, uint8_t *smem, const TcLayout &L) {
    uint4 *xfh = reinterpret_cast<uint4 *>(smem + L.xfh);
    uint4 *xfl = reinterpret_cast<uint4 *>(smem + L.xfl);
    uint2 *xcorr = reinterpret_cast<uint2 *>(smem + L.xcorr);
    float *xsum = reinterpret_cast<float *>(smem + L.xsum);
    for (int t = threadIdx.x; t < p.nbs * p.batch; t += blockDim.x) {
        const int bl = t / p.batch, n = t - bl * p.batch;
        const int gb = kb0 + bl;                        // global block index
        const float *xr = p.x + size_t(n) * p.ncols + size_t(gb) * 32;
        float v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 q = __ldg(reinterpret_cast<const float4 *>(xr) + i);
            v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
        }
        // Q4_0 pairs realign the even block's words; Q4_1 blocks are all aligned
        const int odd = (F == FMT_Q4_1) ? 1 : (gb & 1);
        float sum = 0.0f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            // MMA order: (lo b0, lo b2), (lo b1, lo b3), (hi b0, hi b2), (hi b1, hi b3)
            const int col[8] = {byte_col(odd, c, 0), byte_col(odd, c, 2), byte_col(odd, c, 1), byte_col(odd, c, 3),
                                16 + byte_col(odd, c, 0), 16 + byte_col(odd, c, 2), 16 + byte_col(odd, c, 1),
                                16 + byte_col(odd, c, 3)};
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
            xfh[(bl * p.batch + n) * 4 + c] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            xfl[(bl * p.batch + n) * 4 + c] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        // correction operand: sum = s0 + s1 + s2 (three bf16 parts)
        const uint16_t s0 = bf16_bits_rn(sum);
        const float r1 = sum - bf16_bits_to_f32(s0);
        const uint16_t s1 = bf16_bits_rn(r1);
        const uint16_t s2 = bf16_bits_rn(r1 - bf16_bits_to_f32(s1));
        xcorr[bl * p.batch + n] = make_uint2(uint32_t(s0) | (uint32_t(s1) << 16), uint32_t(s2));
        if constexpr (F == FMT_Q4_1) {
            float s = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) s += v[i];
            xsum[bl * p.batch + n] = s;
        }
    }
}

template <int F>
__global__ void __launch_bounds__(kTcWarps * 32, 1)
gemv_tc_kernel(const TcParams p) {
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
    const int u_begin = static_cast<int>((static_cast<int64_t>(units) * wid) / kTcWarps);
    const int u_end = static_cast<int>((static_cast<int64_t>(units) * (wid + 1)) / kTcWarps);
    const int my_units = u_end - u_begin;
    const int64_t rowbytes = static_cast<int64_t>(p.nb) * BB;

    // copy cursor (tile, chunk) of the next unit to issue; lanes 0..15 each copy one row
    int f_t = u_begin / nch;
    int f_k = u_begin - f_t * nch;
    auto issue_next = [&](int slot) {
        const int row = f_t * kTile + lane;             // cluster-local row of this lane
        const int valid = min(kTile, nrc - f_t * kTile);
        if (lane == 0) mbar_arrive_expect_tx(&wbar[slot], static_cast<uint32_t>(valid * kRowBytes));
        __syncwarp();
        if (lane < valid) {
            const uint8_t *src = p.W + static_cast<int64_t>(rc0 + row) * rowbytes +
                                 static_cast<int64_t>(kb0 + f_k * kCB) * BB;
            bulk_g2s(wring + size_t(slot) * kSlotBytes + lane * kRowBytes, src, kRowBytes, &wbar[slot]);
        }
        if (++f_k == nch) { f_k = 0; ++f_t; }
    };

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&wbar[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    {
        const int n0 = min(S, my_units);
        for (int i = 0; i < n0; ++i) issue_next(i);
    }

    stage_x_frags<F>(p, kb0, smem, L);
    {
        const int np = (kTcWarps + p.max_tiles) * kTile * 8;
        for (int i = threadIdx.x; i < np; i += blockDim.x) part[i] = 0.0f;
    }
    __syncthreads();

    const uint4 *xfh = reinterpret_cast<const uint4 *>(smem + L.xfh);
    const uint4 *xfl = reinterpret_cast<const uint4 *>(smem + L.xfl);
    const uint2 *xcorr = reinterpret_cast<const uint2 *>(smem + L.xcorr);
    const float *xsum = reinterpret_cast<const float *>(smem + L.xsum);

    // opaque constants (kept in registers)
    uint32_t magic = 0x43004300u;                       // bf16 pair (128, 128)
    asm volatile("" : "+r"(magic));
    // correction A fragment: -(128 + OFF) on k-slots 0, 1 and 8 (lane c == 0)
    uint32_t acorr_lo = 0, acorr_hi = 0;
    if (c == 0) {
        const uint32_t m = bf16_bits_rn(-TcFmt<F>::kOff);
        acorr_lo = m | (m << 16);
        acorr_hi = m;
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
        const uint8_t *r0p = sl + g * kRowBytes;         // row g of the tile
        const uint8_t *r1p = sl + (g + 8) * kRowBytes;   // row g + 8
#pragma unroll
        for (int pr = 0; pr < kCB / 2; ++pr) {
            const int bl = kc * kCB + 2 * pr;            // block (within the CTA slice) of the even block
            // ---- words of the pair for rows g and g+8
            uint32_t we[2], wo[2];
            float de[2], dd[2], me[2], md[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t *s = reinterpret_cast<const uint32_t *>((h ? r1p : r0p) + 2 * pr * BB);
                if constexpr (F == FMT_Q4_0) {
                    const uint32_t W0 = s[0], W4 = s[4];
                    const uint32_t Wc = s[c];
                    // even block word of lane c: c = 0 -> qs[0,1,14,15], else the aligned word
                    we[h] = __byte_perm(Wc, W4, c == 0 ? 0x5432 : 0x3210);
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
#pragma unroll
            for (int ob = 0; ob < 2; ++ob) {             // even block, then odd block
                const int blk = bl + ob;
                const uint32_t E0 = ob ? wo[0] : we[0];  // row g
                const uint32_t E1 = ob ? wo[1] : we[1];  // row g + 8
                uint4 bh = make_uint4(0, 0, 0, 0), blo = make_uint4(0, 0, 0, 0);
                uint2 bc = make_uint2(0, 0);
                if (nvalid) {
                    bh = xfh[(blk * p.batch + g) * 4 + c];
                    blo = xfl[(blk * p.batch + g) * 4 + c];
                    if (c == 0) bc = xcorr[blk * p.batch + g];
                }
                float cb[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                uint32_t a[4];
                // k-step 0: low nibbles
                a[0] = and_or<0x000f000fu>(E0, magic);
                a[1] = and_or<0x000f000fu>(E1, magic);
                a[2] = and_or<0x000f000fu>(E0 >> 8, magic);
                a[3] = and_or<0x000f000fu>(E1 >> 8, magic);
                mma_bf16(cb, a, bh.x, bh.y);
                mma_bf16(cb, a, blo.x, blo.y);
                // k-step 1: high nibbles
                a[0] = and_or<0x000f000fu>(E0 >> 4, magic);
                a[1] = and_or<0x000f000fu>(E1 >> 4, magic);
                a[2] = and_or<0x000f000fu>(E0 >> 12, magic);
                a[3] = and_or<0x000f000fu>(E1 >> 12, magic);
                mma_bf16(cb, a, bh.z, bh.w);
                mma_bf16(cb, a, blo.z, blo.w);
                // offset correction
                a[0] = acorr_lo; a[1] = acorr_lo; a[2] = acorr_hi; a[3] = acorr_hi;
                mma_bf16(cb, a, bc.x, bc.y);
                const float d0 = ob ? dd[0] : de[0];
                const float d1 = ob ? dd[1] : de[1];
                acc[0] = fmaf(d0, cb[0], acc[0]);
                acc[1] = fmaf(d0, cb[1], acc[1]);
                acc[2] = fmaf(d1, cb[2], acc[2]);
                acc[3] = fmaf(d1, cb[3], acc[3]);
                if constexpr (F == FMT_Q4_1) {
                    const float m0 = ob ? md[0] : me[0];
                    const float m1 = ob ? md[1] : me[1];
                    const int n0 = 2 * c, n1 = 2 * c + 1;
                    const float s0 = n0 < p.batch ? xsum[blk * p.batch + n0] : 0.0f;
                    const float s1 = n1 < p.batch ? xsum[blk * p.batch + n1] : 0.0f;
                    acc[0] = fmaf(m0, s0, acc[0]);
                    acc[1] = fmaf(m0, s1, acc[1]);
                    acc[2] = fmaf(m1, s0, acc[2]);
                    acc[3] = fmaf(m1, s1, acc[3]);
                }
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
        for (int w = 0; w < kTcWarps; ++w) {
            const int ub = static_cast<int>((static_cast<int64_t>(units) * w) / kTcWarps);
            const int ue = static_cast<int>((static_cast<int64_t>(units) * (w + 1)) / kTcWarps);
            if (ue > ub && ub / nch <= tt && (ue - 1) / nch >= tt) {
                s += part[(size_t(w + tt) * kTile + rr) * 8 + n];
            }
        }
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
            cudaError_t e = cudaFuncSetAttribute(gemv_tc_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(budget));
            if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_tc_kernel<F>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
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
        if (cudaOccupancyMaxActiveClusters(&active, gemv_tc_kernel<F>, &qcfg) != cudaSuccess || active < 1) {
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
        cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_tc_kernel<F>, p);
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
