// gemv_tc.cu -- block-quantized GEMV on the tensor cores (mma.sync m16n8k16,
// fp16 operands, fp32 accumulation):  y[b][r] = sum_k w[r][k] * x[b][k],
// batch 1..8, Q4_0 / Q4_1 / Q8_0 (the batch-1 dequantize_mul_mat_vec path of
// the "llama_cpp 0.12.1 -> 0.12.2" ggml-cuda.cu diff, extended to small
// batches; block formulas from the dequantize_block_q4_0 / _q4_1 /
// _q8_0_f16 hunks of the same diff).
//
// Why tensor cores for a bandwidth-bound product: decoding 4-bit weights and
// multiplying them on the CUDA cores costs >= 2.5 instructions per weight,
// about what the SMs can issue while HBM delivers 6+ TB/s.  Here one logic
// instruction (or one byte permute) turns two quantized values into two exact
// fp16 numbers and the products and sums go to the tensor pipe; the batch
// (<= 8) rides along in the MMA's N dimension for free.
//
// Exactness of the operands:
//  - A (weights): Q4: (word & 0x000f000f) | 0x64006400 is the fp16 pair
//    (1024 + q_lo0, 1024 + q_lo1); the high nibbles are taken in place,
//    (word & 0x00f000f0) | 0x64006400 = (1024 + 16 q), and meet x / 16.
//    Q8_0: bytes biased to u = q + 128 (xor 0x80) and permuted under 0x64,
//    giving 1024 + u.  All exact.
//  - The offsets (1024 + 8, 1024 + 128 for the x/16 slots, 1024 + 128 for
//    Q8_0, 1024 for Q4_1) times the block's sums of the rounded x values are
//    the block accumulator's initial value (-T, computed in fp32 when x is
//    staged), so the MMAs' fp32 sums come out as sum_k (q_k - offset) x_k.
//  - B (activations): x * 2^e rounded to fp16 (relative error <= 2^-11), with
//    e chosen per (warp, batch column, 64-block chunk) so that the largest |x|
//    of those values lands in [2^9, 2^10): no overflow, no subnormals for the
//    large values.  Each chunk's partial sums are scaled back by 2^-e (exact).
//  - Each block's fp32 partial is scaled by its fp16 d on the CUDA cores (for
//    Q4_1, m times the block's fp32 sum of x is added).
//
// Data movement: a cluster of cs CTAs owns a balanced range of rows; CTA j of
// the cluster takes the j-th 1/cs of the columns (cs = 1 unless the staged x
// of a larger batch does not fit).  Rows go in tiles of 16 (the MMA's M); the
// last tile of a range is moved back to end at the range's last row,
// overlapping the tile before it (those rows come from L2 and are not written
// twice).  A unit is one tile x 64 blocks: one 3-D TMA copy (64-byte rows,
// 64-byte swizzle) that lands conflict-free for the fragment loads.  Units
// stream through a CTA-wide ring of mbarrier-completed slots fed by one
// producer warp; each of the 16 consumer warps decodes two block pairs of
// every unit and stages the B operands of exactly those blocks itself.  Per-
// warp partials of a tile are summed in a fixed order, then the cs partial
// vectors of the cluster are summed in rank order through distributed shared
// memory: the result is deterministic.
//
// The kernel is launched with programmatic stream serialization: it may start
// while the previous kernel of the stream drains, waits (griddepcontrol.wait)
// before it touches x or y, and -- only when the caller declared its weights
// static (qgemv_set_option) -- starts the weight copies before that wait.
//
// mma.sync fragment layout (m16n8k16, g = lane/4, c = lane%4):
//   A: a0 = (row g,   k 2c..2c+1)  a1 = (row g+8, k 2c..2c+1)
//      a2 = (row g,   k 2c+8..+9)  a3 = (row g+8, k 2c+8..+9)
//   B: b0 = (k 2c..2c+1, n g)      b1 = (k 2c+8..+9, n g)
//   C: c0 = (g, 2c) c1 = (g, 2c+1) c2 = (g+8, 2c) c3 = (g+8, 2c+1)
// The k order inside a block is free as long as A and B agree; lane c holds
// four qs bytes (Q4) or eight (Q8_0) of each of its rows, at the block columns
// listed with stage_x below, and B is staged in exactly that order.
#include <cuda.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "qgemv_common.cuh"

namespace qg {

// Process-wide launch option (qgemv_set_option): weights are never written by
// the kernel that precedes a GEMV on its stream.
int g_opt_weights_static = 0;

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;    // + one producer warp
constexpr int kPairSlots = 32 / kConsumerWarps;        // block pairs per consumer warp per unit
constexpr int kTile = 16;                               // rows per MMA tile
constexpr int kMaxSlots = 24;
#ifndef QG_TC_EARLY_UNITS
#define QG_TC_EARLY_UNITS 2
#endif
constexpr int kEarlyUnits = QG_TC_EARLY_UNITS;  // weight copies started before the stream dependency resolves

template <int F> struct TcFmt;
template <> struct TcFmt<FMT_Q4_0> { static constexpr int BB = 18; };
template <> struct TcFmt<FMT_Q4_1> { static constexpr int BB = 20; };
template <> struct TcFmt<FMT_Q8_0> { static constexpr int BB = 34; };

// A unit is one 16-row tile x 64 blocks = 32 block pairs (consumer warp w
// decodes pairs w + 8 j, j = 0..3); a column slice whose block count is 32
// mod 64 ends each tile with a half unit of 32 blocks (pairs j = 0, 1 only).
constexpr int kUnitBlocks = 64;
__host__ __device__ constexpr int slot_bytes(int F) { return kUnitBlocks * block_bytes(F) / 64 * 1024; }

struct TcParams {
    const float *x;
    float *y;
    unsigned *err;
    int nrows, ncols, batch;
    int cs;              // CTAs per cluster (column split)
    int rows_lo, extra;  // balanced rows per cluster: rows_lo, the first `extra` get one more
    int nbs;             // blocks per CTA column slice (a multiple of 32)
    int nch;             // units per tile: nbs / 64 rounded up
    int half;            // the last unit of each tile is a half unit
    int ns;              // ring slots
    int max_rows;        // rows of the largest cluster range
    int early;           // start the weight copies before waiting on the preceding kernel
};

// Shared-memory layout of one CTA (offsets from a 1024-byte aligned base).
// Each consumer warp owns the B operands of its own blocks: for unit chunk k,
// pair slot j and block beta of the pair, item ((k * kPairSlots + j) * 2 +
// beta) * batch + n.
struct TcLayout {
    uint32_t ring, xf, xc, xs, us, part, ypart, bars, issued, flag, total;
    uint32_t warp_items;   // (block, column) items per warp: nch * 2 * kPairSlots * batch
};

__host__ __device__ inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline TcLayout tc_layout(int F, int nch, int batch, int ns, int max_rows, int cs) {
    TcLayout L;
    L.warp_items = static_cast<uint32_t>(nch) * 2 * kPairSlots * batch;
    const uint32_t items = L.warp_items * kConsumerWarps;
    uint32_t o = 0;
    L.ring = o;  o += static_cast<uint32_t>(ns) * slot_bytes(F);
    L.xf = o;    o += items * 64;                                   // B fragments [item][c] x 16 B
    L.xc = o;    o += items * 4;                                    // -T per item (offset term)
    L.xs = o;    o += F == FMT_Q4_1 ? items * 4 : 0;                // fp32 block sums of x (Q4_1)
    L.us = o;    o += static_cast<uint32_t>(nch) * batch * kConsumerWarps * 4;   // 2^-e per (warp, chunk, column)
    L.part = o;  o += 2u * kConsumerWarps * kTile * batch * 4;      // per-warp tile partials, double buffered
    L.ypart = o; o += cs > 1 ? align_up(static_cast<uint32_t>((max_rows + kTile - 1) / kTile * kTile) * batch * 4, 16) : 0;
    L.bars = o;  o += static_cast<uint32_t>(ns) * 16;               // full[ns], empty[ns]
    L.issued = o; o += align_up(static_cast<uint32_t>(ns) * 4, 16);
    L.flag = o;  o += 16;
    L.total = o;
    return L;
}

// ------------------------------------------------------------ device helpers
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void consumer_bar() {
    asm volatile("bar.sync 1, %0;" :: "n"(kConsumerWarps * 32) : "memory");
}
// Barrier 2: the consumers signal that their first x loads are in flight; the
// producer waits for it before the bulk of the weight copies, so those loads
// do not queue behind megabytes of weights.
__device__ __forceinline__ void xissued_arrive() {
    asm volatile("bar.arrive 2, %0;" :: "n"(kThreads) : "memory");
}
__device__ __forceinline__ void xissued_wait() {
    asm volatile("bar.sync 2, %0;" :: "n"(kThreads) : "memory");
}
// 32-bit shared-memory load (an ordinary C++ load of a pointer into the
// dynamic shared array, so the compiler emits LDS and may schedule it freely
// between the barrier waits).
__device__ __forceinline__ uint32_t lds32(const uint8_t *base, uint32_t off) {
    return *reinterpret_cast<const uint32_t *>(base + off);
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *tmap, int c0, int c1, int c2,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// (a & MASK) | c, one three-input logic instruction.
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ void mma_f16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A B + C with C = (ce, co, ce, co): the first MMA of a block reads its
// initial accumulator straight from the registers holding -T.
__device__ __forceinline__ void mma_f16_init(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1, float ce,
                                             float co) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %10, %11};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(ce), "f"(co));
}

__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float f16lo(uint32_t u) { return __half2float(__ushort_as_half(static_cast<unsigned short>(u & 0xffffu))); }
__device__ __forceinline__ float f16hi(uint32_t u) { return __half2float(__ushort_as_half(static_cast<unsigned short>(u >> 16))); }

// Exponent e with m * 2^e in [2^9, 2^10), from the bits of m = max|x| >= 0
// (biased exponent be: m in [2^(be-127), 2^(be-126)), so e = 136 - be); 0 for
// zero or non-finite m, 120 for subnormal m, so 2^e and 2^-e stay normal.
__device__ __forceinline__ int x_exponent_bits(uint32_t mbits) {
    const int be = static_cast<int>(mbits >> 23);
    if (be == 255 || mbits == 0u) return 0;
    return be == 0 ? 120 : 136 - be;
}
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// Byte offset inside a slot of the 32-bit word at byte `o` of row `y` of a
// unit: the slot is [64-byte chunk][row][64 bytes] with the 64-byte swizzle
// (16-byte units xor-ed with bits 1..2 of the row).
__device__ __forceinline__ uint32_t slot_off(int o, int y) {
    return static_cast<uint32_t>((o >> 6) * 1024 + y * 64 + ((o & 63) ^ (((y >> 1) & 3) << 4)));
}

// ------------------------------------------------------------ x staging
__device__ __forceinline__ float rsum(uint32_t w) { return f16lo(w) + f16hi(w); }

// One consumer warp stages the B operands of its own blocks.  For unit chunk
// k the warp owns 8 blocks (pair slots j = 0..3, pair w + 8 j, even / odd
// block); lane l builds fragment c = l % 4 of block l / 4, loading exactly
// the eight x values that fragment holds as four 8-byte pieces at per-lane
// offsets, so every lane runs the same instructions.  Columns held by lane c
// (fragment words w0..w3 = (p0.x, p1.x) (p0.y, p1.y) (p2.x, p3.x) (p2.y, p3.y)
// for Q4, (p0) (p1) (p2) (p3) for Q8_0, p_i the pieces in load order):
//   Q4 aligned blocks (odd Q4_0 blocks, all Q4_1): low nibbles of qs[4c..4c+3]
//     (pieces x[4c..], x[4c+2..]), high nibbles x[16+4c..], x[18+4c..]
//     (stored as x / 16);
//   Q4_0 even blocks (read at a 2-byte offset and realigned): c = 0 holds
//     qs[0, 1, 14, 15] (pieces x[0], x[14], x[16], x[30]), c >= 1 holds
//     qs[4c-2 .. 4c+1] (pieces x[4c-2], x[4c], x[4c+14], x[4c+16]);
//   Q8_0 odd blocks: q[8c .. 8c+7]; even blocks: c < 3 hold q[8c+2 .. 8c+9],
//     c = 3 holds q[26..29], q[0], q[1], q[30], q[31].
// Fragment words are ordered (k-step 0: b0, b1; k-step 1: b0, b1) to match the
// A registers built by decode_pair.  Per (batch column, chunk) the warp finds
// max |x| of its 256 values and scales them by 2^e (2^-e is kept and applied
// to the chunk's partial sums).  Per block it also stores -T, the offset term
// the MMA must remove (the initial value of that block's accumulator):
// T = 1032 * (sum of the rounded low-slot x) + 1152 * (sum of the rounded
// high-slot x / 16) for Q4_0, 1024 * (both sums) for Q4_1, 1152 * (sum of all
// rounded x) for Q8_0; and, for Q4_1, the fp32 block sum of x.  All the
// warp's loads of one batch column are issued before any is used.
template <int F>
__device__ __forceinline__ void stage_x(const TcParams &p, int kb0, int wid, int lane, uint8_t *smem,
                                        const TcLayout &L) {
    const int blk = lane >> 2, c = lane & 3;
    const int j = blk >> 1, beta = blk & 1;
    const int nch = p.nch;
    uint4 *frag = reinterpret_cast<uint4 *>(smem + L.xf) + wid * L.warp_items * 4;
    float *negt = reinterpret_cast<float *>(smem + L.xc) + wid * L.warp_items;
    float *xsum = reinterpret_cast<float *>(smem + L.xs) + wid * L.warp_items;
    float *uns = reinterpret_cast<float *>(smem + L.us) + wid * nch * p.batch;
    // offsets (in floats, inside the block) of this lane's four pieces
    int off[4];
    if constexpr (F == FMT_Q8_0) {
        if (beta || c < 3) {
            const int b0 = beta ? 8 * c : 8 * c + 2;
            off[0] = b0; off[1] = b0 + 2; off[2] = b0 + 4; off[3] = b0 + 6;
        } else {
            off[0] = 26; off[1] = 28; off[2] = 0; off[3] = 30;
        }
    } else {
        if (F == FMT_Q4_1 || beta) {
            off[0] = 4 * c; off[1] = 4 * c + 2; off[2] = 16 + 4 * c; off[3] = 18 + 4 * c;
        } else if (c == 0) {
            off[0] = 0; off[1] = 14; off[2] = 16; off[3] = 30;
        } else {
            off[0] = 4 * c - 2; off[1] = 4 * c; off[2] = 4 * c + 14; off[3] = 4 * c + 16;
        }
    }
    // this lane's block inside the warp's blocks of a chunk exists (a half
    // unit has pair slots 0 and 1 only)
    auto valid_k = [&](int k) { return !(p.half && k == nch - 1 && j >= kPairSlots / 2); };
    const size_t bcol = static_cast<size_t>(kb0 + 2 * (wid + kConsumerWarps * j) + beta) * 32;
    constexpr int kMaxLoad = 8;                 // chunks whose loads are in flight at once
    for (int n = 0; n < p.batch; ++n) {
        const float *xr = p.x + static_cast<size_t>(n) * p.ncols + bcol;
        for (int k0 = 0; k0 < nch; k0 += kMaxLoad) {
            float2 v[kMaxLoad][4];
#pragma unroll
            for (int i = 0; i < kMaxLoad; ++i) {
                const int k = k0 + i;
                const bool ld = k < nch && valid_k(k);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    v[i][h] = ld ? __ldg(reinterpret_cast<const float2 *>(xr + k * kUnitBlocks * 32 + off[h]))
                                 : make_float2(0.0f, 0.0f);
                }
            }
            if (n == 0 && k0 == 0) xissued_arrive();
#pragma unroll
            for (int i = 0; i < kMaxLoad; ++i) {
                const int k = k0 + i;
                if (k >= nch) break;                 // warp-uniform
                float m = 0.0f;
#pragma unroll
                for (int h = 0; h < 4; ++h) m = fmaxf(m, fmaxf(fabsf(v[i][h].x), fabsf(v[i][h].y)));
                const int e = x_exponent_bits(__reduce_max_sync(0xffffffffu, __float_as_uint(m)));
                if (lane == 0) uns[k * p.batch + n] = pow2f(-e);
                const float sc = pow2f(e);
                uint32_t w0, w1, w2, w3;
                float slo, shi;
                if constexpr (F == FMT_Q8_0) {
                    w0 = f16x2_rn(v[i][0].x * sc, v[i][0].y * sc);
                    w1 = f16x2_rn(v[i][1].x * sc, v[i][1].y * sc);
                    w2 = f16x2_rn(v[i][2].x * sc, v[i][2].y * sc);
                    w3 = f16x2_rn(v[i][3].x * sc, v[i][3].y * sc);
                    slo = (rsum(w0) + rsum(w1)) + (rsum(w2) + rsum(w3));
                    shi = 0.0f;
                } else {
                    const float sh = sc * 0.0625f;   // high-nibble slots carry x / 16
                    w0 = f16x2_rn(v[i][0].x * sc, v[i][1].x * sc);
                    w1 = f16x2_rn(v[i][0].y * sc, v[i][1].y * sc);
                    w2 = f16x2_rn(v[i][2].x * sh, v[i][3].x * sh);
                    w3 = f16x2_rn(v[i][2].y * sh, v[i][3].y * sh);
                    slo = rsum(w0) + rsum(w1);
                    shi = rsum(w2) + rsum(w3);
                }
                // block sums of the rounded values over lanes c = 0..3 (fixed tree)
                slo += __shfl_xor_sync(0xffffffffu, slo, 1);
                slo += __shfl_xor_sync(0xffffffffu, slo, 2);
                if constexpr (F != FMT_Q8_0) {
                    shi += __shfl_xor_sync(0xffffffffu, shi, 1);
                    shi += __shfl_xor_sync(0xffffffffu, shi, 2);
                }
                const int item = ((k * kPairSlots + j) * 2 + beta) * p.batch + n;
                const bool valid = valid_k(k);
                if (valid) frag[item * 4 + c] = make_uint4(w0, w1, w2, w3);
                if (valid && c == 0) {
                    float T;
                    if constexpr (F == FMT_Q4_0) T = fmaf(1032.0f, slo, 1152.0f * shi);
                    else if constexpr (F == FMT_Q4_1) T = 1024.0f * (slo + shi);
                    else T = 1152.0f * slo;
                    negt[item] = -T;
                }
                if constexpr (F == FMT_Q4_1) {
                    float t = 0.0f;
#pragma unroll
                    for (int h = 0; h < 4; ++h) t += (v[i][h].x + v[i][h].y) * sc;
                    t += __shfl_xor_sync(0xffffffffu, t, 1);
                    t += __shfl_xor_sync(0xffffffffu, t, 2);
                    if (valid && c == 0) xsum[item] = t;
                }
            }
        }
    }
    __syncwarp();
}

// Per-lane word offsets (inside a slot) of one block pair of a unit, for row
// g; row g + 8 is 512 bytes further (same swizzle phase).
template <int F> struct PairOffsets;

template <> struct PairOffsets<FMT_Q4_0> {
    uint32_t w0, w4, wc, w5c;          // pair words s[0], s[4], s[c], s[5 + c]
    __device__ __forceinline__ void init(int pr, int g, int c) {
        const int o = 36 * pr;
        w0 = slot_off(o, g);
        w4 = slot_off(o + 16, g);
        wc = slot_off(o + 4 * c, g);
        w5c = slot_off(o + 20 + 4 * c, g);
    }
};
template <> struct PairOffsets<FMT_Q4_1> {
    uint32_t w0, w5, w1c, w6c;         // s[0], s[5], s[1 + c], s[6 + c]
    __device__ __forceinline__ void init(int pr, int g, int c) {
        const int o = 40 * pr;
        w0 = slot_off(o, g);
        w5 = slot_off(o + 20, g);
        w1c = slot_off(o + 4 + 4 * c, g);
        w6c = slot_off(o + 24 + 4 * c, g);
    }
};
template <> struct PairOffsets<FMT_Q8_0> {
    uint32_t w0, w8, ea, eb, oa, ob;   // s[0], s[8], even words, odd words
    __device__ __forceinline__ void init(int pr, int g, int c) {
        const int o = 68 * pr;
        w0 = slot_off(o, g);
        w8 = slot_off(o + 32, g);
        ea = slot_off(o + 4 * (c < 3 ? 1 + 2 * c : 7), g);
        eb = slot_off(o + 4 * (c < 3 ? 2 + 2 * c : 0), g);
        oa = slot_off(o + 4 * (9 + 2 * c), g);
        ob = slot_off(o + 4 * (10 + 2 * c), g);
    }
};

// A fragments (k-step 0 and 1) of the even and the odd block of a pair for
// rows g and g + 8, and their scales.
struct PairA {
    uint32_t e0[4], e1[4], o0[4], o1[4];
    float de[2], dd[2], me[2], md[2];
};

// Pair words: Q4_0 (36 bytes) s[0] = (d_e, qs_e[0..1]), s[1..3] = qs_e[2..13],
// s[4] = (qs_e[14..15], d_o), s[5..8] = qs_o; Q4_1 (40 bytes) s[0] = (d_e, m_e),
// s[1..4] = qs_e, s[5] = (d_o, m_o), s[6..9] = qs_o; Q8_0 (68 bytes) s[0] =
// (d_e, q_e[0..1]), s[1..7] = q_e[2..29], s[8] = (q_e[30..31], d_o),
// s[9..16] = q_o.  `sel` realigns the word that straddles the even block's
// 2-byte offset (Q4_0 lane 0, Q8_0 lane 3).
template <int F>
__device__ __forceinline__ void decode_pair(const uint8_t *sb, const PairOffsets<F> &po, uint32_t sel, PairA &A) {
    constexpr uint32_t kMagic = 0x64006400u;          // fp16 (1024, 1024)
    if constexpr (F == FMT_Q8_0) {
        uint32_t ea[2], eb[2], oa[2], ob[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint8_t *r = sb + 512 * h;
            const uint32_t s0 = lds32(r, po.w0), s8 = lds32(r, po.w8);
            ea[h] = lds32(r, po.ea) ^ 0x80808080u;
            eb[h] = prmt(lds32(r, po.eb), s8, sel) ^ 0x80808080u;
            oa[h] = lds32(r, po.oa) ^ 0x80808080u;
            ob[h] = lds32(r, po.ob) ^ 0x80808080u;
            A.de[h] = fp16_bits_to_f32(s0);
            A.dd[h] = fp16_bits_to_f32(s8 >> 16);
        }
        constexpr uint32_t K = 0x64646464u;
        A.e0[0] = prmt(ea[0], K, 0x4140); A.e0[1] = prmt(ea[1], K, 0x4140);
        A.e0[2] = prmt(ea[0], K, 0x4342); A.e0[3] = prmt(ea[1], K, 0x4342);
        A.e1[0] = prmt(eb[0], K, 0x4140); A.e1[1] = prmt(eb[1], K, 0x4140);
        A.e1[2] = prmt(eb[0], K, 0x4342); A.e1[3] = prmt(eb[1], K, 0x4342);
        A.o0[0] = prmt(oa[0], K, 0x4140); A.o0[1] = prmt(oa[1], K, 0x4140);
        A.o0[2] = prmt(oa[0], K, 0x4342); A.o0[3] = prmt(oa[1], K, 0x4342);
        A.o1[0] = prmt(ob[0], K, 0x4140); A.o1[1] = prmt(ob[1], K, 0x4140);
        A.o1[2] = prmt(ob[0], K, 0x4342); A.o1[3] = prmt(ob[1], K, 0x4342);
    } else {
        uint32_t we[2], wo[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint8_t *r = sb + 512 * h;
            if constexpr (F == FMT_Q4_0) {
                const uint32_t W0 = lds32(r, po.w0), W4 = lds32(r, po.w4);
                we[h] = prmt(lds32(r, po.wc), W4, sel);
                wo[h] = lds32(r, po.w5c);
                A.de[h] = fp16_bits_to_f32(W0);
                A.dd[h] = fp16_bits_to_f32(W4 >> 16);
            } else {
                const uint32_t W0 = lds32(r, po.w0), W5 = lds32(r, po.w5);
                we[h] = lds32(r, po.w1c);
                wo[h] = lds32(r, po.w6c);
                A.de[h] = fp16_bits_to_f32(W0);
                A.me[h] = fp16_bits_to_f32(W0 >> 16);
                A.dd[h] = fp16_bits_to_f32(W5);
                A.md[h] = fp16_bits_to_f32(W5 >> 16);
            }
        }
        const uint32_t we8 = we[0] >> 8, we8b = we[1] >> 8, wo8 = wo[0] >> 8, wo8b = wo[1] >> 8;
        A.e0[0] = and_or<0x000f000fu>(we[0], kMagic); A.e0[1] = and_or<0x000f000fu>(we[1], kMagic);
        A.e0[2] = and_or<0x000f000fu>(we8, kMagic);   A.e0[3] = and_or<0x000f000fu>(we8b, kMagic);
        A.e1[0] = and_or<0x00f000f0u>(we[0], kMagic); A.e1[1] = and_or<0x00f000f0u>(we[1], kMagic);
        A.e1[2] = and_or<0x00f000f0u>(we8, kMagic);   A.e1[3] = and_or<0x00f000f0u>(we8b, kMagic);
        A.o0[0] = and_or<0x000f000fu>(wo[0], kMagic); A.o0[1] = and_or<0x000f000fu>(wo[1], kMagic);
        A.o0[2] = and_or<0x000f000fu>(wo8, kMagic);   A.o0[3] = and_or<0x000f000fu>(wo8b, kMagic);
        A.o1[0] = and_or<0x00f000f0u>(wo[0], kMagic); A.o1[1] = and_or<0x00f000f0u>(wo[1], kMagic);
        A.o1[2] = and_or<0x00f000f0u>(wo8, kMagic);   A.o1[3] = and_or<0x00f000f0u>(wo8b, kMagic);
    }
}

// One block pair for rows g and g + 8: A from the unit in slot sb, B from this
// warp's staged fragments (fb: the even block's uint4 for this lane, the odd
// block's `bstep` items further; nt: the blocks' -T for C columns n0 / n1,
// the accumulators' initial values, which remove the magic offsets), scaled
// partials into acc.
template <int F, bool B1>
__device__ __forceinline__ void pair_mma(const uint8_t *sb, const PairOffsets<F> &po, uint32_t sel,
                                         const uint4 *fb, const float *nt, const float *xsb, int bstep,
                                         int n0, int n1, float acc[4]) {
    PairA A;
    decode_pair<F>(sb, po, sel, A);
    const uint4 bhe = fb[0], bho = fb[bstep * 4];
    float te0, to0, te1, to1;
    if constexpr (B1) {     // even and odd block adjacent: one 8-byte load
        const float2 t = *reinterpret_cast<const float2 *>(nt);
        te0 = te1 = t.x;
        to0 = to1 = t.y;
    } else {
        te0 = nt[n0]; to0 = nt[bstep + n0];
        te1 = nt[n1]; to1 = nt[bstep + n1];
    }
    float ce[4], co[4];
    mma_f16_init(ce, A.e0, bhe.x, bhe.y, te0, te1);
    mma_f16_init(co, A.o0, bho.x, bho.y, to0, to1);
    mma_f16(ce, A.e1, bhe.z, bhe.w);
    mma_f16(co, A.o1, bho.z, bho.w);
    acc[0] = fmaf(A.de[0], ce[0], acc[0]);
    acc[2] = fmaf(A.de[1], ce[2], acc[2]);
    acc[0] = fmaf(A.dd[0], co[0], acc[0]);
    acc[2] = fmaf(A.dd[1], co[2], acc[2]);
    if constexpr (!B1) {
        acc[1] = fmaf(A.de[0], ce[1], acc[1]);
        acc[3] = fmaf(A.de[1], ce[3], acc[3]);
        acc[1] = fmaf(A.dd[0], co[1], acc[1]);
        acc[3] = fmaf(A.dd[1], co[3], acc[3]);
    }
    if constexpr (F == FMT_Q4_1) {
        const float se0 = xsb[n0], so0 = xsb[bstep + n0];
        acc[0] = fmaf(A.me[0], se0, fmaf(A.md[0], so0, acc[0]));
        acc[2] = fmaf(A.me[1], se0, fmaf(A.md[1], so0, acc[2]));
        if constexpr (!B1) {
            const float se1 = xsb[n1], so1 = xsb[bstep + n1];
            acc[1] = fmaf(A.me[0], se1, fmaf(A.md[0], so1, acc[1]));
            acc[3] = fmaf(A.me[1], se1, fmaf(A.md[1], so1, acc[3]));
        }
    }
}

// Pair slots j and j + 2 of a unit are 16 pairs (a multiple of 64 bytes per
// row) apart, so their words sit a constant distance apart in the slot.
template <int F>
__host__ __device__ constexpr int pair_slot2_bytes() { return 16 * 2 * block_bytes(F) / 64 * 1024; }

// NP pair slots (4 for a full unit, 2 for a half unit) of one unit.
template <int F, bool B1, int NP>
__device__ __forceinline__ void unit_mma(const uint8_t *sb, const PairOffsets<F> (&po)[2], uint32_t sel,
                                         const uint4 *fb, const float *nt, const float *xsb, int batch, int n0,
                                         int n1, float ak[4]) {
    constexpr int kJ2 = pair_slot2_bytes<F>();
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        pair_mma<F, B1>(sb + (j >> 1) * kJ2, po[j & 1], sel, fb + 2 * j * batch * 4, nt + 2 * j * batch,
                        xsb + 2 * j * batch, batch, n0, n1, ak);
    }
}

// ------------------------------------------------------------------ kernel
// B1: batch == 1 (only C column 0 is accumulated).
template <int F, bool B1>
__global__ void __launch_bounds__(kThreads, 1)
gemv_tc_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_half,
               const TcParams p) {
    constexpr int BB = TcFmt<F>::BB;
    constexpr int SLOT = slot_bytes(F);
    extern __shared__ __align__(16) uint8_t smem_raw[];
    // the swizzle pattern follows absolute shared-memory address bits: align
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int g = lane >> 2, c = lane & 3;
    const bool producer = wid == kConsumerWarps;

    // the next kernel of the stream may be scheduled as our CTAs retire
    griddep_launch_dependents();

    uint32_t rank = 0;
    if (p.cs > 1) asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const int cl = blockIdx.x / p.cs;
    const int rc0 = cl * p.rows_lo + min(cl, p.extra);
    const int nrc = p.rows_lo + (cl < p.extra ? 1 : 0);
    const int ntiles = (nrc + kTile - 1) / kTile;
    const int kb0 = static_cast<int>(rank) * p.nbs;
    const int nch = p.nch;
    const int U = ntiles * nch;
    const int NS = p.ns;
    const TcLayout L = tc_layout(F, nch, p.batch, NS, p.max_rows, p.cs);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + NS;
    int *issued = reinterpret_cast<int *>(smem + L.issued);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.flag);
    float *ypart = reinterpret_cast<float *>(smem + L.ypart);

    // first (local) row of tile t; the last tile ends at the range's last row
    auto tile_row0 = [&](int t) { return t == ntiles - 1 ? nrc - kTile : t * kTile; };

    // producer lane: copy unit u (tile u / nch, chunk u % nch) into its slot
    // (no proxy fence: the consumers' reads of the slot are ordered before the
    // copy by the release/acquire pair on the empty barrier)
    auto issue = [&](int u) {
        const int s = u % NS;
        const int t = u / nch, k = u - t * nch;
        const bool half = p.half && k == nch - 1;
        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(half ? SLOT / 2 : SLOT));
        tma_load_3d(smem_u32(smem + L.ring) + static_cast<uint32_t>(s) * SLOT, half ? &tmap_half : &tmap, 0,
                    rc0 + tile_row0(t), ((kb0 + k * kUnitBlocks) * BB) >> 6, &full[s]);
        issued[s] += 1;
    };

    if (producer && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
            issued[s] = 0;
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int first = min(NS, U);
    if (producer) {
        const int early = p.early ? min(first, kEarlyUnits) : 0;
        if (lane == 0) {
            for (int u = 0; u < early; ++u) issue(u);
        }
        griddep_wait();
        xissued_wait();
        if (lane == 0) {
            for (int u = early; u < first; ++u) issue(u);
            // refill each slot as soon as all consumer warps released it
            for (int u = first; u < U; ++u) {
                const int s = u % NS;
                if (!mbar_wait_sleep(&empty[s], static_cast<uint32_t>(u / NS - 1) & 1u, p.err) || *abort_flag) {
                    *abort_flag = 1;
                    break;
                }
                issue(u);
            }
        }
    } else {
        griddep_wait();                    // x, y: only after the preceding kernel completed
        stage_x<F>(p, kb0, wid, lane, smem, L);

        PairOffsets<F> po[2];                       // pair slots 0, 1 (2, 3 are a constant further)
        po[0].init(wid, g, c);
        po[1].init(wid + kConsumerWarps, g, c);
        const uint32_t sel = (F == FMT_Q4_0) ? (c == 0 ? 0x5432u : 0x3210u) : (c == 3 ? 0x5432u : 0x3210u);
        const int batch = B1 ? 1 : p.batch;
        const int ncol = min(g, batch - 1);         // B columns past the batch repeat the last one
        const int n0 = min(2 * c, batch - 1), n1 = min(2 * c + 1, batch - 1);
        // this lane's B operands of (chunk 0, pair slot 0, even block); the odd
        // block is batch items further, pair slot j 2 j batch, the next chunk
        // 2 kPairSlots batch
        const uint4 *fb0 = reinterpret_cast<const uint4 *>(smem + L.xf) + (wid * L.warp_items + ncol) * 4 + c;
        const float *nt0 = reinterpret_cast<const float *>(smem + L.xc) + wid * L.warp_items;
        const float *xs0 = reinterpret_cast<const float *>(smem + L.xs) + wid * L.warp_items;
        const float *us0p = reinterpret_cast<const float *>(smem + L.us) + wid * nch * batch;

        int s = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = 0; t < ntiles; ++t) {
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            const uint4 *fb = fb0;
            const float *nt = nt0;
            const float *xsb = xs0;
            const float *usp = us0p;
            for (int k = 0; k < nch; ++k) {
                float ak[4] = {0.0f, 0.0f, 0.0f, 0.0f};     // this chunk, in units of x * 2^e
                if (ok) {
                    ok = __all_sync(0xffffffffu, mbar_wait_sleep(&full[s], phase, p.err));
                    if (!ok && lane == 0) *abort_flag = 1;
                }
                if (ok) {
                    const uint8_t *sb = smem + L.ring + s * SLOT;
                    if (p.half && k == nch - 1) unit_mma<F, B1, kPairSlots / 2>(sb, po, sel, fb, nt, xsb, batch, n0, n1, ak);
                    else unit_mma<F, B1, kPairSlots>(sb, po, sel, fb, nt, xsb, batch, n0, n1, ak);
                    const float u0 = usp[n0];
                    acc[0] = fmaf(ak[0], u0, acc[0]);
                    acc[2] = fmaf(ak[2], u0, acc[2]);
                    if constexpr (!B1) {
                        const float u1 = usp[n1];
                        acc[1] = fmaf(ak[1], u1, acc[1]);
                        acc[3] = fmaf(ak[3], u1, acc[3]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                fb += 2 * kPairSlots * batch * 4;
                nt += 2 * kPairSlots * batch;
                xsb += 2 * kPairSlots * batch;
                usp += batch;
                if (++s == NS) { s = 0; phase ^= 1u; }
            }
            // ---- end of tile t: fixed-order sum of the warp partials
            float *pw = reinterpret_cast<float *>(smem + L.part) + ((t & 1) * kConsumerWarps + wid) * kTile * batch;
            if (2 * c < batch) {
                pw[g * batch + 2 * c] = acc[0];
                pw[(g + 8) * batch + 2 * c] = acc[2];
            }
            if (2 * c + 1 < batch) {
                pw[g * batch + 2 * c + 1] = acc[1];
                pw[(g + 8) * batch + 2 * c + 1] = acc[3];
            }
            consumer_bar();
            if (tid < kTile * batch) {
                const int rr = tid / batch, n = tid - rr * batch;
                const float *pb = reinterpret_cast<const float *>(smem + L.part) +
                                  (t & 1) * kConsumerWarps * kTile * batch + rr * batch + n;
                float sum = 0.0f;
#pragma unroll 4
                for (int w = 0; w < kConsumerWarps; ++w) sum += pb[w * kTile * batch];
                const int r = tile_row0(t) + rr;      // local row; rows below 16 t belong to earlier tiles
                if (r >= kTile * t) {
                    if (p.cs == 1) p.y[static_cast<int64_t>(n) * p.nrows + rc0 + r] = sum;
                    else ypart[r * batch + n] = sum;
                }
            }
        }
    }
    __syncthreads();
    if (*abort_flag && tid == 0) {
        // a wait gave up: let every copy still in flight land before exiting
        for (int s = 0; s < NS; ++s) {
            if (issued[s] > 0) mbar_wait_bounded(&full[s], static_cast<uint32_t>(issued[s] - 1) & 1u, p.err);
        }
    }
    if (p.cs == 1) return;

    // ---- cluster: CTA j sums its share of the rows over all ranks, in rank order
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    const int rpc = (nrc + p.cs - 1) / p.cs;
    const int rb = static_cast<int>(rank) * rpc;
    const int re = min(nrc, rb + rpc);
    const uint32_t ypart_s = smem_u32(ypart);
    for (int e = tid; e < (re - rb) * p.batch; e += kThreads) {
        const int r = rb + e / p.batch, n = e % p.batch;
        const uint32_t off = static_cast<uint32_t>((r * p.batch + n) * 4);
        float sum = 0.0f;
        for (int q = 0; q < p.cs; ++q) {
            uint32_t remote;
            float v;
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(ypart_s + off), "r"(q));
            asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
            sum += v;
        }
        p.y[static_cast<int64_t>(n) * p.nrows + rc0 + r] = sum;
    }
    // nobody leaves while a peer may still read its shared memory
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Tensor maps of weight matrices, cached by (address, rows, row bytes, unit
// chunks): the map is host data passed by value to the kernel.  The view is
// 3-D -- (64 bytes, row, 64-byte chunk of the row) with strides (1, row
// bytes, 64) -- so that one box of (64, 16, nz) lands as [chunk][row][64 B]
// with the 64-byte swizzle.
struct WMapEntry {
    const void *ptr = nullptr;
    int64_t nrows = 0, rowbytes = 0;
    int nz = 0;
    CUtensorMap map;
};
constexpr int kWMapCache = 32;
std::mutex g_wmap_mutex;
WMapEntry g_wmap[kWMapCache];
int g_wmap_next = 0;
EncodeTiledFn g_encode_w = nullptr;

qgemv_status weight_map(const void *W, int64_t nrows, int64_t rowbytes, int nz, CUtensorMap *out) {
    std::lock_guard<std::mutex> lk(g_wmap_mutex);
    for (int i = 0; i < kWMapCache; ++i) {
        const WMapEntry &e = g_wmap[i];
        if (e.ptr == W && e.nrows == nrows && e.rowbytes == rowbytes && e.nz == nz) {
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
    const cuuint64_t gdim[3] = {64u, static_cast<cuuint64_t>(nrows), static_cast<cuuint64_t>(rowbytes / 64)};
    const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(rowbytes), 64u};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(kTile), static_cast<cuuint32_t>(nz)};
    const cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = g_encode_w(&e.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(W), gdim, gstride, box,
                            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        e.ptr = nullptr;
        set_last_error("cuTensorMapEncodeTiled(weights) failed (%d)", static_cast<int>(r));
        return QGEMV_ERR_CUDA;
    }
    e.ptr = W;
    e.nrows = nrows;
    e.rowbytes = rowbytes;
    e.nz = nz;
    *out = e.map;
    return QGEMV_OK;
}

int env_int(const char *name, int dflt) {
    const char *v = getenv(name);
    return (v && *v) ? atoi(v) : dflt;
}

template <int F, bool B1>
qgemv_status launch_cfg(const CUtensorMap &wmap, const CUtensorMap &wmap_half, const TcParams &p, int ncl,
                        size_t smem, cudaStream_t s) {
    auto kern = gemv_tc_kernel<F, B1>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ncl * p.cs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, wmap, wmap_half, p);
    if (e != cudaSuccess) {
        set_last_error("qgemv(tensor core) launch: %s", cudaGetErrorString(e));
        return QGEMV_ERR_LAUNCH;
    }
    return check_launch("qgemv(tensor core)");
}

// Active clusters of `cs` CTAs with `smem` bytes each (0 if none fit).  Also
// raises the kernel's dynamic shared-memory limit on the current device.
template <int F, bool B1>
int active_clusters(int cs, size_t smem, const DevInfo &di) {
    auto kern = gemv_tc_kernel<F, B1>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(di.smem_optin)) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (cs > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(static_cast<unsigned>(di.sm_count / cs * cs));
    q.blockDim = dim3(kThreads);
    q.dynamicSmemBytes = smem;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = static_cast<unsigned>(cs);
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    q.attrs = a;
    q.numAttrs = 1;
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, kern, &q) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return active;
}

// Launch plan for one cluster size, cached per (device, format, shape, batch,
// cs): the occupancy query is not free.  ncl == 0 means it does not fit.
struct TcChoice {
    int dev = -1, fmt = -1, batch = 0, cs = 0;
    int64_t nrows = 0, ncols = 0;
    int ncl = 0, ns = 0, max_rows = 0;
    size_t smem = 0;
};
constexpr int kChoiceCache = 64;
std::mutex g_choice_mutex;
TcChoice g_choice[kChoiceCache];
int g_choice_next = 0;

template <int F, bool B1>
bool plan(int64_t nrows, int64_t ncols, int batch, int cs, const DevInfo &di, TcChoice *out) {
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lk(g_choice_mutex);
        for (int i = 0; i < kChoiceCache; ++i) {
            const TcChoice &c = g_choice[i];
            if (c.dev == dev && c.fmt == F && c.batch == batch && c.cs == cs && c.nrows == nrows && c.ncols == ncols) {
                *out = c;
                return c.ncl > 0;
            }
        }
    }
    TcChoice ch;
    ch.dev = dev;
    ch.fmt = F;
    ch.batch = batch;
    ch.cs = cs;
    ch.nrows = nrows;
    ch.ncols = ncols;
    const int nbs = static_cast<int>(ncols / 32) / cs;
    const int nch = (nbs + kUnitBlocks - 1) / kUnitBlocks;
    const size_t budget = di.smem_optin;
    const int slot = slot_bytes(F);
    int ncl = di.sm_count / cs;
    for (int pass = 0; pass < 2; ++pass) {
        if (nrows < ncl) ncl = static_cast<int>(nrows);
        const int max_rows = static_cast<int>((nrows + ncl - 1) / ncl);
        const TcLayout L0 = tc_layout(F, nch, batch, 0, max_rows, cs);
        if (static_cast<size_t>(L0.total) + 1024 + 2u * (slot + 20) > budget) break;
        int ns = static_cast<int>((budget - 1024 - L0.total) / (slot + 20));
        if (ns > kMaxSlots) ns = kMaxSlots;
        const int forced = env_int("QGEMV_TC_SLOTS", 0);
        if (forced >= 2 && forced < ns) ns = forced;
        const TcLayout L = tc_layout(F, nch, batch, ns, max_rows, cs);
        const size_t smem = static_cast<size_t>(L.total) + 1024;
        if (smem > budget) break;
        const int active = active_clusters<F, B1>(cs, smem, di);
        if (active < 1) break;
        if (pass == 0 && active < ncl) {
            ncl = active;               // fewer clusters fit: more rows each, resize
            continue;
        }
        ch.ncl = ncl;
        ch.ns = ns;
        ch.max_rows = max_rows;
        ch.smem = smem;
        break;
    }
    {
        std::lock_guard<std::mutex> lk(g_choice_mutex);
        g_choice[g_choice_next] = ch;
        g_choice_next = (g_choice_next + 1) % kChoiceCache;
    }
    *out = ch;
    return ch.ncl > 0;
}

template <int F, bool B1>
qgemv_status launch_tc_b(const void *W, const float *x, float *y, int64_t nrows, int64_t ncols, int batch,
                         cudaStream_t s, const DevInfo &di, unsigned *err, bool *taken) {
    const int nb = static_cast<int>(ncols / 32);
    // Cluster size: 1 when everything fits (no cluster reduction; each CTA
    // reads all of x, with coalesced loads), else the smallest that fits.
    // QGEMV_TC_CS forces one (tuning sweeps).
    const int forced = env_int("QGEMV_TC_CS", 0);
    TcChoice ch;
    bool found = false;
    for (int cs : {1, 2, 4, 7, 8, 14, 16}) {
        if (nb % (32 * cs) != 0 || cs > di.sm_count) continue;
        if (forced && cs != forced) continue;
        if (plan<F, B1>(nrows, ncols, batch, cs, di, &ch)) {
            found = true;
            break;
        }
    }
    if (!found) return QGEMV_OK;                       // not taken
    TcParams p;
    p.x = x;
    p.y = y;
    p.err = err;
    p.nrows = static_cast<int>(nrows);
    p.ncols = static_cast<int>(ncols);
    p.batch = batch;
    p.cs = ch.cs;
    p.rows_lo = static_cast<int>(nrows / ch.ncl);
    p.extra = static_cast<int>(nrows % ch.ncl);
    p.nbs = nb / ch.cs;
    p.nch = (p.nbs + kUnitBlocks - 1) / kUnitBlocks;
    p.half = (p.nbs % kUnitBlocks) != 0;
    p.ns = ch.ns;
    p.max_rows = ch.max_rows;
    p.early = g_opt_weights_static;
    const int64_t rowbytes = static_cast<int64_t>(nb) * block_bytes(F);
    CUtensorMap wmap, wmap_half;
    qgemv_status ms = weight_map(W, nrows, rowbytes, block_bytes(F), &wmap);
    if (ms == QGEMV_OK) ms = weight_map(W, nrows, rowbytes, block_bytes(F) / 2, &wmap_half);
    if (ms != QGEMV_OK) return ms;
    *taken = true;
    return launch_cfg<F, B1>(wmap, wmap_half, p, ch.ncl, ch.smem, s);
}

template <int F>
qgemv_status launch_tc_fmt(const void *W, const float *x, float *y, int64_t nrows, int64_t ncols, int batch,
                           cudaStream_t s, const DevInfo &di, unsigned *err, bool *taken) {
    *taken = false;
    const int nb = static_cast<int>(ncols / 32);
    if (nb % 32 != 0 || nrows < 1 || nrows > (1 << 30) || ncols > (1 << 30)) return QGEMV_OK;
    return batch == 1 ? launch_tc_b<F, true>(W, x, y, nrows, ncols, batch, s, di, err, taken)
                      : launch_tc_b<F, false>(W, x, y, nrows, ncols, batch, s, di, err, taken);
}

}  // namespace

qgemv_status launch_gemv_tc(int fmt, const void *W, const float *x, float *y, int64_t nrows, int64_t ncols,
                            int batch, cudaStream_t s, const DevInfo &di, unsigned *err, bool *taken) {
    switch (fmt) {
    case FMT_Q4_0: return launch_tc_fmt<FMT_Q4_0>(W, x, y, nrows, ncols, batch, s, di, err, taken);
    case FMT_Q4_1: return launch_tc_fmt<FMT_Q4_1>(W, x, y, nrows, ncols, batch, s, di, err, taken);
    case FMT_Q8_0: return launch_tc_fmt<FMT_Q8_0>(W, x, y, nrows, ncols, batch, s, di, err, taken);
    default:
        *taken = false;
        return QGEMV_OK;
    }
}

}  // namespace qg
