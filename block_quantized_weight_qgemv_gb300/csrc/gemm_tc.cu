// gemm_tc.cu -- prefill matmul on the 5th-generation tensor cores:
//   Y[i][n] = sum_k X[i][k] * w[n][k],   X bf16 [m][ncols], Y fp32 [m][nrows]
// (the many-token role of mul_mat_q in the "llama_cpp 0.12.1 -> 0.12.2"
// ggml-cuda.cu diff), for Q4_0 / Q4_1 / Q8_0 weights.
//
// Operands.  tcgen05.mma kind::f16 takes A and B of one 16-bit type.  X
// arrives as bf16; w = d*(q-8) (etc.) has up to 15 significant bits and is
// exact in neither 16-bit type.  fp16 is used for both: a pre-pass scales
// each token row of X by the power of two 2^e_i that puts its largest
// magnitude in [2^14, 2^15) and rounds it to fp16 in a library-owned
// workspace (exact for every value >= 2^-28 times the row's largest; bf16
// has 8 significant bits), and the kernel rounds each dequantized weight once
// to fp16 (relative error <= 2^-11) and multiplies each output row by
// 2^-e_i, so |Y - exact| <= 2^-11 * sum_k |w_k x_k| plus the fp32 accumulation
// error -- inside the 1e-3 bound -- for every finite X whose rows keep their
// nonzero magnitudes within 2^28 of the row's largest.
//
// Tiling.  One CTA owns 192 weight rows (MMA N, B = W) and up to 256 tokens
// (two MMA M-tiles of 128, A = X), with two fp32 accumulators of 192 columns
// in TMEM: each X tile feeds 192 weight rows and each weight tile is
// dequantized once per 256 tokens.  The 512 x 14336 prefill is
// 2 x ceil(14336 / 192) = 150 CTAs: one wave on 152 SMs.  K is walked in
// chunks of 64 (one 128-byte swizzle row of fp16) through a 3-stage operand
// ring (the X tiles + the dequantized W tile per stage):
//   warp 0      : TMA 2-D loads of the X tiles (128-byte swizzle);
//   warp 1      : TMEM allocation; one thread issues the MMAs and commits each
//                 stage back to the producers (tcgen05.commit -> mbarrier);
//   warps 2-9   : dequantize the raw weight bytes of each chunk into the
//                 swizzled K-major W tile (3 half-blocks, or for Q8_0 6
//                 quarter-blocks, per thread), then run the epilogue
//                 (tcgen05.ld of TMEM -> fp32 stores; each warp one TMEM lane
//                 quarter of one M-tile).  Rows of a multiple of 16 bytes that
//                 hold whole superchunks (ncols % 256 for Q4_0 / Q8_0, % 128
//                 for Q4_1): the raw bytes arrive by TMA in superchunks of
//                 several chunks (see SupF) in a 2- or 3-stage ring, whose
//                 stages the warps release with one arrival each; otherwise
//                 the warps copy each chunk's raw bytes themselves with
//                 coalesced 4-byte cp.async copies into a 3- or 4-stage ring
//                 (and meet at a named barrier per chunk);
//   warp 10     : issues the raw superchunk copies (TMA path).
// The matmul is launched with programmatic dependent launch on the X
// conversion: its set-up and weight-side work overlap that kernel, and only
// the X producer and the epilogue (the row scales) wait for it.
// Every wait is a bounded mbarrier probe; on expiry the error word is set, the
// roles stop issuing work, and the CTA still frees its TMEM before exiting.
#include <cuda.h>

#include <cstring>
#include <mutex>

#include "qgemv_common.cuh"
#include "tc_ptx.cuh"

namespace qg {
namespace {

constexpr int kTok = 128;              // tokens of an MMA M-tile
constexpr int kTM = 2;                 // M-tiles of a CTA: up to 256 tokens
constexpr int kRowsW = 192;            // weight rows per CTA (MMA N)
constexpr int kKC = 64;                // K per stage (one 128-byte fp16 swizzle row)
constexpr int kStages = 3;             // operand stages (X tiles + dequantized W)
constexpr int kWarps = 11;             // + warp 10: raw weight superchunks by TMA (Q4_0)
constexpr int kDqThreads = 256;        // warps 2..9
constexpr int kXTileBytes = kTok * kKC * 2;       // 16 KB per M-tile
constexpr int kXStageBytes = kTM * kXTileBytes;   // 32 KB
constexpr int kWTileBytes = kRowsW * kKC * 2;     // 24 KB
constexpr int kTmemCols = 512;                    // >= kTM * kRowsW = 384

struct GemmParams {
    const uint8_t *W;
    float *Y;
    const float *rscale;   // 2^-e_i of each token row (the pre-pass's scale, undone in the epilogue)
    unsigned *err;
    int nrows, ncols, m;
    int mgroups;           // token groups of up to kTM * kTok tokens
    int nchunks;           // ncols / 64
    int rawtma;            // 1: raw weights by TMA in superchunks (rows of a multiple of 16 bytes; see raw_path)
};

// Byte offset of (row r, 16-byte chunk ch) in a K-major, 128-byte-swizzled
// tile: rows of 128 B, 8-row atoms of 1024 B, chunk index XOR (row % 8).
__device__ __forceinline__ uint32_t sw128_off(int r, int ch) {
    return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// Raw words of one block, loaded from global memory (4-byte aligned loads).
template <int F> struct RawBlock;
template <> struct RawBlock<FMT_Q4_0> { uint32_t w[5]; };
template <> struct RawBlock<FMT_Q4_1> { uint32_t w[5]; };
template <> struct RawBlock<FMT_Q8_0> { uint32_t w[9]; };

// Loads block `b` of row `n` (zeros for rows past the end).  18- and 34-byte
// blocks start 2 bytes past a 4-byte boundary when b is odd (rows are a whole
// number of block pairs long), so the enclosing aligned words are loaded.
template <int F>
__device__ __forceinline__ void load_block(const GemmParams &p, int n, int b, RawBlock<F> &rb) {
    constexpr int BB = FmtInfo<F>::kBytes;
    constexpr int NW = sizeof(rb.w) / 4;
    if (n >= p.nrows) {
#pragma unroll
        for (int i = 0; i < NW; ++i) rb.w[i] = 0u;
        return;
    }
    const int64_t rowbytes = static_cast<int64_t>(p.ncols / 32) * BB;
    const int64_t off = static_cast<int64_t>(n) * rowbytes + static_cast<int64_t>(b) * BB;
    const uint32_t *src = reinterpret_cast<const uint32_t *>(p.W + (off & ~int64_t(3)));
#pragma unroll
    for (int i = 0; i < NW; ++i) rb.w[i] = __ldg(src + i);
}

// Dequantizes one block to 32 fp16 values in element order, as four 16-byte
// chunks (elements 8j .. 8j+7 in out[j]).
//  Q4_0: w = fp16(d * (q - 8)): (q - 8) is exact in fp16, the product is
//        rounded once (round-to-nearest-even).
//  Q4_1: w = fp16(d * q + m), one fused rounding.
//  Q8_0: w = fp16(d * q).
// Nibbles/bytes become fp16 with the exponent trick: (bits & mask) | 0x6400
// is 1024 + v for v in the low 10 mantissa bits (a high nibble sits 4 bits up
// and reads as 1024 + 16 v).
template <int F>
__device__ __forceinline__ void dequant_block_f16(const RawBlock<F> &rb, int odd, uint4 out[4]) {
    const uint32_t magic = 0x64006400u;
    if constexpr (F == FMT_Q8_0) {
        const uint32_t sh = odd ? 32u : 16u;   // odd blocks start 2 bytes into the first word
        const float df = fp16_bits_to_f32(odd ? (rb.w[0] >> 16) : rb.w[0]);
        const __half2 d2 = __float2half2_rn(df);
        const __half2 off = __float2half2_rn(1152.0f);          // 1024 + 128 (sign bias)
        uint32_t h[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t Q = __funnelshift_rc(rb.w[k], rb.w[k + 1], sh) ^ 0x80808080u;
            const uint32_t t01 = __byte_perm(Q, 0u, 0x4140);   // [b0, 0, b1, 0]
            const uint32_t t23 = __byte_perm(Q, 0u, 0x4342);   // [b2, 0, b3, 0]
            h[2 * k] = h2u(__hmul2(__hsub2(u2h(lop3_and_or(t01, 0x00ff00ffu, magic)), off), d2));
            h[2 * k + 1] = h2u(__hmul2(__hsub2(u2h(lop3_and_or(t23, 0x00ff00ffu, magic)), off), d2));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) out[j] = make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
    } else {
        uint32_t Q[4];
        __half2 d2, m2;
        if constexpr (F == FMT_Q4_0) {
            const uint32_t sh = odd ? 32u : 16u;
#pragma unroll
            for (int k = 0; k < 4; ++k) Q[k] = __funnelshift_rc(rb.w[k], rb.w[k + 1], sh);
            d2 = __float2half2_rn(fp16_bits_to_f32(odd ? (rb.w[0] >> 16) : rb.w[0]));
            m2 = __float2half2_rn(0.0f);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) Q[k] = rb.w[1 + k];
            d2 = __float2half2_rn(fp16_bits_to_f32(rb.w[0]));
            m2 = __float2half2_rn(fp16_bits_to_f32(rb.w[0] >> 16));
        }
        // low nibble: 1024 + q;  high nibble: 1024 + 16 q
        constexpr float lo_off = (F == FMT_Q4_0) ? 1032.0f : 1024.0f;   // q - 8 or q
        constexpr float hi_off = (F == FMT_Q4_0) ? 72.0f : 64.0f;
        const __half2 lo_sub = __float2half2_rn(lo_off);
        const __half2 sixteenth = __float2half2_rn(0.0625f);
        const __half2 hi_sub = __float2half2_rn(-hi_off);
        uint32_t lo[8], hi[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t t01 = __byte_perm(Q[k], 0u, 0x4140);
            const uint32_t t23 = __byte_perm(Q[k], 0u, 0x4342);
            const __half2 l01 = __hsub2(u2h(lop3_and_or(t01, 0x000f000fu, magic)), lo_sub);
            const __half2 l23 = __hsub2(u2h(lop3_and_or(t23, 0x000f000fu, magic)), lo_sub);
            const __half2 h01 = __hfma2(u2h(lop3_and_or(t01, 0x00f000f0u, magic)), sixteenth, hi_sub);
            const __half2 h23 = __hfma2(u2h(lop3_and_or(t23, 0x00f000f0u, magic)), sixteenth, hi_sub);
            if constexpr (F == FMT_Q4_0) {
                lo[2 * k] = h2u(__hmul2(l01, d2));
                lo[2 * k + 1] = h2u(__hmul2(l23, d2));
                hi[2 * k] = h2u(__hmul2(h01, d2));
                hi[2 * k + 1] = h2u(__hmul2(h23, d2));
            } else {
                lo[2 * k] = h2u(__hfma2(l01, d2, m2));
                lo[2 * k + 1] = h2u(__hfma2(l23, d2, m2));
                hi[2 * k] = h2u(__hfma2(h01, d2, m2));
                hi[2 * k + 1] = h2u(__hfma2(h23, d2, m2));
            }
        }
        out[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);   // elements 0..7
        out[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);   // 8..15
        out[2] = make_uint4(hi[0], hi[1], hi[2], hi[3]);   // 16..23
        out[3] = make_uint4(hi[4], hi[5], hi[6], hi[7]);   // 24..31
    }
}

// Raw weight bytes of one K-chunk (384 rows x 2 blocks) are staged in shared
// memory with coalesced 4-byte cp.async copies: word w of the chunk (row w/NW,
// word w%NW) is copied by producer thread w % 256, so a warp's 32 copies cover
// consecutive words of 3-4 rows.  Rows past the end are zero-filled.
// Raw weights by TMA (rows whose byte length is a multiple of 16): superchunks
// of SupF<F>::kChunks K chunks (kChunks * 2 blocks of each of kRowsW rows),
// in a ring of SupF<F>::kStages stages filled by the raw-issuer warp and
// released by the dequantizing warps.  A TMA box starts at a multiple of 16
// bytes: superchunk j's bytes [j * S, (j + 1) * S) of a row (S =
// sup_row_bytes) are copied as the kBoxBytes-wide box starting at
// (j * S) & ~15, and the dequantizer skips the first (j * S) & 15 bytes.
//   Q4_0: 4 chunks, S = 144 (always aligned), 2 stages.
//   Q4_1: 2 chunks, S = 80 (always aligned), 3 stages.
//   Q8_0: 2 chunks, S = 136 (odd superchunks start 8 bytes in), 144-byte
//         boxes, 2 stages.
template <int F> struct SupF;
template <> struct SupF<FMT_Q4_0> { static constexpr int kChunks = 4, kStages = 2, kBoxBytes = 144; };
template <> struct SupF<FMT_Q4_1> { static constexpr int kChunks = 2, kStages = 3, kBoxBytes = 80; };
template <> struct SupF<FMT_Q8_0> { static constexpr int kChunks = 2, kStages = 2, kBoxBytes = 144; };
template <int F> constexpr int sup_row_bytes() { return SupF<F>::kChunks * 2 * FmtInfo<F>::kBytes; }   // 144 / 80 / 136
template <int F> constexpr int sup_stage_bytes() { return kRowsW * SupF<F>::kBoxBytes; }      // 27,648 / 15,360 / 27,648
constexpr int kMaxSupStages = 3;
static_assert(SupF<FMT_Q4_0>::kBoxBytes % 16 == 0 && SupF<FMT_Q4_1>::kBoxBytes % 16 == 0 &&
                  SupF<FMT_Q8_0>::kBoxBytes % 16 == 0, "TMA boxes of 16-byte multiples");
static_assert(sup_row_bytes<FMT_Q4_0>() + 0 <= SupF<FMT_Q4_0>::kBoxBytes &&
                  sup_row_bytes<FMT_Q4_1>() + 0 <= SupF<FMT_Q4_1>::kBoxBytes &&
                  sup_row_bytes<FMT_Q8_0>() + 8 <= SupF<FMT_Q8_0>::kBoxBytes, "box covers the shifted superchunk");
static_assert(SupF<FMT_Q4_0>::kStages <= kMaxSupStages && SupF<FMT_Q4_1>::kStages <= kMaxSupStages &&
                  SupF<FMT_Q8_0>::kStages <= kMaxSupStages, "barrier slots");
// Barriers (3 x kStages + accumulator + TMEM slot + 2 x kMaxSupStages) in
// front of the raw ring.
constexpr int kBarRegion = 256;
static_assert(8 * (3 * kStages + 2 + 2 * kMaxSupStages) <= kBarRegion, "barrier region");
// MMA descriptors are formed as base + offset / 16 (see the MMA loop): every
// operand address, offset included, must stay below 2^18 bytes.
static_assert(1024 + kStages * (kXStageBytes + kWTileBytes) < (1 << 18), "operand tiles within the 18-bit field");

template <int F> struct RawFmt {
    static constexpr int kRowWords = 2 * FmtInfo<F>::kBytes / 4;      // 9 / 10 / 17 words per row
    static constexpr int kStageBytes = kRowsW * kRowWords * 4;
    static constexpr int kStages = (F == FMT_Q8_0) ? 3 : 4;
    static constexpr int kPerThread = (kRowsW * kRowWords + kDqThreads - 1) / kDqThreads;
};

__device__ __forceinline__ void cp_async4(void *dst, const void *src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;"
                 :: "r"(smem_u32(dst)), "l"(src), "r"(valid ? 4 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }
// Makes every later use of r depend on this point of the program: placed
// after tcgen05.wait::ld, it keeps the compiler from reading registers that a
// TMEM load is still filling.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) asm volatile("" : "+r"(r[j]));
}
static_assert(kRowsW % 64 == 0, "the epilogue reads TMEM in pairs of 32-column slices");

// Programmatic dependent launch: the matmul is launched while the activation
// conversion before it may still run; only what reads that kernel's output
// (the X copy, the row scales) waits for it.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier over the kDqThreads producer threads (warps 2..9) that also
// ORs a per-thread flag, so that all of them take the same exit decision.
__device__ __forceinline__ bool producers_sync_any(bool flag) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"(flag ? 1u : 0u), "n"(kDqThreads) : "memory");
    return r != 0;
}

template <int F>
__device__ __forceinline__ void issue_raw_chunk(const GemmParams &p, int n0, int chunk, int t, uint8_t *raw) {
    using R = RawFmt<F>;
    constexpr int BB = FmtInfo<F>::kBytes;
    const int64_t rowbytes = static_cast<int64_t>(p.ncols / 32) * BB;
#pragma unroll
    for (int j = 0; j < R::kPerThread; ++j) {
        const int w = t + kDqThreads * j;
        if (w < kRowsW * R::kRowWords) {
            const int r = w / R::kRowWords, wi = w - r * R::kRowWords;
            const int n = n0 + r;
            const bool valid = n < p.nrows;
            const uint8_t *src = p.W + (valid ? static_cast<int64_t>(n) * rowbytes : 0) +
                                 static_cast<int64_t>(chunk) * 2 * BB + 4 * wi;
            cp_async4(raw + 4 * w, src, valid);
        }
    }
}

// Dequantizes this thread's block items of the staged chunk into the
// swizzled W tile: item i = t + 256 j (< 384) -> row i/2, block i%2 of the
// chunk.
template <int F>
__device__ __forceinline__ void dequant_chunk(const uint8_t *raw, uint8_t *wtile, int t, int row_words = RawFmt<F>::kRowWords,
                                              int word_off = 0) {
    constexpr int BB = FmtInfo<F>::kBytes;
#pragma unroll
    for (int j = 0; j < (2 * kRowsW + kDqThreads - 1) / kDqThreads; ++j) {
        const int i = t + kDqThreads * j;
        if (i >= 2 * kRowsW) break;
        const int r = i >> 1, blk = i & 1;
        // the odd block of a pair starts at byte BB: aligned words from BB/4 on
        const uint32_t src = smem_u32(raw) + 4u * static_cast<uint32_t>(r * row_words + word_off + blk * (BB >> 2));
        RawBlock<F> rb;
#pragma unroll
        for (int k = 0; k < static_cast<int>(sizeof(rb.w) / 4); ++k) {
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(rb.w[k]) : "r"(src + 4u * k) : "memory");
        }
        uint4 v[4];
        dequant_block_f16<F>(rb, blk, v);
        const uint32_t base = smem_u32(wtile);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                         :: "r"(base + sw128_off(r, 4 * blk + c)), "r"(v[c].x), "r"(v[c].y), "r"(v[c].z), "r"(v[c].w)
                         : "memory");
        }
    }
}

// W tile (Q4_0 / Q4_1) from a raw superchunk in half-blocks: half h of block
// b of a row holds quant bytes 8h .. 8h+7, i.e. elements 8h .. 8h+7 (low
// nibbles) and 16+8h .. 16+8h+7 (high nibbles) -- two 16-byte pieces of the
// swizzled row.  The 192 x 2 x 2 = 768 half-blocks of a chunk are 3 per
// producer thread.  Within a warp, lane bits 0-2 pick one of 8 consecutive
// rows and bits 3-4 the half-block (h, b), so the 8 lanes of each store
// phase write the same chunk index of 8 rows: 8 distinct swizzled 16-byte
// slots.  The arithmetic is that of dequant_block_f16 for the same elements.
template <int F>
__device__ __forceinline__ void dequant_chunk_halves(const uint8_t *raw, uint8_t *wtile, int t, int row_words,
                                                     int word_off) {
    static_assert(F == FMT_Q4_0 || F == FMT_Q4_1, "4-bit formats");
    const uint32_t magic = 0x64006400u;
    // low nibble reads 1024 + q, high nibble (1024 + 16 q) / 16 = 64 + q
    const __half2 lo_sub = __float2half2_rn(F == FMT_Q4_0 ? 1032.0f : 1024.0f);   // q - 8 or q
    const __half2 sixteenth = __float2half2_rn(0.0625f);
    const __half2 hi_sub = __float2half2_rn(F == FMT_Q4_0 ? -72.0f : -64.0f);
    const int lane = t & 31, wq = t >> 5;
    const int h = (lane >> 3) & 1, blk = lane >> 4;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const int r = 8 * (wq + 8 * j) + (lane & 7);
        uint32_t Q0, Q1;
        __half2 d2, m2;
        if constexpr (F == FMT_Q4_0) {
            // the odd block of a pair starts 2 bytes into word 4 of the pair
            const uint32_t src = smem_u32(raw) + 4u * static_cast<uint32_t>(r * row_words + word_off + 4 * blk);
            uint32_t w0, wa, wb, wc;
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w0) : "r"(src) : "memory");
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(wa) : "r"(src + 8u * h) : "memory");
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(wb) : "r"(src + 8u * h + 4u) : "memory");
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(wc) : "r"(src + 8u * h + 8u) : "memory");
            const uint32_t sh = blk ? 32u : 16u;
            Q0 = __funnelshift_rc(wa, wb, sh);          // quant bytes 8h .. 8h+3
            Q1 = __funnelshift_rc(wb, wc, sh);          // quant bytes 8h+4 .. 8h+7
            d2 = __float2half2_rn(fp16_bits_to_f32(blk ? (w0 >> 16) : w0));
            m2 = __float2half2_rn(0.0f);
        } else {
            // 20-byte blocks: word 0 = d | m << 16, words 1-4 = quant bytes 0-15
            const uint32_t src = smem_u32(raw) + 4u * static_cast<uint32_t>(r * row_words + word_off + 5 * blk);
            uint32_t w0;
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w0) : "r"(src) : "memory");
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(Q0) : "r"(src + 4u + 8u * h) : "memory");
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(Q1) : "r"(src + 8u + 8u * h) : "memory");
            d2 = __float2half2_rn(fp16_bits_to_f32(w0));
            m2 = __float2half2_rn(fp16_bits_to_f32(w0 >> 16));
        }
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint32_t Qk = k ? Q1 : Q0;
            const uint32_t t01 = __byte_perm(Qk, 0u, 0x4140);
            const uint32_t t23 = __byte_perm(Qk, 0u, 0x4342);
            const __half2 l01 = __hsub2(u2h(lop3_and_or(t01, 0x000f000fu, magic)), lo_sub);
            const __half2 l23 = __hsub2(u2h(lop3_and_or(t23, 0x000f000fu, magic)), lo_sub);
            const __half2 h01 = __hfma2(u2h(lop3_and_or(t01, 0x00f000f0u, magic)), sixteenth, hi_sub);
            const __half2 h23 = __hfma2(u2h(lop3_and_or(t23, 0x00f000f0u, magic)), sixteenth, hi_sub);
            if constexpr (F == FMT_Q4_0) {
                lo[2 * k] = h2u(__hmul2(l01, d2));
                lo[2 * k + 1] = h2u(__hmul2(l23, d2));
                hi[2 * k] = h2u(__hmul2(h01, d2));
                hi[2 * k + 1] = h2u(__hmul2(h23, d2));
            } else {
                lo[2 * k] = h2u(__hfma2(l01, d2, m2));
                lo[2 * k + 1] = h2u(__hfma2(l23, d2, m2));
                hi[2 * k] = h2u(__hfma2(h01, d2, m2));
                hi[2 * k + 1] = h2u(__hfma2(h23, d2, m2));
            }
        }
        const uint32_t base = smem_u32(wtile);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                     :: "r"(base + sw128_off(r, 4 * blk + h)), "r"(lo[0]), "r"(lo[1]), "r"(lo[2]), "r"(lo[3]) : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                     :: "r"(base + sw128_off(r, 4 * blk + 2 + h)), "r"(hi[0]), "r"(hi[1]), "r"(hi[2]), "r"(hi[3])
                     : "memory");
    }
}

// Q8_0 W tile from a raw superchunk in quarter-blocks: quarter u of block b
// of a row holds quant bytes 8u .. 8u+7, i.e. elements 8u .. 8u+7 -- one
// 16-byte piece of the swizzled row.  The 192 x 2 x 4 = 1536 quarter-blocks
// of a chunk are 6 per producer thread.  Within a warp, lane bits 0-2 pick
// one of 8 consecutive rows and bits 3-4 (with the iteration) the quarter,
// so the 8 lanes of each store phase write the same chunk index of 8 rows.
// `word_off` is the word holding the chunk's first byte; an odd block starts
// 2 bytes into a word.  The arithmetic is that of dequant_block_f16.
__device__ __forceinline__ void dequant_chunk_q8_0_quarters(const uint8_t *raw, uint8_t *wtile, int t, int row_words,
                                                            int word_off) {
    const uint32_t magic = 0x64006400u;
    const __half2 off = __float2half2_rn(1152.0f);      // 1024 + 128 (sign bias)
    const int lane = t & 31, wq = t >> 5;
#pragma unroll
    for (int j = 0; j < 6; ++j) {
        const int wv = wq + 8 * j;                        // 0 .. 47
        const int r = 8 * (wv % 24) + (lane & 7);
        const int combo = (lane >> 3) + 4 * (wv / 24);    // 0 .. 7
        const int blk = combo >> 2, qu = combo & 3;
        // block blk starts at byte 34 * blk of the chunk: word 8 * blk, plus 2 bytes if odd
        const uint32_t src = smem_u32(raw) + 4u * static_cast<uint32_t>(r * row_words + word_off + 8 * blk);
        uint32_t w0, wa, wb, wc;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w0) : "r"(src) : "memory");
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(wa) : "r"(src + 8u * qu) : "memory");
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(wb) : "r"(src + 8u * qu + 4u) : "memory");
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(wc) : "r"(src + 8u * qu + 8u) : "memory");
        const uint32_t sh = blk ? 32u : 16u;
        const __half2 d2 = __float2half2_rn(fp16_bits_to_f32(blk ? (w0 >> 16) : w0));
        uint32_t h[4];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint32_t Q = __funnelshift_rc(k ? wb : wa, k ? wc : wb, sh) ^ 0x80808080u;   // quant bytes 8u+4k ..
            const uint32_t t01 = __byte_perm(Q, 0u, 0x4140);
            const uint32_t t23 = __byte_perm(Q, 0u, 0x4342);
            h[2 * k] = h2u(__hmul2(__hsub2(u2h(lop3_and_or(t01, 0x00ff00ffu, magic)), off), d2));
            h[2 * k + 1] = h2u(__hmul2(__hsub2(u2h(lop3_and_or(t23, 0x00ff00ffu, magic)), off), d2));
        }
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                     :: "r"(smem_u32(wtile) + sw128_off(r, 4 * blk + qu)), "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3])
                     : "memory");
    }
}

template <int F>
__global__ void __launch_bounds__(kWarps * 32, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
               const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *xtiles = smem;                                        // kStages x kTM x 16 KB
    uint8_t *wtiles = smem + kStages * kXStageBytes;               // kStages x 12 KB
    uint64_t *bars = reinterpret_cast<uint64_t *>(wtiles + kStages * kWTileBytes);
    uint64_t *full_x = bars;
    uint64_t *full_w = bars + kStages;
    uint64_t *empty = bars + 2 * kStages;
    uint64_t *accum = bars + 3 * kStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * kStages + 1);
    uint64_t *rawfull = bars + 3 * kStages + 2;                    // raw superchunk stages (TMA path)
    uint64_t *rawempty = rawfull + kMaxSupStages;
    uint8_t *rawring = reinterpret_cast<uint8_t *>(bars) + kBarRegion;          // raw stages of either path
    __shared__ int s_fail;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int mg = blockIdx.x % p.mgroups;         // token group
    const int nt = blockIdx.x / p.mgroups;         // weight-row tile
    const int tok0 = mg * kTM * kTok;
    const int tm = min(kTM, (p.m - tok0 + kTok - 1) / kTok);   // M-tiles of this CTA
    const int n0 = nt * kRowsW;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_x[s], 1);
            mbar_init(&full_w[s], kDqThreads);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accum, 1);
        for (int k = 0; k < SupF<F>::kStages; ++k) {
            mbar_init(&rawfull[k], 1);
            mbar_init(&rawempty[k], kDqThreads / 32);               // one arrival per dequantizing warp
        }
        fence_mbar_init();
        s_fail = 0;
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    cta_sync();
    tc::fence_after_sync();
    const uint32_t taddr = *tmem_slot;
    // epilogue of the dequantizing warps: TMEM -> Y (tcgen05.ld needs the whole warp)
    auto epilogue = [&](bool ok) {
        griddep_wait();                                  // the row scales come from the conversion kernel
        const bool ready = ok && mbar_wait_sleep(accum, 0u, p.err);
        if (__all_sync(0xffffffffu, ready)) {
            tc::fence_after_sync();
            const int q = warp & 3;                     // TMEM lane quarter this warp may access
            const int i = (warp - 2) >> 2;              // M-tile of this warp
            const bool vec = (p.nrows & 3) == 0;
            if (i < tm) {
                const int tok = tok0 + i * kTok + 32 * q + lane;
                const float rs = tok < p.m ? p.rscale[tok] : 0.0f;
                const uint32_t tbase = taddr + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(i * kRowsW);
                auto store = [&](const uint32_t (&r)[32], int cc) {
                    const int n = n0 + cc;
                    if (tok < p.m && n < p.nrows) {
                        float *yr = p.Y + static_cast<int64_t>(tok) * p.nrows + n;
                        if (vec && n + 32 <= p.nrows) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                __stcs(reinterpret_cast<float4 *>(yr) + j,
                                       make_float4(__uint_as_float(r[4 * j]) * rs, __uint_as_float(r[4 * j + 1]) * rs,
                                                   __uint_as_float(r[4 * j + 2]) * rs, __uint_as_float(r[4 * j + 3]) * rs));
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j) {      // constant indices: r stays in registers
                                if (n + j < p.nrows) yr[j] = __uint_as_float(r[j]) * rs;
                            }
                        }
                    }
                };
                // two register buffers: the stores of one 32-column slice overlap
                // the TMEM load of the next
                uint32_t ra[32], rb[32];
                tc::tmem_ld32(tbase, ra);
                tc::tmem_ld_wait();
                reg_fence(ra);
#pragma unroll
                for (int cc = 0; cc < kRowsW; cc += 64) {
                    tc::tmem_ld32(tbase + static_cast<uint32_t>(cc + 32), rb);
                    store(ra, cc);
                    tc::tmem_ld_wait();
                    reg_fence(rb);
                    if (cc + 64 < kRowsW) tc::tmem_ld32(tbase + static_cast<uint32_t>(cc + 64), ra);
                    store(rb, cc + 32);
                    if (cc + 64 < kRowsW) {
                        tc::tmem_ld_wait();
                        reg_fence(ra);
                    }
                }
            }
        } else {
            s_fail = 1;
        }
    };

    // Failure handling: a role whose bounded wait expires sets s_fail and stops;
    // it then no longer arrives on (or commits to) the barriers the others wait
    // for, so their bounded waits expire in turn and every role ends.  The
    // per-chunk loops do not poll s_fail: a shared load per chunk on these
    // paths measurably delayed the next MMAs and W tiles.
    if (warp == 0) {
        // ---------------- X tiles by TMA
        if (lane == 0) {
            griddep_wait();                              // the X copy comes from the conversion kernel
            for (int c = 0; c < p.nchunks; ++c) {
                const int s = c % kStages, f = c / kStages;
                // a sleeping wait: this warp shares a scheduler with two dequantizing warps
                if (f > 0 && !mbar_wait_sleep(&empty[s], static_cast<uint32_t>((f - 1) & 1), p.err)) {
                    s_fail = 1;
                    break;
                }
                mbar_arrive_expect_tx(&full_x[s], static_cast<uint32_t>(tm) * kXTileBytes);
                for (int i = 0; i < tm; ++i) {
                    tc::tma_load_2d(xtiles + s * kXStageBytes + i * kXTileBytes, &tmap_x, c * kKC, tok0 + i * kTok,
                                    &full_x[s]);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issue (one thread)
        if (lane == 0) {
            const uint32_t idn = tc::idesc_f16_f32(kTok, kRowsW);
            bool ok = true;
            for (int c = 0; c < p.nchunks && ok; ++c) {
                const int s = c % kStages, f = c / kStages;
                const uint32_t par = static_cast<uint32_t>(f & 1);
                ok = mbar_wait_sleep(&full_x[s], par, p.err) && mbar_wait_sleep(&full_w[s], par, p.err);
                if (!ok) {
                    s_fail = 1;
                    break;
                }
                tc::fence_after_sync();
                // Descriptors of the stage's tiles; the start-address field is
                // address / 16 in the low 14 bits (shared addresses stay below
                // 2^18), so an offset within the stage adds offset / 16 to it
                // without a carry into the other fields.
                const uint64_t a_base = tc::sdesc_sw128(smem_u32(xtiles + s * kXStageBytes));
                const uint64_t b_base = tc::sdesc_sw128(smem_u32(wtiles + s * kWTileBytes));
#pragma unroll
                for (int ks = 0; ks < kKC / 16; ++ks) {
                    const uint64_t bdesc = b_base + static_cast<uint64_t>(ks * 32 / 16);
                    const uint32_t acc = (c > 0 || ks > 0) ? 1u : 0u;
#pragma unroll
                    for (int i = 0; i < kTM; ++i) {
                        if (i >= tm) break;
                        // M-tile i: accumulator columns i * kRowsW .. + kRowsW - 1
                        const uint64_t adesc = a_base + static_cast<uint64_t>((i * kXTileBytes + ks * 32) / 16);
                        tc::mma_f16(taddr + static_cast<uint32_t>(i * kRowsW), adesc, bdesc, idn, acc);
                    }
                }
                tc::mma_commit(&empty[s]);              // stage s may be refilled once these MMAs are done
            }
            tc::mma_commit(accum);                      // accumulators complete
        }
        __syncwarp();
    } else if (warp == kWarps - 1) {
        // ---------------- raw weight superchunks by TMA (one thread)
        if (lane == 0 && p.rawtma) {
            constexpr int SUP = SupF<F>::kChunks, SS = SupF<F>::kStages;
            const int nsup = p.nchunks / SUP;
            int issued = 0;
            for (int j = 0; j < nsup; ++j) {
                const int js = j % SS;
                if (j >= SS && !mbar_wait_sleep(&rawempty[js], static_cast<uint32_t>(((j - SS) / SS) & 1), p.err)) {
                    s_fail = 1;
                    break;
                }
                if (*reinterpret_cast<volatile int *>(&s_fail)) break;
                mbar_arrive_expect_tx(&rawfull[js], sup_stage_bytes<F>());
                tc::tma_load_2d(rawring + js * sup_stage_bytes<F>(), &tmap_w, (j * sup_row_bytes<F>()) & ~15, n0,
                                &rawfull[js]);
                ++issued;
            }
            if (*reinterpret_cast<volatile int *>(&s_fail)) {
                // let the copies still in flight land before the CTA exits
                for (int j = issued > SS ? issued - SS : 0; j < issued; ++j)
                    mbar_wait_bounded(&rawfull[j % SS], static_cast<uint32_t>((j / SS) & 1), p.err);
            }
        }
        __syncwarp();
    } else if (p.rawtma) {
        // ---------------- W tiles from raw superchunks (TMA path)
        constexpr int SUP = SupF<F>::kChunks, SS = SupF<F>::kStages;
        const int t = threadIdx.x - 64;
        bool ok = true;
        for (int c = 0; c < p.nchunks; ++c) {
            const int s = c % kStages, f = c / kStages;
            const int j = c / SUP, js = j % SS;
            bool fail = false;
            if (c % SUP == 0 && !mbar_wait_sleep(&rawfull[js], static_cast<uint32_t>((j / SS) & 1), p.err)) fail = true;
            if (f > 0 && !mbar_wait_sleep(&empty[s], static_cast<uint32_t>((f - 1) & 1), p.err)) fail = true;
            if (__any_sync(0xffffffffu, fail)) {           // warp-uniform exit
                s_fail = 1;
                ok = false;
                break;
            }
            // word of the stage row holding the chunk's first byte (box start shift + chunk offset)
            const int woff = (((j * sup_row_bytes<F>()) & 15) + (c % SUP) * 2 * FmtInfo<F>::kBytes) / 4;
            if constexpr (F == FMT_Q8_0)
                dequant_chunk_q8_0_quarters(rawring + js * sup_stage_bytes<F>(), wtiles + s * kWTileBytes, t,
                                            SupF<F>::kBoxBytes / 4, woff);
            else
                dequant_chunk_halves<F>(rawring + js * sup_stage_bytes<F>(), wtiles + s * kWTileBytes, t,
                                        SupF<F>::kBoxBytes / 4, woff);
            fence_proxy_async_smem();                   // generic-proxy stores -> tensor-core reads
            mbar_arrive(&full_w[s]);
            if (c % SUP == SUP - 1) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&rawempty[js]);   // this warp is done with the superchunk
            }
        }
        epilogue(ok);
    } else {
        // ---------------- W tiles: dequantize into the swizzled layout
        using R = RawFmt<F>;
        const int t = threadIdx.x - 64;
        // prologue: raw chunks 0 .. RS-2 in flight
#pragma unroll
        for (int c = 0; c < R::kStages - 1; ++c) {
            if (c < p.nchunks) issue_raw_chunk<F>(p, n0, c, t, rawring + c * R::kStageBytes);
            cp_async_commit();
        }
        bool ok = true;
        for (int c = 0; c < p.nchunks; ++c) {
            const int s = c % kStages, f = c / kStages;
            bool fail = false;
            if (f > 0 && !mbar_wait_sleep(&empty[s], static_cast<uint32_t>((f - 1) & 1), p.err)) fail = true;
            cp_async_wait<R::kStages - 2>();           // this thread's copies of chunk c are done
            // ... and everyone's; chunk c-1's raw stage is free; common exit decision
            if (producers_sync_any(fail)) {
                s_fail = 1;
                ok = false;
                break;
            }
            {
                const int cn = c + R::kStages - 1;     // refill the stage chunk c-1 used
                if (cn < p.nchunks) issue_raw_chunk<F>(p, n0, cn, t, rawring + (cn % R::kStages) * R::kStageBytes);
                cp_async_commit();
            }
            dequant_chunk<F>(rawring + (c % R::kStages) * R::kStageBytes, wtiles + s * kWTileBytes, t);
            fence_proxy_async_smem();                   // generic-proxy stores -> tensor-core reads
            mbar_arrive(&full_w[s]);
        }
        cp_async_wait<0>();
        epilogue(ok);
    }

    tc::fence_before_sync();
    cta_sync();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(taddr, kTmemCols);
    }
}

// Activations bf16 -> fp16, one token row per CTA-iteration: the row's
// largest magnitude (bit patterns, so inf / nan count as largest) sets 2^e
// (largest * 2^e in [2^14, 2^15); e = 0 for an all-zero or non-finite row),
// every element is multiplied by 2^e (as two exact power-of-two factors, e
// reaching 140 for subnormal rows) and rounded to nearest even, and 2^-e goes
// to rscale[row].  ncols is a multiple of 64: whole 16-byte vectors.
constexpr int kScaleThreads = 256;
__global__ void __launch_bounds__(kScaleThreads) x_rows_to_f16_kernel(const uint4 *__restrict__ src,
                                                                      uint4 *__restrict__ dst,
                                                                      float *__restrict__ rscale, int m, int ncols) {
    __shared__ uint32_t red[kScaleThreads / 32];
    griddep_launch_dependents();                      // the matmul may start its weight-only work
    const int v8 = ncols / 8;                         // 16-byte vectors per row
    for (int row = blockIdx.x; row < m; row += gridDim.x) {
        const uint4 *s = src + static_cast<int64_t>(row) * v8;
        uint32_t mx = 0u;
        for (int i = threadIdx.x; i < v8; i += kScaleThreads) {
            const uint4 v = __ldg(s + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) mx = max(mx, max(w[k] & 0x7fffu, (w[k] >> 16) & 0x7fffu));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
        __syncthreads();
        mx = red[0];
#pragma unroll
        for (int w = 1; w < kScaleThreads / 32; ++w) mx = max(mx, red[w]);
        __syncthreads();                              // red is reused by the next row
        const int be = static_cast<int>(mx >> 7);     // bf16 biased exponent of the largest magnitude
        const int e = (mx == 0u || be == 255) ? 0 : 141 - max(be, 1);
        const float s1 = __int_as_float((127 + e / 2) << 23), s2 = __int_as_float((127 + e - e / 2) << 23);
        uint4 *d = dst + static_cast<int64_t>(row) * v8;
        for (int i = threadIdx.x; i < v8; i += kScaleThreads) {
            const uint4 v = __ldg(s + i);
            const uint32_t in[4] = {v.x, v.y, v.z, v.w};
            uint32_t out[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float a = __uint_as_float(in[k] << 16) * s1 * s2;
                const float b = __uint_as_float(in[k] & 0xffff0000u) * s1 * s2;
                out[k] = h2u(__floats2half2_rn(a, b));
            }
            d[i] = make_uint4(out[0], out[1], out[2], out[3]);
        }
        if (threadIdx.x == 0) {
            // 2^-e, e in [-113, 140]: a subnormal for e > 126
            rscale[row] = e > 126 ? __int_as_float(1 << (149 - e)) : __int_as_float((127 - e) << 23);
        }
    }
}

// ------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DevWorkspace {
    void *ptr = nullptr;
    size_t bytes = 0;
    // tensor map of the fp16 activation copy, cached by its shape
    CUtensorMap tmap;
    void *tmap_ptr = nullptr;
    int tmap_m = -1, tmap_k = -1;
};

constexpr int kMaxDev = 64;
std::mutex g_ws_mutex;
DevWorkspace g_ws[kMaxDev];
EncodeTiledFn g_encode = nullptr;

qgemv_status get_encoder() {
    if (g_encode) return QGEMV_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
        set_last_error("cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(e));
        return QGEMV_ERR_CUDA;
    }
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    return QGEMV_OK;
}

// Workspace on device `dev` for an [m][k] fp16 copy of the activations
// followed by m row scales (grown on demand; a growth synchronizes the
// device), with the tensor map of the copy.
size_t rscale_offset(int m, int k) { return (static_cast<size_t>(m) * k * 2 + 255) & ~size_t(255); }
qgemv_status workspace_for(int dev, int m, int k, DevWorkspace **out) {
    const size_t bytes = rscale_offset(m, k) + static_cast<size_t>(m) * 4;
    DevWorkspace &w = g_ws[dev];
    if (w.bytes < bytes) {
        if (w.ptr) {
            cudaError_t e = cudaFree(w.ptr);
            w.ptr = nullptr;
            w.bytes = 0;
            if (e != cudaSuccess) {
                set_last_error("cudaFree(workspace): %s", cudaGetErrorString(e));
                return QGEMV_ERR_CUDA;
            }
        }
        const size_t want = (bytes + (size_t(1) << 20) - 1) & ~((size_t(1) << 20) - 1);
        cudaError_t e = cudaMalloc(&w.ptr, want);
        if (e != cudaSuccess) {
            w.ptr = nullptr;
            set_last_error("cudaMalloc(workspace, %zu): %s", want, cudaGetErrorString(e));
            return QGEMV_ERR_CUDA;
        }
        w.bytes = want;
        w.tmap_m = -1;
    }
    if (w.tmap_m != m || w.tmap_k != k || w.tmap_ptr != w.ptr) {
        qgemv_status st = get_encoder();
        if (st != QGEMV_OK) return st;
        const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(m)};
        const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(k) * 2};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(kKC), static_cast<cuuint32_t>(kTok)};
        const cuuint32_t estride[2] = {1, 1};
        CUresult r = g_encode(&w.tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w.ptr, gdim, gstride, box, estride,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            set_last_error("cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
            return QGEMV_ERR_CUDA;
        }
        w.tmap_ptr = w.ptr;
        w.tmap_m = m;
        w.tmap_k = k;
    }
    *out = &w;
    return QGEMV_OK;
}

// Tensor map of a Q4_0 / Q4_1 matrix's raw bytes, [nrows][rowbytes], in
// boxes of sup_row_bytes x kRowsW (the raw superchunks of the TMA path); rows
// past nrows read as zero.  Cached by (address, format, shape).
struct WMapEntry {
    const void *ptr = nullptr;
    int fmt = -1;
    int64_t nrows = 0, ncols = 0;
    CUtensorMap map;
};
std::mutex g_wmap_mutex;
WMapEntry g_wmaps[16];
int g_wmap_next = 0;

template <int F>
qgemv_status raw_weight_map(const void *W, int64_t nrows, int64_t ncols, CUtensorMap *out) {
    std::lock_guard<std::mutex> lk(g_wmap_mutex);
    for (const WMapEntry &e : g_wmaps) {
        if (e.ptr == W && e.fmt == F && e.nrows == nrows && e.ncols == ncols) {
            *out = e.map;
            return QGEMV_OK;
        }
    }
    qgemv_status st = get_encoder();
    if (st != QGEMV_OK) return st;
    WMapEntry &e = g_wmaps[g_wmap_next];
    g_wmap_next = (g_wmap_next + 1) % 16;
    const int64_t rowbytes = ncols / 32 * FmtInfo<F>::kBytes;
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(rowbytes), static_cast<cuuint64_t>(nrows)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(rowbytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(SupF<F>::kBoxBytes), static_cast<cuuint32_t>(kRowsW)};
    const cuuint32_t estride[2] = {1, 1};
    CUresult r = g_encode(&e.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(W), gdim, gstride, box, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        e.ptr = nullptr;
        set_last_error("cuTensorMapEncodeTiled(raw weights) failed (%d)", static_cast<int>(r));
        return QGEMV_ERR_CUDA;
    }
    e.ptr = W;
    e.fmt = F;
    e.nrows = nrows;
    e.ncols = ncols;
    *out = e.map;
    return QGEMV_OK;
}

// The raw-weight map and path flag of a launch: the TMA path when rows hold
// whole superchunks and a multiple of 16 bytes (Q4_0: ncols % 256 == 0,
// Q4_1: % 128, Q8_0: % 256, so an even number of 8-byte-shifted Q8_0
// superchunks and the last box of a row ends at the row's end) at a
// 16-byte aligned address, else a zeroed map (unused) and the cp.async path.
template <int F>
qgemv_status raw_path(const void *W, int64_t nrows, int64_t ncols, CUtensorMap *map, int *rawtma) {
    memset(map, 0, sizeof(*map));
    *rawtma = 0;
    const int64_t rowbytes = ncols / 32 * FmtInfo<F>::kBytes;
    if (ncols % (SupF<F>::kChunks * kKC) != 0 || rowbytes % 16 != 0 || reinterpret_cast<uintptr_t>(W) % 16 != 0)
        return QGEMV_OK;
    qgemv_status st = raw_weight_map<F>(W, nrows, ncols, map);
    if (st == QGEMV_OK) *rawtma = 1;
    return st;
}

template <int F>
constexpr size_t raw_region_bytes() {
    return size_t(SupF<F>::kStages) * sup_stage_bytes<F>() >
                               size_t(RawFmt<F>::kStages) * RawFmt<F>::kStageBytes
               ? size_t(SupF<F>::kStages) * sup_stage_bytes<F>()
               : size_t(RawFmt<F>::kStages) * RawFmt<F>::kStageBytes;
}
template <int F>
constexpr size_t gemm_smem() {
    static_assert(1024 + kStages * (kXStageBytes + kWTileBytes) + kBarRegion + raw_region_bytes<F>() <= 232448,
                  "prefill shared memory exceeds 227 KB");
    return 1024 + kStages * (kXStageBytes + kWTileBytes) + kBarRegion + raw_region_bytes<F>();
}

// The matmul launch: programmatic dependent launch on the conversion kernel.
template <int F>
qgemv_status launch_matmul(int64_t grid, size_t smem, cudaStream_t s, const CUtensorMap &tmap_x,
                           const CUtensorMap &tmap_w, const GemmParams &p, const char *what) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_tc_kernel<F>, tmap_x, tmap_w, p);
    if (e != cudaSuccess) {
        set_last_error("%s launch: %s", what, cudaGetErrorString(e));
        return QGEMV_ERR_LAUNCH;
    }
    return check_launch(what);
}

template <int F>
qgemv_status launch_tc(const void *W, const void *X, float *Y, int64_t nrows, int64_t ncols, int64_t m,
                       cudaStream_t s, const DevInfo &di, int dev, unsigned *err) {
    constexpr size_t kGemmSmem = gemm_smem<F>();
    if (kGemmSmem > di.smem_optin) {
        set_last_error("prefill kernel needs %zu bytes of shared memory", kGemmSmem);
        return QGEMV_ERR_ARCH;
    }
    std::lock_guard<std::mutex> lk(g_ws_mutex);
    DevWorkspace *ws = nullptr;
    qgemv_status st = workspace_for(dev, static_cast<int>(m), static_cast<int>(ncols), &ws);
    if (st != QGEMV_OK) return st;

    // 1) activations to fp16 (the tensor-core operand type), scaled per row
    float *rscale = reinterpret_cast<float *>(static_cast<char *>(ws->ptr) +
                                              rscale_offset(static_cast<int>(m), static_cast<int>(ncols)));
    const int64_t cblocks = m < static_cast<int64_t>(di.sm_count) * 4 ? m : static_cast<int64_t>(di.sm_count) * 4;
    x_rows_to_f16_kernel<<<static_cast<unsigned>(cblocks), kScaleThreads, 0, s>>>(
        static_cast<const uint4 *>(X), static_cast<uint4 *>(ws->ptr), rscale, static_cast<int>(m), static_cast<int>(ncols));
    st = check_launch("qgemm(activation conversion)");
    if (st != QGEMV_OK) return st;

    // 2) the matmul
    static bool attr_set[kMaxDev] = {false};
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kGemmSmem));
        if (e != cudaSuccess) {
            set_last_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            return QGEMV_ERR_CUDA;
        }
        attr_set[dev] = true;
    }
    GemmParams p;
    p.W = static_cast<const uint8_t *>(W);
    p.Y = Y;
    p.rscale = rscale;
    p.err = err;
    p.nrows = static_cast<int>(nrows);
    p.ncols = static_cast<int>(ncols);
    p.m = static_cast<int>(m);
    p.mgroups = static_cast<int>((m + kTM * kTok - 1) / (kTM * kTok));
    p.nchunks = static_cast<int>(ncols / kKC);
    CUtensorMap wmap;
    st = raw_path<F>(W, nrows, ncols, &wmap, &p.rawtma);
    if (st != QGEMV_OK) return st;
    const int64_t ntiles = (nrows + kRowsW - 1) / kRowsW;
    const int64_t grid = ntiles * p.mgroups;
    if (grid > 0x7fffffff) {
        set_last_error("prefill grid too large");
        return QGEMV_ERR_SHAPE;
    }
    return launch_matmul<F>(grid, kGemmSmem, s, ws->tmap, wmap, p, "qgemm(tensor core)");
}

}  // namespace

qgemv_status launch_gemm_tc(int fmt, const void *W, const void *X, float *Y, int64_t nrows, int64_t ncols,
                            int64_t m, cudaStream_t s, const DevInfo &di, int dev, unsigned *err) {
    if (dev < 0 || dev >= kMaxDev) {
        set_last_error("device ordinal %d out of range", dev);
        return QGEMV_ERR_CUDA;
    }
    switch (fmt) {
    case FMT_Q4_0: return launch_tc<FMT_Q4_0>(W, X, Y, nrows, ncols, m, s, di, dev, err);
    case FMT_Q4_1: return launch_tc<FMT_Q4_1>(W, X, Y, nrows, ncols, m, s, di, dev, err);
    case FMT_Q8_0: return launch_tc<FMT_Q8_0>(W, X, Y, nrows, ncols, m, s, di, dev, err);
    default:
        set_last_error("unknown format %d", fmt);
        return QGEMV_ERR_DTYPE;
    }
}

void gemm_release_workspaces() {
    std::lock_guard<std::mutex> lk(g_ws_mutex);
    int cur = 0;
    cudaGetDevice(&cur);
    for (int d = 0; d < kMaxDev; ++d) {
        if (g_ws[d].ptr) {
            cudaSetDevice(d);
            cudaFree(g_ws[d].ptr);
            g_ws[d] = DevWorkspace();
        }
    }
    cudaSetDevice(cur);
}


// --------------------------------------------------------------------------
// Allocation-free variant of the Q4_0 prefill (qgemm_q4_0_noalloc).
//
// Some callers cannot let a library call cudaMalloc: runtimes that reserve all
// of their device memory up front and treat any later allocation as a fault,
// and latency-critical callers for which the device-wide synchronization that
// cudaMalloc / cudaFree can imply is unacceptable.  For them the fp16 copy of
// the activations lives in this fixed array instead of the grown workspace.
// Every GPU that loads the library holds it until the process exits.  All
// calls on a device share it and each call overwrites the part it uses (so
// nothing needs clearing), which means calls that overlap on the GPU (e.g. on
// two streams) race on it.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;       // 8 MiB: m * ncols * 2 bytes at most
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
// row scales: ncols >= 64 bounds m by 8 MiB / 128 bytes
constexpr size_t kNoAllocMaxRows = kNoAllocScratchBytes / 128;
__device__ __align__(256) float g_noalloc_rscale[kNoAllocMaxRows];

struct NoAllocState {
    bool ready = false;
    void *scratch = nullptr;     // device address of g_noalloc_scratch on this device
    float *rscale = nullptr;     // device address of g_noalloc_rscale on this device
    CUtensorMap tmap;
    int tmap_m = -1, tmap_k = -1;
};
std::mutex g_noalloc_mutex;
NoAllocState g_noalloc[kMaxDev];

}  // namespace

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

qgemv_status launch_gemm_q4_0_noalloc(const void *W, const void *X, float *Y, int64_t nrows, int64_t ncols,
                                      int64_t m, cudaStream_t s, const DevInfo &di, int dev, unsigned *err) {
    if (dev < 0 || dev >= kMaxDev) {
        set_last_error("device ordinal %d out of range", dev);
        return QGEMV_ERR_CUDA;
    }
    const size_t need = static_cast<size_t>(m) * static_cast<size_t>(ncols) * 2;
    if (need > kNoAllocScratchBytes) {
        set_last_error("qgemm_q4_0_noalloc: m * ncols * 2 = %zu bytes exceeds its fixed %zu-byte scratch",
                       need, kNoAllocScratchBytes);
        return QGEMV_ERR_SHAPE;
    }
    constexpr size_t kSmem = gemm_smem<FMT_Q4_0>();
    if (kSmem > di.smem_optin) {
        set_last_error("prefill kernel needs %zu bytes of shared memory", kSmem);
        return QGEMV_ERR_ARCH;
    }
    std::lock_guard<std::mutex> lk(g_noalloc_mutex);
    NoAllocState &st = g_noalloc[dev];
    if (!st.ready) {
        // once per device, with that device current: the device address of
        // the fixed array (its host-side name is not a device address)
        void *addr = nullptr, *raddr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
        if (e == cudaSuccess) e = cudaGetSymbolAddress(&raddr, g_noalloc_rscale);
        if (e != cudaSuccess || addr == nullptr || raddr == nullptr) {
            set_last_error("cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
            return QGEMV_ERR_CUDA;
        }
        e = cudaFuncSetAttribute(gemm_tc_kernel<FMT_Q4_0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmem));
        if (e != cudaSuccess) {
            set_last_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            return QGEMV_ERR_CUDA;
        }
        st.scratch = addr;
        st.rscale = static_cast<float *>(raddr);
        st.ready = true;
    }
    if (st.tmap_m != m || st.tmap_k != ncols) {
        qgemv_status es = get_encoder();
        if (es != QGEMV_OK) return es;
        const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(ncols), static_cast<cuuint64_t>(m)};
        const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(ncols) * 2};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(kKC), static_cast<cuuint32_t>(kTok)};
        const cuuint32_t estride[2] = {1, 1};
        CUresult r = g_encode(&st.tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, st.scratch, gdim, gstride, box, estride,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            st.tmap_m = -1;
            set_last_error("cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
            return QGEMV_ERR_CUDA;
        }
        st.tmap_m = static_cast<int>(m);
        st.tmap_k = static_cast<int>(ncols);
    }

    const int64_t cblocks = m < static_cast<int64_t>(di.sm_count) * 4 ? m : static_cast<int64_t>(di.sm_count) * 4;
    x_rows_to_f16_kernel<<<static_cast<unsigned>(cblocks), kScaleThreads, 0, s>>>(
        static_cast<const uint4 *>(X), static_cast<uint4 *>(st.scratch), st.rscale, static_cast<int>(m),
        static_cast<int>(ncols));
    qgemv_status cs = check_launch("qgemm_q4_0_noalloc(activation conversion)");
    if (cs != QGEMV_OK) return cs;

    GemmParams p;
    p.W = static_cast<const uint8_t *>(W);
    p.Y = Y;
    p.rscale = st.rscale;
    p.err = err;
    p.nrows = static_cast<int>(nrows);
    p.ncols = static_cast<int>(ncols);
    p.m = static_cast<int>(m);
    p.mgroups = static_cast<int>((m + kTM * kTok - 1) / (kTM * kTok));
    p.nchunks = static_cast<int>(ncols / kKC);
    CUtensorMap wmap;
    cs = raw_path<FMT_Q4_0>(W, nrows, ncols, &wmap, &p.rawtma);
    if (cs != QGEMV_OK) return cs;
    const int64_t grid = ((nrows + kRowsW - 1) / kRowsW) * p.mgroups;
    if (grid > 0x7fffffff) {
        set_last_error("prefill grid too large");
        return QGEMV_ERR_SHAPE;
    }
    return launch_matmul<FMT_Q4_0>(grid, kSmem, s, st.tmap, wmap, p, "qgemm_q4_0_noalloc");
}

}  // namespace qg
