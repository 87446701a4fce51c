// gemv.cu -- decode / small-batch GEMV on block-quantized weights:
//   y[b][r] = sum_k w[r][k] * x[b][k]
// (the batch-1 fused dequantize + dot product named dequantize_mul_mat_vec in
// the "llama_cpp 0.12.1 -> 0.12.2" ggml-cuda.cu diff, extended to batch <= 8).
//
// Kernels (the tensor-core GEMV, the default where it applies, lives in
// gemv_sk.cu):
//
// 1. gemv_stream_kernel (rows whose byte length is a multiple of 16, i.e.
//    ncols/32 a multiple of 8 -- every shape that matters):
//    - one CTA per SM owns a balanced, contiguous range of rows;
//    - the CTA's rows are cut into chunks of up to 64 blocks; each warp owns
//      a contiguous run of chunks and streams them with 1-D bulk async copies
//      (TMA) into a private ring of shared-memory slots, each completed on its
//      own mbarrier (bounded waits; a timeout sets the error word);
//    - x is staged once per CTA in shared memory (its loads are issued before
//      the weight copies), in natural order, padded by 16 bytes per block pair
//      so the lanes' 16-byte loads hit distinct banks;
//    - each lane decodes one PAIR of blocks per chunk: a pair is 36 / 40 / 68
//      bytes at a 4-byte-aligned offset, read as aligned 32-bit words (the odd
//      half of an 18- or 34-byte pair is realigned with funnel shifts);
//    - a nibble becomes an exact float with the exponent trick
//      ((bits & mask) | 0x4b000000 == 2^23 + q * 2^s) and one packed FMA
//      removes the offset and the 2^s scale: (q - 8) (Q4_0), q (Q4_1) or
//      q (Q8_0, bytes via PRMT after a sign-bias xor); products accumulate with
//      packed fp32 FMAs (__ffma2_rn) over adjacent-element pairs, one partial
//      per block, then scaled by d
//      (Q4_1 adds m * sum(x of the block), precomputed during staging);
//    - per (row, warp) partial sums go to shared memory and are summed in a
//      fixed order (deterministic), then written to y.
// 2. gemv_rowwarp_kernel: one warp per row, plain decode + fp32 FMA; the
//    general path for any ncols % 32 == 0 (and batches the stream kernel does
//    not take).
#include <cstdlib>
#include <cstring>

#include "qgemv_common.cuh"

namespace qg {

// Process-wide launch option (qgemv_set_option): weights are never written by
// the kernel that precedes a GEMV on its stream.
int g_opt_weights_static = 0;

namespace {

// ============================================================ general path
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

// ============================================================ stream path
constexpr int kStreamWarps = 16;          // warps per CTA
constexpr int kMaxRowsPerCta = 128;       // bounds the partial-sum table
constexpr int kMaxStages = 16;

struct StreamParams {
    const uint8_t *W;
    const float *x;
    float *y;
    unsigned *err;
    int nrows;
    int ncols;
    int nb;               // blocks per row
    int nch;              // chunks per row
    int rows_per_cta_lo;  // balanced split: first `extra` CTAs get one more row
    int extra;
    int stages;           // ring slots per warp
    int x_floats;         // floats of staged x per batch (padded)
};

// x layout in shared memory: natural order, with 4 floats of padding after
// every pair of blocks (68 floats per 64).  Lane l reads the pair starting
// 272*l bytes in, so the 8 lanes of a quarter-warp hit 8 distinct 16-byte bank
// groups, and every load of a block is an immediate offset from one pointer.
__host__ __device__ __forceinline__ int xs_pair_off(int b_even) { return (b_even >> 1) * 68; }
__host__ __device__ __forceinline__ int xs_floats(int ncols) { return (ncols / 64) * 68 + ((ncols % 64) ? 68 : 0); }

// Shared-memory layout (dynamic):
//   xs    : NB * xs_floats(ncols) floats (natural order, padded per block pair)
//   sx    : NB * nb floats (sum of x over each block; Q4_1 only)
//   part  : kMaxRowsPerCta * kStreamWarps * NB floats (per row, per warp)
// A chunk (one ring slot) is 64*P blocks of one row: every lane decodes P
// block pairs per chunk, which amortizes the per-chunk bookkeeping.
//   bars  : kStreamWarps * stages mbarriers
//   ring  : kStreamWarps * stages * chunk_bytes
template <int F, int NB, int P>
struct StreamLayout {
    static constexpr int BB = FmtInfo<F>::kBytes;
    static constexpr int kChunkBlocks = 64 * P;
    static constexpr int kChunkBytes = kChunkBlocks * BB;
    __host__ __device__ static size_t xs_bytes(int ncols) { return size_t(NB) * xs_floats(ncols) * 4; }
    __host__ __device__ static size_t sx_bytes(int nb) { return F == FMT_Q4_1 ? ((size_t(NB) * nb * 4 + 15) & ~size_t(15)) : 0; }
    __host__ __device__ static size_t part_bytes() { return size_t(kMaxRowsPerCta) * kStreamWarps * NB * 4; }
    __host__ __device__ static size_t bar_bytes(int stages) { return ((size_t(kStreamWarps) * stages * 8 + 127) & ~size_t(127)); }
    __host__ __device__ static size_t ring_bytes(int stages) { return size_t(kStreamWarps) * stages * kChunkBytes; }
    __host__ __device__ static size_t total(int ncols, int nb, int stages) {
        return xs_bytes(ncols) + sx_bytes(nb) + part_bytes() + bar_bytes(stages) + ring_bytes(stages);
    }
};

// x staging, in rounds of kXRound float4 per thread: a round's loads are all
// issued before its stores, and the first round is issued before the weight
// copies so these loads do not queue behind the weight stream.
constexpr int kXRound = 10;

template <int NB>
struct XStager {
    float4 v[kXRound];
    int n4;        // float4 units per batch row of x (ncols / 4)

    __device__ __forceinline__ void load(const StreamParams &p, int round) {
        const int total = NB * n4;
#pragma unroll
        for (int k = 0; k < kXRound; ++k) {
            const int i = (round * kXRound + k) * blockDim.x + threadIdx.x;
            if (i < total) {
                const int bb = i / n4, g = i - bb * n4;
                v[k] = __ldg(reinterpret_cast<const float4 *>(p.x + size_t(bb) * p.ncols) + g);
            }
        }
    }
    __device__ __forceinline__ void store(const StreamParams &p, float *xs, int round) {
        const int total = NB * n4;
#pragma unroll
        for (int k = 0; k < kXRound; ++k) {
            const int i = (round * kXRound + k) * blockDim.x + threadIdx.x;
            if (i < total) {
                const int bb = i / n4, g = i - bb * n4;
                const int b = g >> 3;   // block, then 16-byte unit within it
                *reinterpret_cast<float4 *>(xs + size_t(bb) * p.x_floats + xs_pair_off(b & ~1) + (b & 1) * 32 + (g & 7) * 4) = v[k];
            }
        }
    }
    __device__ __forceinline__ int rounds() const {
        return (NB * n4 + kXRound * static_cast<int>(blockDim.x) - 1) / (kXRound * static_cast<int>(blockDim.x));
    }
};

// sum of x over each block (fixed order), from the staged copy (Q4_1 only)
template <int NB>
__device__ void block_sums(const StreamParams &p, const float *xs, float *sx) {
    for (int i = threadIdx.x; i < NB * p.nb; i += blockDim.x) {
        const int bb = i / p.nb, b = i - bb * p.nb;
        const float4 *xb = reinterpret_cast<const float4 *>(xs + size_t(bb) * p.x_floats);
        float s = 0.0f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float4 q = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(xb) + xs_pair_off(b & ~1) + (b & 1) * 32 + u * 4);
            s += q.x; s += q.y; s += q.z; s += q.w;
        }
        sx[i] = s;
    }
}


// Packed fp32 helpers on 64-bit register pairs (.x in the low half).
__device__ __forceinline__ uint64_t pk(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t pk_u32(uint32_t lo, uint32_t hi) {
    return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ float2 upk(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Constants of the decode, held in registers for the whole kernel.  They pass
// once through an empty asm statement, which makes them opaque to the
// compiler: it then keeps them live (the float pairs as aligned 64-bit
// registers) instead of re-materializing them before every use.
struct DecodeConsts {
    uint32_t magic;          // 0x4b000000 = bits of 2^23
    uint64_t magic2;         // {2^23, 2^23} bit patterns
    uint64_t sc[4], of[4];   // Q4: scale / offset pairs for v[0..3] below
    uint64_t of8;            // Q8_0: offset pair
};

template <int F>
__device__ __forceinline__ DecodeConsts make_consts() {
    constexpr float o = (F == FMT_Q4_0) ? 8.0f : 0.0f;
    DecodeConsts c;
    c.magic = 0x4b000000u;
    c.magic2 = 0x4b0000004b000000ull;
    c.sc[0] = pk(1.0f, 0x1p-8f);      c.of[0] = pk(-(0x1p23f + o), -(0x1p15f + o));   // s = 0, 8
    c.sc[1] = pk(0x1p-4f, 0x1p-12f);  c.of[1] = pk(-(0x1p19f + o), -(0x1p11f + o));   // s = 4, 12
    c.sc[2] = pk(0x1p-4f, 0x1p-12f);  c.of[2] = pk(-(0x1p19f + o), -(0x1p11f + o));   // s = 4, 12
    c.sc[3] = pk(0x1p-8f, 0x1p-16f);  c.of[3] = pk(-(0x1p15f + o), -(0x1p7f + o));    // s = 8, 16
    c.of8 = pk(-(0x1p23f + 128.0f), -(0x1p23f + 128.0f));
    asm volatile("" : "+l"(c.magic2));
    asm volatile("" : "+r"(c.magic));
#pragma unroll
    for (int i = 0; i < 4; ++i) asm volatile("" : "+l"(c.sc[i]), "+l"(c.of[i]));
    asm volatile("" : "+l"(c.of8));
    return c;
}

// Exact (q - OFF) for the 8 nibbles of a little-endian qs word E (bytes
// b0..b3, holding elements 4i+j (low nibble of bj) and 4i+j+16 (high nibble)
// when E is qs[4i..4i+3]), as four packed float pairs:
//   v[0] = (lo b0, lo b1)  v[1] = (lo b2, lo b3)  v[2] = (hi b0, hi b1)  v[3] = (hi b2, hi b3)
// so each pair multiplies two adjacent floats of x.  Each nibble is isolated in
// place and OR-ed into the exponent of 2^23, giving 2^23 + q * 2^s; one packed
// FMA multiplies by 2^-s and subtracts 2^(23-s) + OFF (exact: the result is a
// small integer; OFF is folded into c.of).
// One packed pair of the decode: lo = (a & MLO) | magic, hi = (a & MHI) | magic
// (three-input logic, truth table 0xEA), then fma.rn.f32x2 with the scale and
// offset pairs.  Kept in one asm block so the two halves are built in place.
template <uint32_t MLO, uint32_t MHI>
__device__ __forceinline__ uint64_t nib_pair(uint32_t a, uint32_t magic, uint64_t sc, uint64_t of) {
    uint64_t d;
    asm("{\n\t.reg .b32 lo, hi;\n\t.reg .b64 t;\n\t"
        "lop3.b32 lo, %1, %5, %2, 0xEA;\n\t"
        "lop3.b32 hi, %1, %6, %2, 0xEA;\n\t"
        "mov.b64 t, {lo, hi};\n\t"
        "fma.rn.f32x2 %0, t, %3, %4;\n\t}"
        : "=l"(d) : "r"(a), "r"(magic), "l"(sc), "l"(of), "n"(MLO), "n"(MHI));
    return d;
}

__device__ __forceinline__ void nibbles_to_f32(uint32_t E, uint64_t v[4], const DecodeConsts &c) {
    const uint32_t T = E >> 12;
    v[0] = nib_pair<0x0000000fu, 0x00000f00u>(E, c.magic, c.sc[0], c.of[0]);   // lo0 s0,  lo1 s8
    v[1] = nib_pair<0x000000f0u, 0x0000f000u>(T, c.magic, c.sc[1], c.of[1]);   // lo2 s4,  lo3 s12
    v[2] = nib_pair<0x000000f0u, 0x0000f000u>(E, c.magic, c.sc[2], c.of[2]);   // hi0 s4,  hi1 s12
    v[3] = nib_pair<0x00000f00u, 0x000f0000u>(T, c.magic, c.sc[3], c.of[3]);   // hi2 s8,  hi3 s16
}

// Exact signed bytes of a qs word as floats (Q8_0): bias to unsigned with an
// xor, put each byte under the exponent of 2^23 (64-bit masks on
// {U, U>>8} and {U>>16, U>>24}), subtract 2^23 + 128.
__device__ __forceinline__ void bytes_to_f32(uint32_t E, uint64_t v[2], const DecodeConsts &c) {
    const uint32_t U = E ^ 0x80808080u;
    const uint64_t A = pk_u32(U, U >> 8);
    const uint64_t B = pk_u32(U >> 16, U >> 24);
    v[0] = fadd2((A & 0x000000ff000000ffull) | c.magic2, c.of8);
    v[1] = fadd2((B & 0x000000ff000000ffull) | c.magic2, c.of8);
}

// sum over one Q4 block of (q - OFF) * x, given its 4 qs words; xb points at
// the block's staged x (8 float4 units).  Two accumulator chains.
__device__ __forceinline__ float q4_block_dot(const uint32_t qw[4], const uint64_t *xb, const DecodeConsts &c) {
    uint64_t accl = 0, acch = 0;                 // bit pattern of (+0.0f, +0.0f)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint64_t v[4];
        nibbles_to_f32(qw[i], v, c);
        // xb[2i], xb[2i+1]: x[4i .. 4i+3] (low nibbles); xb[8+2i], xb[9+2i]: x[16+4i ..] (high)
        accl = ffma2(v[0], xb[2 * i], accl);
        acch = ffma2(v[2], xb[8 + 2 * i], acch);
        accl = ffma2(v[1], xb[2 * i + 1], accl);
        acch = ffma2(v[3], xb[9 + 2 * i], acch);
    }
    const float2 t = upk(fadd2(accl, acch));
    return t.x + t.y;
}

__device__ __forceinline__ float q8_block_dot(const uint32_t qw[8], const uint64_t *xb, const DecodeConsts &c) {
    uint64_t acc0 = 0, acc1 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint64_t v[2];
        bytes_to_f32(qw[i], v, c);
        acc0 = ffma2(v[0], xb[2 * i], acc0);
        acc1 = ffma2(v[1], xb[2 * i + 1], acc1);
    }
    const float2 t = upk(fadd2(acc0, acc1));
    return t.x + t.y;
}

// One lane's contribution from block pair `pr` (blocks 2pr, 2pr+1 of the
// chunk) for all NB batches.  gb0 = global block index of the chunk's first
// block (a multiple of 64).
template <int F, int NB>
__device__ __forceinline__ void consume_pair(const uint8_t *slot, int pr, int gb0, const float *xs, int xstride,
                                             const float *sx, int nb, float acc[NB], const DecodeConsts &c) {
    const int be = gb0 + 2 * pr;                 // even block (global index)
    if constexpr (F == FMT_Q4_0) {
        const uint32_t *s = reinterpret_cast<const uint32_t *>(slot + 36 * pr);
        uint32_t w[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) w[i] = s[i];
        uint32_t qe[4], qo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) qe[i] = __funnelshift_r(w[i], w[i + 1], 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) qo[i] = w[5 + i];
        const float de = fp16_bits_to_f32(w[0]);
        const float dd = fp16_bits_to_f32(w[4] >> 16);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const uint64_t *xb = reinterpret_cast<const uint64_t *>(xs + size_t(b) * xstride + xs_pair_off(be));
            const float se = q4_block_dot(qe, xb, c);
            const float so = q4_block_dot(qo, xb + 16, c);
            acc[b] = fmaf(de, se, acc[b]);
            acc[b] = fmaf(dd, so, acc[b]);
        }
    } else if constexpr (F == FMT_Q4_1) {
        const uint32_t *s = reinterpret_cast<const uint32_t *>(slot + 40 * pr);
        uint32_t w[10];
#pragma unroll
        for (int i = 0; i < 10; ++i) w[i] = s[i];
        const float de = fp16_bits_to_f32(w[0]), me = fp16_bits_to_f32(w[0] >> 16);
        const float dd = fp16_bits_to_f32(w[5]), md = fp16_bits_to_f32(w[5] >> 16);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const uint64_t *xb = reinterpret_cast<const uint64_t *>(xs + size_t(b) * xstride + xs_pair_off(be));
            const float se = q4_block_dot(w + 1, xb, c);
            const float so = q4_block_dot(w + 6, xb + 16, c);
            acc[b] = fmaf(de, se, acc[b]);
            acc[b] = fmaf(me, sx[b * nb + be], acc[b]);
            acc[b] = fmaf(dd, so, acc[b]);
            acc[b] = fmaf(md, sx[b * nb + be + 1], acc[b]);
        }
    } else {
        const uint32_t *s = reinterpret_cast<const uint32_t *>(slot + 68 * pr);
        uint32_t w[17];
#pragma unroll
        for (int i = 0; i < 17; ++i) w[i] = s[i];
        uint32_t qe[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) qe[i] = __funnelshift_r(w[i], w[i + 1], 16);
        const float de = fp16_bits_to_f32(w[0]);
        const float dd = fp16_bits_to_f32(w[8] >> 16);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const uint64_t *xb = reinterpret_cast<const uint64_t *>(xs + size_t(b) * xstride + xs_pair_off(be));
            const float se = q8_block_dot(qe, xb, c);
            const float so = q8_block_dot(w + 9, xb + 16, c);
            acc[b] = fmaf(de, se, acc[b]);
            acc[b] = fmaf(dd, so, acc[b]);
        }
    }
}

template <int F, int NB, int P>
__global__ void __launch_bounds__(kStreamWarps * 32, 1)
gemv_stream_kernel(const StreamParams p) {
    using L = StreamLayout<F, NB, P>;
    constexpr int kChunkBlocks = L::kChunkBlocks;
    constexpr int BB = FmtInfo<F>::kBytes;
    extern __shared__ __align__(128) uint8_t smem[];
    float *xs = reinterpret_cast<float *>(smem);
    float *sx = reinterpret_cast<float *>(smem + L::xs_bytes(p.ncols));
    float *part = reinterpret_cast<float *>(smem + L::xs_bytes(p.ncols) + L::sx_bytes(p.nb));
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(part) + L::part_bytes());
    uint8_t *ring = reinterpret_cast<uint8_t *>(bars) + L::bar_bytes(p.stages);

    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int S = p.stages;

    // rows of this CTA
    const int cta = blockIdx.x;
    const int r0 = cta * p.rows_per_cta_lo + min(cta, p.extra);
    const int nrows_cta = p.rows_per_cta_lo + (cta < p.extra ? 1 : 0);
    const int units = nrows_cta * p.nch;
    const int u_begin = static_cast<int>((static_cast<int64_t>(units) * wid) / kStreamWarps);
    const int u_end = static_cast<int>((static_cast<int64_t>(units) * (wid + 1)) / kStreamWarps);
    const int my_units = u_end - u_begin;

    uint64_t *wbar = bars + wid * S;
    uint8_t *wring = ring + size_t(wid) * S * L::kChunkBytes;
    const int64_t rowbytes = static_cast<int64_t>(p.nb) * BB;

    // chunk cursor (row-local index, chunk within the row) for the copies
    int f_rl = u_begin / p.nch;
    int f_ch = u_begin - f_rl * p.nch;
    auto issue_next = [&](int slot) {
        const int nblk = min(kChunkBlocks, p.nb - f_ch * kChunkBlocks);
        const uint32_t bytes = static_cast<uint32_t>(nblk * BB);
        const uint8_t *src = p.W + static_cast<int64_t>(r0 + f_rl) * rowbytes + static_cast<int64_t>(f_ch) * L::kChunkBytes;
        mbar_arrive_expect_tx(&wbar[slot], bytes);
        bulk_g2s(wring + size_t(slot) * L::kChunkBytes, src, bytes, &wbar[slot]);
        if (++f_ch == p.nch) { f_ch = 0; ++f_rl; }
    };

    // ---- x loads first (round 0), then this warp's first weight chunks
    XStager<NB> xst;
    xst.n4 = p.ncols / 4;
    xst.load(p, 0);
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&wbar[s], 1);
        fence_mbar_init();
        const int n0 = min(S, my_units);
        for (int i = 0; i < n0; ++i) issue_next(i);
    }
    xst.store(p, xs, 0);
    for (int r = 1; r < xst.rounds(); ++r) {
        xst.load(p, r);
        xst.store(p, xs, r);
    }
    for (int i = threadIdx.x; i < nrows_cta * kStreamWarps * NB; i += blockDim.x) part[i] = 0.0f;
    if constexpr (F == FMT_Q4_1) {
        cta_sync();
        block_sums<NB>(p, xs, sx);
    }
    cta_sync();

    // ---- consume
    const DecodeConsts dc = make_consts<F>();
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
    bool ok = true;
    int i = 0;
    int slot = 0;
    uint32_t phase = 0;
    int rl = u_begin / p.nch;
    int ch = u_begin - rl * p.nch;
    for (; i < my_units; ++i) {
        const bool got = mbar_wait_bounded(&wbar[slot], phase, p.err);
        if (!__all_sync(0xffffffffu, got)) {     // warp-uniform decision
            ok = false;
            break;
        }
        const int nblk = min(kChunkBlocks, p.nb - ch * kChunkBlocks);
        const uint8_t *sl = wring + size_t(slot) * L::kChunkBytes;
#pragma unroll
        for (int q = 0; q < P; ++q) {
            const int pr = lane + 32 * q;
            if (2 * pr < nblk) consume_pair<F, NB>(sl, pr, ch * kChunkBlocks, xs, p.x_floats, sx, p.nb, acc, dc);
        }
        __syncwarp();
        // refill this slot with the chunk S ahead
        if (lane == 0 && i + S < my_units) {
            fence_proxy_async_smem();
            issue_next(slot);
        }
        // end of a row (or of this warp's run): reduce and park the partial
        if (ch == p.nch - 1 || i == my_units - 1) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float s = warp_sum(acc[b]);
                if (lane == 0) part[(rl * kStreamWarps + wid) * NB + b] = s;
                acc[b] = 0.0f;
            }
        }
        if (++slot == S) { slot = 0; phase ^= 1u; }
        if (++ch == p.nch) { ch = 0; ++rl; }
    }
    if (!ok) {
        // drain the copies still in flight into this warp's ring (bounded)
        for (int j = i; j < my_units && j < i + S; ++j) {
            mbar_wait_bounded(&wbar[slot], phase, p.err);
            if (++slot == S) { slot = 0; phase ^= 1u; }
        }
    }
    cta_sync();

    // ---- fixed-order sum of the per-warp partials of each row
    for (int t = threadIdx.x; t < nrows_cta * NB; t += blockDim.x) {
        const int rl = t / NB, b = t - rl * NB;
        float s = 0.0f;
#pragma unroll 4
        for (int w = 0; w < kStreamWarps; ++w) s += part[(rl * kStreamWarps + w) * NB + b];
        p.y[static_cast<int64_t>(b) * p.nrows + r0 + rl] = s;
    }
}

template <int F, int NB, int P>
qgemv_status launch_stream(const void *W, const float *x, float *y, int64_t nrows, int64_t ncols,
                           cudaStream_t s, const DevInfo &di, unsigned *err, bool *taken) {
    using L = StreamLayout<F, NB, P>;
    *taken = false;
    const int nb = static_cast<int>(ncols / 32);
    int ctas = di.sm_count;
    if (nrows < ctas) ctas = static_cast<int>(nrows);
    if (nrows > static_cast<int64_t>(ctas) * kMaxRowsPerCta) {
        ctas = static_cast<int>((nrows + kMaxRowsPerCta - 1) / kMaxRowsPerCta);
    }
    const size_t budget = di.smem_optin;
    const size_t fixed = L::total(static_cast<int>(ncols), nb, 0);
    if (fixed >= budget) return QGEMV_OK;                 // x does not fit: not taken
    int stages = static_cast<int>((budget - fixed - 128) / (size_t(kStreamWarps) * (L::kChunkBytes + 8)));
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return QGEMV_OK;                      // not taken
    const size_t smem = L::total(static_cast<int>(ncols), nb, stages);
    if (smem > budget) return QGEMV_OK;

    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemv_stream_kernel<F, NB, P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(budget));
        if (e != cudaSuccess) {
            set_last_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            return QGEMV_ERR_CUDA;
        }
        attr_set[dev] = true;
    }
    StreamParams p;
    p.W = static_cast<const uint8_t *>(W);
    p.x = x;
    p.y = y;
    p.err = err;
    p.nrows = static_cast<int>(nrows);
    p.ncols = static_cast<int>(ncols);
    p.nb = nb;
    p.nch = (nb + L::kChunkBlocks - 1) / L::kChunkBlocks;
    p.rows_per_cta_lo = static_cast<int>(nrows / ctas);
    p.extra = static_cast<int>(nrows % ctas);
    p.stages = stages;
    p.x_floats = xs_floats(static_cast<int>(ncols));
    *taken = true;
    gemv_stream_kernel<F, NB, P><<<ctas, kStreamWarps * 32, smem, s>>>(p);
    return check_launch("qgemv(stream)");
}

template <int F, int NB>
qgemv_status launch_rowwarp(const void *W, const float *x, float *y, int64_t nrows, int64_t ncols,
                            cudaStream_t s, const DevInfo &di) {
    int64_t ctas = (nrows + kRowWarps - 1) / kRowWarps;
    const int64_t cap = static_cast<int64_t>(di.sm_count) * 8;
    if (ctas > cap) ctas = cap;
    gemv_rowwarp_kernel<F, NB><<<static_cast<unsigned>(ctas), kRowWarps * 32, 0, s>>>(
        static_cast<const uint8_t *>(W), x, y, nrows, static_cast<int>(ncols));
    return check_launch("qgemv(rowwarp)");
}

// Kernel choice: QGEMV_GEMV_PATH=fx|sk|stream|rowwarp forces one (read once;
// the path tests use it; a kernel that cannot take a shape passes it on to
// the next).  By default every shape the stream-K tensor-core kernel takes
// (ncols a multiple of 1024) goes there, then the streamed CUDA-core kernel
// (batch <= 2, ncols a multiple of 256), and everything else to the general
// warp-per-row kernel.  The fixed-point dp4a kernel of gemv_int.cu (row
// bytes a multiple of 16, ncols of 64, batch columns in groups of up to
// four) is taken only when forced.
enum GemvPath { PATH_AUTO = 0, PATH_STREAM = 2, PATH_ROWWARP = 3, PATH_SK = 4, PATH_FX = 5 };

GemvPath gemv_path_override() {
    static int cached = -1;
    if (cached < 0) {
        const char *e = getenv("QGEMV_GEMV_PATH");
        int v = PATH_AUTO;
        if (e) {
            if (!strcmp(e, "fx")) v = PATH_FX;
            else if (!strcmp(e, "sk")) v = PATH_SK;
            else if (!strcmp(e, "stream")) v = PATH_STREAM;
            else if (!strcmp(e, "rowwarp")) v = PATH_ROWWARP;
        }
        cached = v;
    }
    return static_cast<GemvPath>(cached);
}

template <int F, int NB>
qgemv_status launch_nb(const void *W, const float *x, float *y, int64_t nrows, int64_t ncols,
                       cudaStream_t s, const DevInfo &di, int dev, unsigned *err) {
    const int nb = static_cast<int>(ncols / 32);
    const GemvPath forced = gemv_path_override();
    if (forced == PATH_FX) {
        bool taken = false;
        qgemv_status st = launch_gemv_fx(F, W, x, y, nrows, ncols, NB, s, di, dev, err, &taken);
        if (st != QGEMV_OK || taken) return st;
    }
    if (forced == PATH_AUTO || forced == PATH_SK || forced == PATH_FX) {
        bool taken = false;
        qgemv_status st = launch_gemv_sk(F, W, x, y, nrows, ncols, NB, s, di, err, &taken);
        if (st != QGEMV_OK || taken) return st;
    }
    if (NB <= 2 && nb % 8 == 0 && forced != PATH_ROWWARP) {
        // largest chunk (64*P blocks, no longer than the row) that leaves at
        // least two ring slots per warp
        constexpr int NBs = (NB <= 2 ? NB : 1);
        bool taken = false;
        qgemv_status st = QGEMV_OK;
        if (nb > 128) {
            st = launch_stream<F, NBs, 4>(W, x, y, nrows, ncols, s, di, err, &taken);
            if (st != QGEMV_OK || taken) return st;
        }
        if (nb > 64) {
            st = launch_stream<F, NBs, 2>(W, x, y, nrows, ncols, s, di, err, &taken);
            if (st != QGEMV_OK || taken) return st;
        }
        st = launch_stream<F, NBs, 1>(W, x, y, nrows, ncols, s, di, err, &taken);
        if (st != QGEMV_OK || taken) return st;
    }
    return launch_rowwarp<F, NB>(W, x, y, nrows, ncols, s, di);
}

template <int F>
qgemv_status launch_fmt(const void *W, const float *x, float *y, int64_t nrows, int64_t ncols, int batch,
                        cudaStream_t s, const DevInfo &di, int dev, unsigned *err) {
    switch (batch) {
    case 1: return launch_nb<F, 1>(W, x, y, nrows, ncols, s, di, dev, err);
    case 2: return launch_nb<F, 2>(W, x, y, nrows, ncols, s, di, dev, err);
    case 3: return launch_nb<F, 3>(W, x, y, nrows, ncols, s, di, dev, err);
    case 4: return launch_nb<F, 4>(W, x, y, nrows, ncols, s, di, dev, err);
    case 5: return launch_nb<F, 5>(W, x, y, nrows, ncols, s, di, dev, err);
    case 6: return launch_nb<F, 6>(W, x, y, nrows, ncols, s, di, dev, err);
    case 7: return launch_nb<F, 7>(W, x, y, nrows, ncols, s, di, dev, err);
    default: return launch_nb<F, 8>(W, x, y, nrows, ncols, s, di, dev, err);
    }
}

}  // namespace

qgemv_status launch_gemv(int fmt, const void *W, const float *x, float *y, int64_t nrows,
                         int64_t ncols, int batch, cudaStream_t s, const DevInfo &di, int dev, unsigned *err) {
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
    case FMT_Q4_0: return launch_fmt<FMT_Q4_0>(W, x, y, nrows, ncols, batch, s, di, dev, err);
    case FMT_Q4_1: return launch_fmt<FMT_Q4_1>(W, x, y, nrows, ncols, batch, s, di, dev, err);
    case FMT_Q8_0: return launch_fmt<FMT_Q8_0>(W, x, y, nrows, ncols, batch, s, di, dev, err);
    default:
        set_last_error("unknown format %d", fmt);
        return QGEMV_ERR_DTYPE;
    }
}

}  // namespace qg
