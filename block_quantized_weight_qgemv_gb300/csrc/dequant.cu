// dequant.cu -- standalone dequantization of Q4_0 / Q4_1 / Q8_0 blocks to
// fp32 or fp16 (the to-fp32 / to-fp16 converters of the "llama_cpp 0.12.1 ->
// 0.12.2" ggml-cuda.cu diff: dequantize_block_q4_0, dequantize_block_q4_1,
// dequantize_block_q8_0_f16).
//
// A pure HBM-bandwidth kernel: it reads 18/20/34 bytes and writes 64 (fp16)
// or 128 (fp32) bytes per 32-weight block.  The whole matrix is one flat run
// of blocks (rows are consecutive, ncols % 32 == 0), so the kernel works on
// "groups" of 32 consecutive blocks:
//   - a warp loads its group (576/640/1088 bytes, a multiple of 16) with
//     coalesced 16-byte loads into a private shared-memory buffer, while the
//     next group's loads are already in flight in registers;
//   - each lane then produces whole 16-byte output chunks so that every warp
//     store instruction writes 512 contiguous bytes (streaming stores, the
//     output does not fit in L2 at the sizes that matter).
// The arithmetic is the IEEE evaluation of the block formula, with no fused
// multiply-add: Q4_0 d*(q-8) (exact), Q4_1 fl(fl(d*q)+m), Q8_0 d*q (exact),
// and fp16 output = round-to-nearest-even of that fp32 value.
#include "qgemv_common.cuh"

namespace qg {
namespace {

constexpr int kWarps = 8;          // warps per CTA
constexpr int kGroup = 32;         // blocks per warp group

template <int F> struct Group {
    static constexpr int kBytes = kGroup * FmtInfo<F>::kBytes;      // 576 / 640 / 1088
    static constexpr int kVec = kBytes / 16;                         // 36 / 40 / 68
    static constexpr int kPerLane = (kVec + 31) / 32;                // 2 / 2 / 3
};

// Reads 4 bytes at an even shared-memory byte offset (two 16-bit loads).
__device__ __forceinline__ uint32_t lds_u32_at_even(const uint8_t *base, int off) {
    const uint16_t *p = reinterpret_cast<const uint16_t *>(base + off);
    return static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 16);
}

__device__ __forceinline__ uint32_t lds_u16(const uint8_t *base, int off) {
    return *reinterpret_cast<const uint16_t *>(base + off);
}

// Four consecutive weights [o, o+4) of block `blk` of the staged group (o a
// multiple of 4), as fp32.
template <int F>
__device__ __forceinline__ float4 dequant4(const uint8_t *g, int blk, int o) {
    constexpr int BB = FmtInfo<F>::kBytes;
    float4 r;
    if constexpr (F == FMT_Q8_0) {
        const float d = fp16_bits_to_f32(lds_u16(g, blk * BB));
        const uint32_t q4 = lds_u32_at_even(g, blk * BB + 2 + o);
        r.x = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(q4 & 0xff)));
        r.y = __fmul_rn(d, static_cast<float>(static_cast<int8_t>((q4 >> 8) & 0xff)));
        r.z = __fmul_rn(d, static_cast<float>(static_cast<int8_t>((q4 >> 16) & 0xff)));
        r.w = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(q4 >> 24)));
    } else {
        const int sh = (o & 16) ? 4 : 0;      // elements 16..31 are the high nibbles
        if constexpr (F == FMT_Q4_0) {
            const float d = fp16_bits_to_f32(lds_u16(g, blk * BB));
            const uint32_t q4 = lds_u32_at_even(g, blk * BB + 2 + (o & 15));
            r.x = __fmul_rn(d, static_cast<float>(static_cast<int>((q4 >> sh) & 15) - 8));
            r.y = __fmul_rn(d, static_cast<float>(static_cast<int>((q4 >> (8 + sh)) & 15) - 8));
            r.z = __fmul_rn(d, static_cast<float>(static_cast<int>((q4 >> (16 + sh)) & 15) - 8));
            r.w = __fmul_rn(d, static_cast<float>(static_cast<int>((q4 >> (24 + sh)) & 15) - 8));
        } else {
            const uint32_t dm = *reinterpret_cast<const uint32_t *>(g + blk * BB);
            const float d = fp16_bits_to_f32(dm);
            const float m = fp16_bits_to_f32(dm >> 16);
            const uint32_t q4 = *reinterpret_cast<const uint32_t *>(g + blk * BB + 4 + (o & 15));
            r.x = __fadd_rn(__fmul_rn(d, static_cast<float>((q4 >> sh) & 15)), m);
            r.y = __fadd_rn(__fmul_rn(d, static_cast<float>((q4 >> (8 + sh)) & 15)), m);
            r.z = __fadd_rn(__fmul_rn(d, static_cast<float>((q4 >> (16 + sh)) & 15)), m);
            r.w = __fadd_rn(__fmul_rn(d, static_cast<float>((q4 >> (24 + sh)) & 15)), m);
        }
    }
    return r;
}

__device__ __forceinline__ uint32_t pack_half2_rn(float a, float b) {
    const uint32_t lo = __half_as_ushort(__float2half_rn(a));
    const uint32_t hi = __half_as_ushort(__float2half_rn(b));
    return lo | (hi << 16);
}

// Writes the dequantized group (nblk <= 32 valid blocks staged in g) to out.
template <int F, bool F16>
__device__ __forceinline__ void emit_group(const uint8_t *g, int nblk, void *out, int64_t elem0, int lane) {
    if constexpr (!F16) {
        float4 *o4 = reinterpret_cast<float4 *>(static_cast<float *>(out) + elem0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {                       // 256 chunks of 4 floats
            const int c = i * 32 + lane;
            const int blk = c >> 3;
            if (blk < nblk) __stcs(o4 + c, dequant4<F>(g, blk, (c & 7) * 4));
        }
    } else {
        uint4 *o4 = reinterpret_cast<uint4 *>(static_cast<__half *>(out) + elem0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {                       // 128 chunks of 8 halves
            const int c = i * 32 + lane;
            const int blk = c >> 2;
            if (blk < nblk) {
                const int o = (c & 3) * 8;
                const float4 a = dequant4<F>(g, blk, o);
                const float4 b = dequant4<F>(g, blk, o + 4);
                uint4 v;
                v.x = pack_half2_rn(a.x, a.y);
                v.y = pack_half2_rn(a.z, a.w);
                v.z = pack_half2_rn(b.x, b.y);
                v.w = pack_half2_rn(b.z, b.w);
                __stcs(o4 + c, v);
            }
        }
    }
}

template <int F, bool F16>
__global__ void __launch_bounds__(kWarps * 32)
dequant_kernel(const uint8_t *__restrict__ W, void *__restrict__ out, int64_t nblocks) {
    using G = Group<F>;
    __shared__ __align__(16) uint8_t stage[kWarps][G::kBytes];
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    uint8_t *g = stage[wid];

    const int64_t nfull = nblocks / kGroup;                       // full groups
    const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kWarps + wid;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;

    const uint4 *src = reinterpret_cast<const uint4 *>(W);
    uint4 v[G::kPerLane];
    int64_t grp = warp0;
    if (grp < nfull) {
#pragma unroll
        for (int i = 0; i < G::kPerLane; ++i) {
            const int idx = i * 32 + lane;
            if (idx < G::kVec) v[i] = __ldcs(src + grp * G::kVec + idx);
        }
    }
    for (; grp < nfull; grp += nwarps) {
        // stage the current group, then put the next group's loads in flight
#pragma unroll
        for (int i = 0; i < G::kPerLane; ++i) {
            const int idx = i * 32 + lane;
            if (idx < G::kVec) reinterpret_cast<uint4 *>(g)[idx] = v[i];
        }
        const int64_t nxt = grp + nwarps;
        if (nxt < nfull) {
#pragma unroll
            for (int i = 0; i < G::kPerLane; ++i) {
                const int idx = i * 32 + lane;
                if (idx < G::kVec) v[i] = __ldcs(src + nxt * G::kVec + idx);
            }
        }
        __syncwarp();
        emit_group<F, F16>(g, kGroup, out, grp * kGroup * 32, lane);
        __syncwarp();
    }

    // ragged tail (< 32 blocks): the last warp of the grid stages it with
    // 16-bit loads (block sizes are even, W is 16-byte aligned)
    const int64_t tail = nblocks - nfull * kGroup;
    if (tail > 0 && warp0 == nwarps - 1) {
        const int nhalf = static_cast<int>(tail) * FmtInfo<F>::kBytes / 2;
        const uint16_t *s16 = reinterpret_cast<const uint16_t *>(W + nfull * G::kBytes);
        for (int i = lane; i < nhalf; i += 32) reinterpret_cast<uint16_t *>(g)[i] = s16[i];
        __syncwarp();
        emit_group<F, F16>(g, static_cast<int>(tail), out, nfull * kGroup * 32, lane);
    }
}

template <int F, bool F16>
qgemv_status launch_one(const void *W, void *out, int64_t nblocks, cudaStream_t s, const DevInfo &di) {
    const int64_t groups = (nblocks + kGroup - 1) / kGroup;
    int64_t ctas = (groups + kWarps - 1) / kWarps;
    const int64_t cap = static_cast<int64_t>(di.sm_count) * 8;   // 8 CTAs x 8 warps = 64 warps / SM
    if (ctas > cap) ctas = cap;
    if (ctas < 1) ctas = 1;
    dequant_kernel<F, F16><<<static_cast<unsigned>(ctas), kWarps * 32, 0, s>>>(
        static_cast<const uint8_t *>(W), out, nblocks);
    return check_launch("qdequant");
}

}  // namespace

qgemv_status launch_dequant(int fmt, const void *W, void *out, int64_t nrows, int64_t ncols,
                            int out_f16, cudaStream_t s, const DevInfo &di) {
    const int64_t nblocks = nrows * (ncols / 32);
    switch (fmt * 2 + (out_f16 ? 1 : 0)) {
    case FMT_Q4_0 * 2 + 0: return launch_one<FMT_Q4_0, false>(W, out, nblocks, s, di);
    case FMT_Q4_0 * 2 + 1: return launch_one<FMT_Q4_0, true>(W, out, nblocks, s, di);
    case FMT_Q4_1 * 2 + 0: return launch_one<FMT_Q4_1, false>(W, out, nblocks, s, di);
    case FMT_Q4_1 * 2 + 1: return launch_one<FMT_Q4_1, true>(W, out, nblocks, s, di);
    case FMT_Q8_0 * 2 + 0: return launch_one<FMT_Q8_0, false>(W, out, nblocks, s, di);
    case FMT_Q8_0 * 2 + 1: return launch_one<FMT_Q8_0, true>(W, out, nblocks, s, di);
    default:
        set_last_error("unknown format %d", fmt);
        return QGEMV_ERR_DTYPE;
    }
}

}  // namespace qg
