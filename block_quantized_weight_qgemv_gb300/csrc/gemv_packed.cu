// gemv_packed.cu -- Q4_0 GEMV on weights rearranged once into MMA fragment
// order ("packed"), and the kernel that rearranges them.
//
// The arithmetic is that of the block-quantized GEMV (Q4_0 blocks as in the
// dequantize_block_q4_0 hunk of the "llama_cpp 0.12.1 -> 0.12.2" ggml-cuda.cu
// diff: w = d * (q - 8), low nibble -> element j, high nibble -> element
// j + 16; y[b][r] = sum_k w[r][k] x[b][k]).  Only the byte order in memory
// differs: the same 18 bytes per block, grouped so that one warp streams a
// 16-row x 2-block group with one coalesced 16-byte load per lane, straight
// into the registers that feed mma.sync -- no shared-memory copy of the
// weights at all.
//
// Packed layout (see qgemv.h): tiles of 16 rows (the last one zero-padded),
// each row of a tile cut into ncols/64 block pairs; record (tile t, pair p)
// is 576 bytes at offset (t * npairs + p) * 576:
//   bytes [16 l, 16 l + 16), lane l = 4 g + c (g = 0..7, c = 0..3):
//       qs[16t+g][2p][4c..4c+3], qs[16t+g+8][2p][4c..4c+3],
//       qs[16t+g][2p+1][4c..4c+3], qs[16t+g+8][2p+1][4c..4c+3]
//   bytes [512 + 8 g, 512 + 8 g + 8):
//       d[16t+g][2p], d[16t+g+8][2p], d[16t+g][2p+1], d[16t+g+8][2p+1]
// (qs[r][b] = the 16 nibble bytes of block b of row r, d its fp16 scale).
//
// GEMV kernel: a CTA of 8 warps takes whole tiles (persistent over tiles,
// two CTAs per SM); warp w takes a contiguous range of the block pairs of
// every tile and stages the fp16 x operands of that range once (scaled per 8
// blocks by a power of two).  Its records of one tile are
// contiguous, so it streams them in chunks of 4 records through a small ring
// of its own in shared memory, one bulk copy per chunk completing on the
// slot's mbarrier.  Per record each lane reads its 16 bytes, decodes them
// into A fragments with one logic instruction per two weights (fp16 1024 + q
// and 1024 + 16 q) and runs 4 mma.sync m16n8k16 whose accumulators start at
// -T (the offset terms).
// Per-warp tile partials are summed in a fixed order: deterministic.
#include <cstdlib>
#include <cstring>

#include <algorithm>
#include <type_traits>

#include "qgemv_common.cuh"

namespace qg {
namespace {

#ifndef QG_PK_WARPS
#define QG_PK_WARPS 8
#endif
constexpr int kPkWarps = QG_PK_WARPS;
constexpr int kPkThreads = kPkWarps * 32;
constexpr int kRecBytes = 576;
constexpr int kGroup = 4;                   // pairs per x scale round
#ifndef QG_PK_RING
#define QG_PK_RING 2
#endif
#ifndef QG_PK_CTAS_PER_SM
#define QG_PK_CTAS_PER_SM 2
#endif
constexpr int kRing = QG_PK_RING;           // chunk slots per warp
constexpr int kCtasPerSm = QG_PK_CTAS_PER_SM;
constexpr int kPkMinBlocks = 16 / kPkWarps; // register cap: two 8-warp CTAs per SM
constexpr int kStageRounds = 8;             // x rounds loaded at once while staging
constexpr uint32_t kChunkBytes = kGroup * kRecBytes;

// ------------------------------------------------------------------ packing
// One thread per (tile, pair, lane) 16-byte piece; the lanes with c == 0 (one
// per row pair g) also write the 8-byte scale pieces.  Rows past nrows are zero.
__global__ void pack_q4_0_kernel(const uint8_t *__restrict__ W, uint8_t *__restrict__ Wp, int64_t nrows, int nb,
                                 int64_t ntiles) {
    const int npairs = nb / 2;
    const int64_t nunits = ntiles * npairs * 32;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nunits;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int l = static_cast<int>(i & 31);
        const int64_t tp = i >> 5;                 // tile * npairs + pair
        const int64_t t = tp / npairs;
        const int p = static_cast<int>(tp - t * npairs);
        const int g = l >> 2, c = l & 3;
        uint32_t w[4];
        uint16_t d[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t r = t * 16 + g + ((q & 1) ? 8 : 0);
            const int b = 2 * p + (q >> 1);
            if (r < nrows) {
                const uint8_t *blk = W + (r * nb + b) * 18;
                w[q] = static_cast<uint32_t>(blk[2 + 4 * c]) | (static_cast<uint32_t>(blk[3 + 4 * c]) << 8) |
                       (static_cast<uint32_t>(blk[4 + 4 * c]) << 16) | (static_cast<uint32_t>(blk[5 + 4 * c]) << 24);
                d[q] = static_cast<uint16_t>(blk[0] | (blk[1] << 8));
            } else {
                w[q] = 0u;
                d[q] = 0u;
            }
        }
        uint8_t *rec = Wp + tp * kRecBytes;
        *reinterpret_cast<uint4 *>(rec + 16 * l) = make_uint4(w[0], w[1], w[2], w[3]);
        if (c == 0) {
            *reinterpret_cast<uint2 *>(rec + 512 + 8 * g) =
                make_uint2(static_cast<uint32_t>(d[0]) | (static_cast<uint32_t>(d[1]) << 16),
                           static_cast<uint32_t>(d[2]) | (static_cast<uint32_t>(d[3]) << 16));
        }
    }
}

// ------------------------------------------------------------ device helpers
template <uint32_t MASK>
__device__ __forceinline__ uint32_t pk_and_or(uint32_t a, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
    return d;
}
__device__ __forceinline__ void pk_mma(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void pk_mma_c(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1, const float4 &cq) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(cq.x), "f"(cq.y), "f"(cq.z),
          "f"(cq.w));
}
// both fp16 halves of a word to f32 (low half -> .x)
__device__ __forceinline__ float2 pk_h2f2(uint32_t w) {
    __half2 h;
    memcpy(&h, &w, sizeof(h));
    return __half22float2(h);
}
__device__ __forceinline__ uint32_t pk_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float pk_rsum(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu))) +
           __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}
// 2^e with m * 2^e in [2^9, 2^10) from the bits of m = max|x|
__device__ __forceinline__ int pk_exponent(uint32_t mbits) {
    const int be = static_cast<int>(mbits >> 23);
    if (be == 255 || mbits == 0u) return 0;
    return be == 0 ? 120 : 136 - be;
}
__device__ __forceinline__ float pk_pow2(int e) { return __int_as_float((127 + e) << 23); }
struct PkParams {
    const uint8_t *Wp;
    const float *x;
    float *y;
    int nrows, ncols, batch;
    int ntiles, npairs;
    int ring;             // chunk slots per warp (2..kRing)
    int early;            // first weight copies before waiting on the preceding kernel
    unsigned *err;        // device error word (wait timeouts)
};

// Shared memory: per warp, its ring of chunk slots and their mbarriers; per
// warp, for each of its blocks (round r of 4 pairs = 8 blocks) and batch
// column n: the lane-c B fragment (uint4 [c]), the accumulator start quads
// (one per block for batch 1, one per (block, lane c) otherwise), the scalar
// -T, and per (round, column) 2^-e; then the per-warp tile partials,
// double-buffered by tile parity.
struct PkLayout {
    uint32_t ring, bars, xf, nq, nt, us, part, total;
    uint32_t warp_rounds;      // rounds per warp (of the largest range)
};

__host__ __device__ inline PkLayout pk_layout(int npairs, int batch, int ring) {
    PkLayout L;
    const int maxp = (npairs + kPkWarps - 1) / kPkWarps;
    L.warp_rounds = static_cast<uint32_t>((maxp + kGroup - 1) / kGroup);
    const uint32_t items = L.warp_rounds * 8 * batch;      // per warp
    uint32_t o = 0;
    L.ring = o; o += kPkWarps * ring * kChunkBytes;
    L.bars = o; o += kPkWarps * ring * 8;
    L.xf = o; o += kPkWarps * items * 64;
    L.nq = o; o += kPkWarps * L.warp_rounds * 8 * (batch == 1 ? 16 : 64);
    L.nt = o; o += kPkWarps * items * 4;
    L.us = o; o += kPkWarps * L.warp_rounds * batch * 4;
    L.part = o; o += 2 * kPkWarps * 16 * batch * 4;
    L.total = o;
    return L;
}

__device__ __forceinline__ void pk_bar_sync() { asm volatile("bar.sync 1, %0;" :: "n"(kPkThreads) : "memory"); }
__device__ __forceinline__ uint4 lds16(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }
__device__ __forceinline__ uint2 lds8(const uint8_t *p) { return *reinterpret_cast<const uint2 *>(p); }

// ------------------------------------------------------------------ kernel
// Each warp streams the records of its pair range [p0, p0 + np) of every tile
// of its CTA (tiles blockIdx.x, + gridDim.x, ...) in chunks of up to 4
// records (one x scale round; a chunk never crosses a tile), through a ring
// of p.ring chunk slots of its own: lane 0 fills a slot with one bulk copy
// completing on the slot's mbarrier, and refills it as soon as the warp has
// read the chunk in it.
template <bool B1>
__global__ void __launch_bounds__(kPkThreads, kPkMinBlocks)
gemv_packed_q4_0_kernel(const PkParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int batch = B1 ? 1 : p.batch;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const PkLayout L = pk_layout(p.npairs, p.batch, p.ring);
    const int nring = p.ring;
    // this warp's pairs: [p0, p0 + np) of every tile
    const int base = p.npairs / kPkWarps, extra = p.npairs % kPkWarps;
    const int np = base + (wid < extra ? 1 : 0);
    const int p0 = wid * base + min(wid, extra);
    const int nrounds = (np + kGroup - 1) / kGroup;
    const uint32_t witems = L.warp_rounds * 8 * p.batch;
    const int t0 = blockIdx.x, tstep = gridDim.x;
    const int ntl = t0 < p.ntiles ? (p.ntiles - 1 - t0) / tstep + 1 : 0;    // tiles of this CTA
    const int nch = ntl * nrounds;                                          // chunks of this warp

    uint8_t *ring = smem + L.ring + wid * nring * kChunkBytes;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L.bars) + wid * nring;
    if (lane == 0) {
        for (int s = 0; s < nring; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    // ---- chunk issue (lane 0): chunk ni = (tile ik, round ir) into slot is
    int ni = 0, ik = 0, ir = 0, is = 0;
    auto issue = [&]() {
        const int cnt = min(kGroup, np - kGroup * ir);
        const uint32_t bytes = static_cast<uint32_t>(cnt * kRecBytes);
        const uint8_t *src =
            p.Wp + (static_cast<int64_t>(t0 + ik * tstep) * p.npairs + p0 + kGroup * ir) * kRecBytes;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bar[is], bytes);
        bulk_g2s(ring + is * kChunkBytes, src, bytes, &bar[is]);
        if (++ir == nrounds) {
            ir = 0;
            ++ik;
        }
        if (++is == nring) is = 0;
        ++ni;
    };
    if (p.early && lane == 0) {
        while (ni < nch && ni < nring) issue();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!p.early && lane == 0) {
        while (ni < nch && ni < nring) issue();
    }

    // ---- stage x for this warp's blocks [2 p0, 2 (p0 + np)): lane l builds
    // fragment c of block l / 4 of each 8-block round (aligned column map:
    // low nibbles x[4c..4c+3], high nibbles x[16+4c..] / 16), scaled per
    // (round, column) by a power of two; -T per block (the offset term the
    // accumulator starts from: 1032 * sum of the rounded low-slot x + 1152 *
    // sum of the rounded high-slot x / 16)
    uint4 *xf = reinterpret_cast<uint4 *>(smem + L.xf) + wid * witems * 4;
    float *ntp = reinterpret_cast<float *>(smem + L.nt) + wid * witems;
    // batch 1: one start quad per block; else one per (block, lane c)
    float4 *ntq = reinterpret_cast<float4 *>(smem + L.nq) + wid * L.warp_rounds * 8 * (B1 ? 1 : 4);
    float *usp = reinterpret_cast<float *>(smem + L.us) + wid * L.warp_rounds * p.batch;
    const int bl = lane >> 2;
    // x[blk * 32 + 4c .. + 3] and x[blk * 32 + 16 + 4c .. + 3] of column n
    // for block bl of round r (zero past the warp's blocks)
    auto xload = [&](int r, int n, float4 &lo, float4 &hi) {
        const int blk = r * 8 + bl;
        if (r < nrounds && blk < 2 * np) {
            const float *xb = p.x + static_cast<size_t>(n) * p.ncols + static_cast<size_t>(2 * p0 + blk) * 32;
            lo = __ldg(reinterpret_cast<const float4 *>(xb + 4 * c));
            hi = __ldg(reinterpret_cast<const float4 *>(xb + 16 + 4 * c));
        } else {
            lo = hi = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
    };
    // round r, column n: scale, fp16 fragments and -T of block bl (stored
    // only for the warp's rounds; the arithmetic runs unconditionally so that
    // the rounds of a group interleave)
    auto stage_round = [&](int r, int n, const float4 &lo, const float4 &hi) {
        const float m = fmaxf(fmaxf(fmaxf(fabsf(lo.x), fabsf(lo.y)), fmaxf(fabsf(lo.z), fabsf(lo.w))),
                              fmaxf(fmaxf(fabsf(hi.x), fabsf(hi.y)), fmaxf(fabsf(hi.z), fabsf(hi.w))));
        const int e = pk_exponent(__reduce_max_sync(0xffffffffu, __float_as_uint(m)));
        const bool keep = r < nrounds;
        if (keep && lane == 0) usp[r * p.batch + n] = pk_pow2(-e);
        const float sc = pk_pow2(e), sh = sc * 0.0625f;
        const uint32_t w0 = pk_f16x2(lo.x * sc, lo.z * sc);
        const uint32_t w1 = pk_f16x2(lo.y * sc, lo.w * sc);
        const uint32_t w2 = pk_f16x2(hi.x * sh, hi.z * sh);
        const uint32_t w3 = pk_f16x2(hi.y * sh, hi.w * sh);
        float slo = pk_rsum(w0) + pk_rsum(w1), shi = pk_rsum(w2) + pk_rsum(w3);
        slo += __shfl_xor_sync(0xffffffffu, slo, 1);
        shi += __shfl_xor_sync(0xffffffffu, shi, 1);
        slo += __shfl_xor_sync(0xffffffffu, slo, 2);
        shi += __shfl_xor_sync(0xffffffffu, shi, 2);
        const int item = (r * 8 + bl) * p.batch + n;
        const float nt = -fmaf(1032.0f, slo, 1152.0f * shi);
        if (keep) {
            xf[item * 4 + c] = make_uint4(w0, w1, w2, w3);
            if constexpr (B1) {
                if (c == 0) ntq[r * 8 + bl] = make_float4(nt, nt, nt, nt);
            } else if (c == 0) {
                ntp[item] = nt;
            }
        }
    };
    {
        // groups of G rounds: all their loads first, then G independent conversions
        auto stage_all = [&](auto group) {
            constexpr int G = decltype(group)::value;
            for (int n = 0; n < p.batch; ++n) {
                for (int r0 = 0; r0 < nrounds; r0 += G) {
                    float4 lo[G], hi[G];
#pragma unroll
                    for (int i = 0; i < G; ++i) xload(r0 + i, n, lo[i], hi[i]);
#pragma unroll
                    for (int i = 0; i < G; ++i) stage_round(r0 + i, n, lo[i], hi[i]);
                }
            }
        };
        if (nrounds <= 2) stage_all(std::integral_constant<int, 2>{});
        else if (nrounds <= 4) stage_all(std::integral_constant<int, 4>{});
        else stage_all(std::integral_constant<int, kStageRounds>{});
        __syncwarp();
        if constexpr (!B1) {
            // accumulator starts of lane c: {-T[n0], -T[n1], -T[n0], -T[n1]} per block
            const int m0 = min(2 * c, p.batch - 1), m1 = min(2 * c + 1, p.batch - 1);
            for (int blk = bl; blk < 2 * np; blk += 8) {
                const float ta = ntp[blk * p.batch + m0], tb = ntp[blk * p.batch + m1];
                ntq[blk * 4 + c] = make_float4(ta, tb, ta, tb);
            }
            __syncwarp();
        }
    }

    // ---- the stream: decode each lane's 16 bytes into A fragments, 4 MMAs
    // per pair from -T, scale by d; fold per 4-pair round by 2^-e
    constexpr uint32_t kMagic = 0x64006400u;      // fp16 (1024, 1024)
    const int ncol = min(g, batch - 1);          // B columns past the batch repeat the last one
    const int n0 = min(2 * c, batch - 1), n1 = min(2 * c + 1, batch - 1);
    const uint4 *fb0 = xf + ncol * 4 + c;
    const float4 *fq0 = ntq + (B1 ? 0 : c);
    constexpr int qstep = B1 ? 1 : 4;
    float *part = reinterpret_cast<float *>(smem + L.part);

    auto compute_pair = [&](const uint4 q, const uint2 d, int blk, float ak[4]) {
        const uint32_t q0 = q.x, q1 = q.y, q2 = q.z, q3 = q.w;
        const uint32_t q0s = q0 >> 8, q1s = q1 >> 8, q2s = q2 >> 8, q3s = q3 >> 8;
        uint32_t e0[4], e1[4], o0[4], o1[4];
        e0[0] = pk_and_or<0x000f000fu>(q0, kMagic); e0[1] = pk_and_or<0x000f000fu>(q1, kMagic);
        e0[2] = pk_and_or<0x000f000fu>(q0s, kMagic); e0[3] = pk_and_or<0x000f000fu>(q1s, kMagic);
        e1[0] = pk_and_or<0x00f000f0u>(q0, kMagic); e1[1] = pk_and_or<0x00f000f0u>(q1, kMagic);
        e1[2] = pk_and_or<0x00f000f0u>(q0s, kMagic); e1[3] = pk_and_or<0x00f000f0u>(q1s, kMagic);
        o0[0] = pk_and_or<0x000f000fu>(q2, kMagic); o0[1] = pk_and_or<0x000f000fu>(q3, kMagic);
        o0[2] = pk_and_or<0x000f000fu>(q2s, kMagic); o0[3] = pk_and_or<0x000f000fu>(q3s, kMagic);
        o1[0] = pk_and_or<0x00f000f0u>(q2, kMagic); o1[1] = pk_and_or<0x00f000f0u>(q3, kMagic);
        o1[2] = pk_and_or<0x00f000f0u>(q2s, kMagic); o1[3] = pk_and_or<0x00f000f0u>(q3s, kMagic);
        const uint4 be = fb0[(blk * batch) * 4], bo = fb0[((blk + 1) * batch) * 4];
        const float4 qe = fq0[blk * qstep], qo = fq0[(blk + 1) * qstep];
        float ce[4], co[4];
        pk_mma_c(ce, e0, be.x, be.y, qe);
        pk_mma_c(co, o0, bo.x, bo.y, qo);
        pk_mma(ce, e1, be.z, be.w);
        pk_mma(co, o1, bo.z, bo.w);
        const float2 de = pk_h2f2(d.x), dd = pk_h2f2(d.y);
        const float de0 = de.x, de1 = de.y, do0 = dd.x, do1 = dd.y;
        ak[0] = fmaf(de0, ce[0], ak[0]);
        ak[2] = fmaf(de1, ce[2], ak[2]);
        ak[0] = fmaf(do0, co[0], ak[0]);
        ak[2] = fmaf(do1, co[2], ak[2]);
        if constexpr (!B1) {
            ak[1] = fmaf(de0, ce[1], ak[1]);
            ak[3] = fmaf(de1, ce[3], ak[3]);
            ak[1] = fmaf(do0, co[1], ak[1]);
            ak[3] = fmaf(do1, co[3], ak[3]);
        }
    };
    // tile k of the CTA done: fixed-order sum of the warp partials
    auto tile_end = [&](int k, const float acc[4]) {
        float *pb = part + (k & 1) * kPkWarps * 16 * batch;
        float *pw = pb + wid * 16 * batch;
        if (2 * c < batch) {
            pw[g * batch + 2 * c] = acc[0];
            pw[(g + 8) * batch + 2 * c] = acc[2];
        }
        if (2 * c + 1 < batch) {
            pw[g * batch + 2 * c + 1] = acc[1];
            pw[(g + 8) * batch + 2 * c + 1] = acc[3];
        }
        pk_bar_sync();
        if (tid < 16 * batch) {
            const int rr = tid / batch, n = tid - rr * batch;
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < kPkWarps; ++w) sum += pb[(w * 16 + rr) * batch + n];
            const int row = (t0 + k * tstep) * 16 + rr;
            if (row < p.nrows) p.y[static_cast<int64_t>(n) * p.nrows + row] = sum;
        }
    };

    // ---- consume the chunks in order: chunk ci sits in slot ci % p.ring,
    // phase (ci / p.ring) & 1.  Every warp (also one without pairs, or one
    // whose wait gave up) reaches tile_end exactly once per tile of the CTA.
    bool aborted = false;
    int cs = 0;
    uint32_t cph = 0;
    for (int k = 0; k < ntl; ++k) {
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int r = 0; r < nrounds; ++r) {
            if (!aborted) {
                const bool ok = __all_sync(0xffffffffu, mbar_wait_sleep(&bar[cs], cph, p.err));
                aborted = !ok;
            }
            if (!aborted) {
                const uint8_t *ch = ring + cs * kChunkBytes + 16 * lane;
                const int dof = 512 + 8 * g - 16 * lane;
                float ak[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                const int blk0 = 2 * kGroup * r;
                if (kGroup * r + kGroup <= np) {
#pragma unroll
                    for (int i = 0; i < kGroup; ++i) {
                        compute_pair(lds16(ch + i * kRecBytes), lds8(ch + i * kRecBytes + dof), blk0 + 2 * i, ak);
                    }
                } else {
                    for (int i = 0; i < np - kGroup * r; ++i) {
                        compute_pair(lds16(ch + i * kRecBytes), lds8(ch + i * kRecBytes + dof), blk0 + 2 * i, ak);
                    }
                }
                const float u0 = usp[r * batch + n0];
                acc[0] = fmaf(ak[0], u0, acc[0]);
                acc[2] = fmaf(ak[2], u0, acc[2]);
                if constexpr (!B1) {
                    const float u1 = usp[r * batch + n1];
                    acc[1] = fmaf(ak[1], u1, acc[1]);
                    acc[3] = fmaf(ak[3], u1, acc[3]);
                }
                __syncwarp();
                if (lane == 0 && ni < nch) issue();      // the slot just read is the next to fill
            }
            if (++cs == nring) {
                cs = 0;
                cph ^= 1u;
            }
        }
        tile_end(k, acc);
    }
    if (aborted && lane == 0) {
        // a wait gave up: let this warp's copies still in flight land before exiting
        for (int ci = ni - nring < 0 ? 0 : ni - nring; ci < ni; ++ci)
            mbar_wait_bounded(&bar[ci % nring], static_cast<uint32_t>(ci / nring) & 1u, p.err);
    }
}

template <bool B1>
qgemv_status launch_packed_b(const void *Wp, const float *x, float *y, int64_t nrows, int64_t ncols, int batch,
                             cudaStream_t s, const DevInfo &di, unsigned *err) {
    auto kern = gemv_packed_q4_0_kernel<B1>;
    const int npairs = static_cast<int>(ncols / 64);
    int ring = kRing;                           // deepest ring that fits
    while (ring > 2 && pk_layout(npairs, batch, ring).total > di.smem_optin) --ring;
    const PkLayout L = pk_layout(npairs, batch, ring);
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(di.smem_optin));
        if (e != cudaSuccess) {
            set_last_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            return QGEMV_ERR_CUDA;
        }
        attr_set[dev] = true;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kPkThreads, L.total) != cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        set_last_error("packed GEMV: no CTA fits (%u bytes of shared memory)", L.total);
        return QGEMV_ERR_LAUNCH;
    }
    PkParams p;
    p.Wp = static_cast<const uint8_t *>(Wp);
    p.x = x;
    p.y = y;
    p.nrows = static_cast<int>(nrows);
    p.ncols = static_cast<int>(ncols);
    p.batch = batch;
    p.ntiles = static_cast<int>((nrows + 15) / 16);
    p.npairs = npairs;
    p.ring = ring;
    p.early = g_opt_weights_static;
    p.err = err;
    // kCtasPerSm CTAs per SM at most (persistent over the remaining tiles)
    const int grid = static_cast<int>(std::min<int64_t>(p.ntiles, static_cast<int64_t>(std::min(per_sm, kCtasPerSm)) * di.sm_count));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kPkThreads);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e != cudaSuccess) {
        set_last_error("qgemv_packed launch: %s", cudaGetErrorString(e));
        return QGEMV_ERR_LAUNCH;
    }
    return check_launch("qgemv_packed");
}

}  // namespace

int64_t packed_bytes_q4_0(int64_t nrows, int64_t ncols) { return (nrows + 15) / 16 * 16 * (ncols / 32) * 18; }

qgemv_status launch_pack_q4_0(const void *W, void *Wp, int64_t nrows, int64_t ncols, cudaStream_t s,
                              const DevInfo &di) {
    const int nb = static_cast<int>(ncols / 32);
    const int64_t ntiles = (nrows + 15) / 16;
    const int64_t units = ntiles * (nb / 2) * 32;
    const int64_t blocks = std::min<int64_t>((units + 255) / 256, static_cast<int64_t>(di.sm_count) * 16);
    pack_q4_0_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<const uint8_t *>(W),
                                                                    static_cast<uint8_t *>(Wp), nrows, nb, ntiles);
    return check_launch("qgemv_pack_q4_0");
}

qgemv_status launch_gemv_packed_q4_0(const void *Wp, const float *x, float *y, int64_t nrows, int64_t ncols,
                                     int batch, cudaStream_t s, const DevInfo &di, unsigned *err) {
    // batch columns per launch: as many as keep the staged x within the cap
    const int npairs = static_cast<int>(ncols / 64);
    int per = batch;
    while (per > 1 && pk_layout(npairs, per, 2).total > di.smem_optin) --per;
    if (pk_layout(npairs, per, 2).total > di.smem_optin) {
        set_last_error("packed GEMV: ncols=%lld needs more shared memory than one CTA has", (long long)ncols);
        return QGEMV_ERR_SHAPE;
    }
    qgemv_status st = QGEMV_OK;
    for (int n0 = 0; n0 < batch; n0 += per) {
        const int nb = std::min(per, batch - n0);
        const float *xs = x + static_cast<int64_t>(n0) * ncols;
        float *ys = y + static_cast<int64_t>(n0) * nrows;
        st = nb == 1 ? launch_packed_b<true>(Wp, xs, ys, nrows, ncols, nb, s, di, err)
                     : launch_packed_b<false>(Wp, xs, ys, nrows, ncols, nb, s, di, err);
        if (st != QGEMV_OK) return st;
    }
    return QGEMV_OK;
}

}  // namespace qg
