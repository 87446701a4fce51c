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
// GEMV kernel: a CTA of 8 warps takes whole tiles (persistent over tiles);
// warp w takes a contiguous range of the block pairs of every tile, stages
// the fp16 x operands of that range once (scaled per 8 blocks by a power of
// two, as in gemv_tc.cu), then per tile streams its records (prefetching the
// next group of four while it computes one), decodes each lane's 16 bytes
// into A fragments with one logic instruction per two weights (fp16 1024 + q
// and 1024 + 16 q), and runs 4 mma.sync m16n8k16 per pair whose accumulators
// start at -T (the offset terms).  Per-warp tile partials are summed in a
// fixed order: deterministic.
#include <cstdlib>
#include <cstring>

#include <algorithm>

#include "qgemv_common.cuh"

namespace qg {
namespace {

constexpr int kPkWarps = 8;
constexpr int kPkThreads = kPkWarps * 32;
constexpr int kRecBytes = 576;
constexpr int kGroup = 4;                   // pairs per prefetch group (= per x scale round)

// ------------------------------------------------------------------ packing
// One thread per (tile, pair, lane) 16-byte piece, and lanes 0..7 also write
// the 8-byte scale pieces.  Rows past nrows are zero.
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
__device__ __forceinline__ void pk_mma_init(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1, float ce,
                                            float co) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %10, %11};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(ce), "f"(co));
}
__device__ __forceinline__ uint32_t pk_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float pk_rsum(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu))) +
           __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}
// 2^e with m * 2^e in [2^9, 2^10) from the bits of m = max|x| (see gemv_tc.cu)
__device__ __forceinline__ int pk_exponent(uint32_t mbits) {
    const int be = static_cast<int>(mbits >> 23);
    if (be == 255 || mbits == 0u) return 0;
    return be == 0 ? 120 : 136 - be;
}
__device__ __forceinline__ float pk_pow2(int e) { return __int_as_float((127 + e) << 23); }
// 16-byte / 8-byte streaming loads of the packed weights (read once).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
// Bulk prefetch of [p, p + bytes) into L2 (a cache hint: it changes no data
// and is ordered with nothing, so it may run before the stream dependency).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint2 ld_stream8(const void *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

struct PkParams {
    const uint8_t *Wp;
    const float *x;
    float *y;
    int nrows, ncols, batch;
    int ntiles, npairs;
    int early;            // first weight loads before waiting on the preceding kernel
};

// Shared memory: per warp, for each of its block pairs' blocks (round r of 4
// pairs = 8 blocks, block i of the round) and batch column n: the lane-c
// fragment (uint4 [c]), -T, and per (round, column) 2^-e; then the per-warp
// tile partials.
struct PkLayout {
    uint32_t xf, nt, us, part, total;
    uint32_t warp_rounds;      // rounds per warp (of the largest range)
};

__host__ __device__ inline PkLayout pk_layout(int npairs, int batch) {
    PkLayout L;
    const int maxp = (npairs + kPkWarps - 1) / kPkWarps;
    L.warp_rounds = static_cast<uint32_t>((maxp + kGroup - 1) / kGroup);
    const uint32_t items = L.warp_rounds * 8 * batch;      // per warp
    uint32_t o = 0;
    L.xf = o; o += kPkWarps * items * 64;
    L.nt = o; o += kPkWarps * items * 4;
    L.us = o; o += kPkWarps * L.warp_rounds * batch * 4;
    L.part = o; o += kPkWarps * 16 * batch * 4;
    L.total = o;
    return L;
}

// ------------------------------------------------------------------ kernel
template <bool B1>
__global__ void __launch_bounds__(kPkThreads, 2)
gemv_packed_q4_0_kernel(const PkParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int batch = B1 ? 1 : p.batch;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const PkLayout L = pk_layout(p.npairs, p.batch);
    // this warp's pairs: [p0, p0 + np) of every tile
    const int base = p.npairs / kPkWarps, extra = p.npairs % kPkWarps;
    const int np = base + (wid < extra ? 1 : 0);
    const int p0 = wid * base + min(wid, extra);
    const int nrounds = (np + kGroup - 1) / kGroup;
    const uint32_t witems = L.warp_rounds * 8 * p.batch;

    // ---- prefetch of one round (4 pairs) of weight records of tile t
    uint4 qa[kGroup], qb[kGroup];
    uint2 da[kGroup], db[kGroup];
    auto load_round = [&](uint4 (&q)[kGroup], uint2 (&d)[kGroup], int t, int r) {
        const uint8_t *rec = p.Wp + (static_cast<int64_t>(t) * p.npairs + p0 + r * kGroup) * kRecBytes;
#pragma unroll
        for (int i = 0; i < kGroup; ++i) {
            if (r * kGroup + i < np) {
                q[i] = ld_stream16(rec + i * kRecBytes + 16 * lane);
                d[i] = ld_stream8(rec + i * kRecBytes + 512 + 8 * g);
            } else {
                q[i] = make_uint4(0u, 0u, 0u, 0u);
                d[i] = make_uint2(0u, 0u);
            }
        }
    };
    const int t0 = blockIdx.x;
    // this warp's records of tile t are contiguous: pull them into L2 ahead
    auto prefetch_tile = [&](int t) {
        if (lane == 0 && np > 0 && t < p.ntiles) {
            prefetch_l2(p.Wp + (static_cast<int64_t>(t) * p.npairs + p0) * kRecBytes,
                        static_cast<uint32_t>(np * kRecBytes));
        }
    };
    prefetch_tile(t0);
    prefetch_tile(t0 + static_cast<int>(gridDim.x));
    if (p.early && t0 < p.ntiles && nrounds > 0) load_round(qa, da, t0, 0);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!p.early && t0 < p.ntiles && nrounds > 0) load_round(qa, da, t0, 0);

    // ---- stage x for this warp's blocks [2 p0, 2 (p0 + np)): lane l builds
    // fragment c of block l / 4 of each 8-block round (aligned column map:
    // low nibbles x[4c..4c+3], high nibbles x[16+4c..] / 16), scaled per
    // (round, column) by a power of two; -T per block (the offset term the
    // accumulator starts from: 1032 * sum of the rounded low-slot x + 1152 *
    // sum of the rounded high-slot x / 16)
    uint4 *xf = reinterpret_cast<uint4 *>(smem + L.xf) + wid * witems * 4;
    float *ntp = reinterpret_cast<float *>(smem + L.nt) + wid * witems;
    float *usp = reinterpret_cast<float *>(smem + L.us) + wid * L.warp_rounds * p.batch;
    {
        const int bl = lane >> 2;
        const int off[4] = {4 * c, 4 * c + 2, 16 + 4 * c, 18 + 4 * c};
        for (int n = 0; n < p.batch; ++n) {
            const float *xr = p.x + static_cast<size_t>(n) * p.ncols + static_cast<size_t>(2 * p0) * 32;
            for (int r0 = 0; r0 < nrounds; r0 += 8) {
                float2 v[8][4];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int blk = (r0 + i) * 8 + bl;
                    const bool ok = r0 + i < nrounds && blk < 2 * np;
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        v[i][h] = ok ? __ldg(reinterpret_cast<const float2 *>(xr + blk * 32 + off[h])) : make_float2(0.0f, 0.0f);
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = r0 + i;
                    if (r >= nrounds) break;             // warp-uniform
                    float m = 0.0f;
#pragma unroll
                    for (int h = 0; h < 4; ++h) m = fmaxf(m, fmaxf(fabsf(v[i][h].x), fabsf(v[i][h].y)));
                    const int e = pk_exponent(__reduce_max_sync(0xffffffffu, __float_as_uint(m)));
                    if (lane == 0) usp[r * p.batch + n] = pk_pow2(-e);
                    const float sc = pk_pow2(e), sh = sc * 0.0625f;
                    const uint32_t w0 = pk_f16x2(v[i][0].x * sc, v[i][1].x * sc);
                    const uint32_t w1 = pk_f16x2(v[i][0].y * sc, v[i][1].y * sc);
                    const uint32_t w2 = pk_f16x2(v[i][2].x * sh, v[i][3].x * sh);
                    const uint32_t w3 = pk_f16x2(v[i][2].y * sh, v[i][3].y * sh);
                    float slo = pk_rsum(w0) + pk_rsum(w1), shi = pk_rsum(w2) + pk_rsum(w3);
                    slo += __shfl_xor_sync(0xffffffffu, slo, 1);
                    shi += __shfl_xor_sync(0xffffffffu, shi, 1);
                    slo += __shfl_xor_sync(0xffffffffu, slo, 2);
                    shi += __shfl_xor_sync(0xffffffffu, shi, 2);
                    const int item = (r * 8 + bl) * p.batch + n;
                    xf[item * 4 + c] = make_uint4(w0, w1, w2, w3);
                    if (c == 0) ntp[item] = -fmaf(1032.0f, slo, 1152.0f * shi);
                }
            }
        }
        __syncwarp();
    }

    // ---- per tile: stream this warp's records, 4 pairs per round, the next
    // round's loads in flight while one is computed
    constexpr uint32_t kMagic = 0x64006400u;      // fp16 (1024, 1024)
    const int ncol = min(g, batch - 1);          // B columns past the batch repeat the last one
    const int n0 = min(2 * c, batch - 1), n1 = min(2 * c + 1, batch - 1);
    const uint4 *fb0 = xf + ncol * 4 + c;
    float *part = reinterpret_cast<float *>(smem + L.part);

    auto compute_round = [&](const uint4 (&q)[kGroup], const uint2 (&d)[kGroup], int r, float acc[4]) {
        float ak[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < kGroup; ++i) {
            if (r * kGroup + i < np) {
                const int blk = r * 8 + 2 * i;
                const uint32_t q0 = q[i].x, q1 = q[i].y, q2 = q[i].z, q3 = q[i].w;
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
                const uint4 be = fb0[(blk * p.batch) * 4], bo = fb0[((blk + 1) * p.batch) * 4];
                float te0, te1, to0, to1;
                if constexpr (B1) {
                    const float2 tt = *reinterpret_cast<const float2 *>(ntp + blk);
                    te0 = te1 = tt.x;
                    to0 = to1 = tt.y;
                } else {
                    te0 = ntp[blk * p.batch + n0]; te1 = ntp[blk * p.batch + n1];
                    to0 = ntp[(blk + 1) * p.batch + n0]; to1 = ntp[(blk + 1) * p.batch + n1];
                }
                float ce[4], co[4];
                pk_mma_init(ce, e0, be.x, be.y, te0, te1);
                pk_mma_init(co, o0, bo.x, bo.y, to0, to1);
                pk_mma(ce, e1, be.z, be.w);
                pk_mma(co, o1, bo.z, bo.w);
                const float de0 = __half2float(__ushort_as_half(static_cast<unsigned short>(d[i].x & 0xffffu)));
                const float de1 = __half2float(__ushort_as_half(static_cast<unsigned short>(d[i].x >> 16)));
                const float do0 = __half2float(__ushort_as_half(static_cast<unsigned short>(d[i].y & 0xffffu)));
                const float do1 = __half2float(__ushort_as_half(static_cast<unsigned short>(d[i].y >> 16)));
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
            }
        }
        const float u0 = usp[r * p.batch + n0];
        acc[0] = fmaf(ak[0], u0, acc[0]);
        acc[2] = fmaf(ak[2], u0, acc[2]);
        if constexpr (!B1) {
            const float u1 = usp[r * p.batch + n1];
            acc[1] = fmaf(ak[1], u1, acc[1]);
            acc[3] = fmaf(ak[3], u1, acc[3]);
        }
    };

    bool inb = false;                           // the current round sits in (qb, db)
    for (int t = t0; t < p.ntiles; t += gridDim.x) {
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (t != t0) prefetch_tile(t + static_cast<int>(gridDim.x));
        for (int r = 0; r < nrounds; ++r) {
            // loads of the next round (this tile's, or the next tile's first)
            const int tn = (r + 1 < nrounds) ? t : t + static_cast<int>(gridDim.x);
            const int rn = (r + 1 < nrounds) ? r + 1 : 0;
            if (inb) {
                if (tn < p.ntiles) load_round(qa, da, tn, rn);
                compute_round(qb, db, r, acc);
            } else {
                if (tn < p.ntiles) load_round(qb, db, tn, rn);
                compute_round(qa, da, r, acc);
            }
            inb = !inb;
        }
        // ---- tile t: fixed-order sum of the warp partials
        float *pw = part + wid * 16 * batch;
        if (2 * c < batch) {
            pw[g * batch + 2 * c] = acc[0];
            pw[(g + 8) * batch + 2 * c] = acc[2];
        }
        if (2 * c + 1 < batch) {
            pw[g * batch + 2 * c + 1] = acc[1];
            pw[(g + 8) * batch + 2 * c + 1] = acc[3];
        }
        __syncthreads();
        if (tid < 16 * batch) {
            const int rr = tid / batch, n = tid - rr * batch;
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < kPkWarps; ++w) sum += part[(w * 16 + rr) * batch + n];
            const int row = t * 16 + rr;
            if (row < p.nrows) p.y[static_cast<int64_t>(n) * p.nrows + row] = sum;
        }
        __syncthreads();
    }
}

// Shared-memory bytes above which the batch is split into several launches.
constexpr uint32_t kPkSmemCap = 110 * 1024;

template <bool B1>
qgemv_status launch_packed_b(const void *Wp, const float *x, float *y, int64_t nrows, int64_t ncols, int batch,
                             cudaStream_t s, const DevInfo &di) {
    auto kern = gemv_packed_q4_0_kernel<B1>;
    const int npairs = static_cast<int>(ncols / 64);
    const PkLayout L = pk_layout(npairs, batch);
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
    p.early = g_opt_weights_static;
    const int grid = static_cast<int>(std::min<int64_t>(p.ntiles, static_cast<int64_t>(per_sm) * di.sm_count));
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
                                     int batch, cudaStream_t s, const DevInfo &di) {
    // batch columns per launch: as many as keep the staged x within the cap
    const int npairs = static_cast<int>(ncols / 64);
    int per = batch;
    while (per > 1 && pk_layout(npairs, per).total > kPkSmemCap) --per;
    if (pk_layout(npairs, per).total > di.smem_optin) {
        set_last_error("packed GEMV: ncols=%lld needs more shared memory than one CTA has", (long long)ncols);
        return QGEMV_ERR_SHAPE;
    }
    for (int n0 = 0; n0 < batch; n0 += per) {
        const int nb = std::min(per, batch - n0);
        const float *xs = x + static_cast<int64_t>(n0) * ncols;
        float *ys = y + static_cast<int64_t>(n0) * nrows;
        qgemv_status st = nb == 1 ? launch_packed_b<true>(Wp, xs, ys, nrows, ncols, nb, s, di)
                                  : launch_packed_b<false>(Wp, xs, ys, nrows, ncols, nb, s, di);
        if (st != QGEMV_OK) return st;
    }
    return QGEMV_OK;
}

}  // namespace qg
