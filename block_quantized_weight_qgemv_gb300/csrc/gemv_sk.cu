// gemv_sk.cu -- block-quantized GEMV on the tensor cores with a stream-K
// split of the weight stream:  y[b][r] = sum_k w[r][k] * x[b][k], batch 1..8,
// Q4_0 / Q4_1 / Q8_0 in ggml's block layout (the batch-1 "dequantize_mul_mat_vec"
// path of the "llama_cpp 0.12.1 -> 0.12.2" ggml-cuda.cu diff, extended to small
// batches; block formulas from its dequantize_block_q4_0 / _q4_1 / _q8_0_f16
// hunks).
//
// Work split.  The weights are cut into units of 16 rows x 64 blocks (one
// 3-D TMA box, 64-byte swizzle).  Units are numbered row group major, k unit
// minor (nu units per row group), and CTA i of G (one per SM) takes the
// contiguous range [floor(i U / G), floor((i+1) U / G)): every SM streams the
// same number of bytes (to within one unit) and decodes / multiplies the same
// number of blocks, whatever the row count.  Each range holds at least
// ceil(nu / 4) units, so a row group falls to at most 5 CTAs.  A row group
// that falls to several CTAs is summed by the first of them (the "owner", for
// which it is the last group of its range): every other CTA covering it has
// it as its first group, finishes its part early, writes the partial to its
// scratch slot and raises the slot's flag (release).  The owner's producer
// warp, once it has issued all its weight copies, waits for those flags
// (acquire), copies the partials into shared memory and clears the flags; the
// owner then adds them to its own partial in CTA order (fixed: the result is
// deterministic).
//
// Arithmetic.  Inside a CTA the 16 consumer warps split each unit by block
// pairs (warp w takes pairs w and w + 16) and multiply with mma.sync
// m16n8k16 (fp16 operands, fp32 accumulation), the batch riding in the MMA's
// N dimension:
//  - A (weights) are the exact small integers q - 8 (Q4_0), q (Q4_1) or q
//    (Q8_0) in fp16: a logic op puts a nibble (byte) under the fp16 exponent
//    of 1024, an fp16 add / fma removes the offset exactly.
//  - B (activations): each warp scales the x values of its four blocks of a
//    k unit ("chunk", per batch column) by one power of two that puts their
//    largest magnitude in [2^9, 2^10) and rounds them to fp16 (relative error
//    <= 2^-11 while the scaled value is >= 2^-14).  A chunk holding a non-
//    finite value, or a nonzero value whose scaled magnitude is below 2^-14
//    (a dynamic range above ~2^23 inside 128 values), is flagged and computed
//    exactly in fp32 on the CUDA cores instead.
//  - each block's fp32 MMA result is multiplied by its fp16 scale d (and for
//    Q4_1 the block's sum of the rounded x times m is added) on the CUDA
//    cores; each chunk's sum is scaled back by the exact power of two.
// Hence |y - exact| <= 2^-11 sum_k |w_k x_k| + fp32 accumulation error.
//
// Data movement.  A producer warp streams units through a ring of NS slots
// (one mbarrier-completed TMA copy each).  When the caller declared its
// weights static, the whole ring is filled before the kernel waits on the
// preceding kernel of its stream (griddepcontrol.wait).  x is then brought
// into a shared-memory area of its own by one bulk copy per 2048-column chunk
// (one mbarrier each), and the consumers convert all of it at once (several
// items in flight per lane) before their first unit.  When x does not fit in shared
// memory next to a ring of four units, the consumers load it directly
// before the loop and only two weight copies go ahead of those loads
// (weight copies in flight delay plain loads).
//
// mma.sync fragment layout (m16n8k16, g = lane/4, c = lane%4):
//   A: a0 = (row g, k 2c..2c+1)  a1 = (row g+8, k 2c..2c+1)
//      a2 = (row g, k 2c+8..+9)  a3 = (row g+8, k 2c+8..+9)
//   B: b0 = (k 2c..2c+1, n g)    b1 = (k 2c+8..+9, n g)
//   C: c0 = (g, 2c) c1 = (g, 2c+1) c2 = (g+8, 2c) c3 = (g+8, 2c+1)
// The k order inside a block is free as long as A and B agree: lane c takes
// four qs bytes (Q4) or eight (Q8_0) of each of its rows, at the columns
// listed with piece_offsets below, and B is staged in exactly that order.
#include <cuda.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "qgemv_common.cuh"

namespace qg {

// Split-row-group scratch: kSkSets independent sets (one per stream, see
// scratch_for), each with one partial slot of 16 x batch floats and one flag
// per CTA.  Zero-initialized; every flag a call raises is cleared by the same
// call.
constexpr int kSkSets = 8;
constexpr int kSkMaxG = 320;
constexpr int kSkSlotFloats = kSkMaxG * 16 * QGEMV_MAX_BATCH;
__device__ float g_sk_part[kSkSets * kSkSlotFloats];
__device__ unsigned g_sk_flag[kSkSets * kSkMaxG];

// Probes of a consumer's wait for a weight copy before it gives up
// (qgemv_set_option(QGEMV_OPT_WAIT_PROBES)); each probe sleeps <= 256 ns.
unsigned g_opt_wait_probes = 1u << 20;
// qgemv_set_option(QGEMV_OPT_TEST_WITHHOLD_COPY): the next launch withholds
// its first weight copy.
int g_opt_withhold_next = 0;

namespace {

constexpr int kCW = 16;                      // consumer warps
constexpr int kThreads = (kCW + 1) * 32;     // + one producer warp
constexpr int kUB = 64;                      // blocks per unit (k)
constexpr int RT = 16;                       // rows per unit
constexpr int kMaxSlots = 12;
constexpr int kMaxPartners = 4;              // other CTAs sharing the owner's last row group

template <int F> struct SkFmt;
template <> struct SkFmt<FMT_Q4_0> { static constexpr int BB = 18; static constexpr int PB = 36; };
template <> struct SkFmt<FMT_Q4_1> { static constexpr int BB = 20; static constexpr int PB = 40; };
template <> struct SkFmt<FMT_Q8_0> { static constexpr int BB = 34; static constexpr int PB = 68; };

__host__ __device__ constexpr uint32_t sk_slot_bytes(int F) { return static_cast<uint32_t>(64 * RT * block_bytes(F)); }

struct SkParams {
    const float *x;
    float *y;
    unsigned *err;
    float *part;       // scratch partial slots of this call's set (16 x batch floats per CTA)
    unsigned *flag;    // scratch flags of this call's set (one per CTA)
    int nrows, ncols, batch;
    int nu;            // k units per row (ncols / 2048)
    int U;             // units in total (row groups x nu)
    int G;             // CTAs
    int ns;            // ring slots
    int early;         // 1: weights may be copied before waiting on the preceding kernel
    int xs;            // 1: x by bulk copies into shared memory; 0: direct loads
    int pre;           // direct loads: units copied ahead of them
    unsigned probes;   // consumer wait limit
    int withhold;      // testing: never copy the first unit (its wait runs out)
};

// Shared-memory layout (offsets from a 1024-byte aligned base).  Warp w's
// staged B fragments for k unit ku and batch column n are 16 uint4 (block of
// the warp blk4 = 0..3, lane c) at xf + ((w nu + ku) batch + n) 256 bytes.
struct SkLayout {
    uint32_t ring, xf, us, wf, xs, part, pp, x32, bars, issued, flag, total;
};

__host__ __device__ inline uint32_t sk_align(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline SkLayout sk_layout(int F, int nu, int batch, int ns, int xs) {
    SkLayout L;
    const uint32_t items = static_cast<uint32_t>(kCW * nu * batch);
    uint32_t o = 0;
    L.ring = o;  o += static_cast<uint32_t>(ns) * sk_slot_bytes(F);
    L.xf = o;    o += items * 256;
    L.us = o;    o += sk_align(items * 4, 16);
    L.wf = o;    o += sk_align(static_cast<uint32_t>(kCW * nu) * 4, 16);
    L.xs = o;    o += F == FMT_Q4_1 ? items * 16 : 0;
    L.part = o;  o += 2u * kCW * RT * batch * 4;
    L.pp = o;    o += static_cast<uint32_t>(kMaxPartners) * RT * batch * 4;
    L.x32 = o;   o += xs ? static_cast<uint32_t>(batch) * nu * 2048u * 4u : 0u;     // fp32 x, [batch][ncols]
    L.bars = o;  o += static_cast<uint32_t>(ns) * 16 + 8 + (xs ? nu * 8 : 0);      // full, empty, ppbar, xbar[nu]
    L.issued = o; o += sk_align(static_cast<uint32_t>(ns) * 4, 16);
    L.flag = o;  o += 16;
    L.total = o;
    return L;
}

// ------------------------------------------------------------ device helpers
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void consumer_bar() {
    asm volatile("bar.sync 1, %0;" :: "n"(kCW * 32) : "memory");
}
// Barrier 2: the consumers signal that x is staged (or, for direct loads,
// that their loads of x are in flight); the producer holds the remaining
// weight copies until then.
__device__ __forceinline__ void xready_arrive() {
    asm volatile("bar.arrive 2, %0;" :: "n"(kThreads) : "memory");
}
__device__ __forceinline__ void xready_wait() {
    asm volatile("bar.sync 2, %0;" :: "n"(kThreads) : "memory");
}
__device__ __forceinline__ uint32_t lds(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ float ldsf(uint32_t a) { return __uint_as_float(lds(a)); }
__device__ __forceinline__ float2 lds64f(uint32_t a) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *tmap, int c0, int c1, int c2,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}
// Non-blocking probe of the phase with the given parity.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// Bounded wait: non-blocking probes separated by sleeps that grow from 32 to
// 256 ns, so waiting warps give their issue slots (and the barrier's shared-
// memory word) to the warps doing work.  (A try_wait with a suspend-time hint
// was measured to return at once on this part, i.e. to spin.)  Gives up after
// `probes` sleeps.
__device__ __forceinline__ bool mbar_wait_hint(uint64_t *bar, uint32_t parity, unsigned probes) {
    if (mbar_test(bar, parity)) return true;
    unsigned ns = 32;
    for (unsigned i = 0; i < probes; ++i) {
        __nanosleep(ns);
        if (mbar_test(bar, parity)) return true;
        if (ns < 256) ns <<= 1;
    }
    return false;
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
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
__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// D = A B (C = 0)
__device__ __forceinline__ void mma0(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                     uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}
// D = A B + D
__device__ __forceinline__ void mma1(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                     uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
// fp16 halves of a 32-bit word as fp32 (one conversion each)
__device__ __forceinline__ float h_lo(uint32_t u) { return __low2float(*reinterpret_cast<const __half2 *>(&u)); }
__device__ __forceinline__ float h_hi(uint32_t u) { return __high2float(*reinterpret_cast<const __half2 *>(&u)); }
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// Byte offset inside a slot of the word at byte `o` of unit row `y`: the slot
// is [64-byte piece][16 rows][64 bytes], 16-byte units xor-ed with bits 1..2
// of the row (TMA's 64-byte swizzle on a 1024-byte aligned slot).
__device__ __forceinline__ uint32_t sk_off(int o, int y) {
    return static_cast<uint32_t>((o >> 6) * (RT * 64) + y * 64 + ((o & 63) ^ (((y >> 1) & 3) << 4)));
}

// Columns (inside a block) of the four 2-float pieces that lane c's fragment
// of a block holds (par: 0 for the even block of a pair, 1 for the odd one).
//  Q4 : pieces (o_a, o_b, 16 + o_a, 16 + o_b); the lane's four qs bytes are
//       qs[o_a], qs[o_a + 1], qs[o_b], qs[o_b + 1] (their low nibbles are
//       columns o_a.., their high nibbles 16 + o_a..).
//  Q8 : pieces (p0, p1, p2, p3); the lane's eight bytes are q[p_i], q[p_i + 1].
// Even Q4_0 / Q8_0 blocks start 2 bytes into a 4-byte word: lanes read the
// aligned words and lane 3 assembles the straddling bytes.
template <int F>
__host__ __device__ inline void piece_offsets(int par, int c, int off[4]) {
    if (F == FMT_Q8_0) {
        if (par || c < 3) {
            const int b0 = par ? 8 * c : 8 * c + 2;
            off[0] = b0; off[1] = b0 + 2; off[2] = b0 + 4; off[3] = b0 + 6;
        } else {
            off[0] = 26; off[1] = 28; off[2] = 0; off[3] = 30;
        }
    } else {
        int oa, ob;
        if (F == FMT_Q4_1 || par) {
            oa = 4 * c; ob = 4 * c + 2;
        } else if (c < 3) {
            oa = 4 * c + 2; ob = 4 * c + 4;
        } else {
            oa = 0; ob = 14;
        }
        off[0] = oa; off[1] = ob; off[2] = 16 + oa; off[3] = 16 + ob;
    }
}

// Byte offsets (inside a pair of blocks, PB bytes) of the words a lane reads.
//  Q4_0: s0 = [d_e, qs_e 0..1], s4 = [qs_e 14..15, d_o], xw = own even word
//        (s_{1+c}, or s0 for c = 3, realigned with s4), ow = s_{5+c}.
//  Q4_1: s0 = [d_e, m_e], s5 = [d_o, m_o], xw = s_{1+c}, ow = s_{6+c}.
//  Q8_0: s0 = [d_e, q_e 0..1], s8 = [q_e 30..31, d_o], ea / eb = own even
//        words (eb realigned with s8 on lane 3), oa / ob = s_{9+2c}, s_{10+2c}.
template <int F> struct PairWords;
template <> struct PairWords<FMT_Q4_0> {
    static constexpr int NW = 4;
    __device__ static void offsets(int c, int o[4]) { o[0] = 0; o[1] = 16; o[2] = c < 3 ? 4 + 4 * c : 0; o[3] = 20 + 4 * c; }
};
template <> struct PairWords<FMT_Q4_1> {
    static constexpr int NW = 4;
    __device__ static void offsets(int c, int o[4]) { o[0] = 0; o[1] = 20; o[2] = 4 + 4 * c; o[3] = 24 + 4 * c; }
};
template <> struct PairWords<FMT_Q8_0> {
    static constexpr int NW = 6;
    __device__ static void offsets(int c, int o[6]) {
        o[0] = 0; o[1] = 32;
        o[2] = 4 * (c < 3 ? 1 + 2 * c : 7);
        o[3] = 4 * (c < 3 ? 2 + 2 * c : 0);
        o[4] = 4 * (9 + 2 * c);
        o[5] = 4 * (10 + 2 * c);
    }
};

template <int F> struct RowWords { uint32_t w[PairWords<F>::NW]; };

// The lane's data words of the even / odd block (Q4: one each; Q8: two each)
// and the scales of one row as fp32.
template <int F> struct LaneBlocks {
    uint32_t e[F == FMT_Q8_0 ? 2 : 1], o[F == FMT_Q8_0 ? 2 : 1];
    float de, dd, me, md;
};
template <int F>
__device__ __forceinline__ LaneBlocks<F> lane_blocks(const RowWords<F> &r, uint32_t sel) {
    LaneBlocks<F> b;
    if constexpr (F == FMT_Q4_0) {
        b.e[0] = prmt(r.w[2], r.w[1], sel);
        b.o[0] = r.w[3];
        b.de = h_lo(r.w[0]);
        b.dd = h_hi(r.w[1]);
        b.me = b.md = 0.0f;
    } else if constexpr (F == FMT_Q4_1) {
        b.e[0] = r.w[2];
        b.o[0] = r.w[3];
        b.de = h_lo(r.w[0]);
        b.me = h_hi(r.w[0]);
        b.dd = h_lo(r.w[1]);
        b.md = h_hi(r.w[1]);
    } else {
        b.e[0] = r.w[2];
        b.e[1] = prmt(r.w[3], r.w[1], sel);
        b.o[0] = r.w[4];
        b.o[1] = r.w[5];
        b.de = h_lo(r.w[0]);
        b.dd = h_hi(r.w[1]);
        b.me = b.md = 0.0f;
    }
    return b;
}

// Exact fp16 operands of one block's data word(s): h[0], h[1] for the first
// k-step (a0/a2 of this row), h[2], h[3] for the second.
template <int F>
__device__ __forceinline__ void decode(const uint32_t (&wd)[F == FMT_Q8_0 ? 2 : 1], uint32_t h[4]) {
    constexpr uint32_t kMagic = 0x64006400u;   // fp16 (1024, 1024)
    if constexpr (F == FMT_Q8_0) {
        constexpr uint32_t K = 0x64646464u, kOff = 0xE480E480u;   // -1152
        const uint32_t a = wd[0] ^ 0x80808080u, b = wd[1] ^ 0x80808080u;
        h[0] = hadd2(prmt(a, K, 0x4140), kOff);
        h[1] = hadd2(prmt(a, K, 0x4342), kOff);
        h[2] = hadd2(prmt(b, K, 0x4140), kOff);
        h[3] = hadd2(prmt(b, K, 0x4342), kOff);
    } else {
        // low nibbles: 1024 + q - (1024 + 8 | 1024); high nibbles (under the
        // magic as 1024 + 16 q): (1024 + 16 q) / 16 - (72 | 64)
        constexpr uint32_t kLo = F == FMT_Q4_0 ? 0xE408E408u : 0xE400E400u;   // -1032 | -1024
        constexpr uint32_t kHi = F == FMT_Q4_0 ? 0xD480D480u : 0xD400D400u;   // -72 | -64
        constexpr uint32_t kSixteenth = 0x2C002C00u;                          // 1/16
        const uint32_t w = wd[0], w8 = wd[0] >> 8;
        h[0] = hadd2(and_or<0x000f000fu>(w, kMagic), kLo);
        h[1] = hadd2(and_or<0x000f000fu>(w8, kMagic), kLo);
        h[2] = hfma2(and_or<0x00f000f0u>(w, kMagic), kSixteenth, kHi);
        h[3] = hfma2(and_or<0x00f000f0u>(w8, kMagic), kSixteenth, kHi);
    }
}

// ------------------------------------------------------------ x staging
// Warp w stages, for the items it = ku * batch + n in [i_lo, i_hi) (k unit ku,
// batch column n), the B fragments of its four blocks of unit ku (pairs w and
// w + 16): lane f = l % 16 builds fragment (blk4 = f / 4, c = f % 4), half-
// warp h = l / 16 takes the items of parity h.  Per item the 16 lanes find the
// largest |x| of their 128 values, scale by 2^e, round to fp16, and flag the
// chunk ku when the fast path would lose more than fp16 rounding (see the file
// header); the caller clears the flags of the chunks first.  x comes from
// shared memory (xs_smem != 0: the bulk-copied [batch][ncols] x) or global
// memory; with `arrive`, the warp arrives on barrier 2 once its first loads
// of global x are in flight.
template <int F>
__device__ __forceinline__ void stage_items(const SkParams &p, int w, int lane, uint8_t *smem, const SkLayout &L,
                                            uint32_t xs_smem, int i_lo, int i_hi, bool arrive) {
    const int f = lane & 15, hw = lane >> 4;
    const int blk4 = f >> 2, c = f & 3;
    const int par = blk4 & 1, j = blk4 >> 1;
    const int bin = 2 * (w + kCW * j) + par;     // block inside a unit
    int off[4];
    piece_offsets<F>(par, c, off);
    const int nu = p.nu, batch = p.batch;
    const int items = nu * batch;
    uint4 *xf = reinterpret_cast<uint4 *>(smem + L.xf) + static_cast<size_t>(w) * items * 16;
    float *us = reinterpret_cast<float *>(smem + L.us) + w * items;
    int *wf = reinterpret_cast<int *>(smem + L.wf) + w * nu;
    float *xs = reinterpret_cast<float *>(smem + L.xs) + w * items * 4;
    constexpr int kIL = 4;                        // items per lane in flight
    bool arrived = !arrive;
    for (int i0 = i_lo; i0 < i_hi; i0 += 2 * kIL) {
        float2 v[kIL][4];
#pragma unroll
        for (int t = 0; t < kIL; ++t) {
            const int it = i0 + 2 * t + hw;
            const bool ld = it < i_hi;
            const int ku = ld ? it / batch : 0, n = ld ? it - ku * batch : 0;
            const size_t base = static_cast<size_t>(n) * p.ncols + static_cast<size_t>(ku * kUB + bin) * 32;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                if (!ld) v[t][h] = make_float2(0.0f, 0.0f);
                else if (xs_smem) v[t][h] = lds64f(xs_smem + static_cast<uint32_t>(base + off[h]) * 4u);
                else v[t][h] = __ldg(reinterpret_cast<const float2 *>(p.x + base + off[h]));
            }
        }
        if (!arrived) {
            xready_arrive();
            arrived = true;
        }
#pragma unroll
        for (int t = 0; t < kIL; ++t) {
            const int it0 = i0 + 2 * t;
            if (it0 >= i_hi) break;                    // warp-uniform
            const int it = it0 + hw;
            const bool valid = it < i_hi;
            float m = 0.0f;
            bool bad = false;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float a = fabsf(v[t][h].x), b = fabsf(v[t][h].y);
                m = fmaxf(m, fmaxf(a, b));
                bad |= !(a <= 3.0e38f) || !(b <= 3.0e38f);     // inf or nan
            }
#pragma unroll
            for (int s = 1; s < 16; s <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
            const uint32_t mb = __float_as_uint(m);
            const int be = static_cast<int>(mb >> 23);
            const int e = (mb == 0u || be >= 255) ? 0 : (be == 0 ? 120 : 136 - be);
            const float sc = pow2f(e);
            float s[8];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                s[2 * h] = v[t][h].x * sc;
                s[2 * h + 1] = v[t][h].y * sc;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) bad |= (s[q] != 0.0f) && (fabsf(s[q]) < 6.103515625e-05f);   // < 2^-14
            uint4 fr;
            if constexpr (F == FMT_Q8_0) {
                fr = make_uint4(f16x2_rn(s[0], s[1]), f16x2_rn(s[2], s[3]), f16x2_rn(s[4], s[5]), f16x2_rn(s[6], s[7]));
            } else {
                // (pa.x, pb.x) (pa.y, pb.y) (pc.x, pd.x) (pc.y, pd.y)
                fr = make_uint4(f16x2_rn(s[0], s[2]), f16x2_rn(s[1], s[3]), f16x2_rn(s[4], s[6]), f16x2_rn(s[5], s[7]));
            }
            const unsigned bal = __ballot_sync(0xffffffffu, bad && valid);
            const bool wide = ((bal >> (16 * hw)) & 0xffffu) != 0u;
            if (valid) {
                xf[it * 16 + f] = fr;
                if (f == 0) {
                    us[it] = pow2f(-e);
                    if (wide) wf[it / batch] = 1;      // any column flags the whole chunk
                }
            }
            if constexpr (F == FMT_Q4_1) {
                // block sum of the rounded values, fixed order, over lanes c
                float t4 = (h_lo(fr.x) + h_hi(fr.x)) + (h_lo(fr.y) + h_hi(fr.y)) +
                           ((h_lo(fr.z) + h_hi(fr.z)) + (h_lo(fr.w) + h_hi(fr.w)));
                t4 += __shfl_xor_sync(0xffffffffu, t4, 1);
                t4 += __shfl_xor_sync(0xffffffffu, t4, 2);
                if (valid && c == 0) xs[it * 4 + blk4] = t4;
            }
        }
    }
    if (!arrived) xready_arrive();
    __syncwarp();
}

// Clears the wide-chunk flags of warp w for k units [k_lo, k_hi).
__device__ __forceinline__ void clear_wide(const SkParams &p, int w, int lane, uint8_t *smem, const SkLayout &L,
                                           int k_lo, int k_hi) {
    int *wf = reinterpret_cast<int *>(smem + L.wf) + w * p.nu;
    for (int k = k_lo + lane; k < k_hi; k += 32) wf[k] = 0;
    __syncwarp();
}

// ------------------------------------------------------------ one unit
// Per-lane word addresses (pair slot j, word i) of row g inside slot 0; row
// g + 8 is 512 bytes further, slot s s * SLOT further.
template <int F> struct LaneCtx {
    uint32_t off[2][PairWords<F>::NW];
    uint32_t sel;
};

// Fast path: both pair slots of the warp in the unit at sb (shared address).
// fb: shared address of this lane's fragment of block 0 for (ku, its column);
// blocks 1..3 follow at +64 bytes.  xs0 / xs1 (Q4_1): shared addresses of the
// four block sums for (ku, n0) / (ku, n1).
template <int F, bool B1>
__device__ __forceinline__ void unit_fast(uint32_t sb, const LaneCtx<F> &lc, uint32_t fb, uint32_t xs0,
                                          uint32_t xs1, float ak[4]) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint4 fe = lds128(fb + (2 * j) * 64), fo = lds128(fb + (2 * j + 1) * 64);
        RowWords<F> r0, r8;
#pragma unroll
        for (int i = 0; i < PairWords<F>::NW; ++i) {
            const uint32_t a = sb + lc.off[j][i];
            r0.w[i] = lds(a);
            r8.w[i] = lds(a + 512);
        }
        const LaneBlocks<F> b0 = lane_blocks<F>(r0, lc.sel);
        const LaneBlocks<F> b8 = lane_blocks<F>(r8, lc.sel);
        uint32_t e0[4], e8[4], o0[4], o8[4];
        decode<F>(b0.e, e0);
        decode<F>(b8.e, e8);
        decode<F>(b0.o, o0);
        decode<F>(b8.o, o8);
        float ce[4], co[4];
        mma0(ce, e0[0], e8[0], e0[1], e8[1], fe.x, fe.y);
        mma0(co, o0[0], o8[0], o0[1], o8[1], fo.x, fo.y);
        mma1(ce, e0[2], e8[2], e0[3], e8[3], fe.z, fe.w);
        mma1(co, o0[2], o8[2], o0[3], o8[3], fo.z, fo.w);
        ak[0] = fmaf(b0.de, ce[0], ak[0]);
        ak[2] = fmaf(b8.de, ce[2], ak[2]);
        ak[0] = fmaf(b0.dd, co[0], ak[0]);
        ak[2] = fmaf(b8.dd, co[2], ak[2]);
        if constexpr (!B1) {
            ak[1] = fmaf(b0.de, ce[1], ak[1]);
            ak[3] = fmaf(b8.de, ce[3], ak[3]);
            ak[1] = fmaf(b0.dd, co[1], ak[1]);
            ak[3] = fmaf(b8.dd, co[3], ak[3]);
        }
        if constexpr (F == FMT_Q4_1) {
            const float se = ldsf(xs0 + (2 * j) * 4), so = ldsf(xs0 + (2 * j + 1) * 4);
            ak[0] = fmaf(b0.me, se, fmaf(b0.md, so, ak[0]));
            ak[2] = fmaf(b8.me, se, fmaf(b8.md, so, ak[2]));
            if constexpr (!B1) {
                const float se1 = ldsf(xs1 + (2 * j) * 4), so1 = ldsf(xs1 + (2 * j + 1) * 4);
                ak[1] = fmaf(b0.me, se1, fmaf(b0.md, so1, ak[1]));
                ak[3] = fmaf(b8.me, se1, fmaf(b8.md, so1, ak[3]));
            }
        }
    }
}

// Exact fp32 path for a flagged chunk (rare: see the file header).  Same
// words as the fast path; x read in fp32 from global memory; each lane sums
// its own columns, the four lanes of a row are reduced with shuffles.
// Results are in unscaled units, returned by value (registers).
struct AkOut { float v[4]; };

template <int F, bool B1>
__device__ __noinline__ AkOut unit_slow(uint32_t sb, const LaneCtx<F> lc, const float *x, int ncols, int batch,
                                        int kb0, int w, int c, int n0, int n1) {
    AkOut out;
    out.v[0] = out.v[1] = out.v[2] = out.v[3] = 0.0f;
    for (int j = 0; j < 2; ++j) {
        for (int h = 0; h < 2; ++h) {
            RowWords<F> r;
            for (int i = 0; i < PairWords<F>::NW; ++i) r.w[i] = lds(sb + lc.off[j][i] + 512u * h);
            const LaneBlocks<F> lb = lane_blocks<F>(r, lc.sel);
            for (int par = 0; par < 2; ++par) {
                const int blk = kb0 + 2 * (w + kCW * j) + par;
                int off[4];
                piece_offsets<F>(par, c, off);
                const float d = par ? lb.dd : lb.de;
                const float mm = par ? lb.md : lb.me;
                for (int n = 0; n < batch; ++n) {
                    const float *xb = x + static_cast<size_t>(n) * ncols + static_cast<size_t>(blk) * 32;
                    float dot = 0.0f, sx = 0.0f;
                    for (int q = 0; q < 8; ++q) {
                        int col, val;
                        if constexpr (F == FMT_Q8_0) {
                            const uint32_t wd = par ? lb.o[q >> 2] : lb.e[q >> 2];
                            const int byte = static_cast<int>((wd >> (8 * (q & 3))) & 0xffu);
                            val = byte >= 128 ? byte - 256 : byte;
                            col = off[q >> 1] + (q & 1);
                        } else {
                            const uint32_t wd = par ? lb.o[0] : lb.e[0];
                            const int bi = q & 3, hi = q >> 2;   // byte bi of the word, low / high nibble
                            const int byte = static_cast<int>((wd >> (8 * bi)) & 0xffu);
                            const int nib = hi ? byte >> 4 : byte & 15;
                            val = F == FMT_Q4_0 ? nib - 8 : nib;
                            // byte bi sits at column off[bi >> 1] + (bi & 1)
                            col = off[bi >> 1] + (bi & 1) + (hi ? 16 : 0);
                        }
                        const float xv = xb[col];
                        dot = fmaf(static_cast<float>(val), xv, dot);
                        sx += xv;
                    }
                    dot += __shfl_xor_sync(0xffffffffu, dot, 1);
                    dot += __shfl_xor_sync(0xffffffffu, dot, 2);
                    float v = d * dot;
                    if constexpr (F == FMT_Q4_1) {
                        sx += __shfl_xor_sync(0xffffffffu, sx, 1);
                        sx += __shfl_xor_sync(0xffffffffu, sx, 2);
                        v = fmaf(mm, sx, v);
                    }
                    if (n == n0) out.v[2 * h] += v;
                    if (!B1 && n == n1) out.v[2 * h + 1] += v;
                }
            }
        }
    }
    return out;
}

// CTA owning linear unit `pos` (ranges [floor(i U / G), floor((i+1) U / G))).
__device__ __forceinline__ int cta_of(int pos, int U, int G) {
    return static_cast<int>((static_cast<int64_t>(pos + 1) * G - 1) / U);
}
__device__ __forceinline__ int range_lo(int i, int U, int G) {
    return static_cast<int>(static_cast<int64_t>(i) * U / G);
}

// The consumer warps' main loop over the CTA's units (SLOW: this warp has a
// flagged chunk, so every unit checks its chunk's flag and may take the exact
// fp32 path; the common instantiation carries neither the check nor the call).
template <int F, bool B1> struct ConsCtx {
    const uint8_t *smem;
    uint64_t *full, *empty, *ppbar;
    volatile int *abort_flag;
    LaneCtx<F> lc;
    const int *wfw;
    uint32_t ring, xfw, usw, xsw, pp;
    float *partb;
    int u0, nunits, nu, tgL, npart, cta, g, c, lane, wid, batch, n0, n1, NS, nv;
    bool owner, ok;
};

template <int F, bool B1, bool SLOW>
__device__ __forceinline__ void consume(const SkParams &p, const ConsCtx<F, B1> &cx) {
    constexpr uint32_t SLOT = sk_slot_bytes(F);
    const LaneCtx<F> &lc = cx.lc;
    uint64_t *full = cx.full, *empty = cx.empty, *ppbar = cx.ppbar;
    volatile int *abort_flag = cx.abort_flag;
    const int *wfw = cx.wfw;
    const uint32_t ring = cx.ring, xfw = cx.xfw, usw = cx.usw, xsw = cx.xsw;
    float *partb = cx.partb;
    const int u0 = cx.u0, nunits = cx.nunits, nu = cx.nu, tgL = cx.tgL, npart = cx.npart, cta = cx.cta;
    const int g = cx.g, c = cx.c, lane = cx.lane, wid = cx.wid, batch = cx.batch, n0 = cx.n0, n1 = cx.n1;
    const int NS = cx.NS, nv = cx.nv;
    const bool owner = cx.owner;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    int s = 0;
    uint32_t phase = 0;
    bool ok = cx.ok;
    int seg = 0;
    int tg = u0 / nu, ku = u0 - tg * nu;
    for (int k = 0; k < nunits; ++k) {
        float ak[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (ok) {
            // (every lane probes the same barrier in the same instruction:
            // `got` is warp-uniform)
            bool got = mbar_test(&full[s], phase);
            unsigned ns = 32;
            for (unsigned i = 0; i < p.probes && !got; ++i) {
                __nanosleep(ns);
                got = mbar_test(&full[s], phase);
                if (ns < 256) ns <<= 1;
                if (*abort_flag) break;
            }
            ok = got;
            if (!ok && lane == 0) {
                *abort_flag = 1;
                atomicOr(p.err, ERRBIT_TIMEOUT);
            }
        }
        float u0s = 1.0f, u1s = 1.0f;
        if (ok) {
            const uint32_t sb = ring + static_cast<uint32_t>(s) * SLOT;
            const int it = ku * p.batch;
            if (!SLOW || wfw[ku] == 0) {
                unit_fast<F, B1>(sb, lc, xfw + static_cast<uint32_t>(it * 256), xsw + static_cast<uint32_t>((it + n0) * 16),
                                 xsw + static_cast<uint32_t>((it + n1) * 16), ak);
                u0s = ldsf(usw + static_cast<uint32_t>((it + n0) * 4));
                u1s = ldsf(usw + static_cast<uint32_t>((it + n1) * 4));
            } else if constexpr (SLOW) {
                const AkOut r = unit_slow<F, B1>(sb, lc, p.x, p.ncols, p.batch, ku * kUB, wid, c, n0, n1);
                ak[0] = r.v[0]; ak[1] = r.v[1]; ak[2] = r.v[2]; ak[3] = r.v[3];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == NS) { s = 0; phase ^= 1u; }
        acc[0] = fmaf(ak[0], u0s, acc[0]);
        acc[2] = fmaf(ak[2], u0s, acc[2]);
        if constexpr (!B1) {
            acc[1] = fmaf(ak[1], u1s, acc[1]);
            acc[3] = fmaf(ak[3], u1s, acc[3]);
        }
        const int u = u0 + k;
        if (k == nunits - 1 || ku == nu - 1) {
            // ---- end of this CTA's part of row group tg: sum the warps
            float *pw = partb + ((seg & 1) * kCW + wid) * nv;
            const int ra = g, rb = g + 8;
            if (B1) {
                if (c == 0) {
                    pw[ra] = acc[0];
                    pw[rb] = acc[2];
                }
            } else {
                if (2 * c < batch) {
                    pw[ra * batch + 2 * c] = acc[0];
                    pw[rb * batch + 2 * c] = acc[2];
                }
                if (2 * c + 1 < batch) {
                    pw[ra * batch + 2 * c + 1] = acc[1];
                    pw[rb * batch + 2 * c + 1] = acc[3];
                }
            }
            acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
            consumer_bar();
            if (wid == 0) {
                const float *pb = partb + (seg & 1) * kCW * nv;
                const bool whole = max(u0, tg * nu) == tg * nu && u + 1 == tg * nu + nu;
                const bool own = !whole && tg == tgL && owner;
                constexpr int kPer = (RT * (B1 ? 1 : QGEMV_MAX_BATCH) + 31) / 32;
                float vals[kPer];
#pragma unroll
                for (int q = 0; q < kPer; ++q) {
                    const int v = lane + 32 * q;
                    float sum = 0.0f;
                    if (v < nv) {
                        sum = pb[v];
#pragma unroll 4
                        for (int ww = 1; ww < kCW; ++ww) sum += pb[ww * nv + v];
                    }
                    vals[q] = sum;
                }
                const int row0 = tg * RT;
                if (whole || own) {
                    if (own && !mbar_wait_hint(ppbar, 0, p.probes) && lane == 0) {
                        *abort_flag = 1;
                        atomicOr(p.err, ERRBIT_TIMEOUT);
                    }
                    const float *pp = reinterpret_cast<const float *>(cx.smem) + cx.pp / 4;
#pragma unroll
                    for (int q = 0; q < kPer; ++q) {
                        const int v = lane + 32 * q;
                        if (v < nv) {
                            float sum = vals[q];
                            if (own) {
                                for (int i = 0; i < npart; ++i) sum += pp[i * nv + v];
                            }
                            const int r = v / batch, n = v - r * batch;
                            if (row0 + r < p.nrows) p.y[static_cast<int64_t>(n) * p.nrows + row0 + r] = sum;
                        }
                    }
                } else {
                    // a later part of a shared row group: publish it for the owner
                    float *mine = p.part + static_cast<size_t>(cta) * nv;
#pragma unroll
                    for (int q = 0; q < kPer; ++q) {
                        const int v = lane + 32 * q;
                        if (v < nv) __stcg(mine + v, vals[q]);
                    }
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) st_release(p.flag + cta, 1u);
                }
            }
            ++seg;
        }
        if (++ku == nu) {
            ku = 0;
            ++tg;
        }
    }
}

// ------------------------------------------------------------------ kernel
template <int F, bool B1>
__global__ void __launch_bounds__(kThreads, 1)
gemv_sk_kernel(const __grid_constant__ CUtensorMap tmap, const SkParams p) {
    constexpr uint32_t SLOT = sk_slot_bytes(F);
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int nu = p.nu, U = p.U, G = p.G, NS = p.ns;
    const int cta = blockIdx.x;
    const int u0 = range_lo(cta, U, G), u1 = range_lo(cta + 1, U, G);
    const int nunits = u1 - u0;
    const SkLayout L = sk_layout(F, nu, p.batch, NS, p.xs);
    const uint32_t ring = smem_u32(smem + L.ring);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + NS;
    uint64_t *ppbar = empty + NS;
    uint64_t *xbar = ppbar + 1;                  // [nu], bulk-copied x only
    int *issued = reinterpret_cast<int *>(smem + L.issued);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.flag);
    const int nv = RT * p.batch;                 // values of one row group's partial

    // the CTA's last row group: whole, or shared with the next CTAs (then
    // this CTA owns it exactly when it holds the group's first unit)
    const int tgL = (u1 - 1) / nu;
    const bool last_split = !(max(u0, tgL * nu) == tgL * nu && u1 == tgL * nu + nu);
    const bool owner = last_split && u0 <= tgL * nu;
    const int npart = owner ? cta_of(tgL * nu + nu - 1, U, G) - cta : 0;

    griddep_launch_dependents();

    auto issue = [&](int k) {
        if (k == 0 && p.withhold && cta == 0) return;     // testing the timeout path
        const int s = k % NS;
        const int u = u0 + k;
        const int tg = u / nu, ku = u - tg * nu;
        mbar_arrive_expect_tx(&full[s], SLOT);
        tma_load_3d(ring + static_cast<uint32_t>(s) * SLOT, &tmap, 0, tg * RT, ku * SkFmt<F>::BB, &full[s]);
        issued[s] += 1;
    };

    if (wid == kCW && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
            issued[s] = 0;
        }
        mbar_init(ppbar, 1);
        if (p.xs) {
            for (int q = 0; q < nu; ++q) mbar_init(&xbar[q], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int first = min(NS, nunits);
    // units copied before x (direct loads: two, so that they do not delay them)
    const int ahead = p.xs ? first : min(first, p.pre);
    if (wid == kCW) {
        // ------------------------------------------------ producer warp
        if (lane == 0 && p.early) {
            for (int k = 0; k < ahead; ++k) issue(k);
        }
        griddep_wait();
        if (lane == 0) {
            if (p.xs) {
                // x chunks in the order this CTA's units need them
                const int ku0 = u0 % nu;
                for (int q = 0; q < nu; ++q) {
                    const int ku = ku0 + q < nu ? ku0 + q : ku0 + q - nu;
                    mbar_arrive_expect_tx(&xbar[ku], static_cast<uint32_t>(p.batch) * 8192u);
                    for (int n = 0; n < p.batch; ++n) {
                        const size_t e0 = static_cast<size_t>(n) * p.ncols + static_cast<size_t>(ku) * 2048;
                        bulk_g2s(smem + L.x32 + e0 * 4, p.x + e0, 8192u, &xbar[ku]);
                    }
                }
            }
            if (!p.early) {
                for (int k = 0; k < ahead; ++k) issue(k);
            }
        }
        if (!p.xs) xready_wait();
        if (lane == 0) {
            for (int k = ahead; k < first; ++k) issue(k);
            // refill each slot as soon as all consumer warps released it
            for (int k = first; k < nunits; ++k) {
                const int s = k % NS;
                if (!mbar_wait_hint(&empty[s], static_cast<uint32_t>(k / NS - 1) & 1u, p.probes) || *abort_flag) {
                    atomicOr(p.err, ERRBIT_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                issue(k);
            }
            if (owner) {
                // partials of the CTAs sharing the last row group, in CTA order
                float *pp = reinterpret_cast<float *>(smem + L.pp);
                for (int q = 0; q < npart; ++q) {
                    const int i = cta + 1 + q;
                    bool got = false;
                    for (unsigned t = 0; t < p.probes && !*abort_flag; ++t) {
                        if (ld_acquire(p.flag + i) != 0u) {
                            got = true;
                            break;
                        }
                        __nanosleep(200);
                    }
                    if (!got) {
                        *abort_flag = 1;
                        atomicOr(p.err, ERRBIT_TIMEOUT);
                        break;
                    }
                    const float *src = p.part + static_cast<size_t>(i) * nv;
                    for (int v = 0; v < nv; ++v) pp[q * nv + v] = __ldcg(src + v);
                    p.flag[i] = 0u;            // cleared for the next call (after this one completes)
                }
            }
            mbar_arrive(ppbar);
        }
    } else {
        // ------------------------------------------------ consumer warps
        griddep_wait();                         // x, y, scratch: after the preceding kernel
        const uint32_t x32 = p.xs ? smem_u32(smem + L.x32) : 0u;
        clear_wide(p, wid, lane, smem, L, 0, nu);
        if (p.xs) {
            // all chunks of x, then all fragments at once (several items in
            // flight per lane)
            bool got = true;
            for (int q = 0; q < nu; ++q) got = got && mbar_wait_hint(&xbar[q], 0, p.probes);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) {
                    *abort_flag = 1;
                    atomicOr(p.err, ERRBIT_TIMEOUT);
                }
            } else {
                stage_items<F>(p, wid, lane, smem, L, x32, 0, nu * p.batch, false);
            }
        } else {
            stage_items<F>(p, wid, lane, smem, L, 0u, 0, nu * p.batch, true);
        }

        LaneCtx<F> lc;
        {
            int o[PairWords<F>::NW];
            PairWords<F>::offsets(c, o);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int pb = SkFmt<F>::PB * (wid + kCW * j);
#pragma unroll
                for (int i = 0; i < PairWords<F>::NW; ++i) lc.off[j][i] = sk_off(pb + o[i], g);
            }
            lc.sel = c == 3 ? 0x5432u : 0x3210u;
        }
        const int batch = B1 ? 1 : p.batch;
        const int items = nu * p.batch;
        const int ncol = min(g, batch - 1);          // B columns past the batch repeat the last one
        const int n0 = min(2 * c, batch - 1), n1 = min(2 * c + 1, batch - 1);
        const uint32_t xfw = smem_u32(smem + L.xf) + static_cast<uint32_t>(wid * items * 256 + ncol * 256 + c * 16);
        const uint32_t usw = smem_u32(smem + L.us) + static_cast<uint32_t>(wid * items * 4);
        const int *wfw = reinterpret_cast<const int *>(smem + L.wf) + wid * nu;
        const uint32_t xsw = smem_u32(smem + L.xs) + static_cast<uint32_t>(wid * items * 16);
        float *partb = reinterpret_cast<float *>(smem + L.part);

        ConsCtx<F, B1> cx;
        cx.smem = smem;
        cx.full = full;
        cx.empty = empty;
        cx.ppbar = ppbar;
        cx.abort_flag = abort_flag;
        cx.lc = lc;
        cx.wfw = wfw;
        cx.ring = ring;
        cx.xfw = xfw;
        cx.usw = usw;
        cx.xsw = xsw;
        cx.pp = L.pp;
        cx.partb = partb;
        cx.u0 = u0;
        cx.nunits = nunits;
        cx.nu = nu;
        cx.tgL = tgL;
        cx.npart = npart;
        cx.cta = cta;
        cx.g = g;
        cx.c = c;
        cx.lane = lane;
        cx.wid = wid;
        cx.batch = batch;
        cx.n0 = n0;
        cx.n1 = n1;
        cx.NS = NS;
        cx.nv = nv;
        cx.owner = owner;
        cx.ok = !*abort_flag;
        // a warp with a flagged chunk (or too many chunks for a mask) runs the
        // loop that can take the exact path
        bool slow = nu > 32;
        for (int q = 0; q < nu && !slow; ++q) slow = wfw[q] != 0;
        if (slow) consume<F, B1, true>(p, cx);
        else consume<F, B1, false>(p, cx);
    }
    __syncthreads();
    if (*abort_flag && tid == 0) {
        // a wait gave up: let every copy still in flight land before exiting
        for (int s = 0; s < NS; ++s) {
            if (issued[s] > 0) mbar_wait_bounded(&full[s], static_cast<uint32_t>(issued[s] - 1) & 1u, p.err);
        }
        if (p.xs) {
            for (int q = 0; q < nu; ++q) mbar_wait_bounded(&xbar[q], 0, p.err);
        }
    }
}

// ------------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Tensor maps of weight matrices, cached by (address, rows, row bytes, box
// pieces).  The view is 3-D -- (64 bytes, row, 64-byte piece of the row) with
// strides (1, row bytes, 64) -- so one box of (64, 16, BB) lands as
// [piece][row][64 B] with the 64-byte swizzle; rows past nrows read as zero.
struct MapEntry {
    const void *ptr = nullptr;
    int64_t nrows = 0, rowbytes = 0;
    int nz = 0;
    CUtensorMap map;
};
constexpr int kMapCache = 32;
std::mutex g_map_mutex;
MapEntry g_maps[kMapCache];
int g_map_next = 0;
EncodeTiledFn g_encode = nullptr;

qgemv_status weight_map(const void *W, int64_t nrows, int64_t rowbytes, int nz, CUtensorMap *out) {
    std::lock_guard<std::mutex> lk(g_map_mutex);
    for (int i = 0; i < kMapCache; ++i) {
        const MapEntry &e = g_maps[i];
        if (e.ptr == W && e.nrows == nrows && e.rowbytes == rowbytes && e.nz == nz) {
            *out = e.map;
            return QGEMV_OK;
        }
    }
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
            set_last_error("cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(e));
            return QGEMV_ERR_CUDA;
        }
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    MapEntry &e = g_maps[g_map_next];
    g_map_next = (g_map_next + 1) % kMapCache;
    const cuuint64_t gdim[3] = {64u, static_cast<cuuint64_t>(nrows), static_cast<cuuint64_t>(rowbytes / 64)};
    const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(rowbytes), 64u};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(RT), static_cast<cuuint32_t>(nz)};
    const cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = g_encode(&e.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(W), gdim, gstride, box,
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

// Scratch set of a (device, stream): streams get sets round-robin in the
// order they are first seen on a device, and keep them.
constexpr int kMaxDev = 64;
constexpr int kStreamTab = 64;
struct StreamSet {
    int dev = -1;
    cudaStream_t s = nullptr;
    int set = 0;
};
std::mutex g_set_mutex;
StreamSet g_stream_tab[kStreamTab];
int g_stream_next = 0;
int g_set_rr[kMaxDev] = {0};
float *g_part_base[kMaxDev] = {nullptr};
unsigned *g_flag_base[kMaxDev] = {nullptr};

qgemv_status scratch_for(int dev, cudaStream_t s, float **part, unsigned **flag) {
    std::lock_guard<std::mutex> lk(g_set_mutex);
    if (!g_part_base[dev]) {
        void *a = nullptr, *b = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&a, g_sk_part);
        if (e == cudaSuccess) e = cudaGetSymbolAddress(&b, g_sk_flag);
        if (e != cudaSuccess) {
            set_last_error("cudaGetSymbolAddress(GEMV scratch): %s", cudaGetErrorString(e));
            return QGEMV_ERR_CUDA;
        }
        g_part_base[dev] = static_cast<float *>(a);
        g_flag_base[dev] = static_cast<unsigned *>(b);
    }
    int set = -1;
    for (int i = 0; i < kStreamTab; ++i) {
        if (g_stream_tab[i].dev == dev && g_stream_tab[i].s == s) {
            set = g_stream_tab[i].set;
            break;
        }
    }
    if (set < 0) {
        set = g_set_rr[dev];
        g_set_rr[dev] = (g_set_rr[dev] + 1) % kSkSets;
        StreamSet &e = g_stream_tab[g_stream_next];
        g_stream_next = (g_stream_next + 1) % kStreamTab;
        e.dev = dev;
        e.s = s;
        e.set = set;
    }
    *part = g_part_base[dev] + static_cast<size_t>(set) * kSkSlotFloats;
    *flag = g_flag_base[dev] + static_cast<size_t>(set) * kSkMaxG;
    return QGEMV_OK;
}

struct SkPlan {
    int dev = -1, fmt = -1, batch = 0;
    int64_t nrows = 0, ncols = 0;
    int ns = 0, G = 0, xs = 0;
    size_t smem = 0;
};
constexpr int kPlanCache = 64;
std::mutex g_plan_mutex;
SkPlan g_plans[kPlanCache];
int g_plan_next = 0;

template <int F, bool B1>
bool set_smem_attr(int dev, size_t optin) {
    static bool done[kMaxDev] = {false};
    if (done[dev]) return true;
    if (cudaFuncSetAttribute(gemv_sk_kernel<F, B1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(optin)) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    done[dev] = true;
    return true;
}

template <int F>
bool make_plan(int dev, int64_t nrows, int64_t ncols, int batch, const DevInfo &di, SkPlan *out) {
    {
        std::lock_guard<std::mutex> lk(g_plan_mutex);
        for (int i = 0; i < kPlanCache; ++i) {
            const SkPlan &q = g_plans[i];
            if (q.dev == dev && q.fmt == F && q.batch == batch && q.nrows == nrows && q.ncols == ncols) {
                *out = q;
                return q.G > 0;
            }
        }
    }
    SkPlan pl;
    pl.dev = dev;
    pl.fmt = F;
    pl.batch = batch;
    pl.nrows = nrows;
    pl.ncols = ncols;
    const int nu = static_cast<int>(ncols / 2048);
    const size_t budget = di.smem_optin;
    const uint32_t slot = sk_slot_bytes(F);
    // x in shared memory when a ring of >= 4 units still fits (and <= 32 chunk
    // barriers), else direct loads
    for (int xs = (nu <= 32 ? 1 : 0); xs >= 0; --xs) {
        const SkLayout L0 = sk_layout(F, nu, batch, 0, xs);
        if (static_cast<size_t>(L0.total) + 1024 + 4u * (slot + 20) > budget) continue;
        int ns = static_cast<int>((budget - 1024 - L0.total) / (slot + 20));
        if (ns > kMaxSlots) ns = kMaxSlots;
        const SkLayout L = sk_layout(F, nu, batch, ns, xs);
        if (static_cast<size_t>(L.total) + 1024 <= budget) {
            const int64_t U = (nrows + RT - 1) / RT * nu;
            // every range holds >= ceil(nu / 4) units: a row group spans <= 5 CTAs
            int64_t G = U / ((nu + 3) / 4);
            if (G > di.sm_count) G = di.sm_count;
            if (G > kSkMaxG) G = kSkMaxG;
            if (G < 1) G = 1;
            pl.ns = ns;
            pl.G = static_cast<int>(G);
            pl.smem = static_cast<size_t>(L.total) + 1024;
            pl.xs = xs;
            break;
        }
    }
    {
        std::lock_guard<std::mutex> lk(g_plan_mutex);
        g_plans[g_plan_next] = pl;
        g_plan_next = (g_plan_next + 1) % kPlanCache;
    }
    *out = pl;
    return pl.G > 0;
}

template <int F, bool B1>
qgemv_status launch_k(const SkPlan &pl, const void *W, const SkParams &p, cudaStream_t s, const DevInfo &di) {
    if (!set_smem_attr<F, B1>(pl.dev, di.smem_optin)) {
        set_last_error("qgemv(stream-K): cannot raise the shared-memory limit");
        return QGEMV_ERR_LAUNCH;
    }
    const int64_t rowbytes = pl.ncols / 32 * block_bytes(F);
    CUtensorMap map;
    qgemv_status ms = weight_map(W, pl.nrows, rowbytes, SkFmt<F>::BB, &map);
    if (ms != QGEMV_OK) return ms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(pl.G));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_sk_kernel<F, B1>, map, p);
    if (e != cudaSuccess) {
        set_last_error("qgemv(stream-K) launch: %s", cudaGetErrorString(e));
        return QGEMV_ERR_LAUNCH;
    }
    return check_launch("qgemv(stream-K)");
}

template <int F>
qgemv_status launch_sk_fmt(const void *W, const float *x, float *y, int64_t nrows, int64_t ncols, int batch,
                           cudaStream_t s, const DevInfo &di, unsigned *err, bool *taken) {
    *taken = false;
    if (ncols % 2048 != 0 || nrows < 1 || nrows > (1 << 28) || ncols > (1 << 24)) return QGEMV_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return QGEMV_OK;
    SkPlan pl;
    if (!make_plan<F>(dev, nrows, ncols, batch, di, &pl)) return QGEMV_OK;
    const int nu = static_cast<int>(ncols / 2048);
    const int64_t ngroups = (nrows + RT - 1) / RT;
    if (ngroups * nu > (int64_t(1) << 30)) return QGEMV_OK;
    SkParams p;
    p.x = x;
    p.y = y;
    p.err = err;
    qgemv_status st = scratch_for(dev, s, &p.part, &p.flag);
    if (st != QGEMV_OK) return st;
    p.nrows = static_cast<int>(nrows);
    p.ncols = static_cast<int>(ncols);
    p.batch = batch;
    p.nu = nu;
    p.U = static_cast<int>(ngroups * nu);
    p.G = pl.G;
    p.ns = pl.ns;
    p.early = g_opt_weights_static;
    p.xs = pl.xs;
    p.pre = 2;
    p.probes = g_opt_wait_probes;
    p.withhold = g_opt_withhold_next;
    g_opt_withhold_next = 0;
    *taken = true;
    return batch == 1 ? launch_k<F, true>(pl, W, p, s, di) : launch_k<F, false>(pl, W, p, s, di);
}

}  // namespace

qgemv_status launch_gemv_sk(int fmt, const void *W, const float *x, float *y, int64_t nrows, int64_t ncols,
                            int batch, cudaStream_t s, const DevInfo &di, unsigned *err, bool *taken) {
    switch (fmt) {
    case FMT_Q4_0: return launch_sk_fmt<FMT_Q4_0>(W, x, y, nrows, ncols, batch, s, di, err, taken);
    case FMT_Q4_1: return launch_sk_fmt<FMT_Q4_1>(W, x, y, nrows, ncols, batch, s, di, err, taken);
    case FMT_Q8_0: return launch_sk_fmt<FMT_Q8_0>(W, x, y, nrows, ncols, batch, s, di, err, taken);
    default:
        *taken = false;
        return QGEMV_OK;
    }
}

// Flags of every scratch set of the current device back to zero (after a
// kernel gave up mid-call, a flag may still be raised).
void gemv_sk_reset_scratch() {
    void *b = nullptr;
    if (cudaGetSymbolAddress(&b, g_sk_flag) == cudaSuccess) {
        cudaMemset(b, 0, sizeof(unsigned) * kSkSets * kSkMaxG);
    }
    cudaGetLastError();
}

}  // namespace qg
