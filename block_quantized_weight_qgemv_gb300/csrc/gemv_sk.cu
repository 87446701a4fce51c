// gemv_sk.cu -- block-quantized GEMV on the tensor cores with a stream-K
// split of the weight stream:  y[b][r] = sum_k w[r][k] * x[b][k], batch 1..8,
// Q4_0 / Q4_1 / Q8_0 in ggml's block layout (the batch-1 "dequantize_mul_mat_vec"
// path of the "llama_cpp 0.12.1 -> 0.12.2" ggml-cuda.cu diff, extended to small
// batches; block formulas from its dequantize_block_q4_0 / _q4_1 / _q8_0_f16
// hunks).
//
// Work split.  The weights are cut into units of 16 rows x 64 blocks (one
// 3-D TMA box, 64-byte swizzle): row group tg, k chunk ku (2048 columns).
// CTA i of G (one per SM) takes the contiguous range [floor(i U / G),
// floor((i+1) U / G)) of the U units: every SM streams the same number of
// bytes (to within one unit).  Two numberings:
//  - row group major, u = tg nu + ku (nu chunks), when the staged x of all
//    chunks fits in shared memory.  A CTA then holds whole row groups
//    (summed in the CTA) plus at most a split group at each end of its range.
//    A split group is summed by the CTA holding its first unit (the owner,
//    for which it is the last group); every other CTA covering it has it as
//    its first group, finishes its part early and publishes it (scratch
//    slot, release flag); the owner's producer warp fetches those partials
//    (acquire) while the consumers still work, and the owner adds them in CTA
//    order.  Every range holds >= ceil(nu / 4) units, so a group falls to at
//    most 5 CTAs.
//  - k chunk major, u = ku NRG + tg (NRG row groups), otherwise (large
//    batches): a range touches one or two chunks, so their staged x fits.
//    Every unit's partial goes to a scratch array; each CTA then announces,
//    once, that its partials are stored (fence, atomic add), and the last M
//    CTAs to announce (M: enough for one pass over y) wait until every CTA
//    has and sum their share of y in k order; the others exit at once.
// Either way y is deterministic, and no CTA waits for another that could
// itself be waiting.
//
// Inside a CTA the 16 consumer warps split each unit by block pairs (warp w
// takes pairs w and w + 16) and accumulate over the units of one row group;
// at the end of the CTA's part of a group they leave their shares in a
// shared-memory slot, and a reducer warp adds them in warp order.
//
// Arithmetic: mma.sync m16n8k16 (fp16 operands, fp32 accumulation), the batch
// riding in the MMA's N dimension:
//  - A (weights) are the exact small integers q - 8 (Q4_0), q - q0 (Q4_1) or
//    q (Q8_0) in fp16: a logic op puts a nibble (byte) under the fp16 exponent
//    of 1024, an fp16 add / fma removes the offset exactly.
//  - B (activations): each warp scales the x values of its four blocks of a
//    k chunk (per batch column) by one power of two that puts their largest
//    magnitude in [2^9, 2^10) and rounds them to fp16 (relative error
//    <= 2^-11 while the scaled value is >= 2^-14).  A chunk holding a non-
//    finite value, or a nonzero value whose scaled magnitude would be below
//    2^-14 (a dynamic range above ~2^23 inside 128 values), is flagged and
//    computed exactly in fp32 on the CUDA cores instead.
//  - each block's fp32 MMA result is multiplied by its fp16 scale d (and for
//    Q4_1, whose codes enter as q - q0 with q0 the code nearest -m/d, the
//    block's sum of the rounded x times m + d q0 is added) on the CUDA
//    cores; each chunk's sum is scaled back by the exact power of two.
// Hence |y - exact| <= 2^-11 sum_k |w_k x_k| + fp32 accumulation error.
//
// Data movement.  A producer warp streams units through a ring of NS slots
// (one mbarrier-completed TMA copy each).  When the caller declared its
// weights static, four units are copied before the kernel waits on the
// preceding kernel of its stream (griddepcontrol.wait); the consumers then
// load their part of x (L2-resident after the first CTA touched it) and
// signal once those loads are in flight, and only then does the producer
// fill the rest of the ring (weight copies in flight delay plain loads).
//
// Expert-selected form (MUL_MAT_ID).  The same body, switched at compile
// time, computes output column b against matrix ids[b] of a stack of
// experts: every CTA scans ids and takes work unit blockIdx.y (up to 8
// columns of one expert, riding in the MMA's N dimension), loads that
// expert's units through a 4-D tensor map (expert outermost), gathers its x
// and y columns, and takes whole row groups only (CTA ranges cut at
// row-group boundaries), so no partial sum crosses CTAs and none of the
// scratch below is used.
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

#include <algorithm>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "qgemv_common.cuh"

namespace qg {

// Scratch: kSkSets independent sets (one per stream, see scratch_for), each
// with
//  - partials: row group major, one slot of 16 x batch floats per CTA (its
//    published part of a split group); k chunk major, [row group][k chunk]
//    [16 x batch] floats;
//  - one publish flag per CTA (row group major; the owner clears it);
//  - two counters (k chunk major: CTAs that stored their partials, finishing
//    CTAs done), each on a line of its own; the last finisher clears them.
// Zero-initialized.
constexpr int kSkSets = 8;
constexpr int kSkPartFloats = 1 << 19;
constexpr int kSkMaxG = 1024;
constexpr int kSkSyncWords = 64;
__device__ float g_sk_part[kSkSets * kSkPartFloats];
__device__ unsigned g_sk_flag[kSkSets * kSkMaxG];
__device__ unsigned g_sk_sync[kSkSets * kSkSyncWords];

// Probes of a wait before it gives up (qgemv_set_option(QGEMV_OPT_WAIT_PROBES));
// each probe sleeps <= 256 ns.
unsigned g_opt_wait_probes = 1u << 20;
// qgemv_set_option(QGEMV_OPT_TEST_WITHHOLD_COPY): the next launch withholds
// its first weight copy.
int g_opt_withhold_next = 0;

namespace {

constexpr int kCW = 16;                      // consumer warps
constexpr int PPW = 32 / kCW;                // block pairs of a unit per consumer warp
constexpr int kNR = 2;                       // reducer warps
constexpr int kProd = kCW;                   // warp index of the producer
constexpr int kRed0 = kCW + 1;               // warp index of the first reducer
constexpr int kThreads = (kCW + 1 + kNR) * 32;
constexpr int kUB = 64;                      // blocks per unit (k)
constexpr int RT = 16;                       // rows per unit
constexpr int kMaxSlots = 12;
constexpr int kMaxPartners = 4;              // other CTAs sharing the owner's last row group
template <bool B1> struct SkPs { static constexpr int v = B1 ? 8 : 4; };   // partial slots (a multiple of kNR)

template <int F> struct SkFmt;
template <> struct SkFmt<FMT_Q4_0> { static constexpr int BB = 18; static constexpr int PB = 36; };
template <> struct SkFmt<FMT_Q4_1> { static constexpr int BB = 20; static constexpr int PB = 40; };
template <> struct SkFmt<FMT_Q8_0> { static constexpr int BB = 34; static constexpr int PB = 68; };

__host__ __device__ constexpr uint32_t sk_slot_bytes(int F) { return static_cast<uint32_t>(64 * RT * block_bytes(F)); }
// Pair slot j of consumer warp w starts PB (w + kCW j) bytes into a unit
// row.  The slot's swizzle depends only on the row and on the byte inside a
// 64-byte piece, so pair slots whose starts differ by a multiple of 64 bytes
// share their word offsets up to a constant: the lane keeps `sets` offset
// sets (pair slots j mod sets) and adds (j / sets) * stride.
template <int F> struct SkPairs {
    static constexpr int span = SkFmt<F>::PB * kCW;            // bytes from pair slot j to j + 1
    static constexpr int sets = span % 64 == 0 ? 1 : ((2 * span) % 64 == 0 ? 2 : PPW);
    static constexpr uint32_t stride = static_cast<uint32_t>(sets * span / 64 * RT * 64);
};

struct SkParams {
    const float *x;
    float *y;
    unsigned *err;
    float *part;       // partials of this call's scratch set
    unsigned *flag;    // publish flags of this call's scratch set (row group major)
    unsigned *sync;    // counters of this call's scratch set: [0] stored, [32] finished (k chunk major)
    int nrows, ncols, batch;
    int nu;            // k chunks (ceil(ncols / 2048); a last chunk may hold 1024 columns)
    int ngr;           // row groups (ceil(nrows / 16))
    int U;             // units in total (ngr x nu)
    int G;             // CTAs
    int kmaj;          // 1: k chunk major numbering, 0: row group major
    int ns;            // ring slots
    int ch;            // k chunk slots staged (row group major: nu)
    int fin;           // finishing CTAs (k chunk major, nu > 1)
    int early;         // 1: weights may be copied before waiting on the preceding kernel
    int pre;           // units copied before the consumers' loads of x
    unsigned probes;   // wait limit
    int withhold;      // testing: never copy the first unit (its wait runs out)
};

// Element offsets of the batch columns in x and y for the expert-selected
// kernel (its columns are gathered); the plain kernel has column n at
// n * ncols and n * nrows.
struct SkCols {
    int64_t xo[QGEMV_MAX_BATCH], yo[QGEMV_MAX_BATCH];
};
template <bool ID> __device__ __forceinline__ int64_t col_x(const SkParams &p, const SkCols &cc, int n) {
    if constexpr (ID) return cc.xo[n];
    else return static_cast<int64_t>(n) * p.ncols;
}
template <bool ID> __device__ __forceinline__ int64_t col_y(const SkParams &p, const SkCols &cc, int n) {
    if constexpr (ID) return cc.yo[n];
    else return static_cast<int64_t>(n) * p.nrows;
}

// Shared-memory layout (offsets from a 1024-byte aligned base).  Warp w's
// staged B fragments for item it = (chunk slot) * batch + n are 2 PPW blocks
// x 4 lanes of 16 bytes at xf + (w ch batch + it) 128 PPW bytes.
struct SkLayout {
    uint32_t ring, xf, us, wf, xs, pslot, pp, bars, issued, flag, total;
};

__host__ __device__ inline uint32_t sk_align(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline SkLayout sk_layout(int F, int ch, int batch, int ns, int ps) {
    SkLayout L;
    const uint32_t items = static_cast<uint32_t>(kCW * ch * batch);
    uint32_t o = 0;
    L.ring = o;  o += static_cast<uint32_t>(ns) * sk_slot_bytes(F);
    L.xf = o;    o += items * 128u * PPW;
    L.us = o;    o += sk_align(items * 4, 16);
    L.wf = o;    o += sk_align(static_cast<uint32_t>(kCW * ch) * 4, 16);
    L.xs = o;    o += F == FMT_Q4_1 ? items * 8u * PPW : 0u;
    L.pslot = o; o += static_cast<uint32_t>(ps) * kCW * RT * batch * 4;
    L.pp = o;    o += static_cast<uint32_t>(kMaxPartners) * RT * batch * 4;
    L.bars = o;  o += static_cast<uint32_t>(2 * ns + 2 * ps + 1) * 8;     // full, empty, pfull, pempty, ppbar
    o = sk_align(o, 16);
    L.issued = o; o += sk_align(static_cast<uint32_t>(ns) * 4, 16);
    L.flag = o;  o += 16;                                   // abort flag, broadcast word
    L.total = o;
    return L;
}

// ------------------------------------------------------------ device helpers
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Barrier 0 with an explicit thread count, so that some warps can arrive
// without waiting (and exit) while the others wait.
template <int N> __device__ __forceinline__ void cta_arrive_all() {
    asm volatile("barrier.arrive 0, %0;" :: "n"(N) : "memory");
}
template <int N> __device__ __forceinline__ void cta_sync_all() {
    asm volatile("barrier.sync 0, %0;" :: "n"(N) : "memory");
}
// Barrier 2 (unaligned form, as cta_sync): the consumers signal that their loads of x are in flight; the
// producer holds the remaining weight copies until then.
constexpr int kXreadyThreads = (kCW + 1) * 32;
__device__ __forceinline__ void xready_arrive() {
    asm volatile("barrier.arrive 2, %0;" :: "n"(kXreadyThreads) : "memory");
}
__device__ __forceinline__ void xready_wait() {
    asm volatile("barrier.sync 2, %0;" :: "n"(kXreadyThreads) : "memory");
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
__device__ __forceinline__ void sts64(uint32_t a, uint32_t lo, uint32_t hi) {
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" :: "r"(a), "r"(lo), "r"(hi) : "memory");
}
__device__ __forceinline__ void st_release_u32(unsigned *a, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned *a) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}
__device__ __forceinline__ void sts(uint32_t a, float v) {
    asm volatile("st.shared.f32 [%0], %1;" :: "r"(a), "f"(v) : "memory");
}
// Weight copies carry an evict-first L2 policy: the weights stream through
// once per call and should not push x, y and the scratch out of L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *tmap, int c0, int c1, int c2,
                                            uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *tmap, int c0, int c1, int c2, int c3,
                                            uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar)),
           "l"(pol)
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
// `probes` sleeps, or early once another warp of the CTA has given up.
__device__ __forceinline__ bool mbar_wait_abortable(uint64_t *bar, uint32_t parity, unsigned probes,
                                                    volatile int *abort_flag) {
    if (mbar_test(bar, parity)) return true;
    unsigned ns = 32;
    for (unsigned i = 0; i < probes; ++i) {
        __nanosleep(ns);
        if (mbar_test(bar, parity)) return true;
        if (ns < 256) ns <<= 1;
        if (*abort_flag) return false;
    }
    return false;
}
// The same on 32-bit shared-memory addresses of barriers.
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
// The waits on the stream itself (consumers for a weight copy, the producer
// for a released slot) sleep a short, fixed 32 ns between probes: a longer
// sleep delays the next copy, and the TMA engine only keeps up with the HBM
// when every slot is refilled promptly.
__device__ __forceinline__ bool mbar_ready(uint32_t bar, uint32_t parity, unsigned probes, volatile int *abort_flag) {
    if (mbar_test_a(bar, parity)) return true;
    for (unsigned i = 0; i < probes; ++i) {
        __nanosleep(32);
        if (mbar_test_a(bar, parity)) return true;
        if (*abort_flag) return false;
    }
    return false;
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
// and the scales of one row as fp32.  Q4_1: the codes enter the MMA as
// q - q0 with q0 the code nearest -m / d (clamped to 0 .. 15), and me / md
// hold m + d q0: every weight d q + m then has a magnitude at least that of
// m + d q0, so neither d * sum((q - q0) x) nor (m + d q0) * sum(x) can be
// much larger than sum |w x| -- no cancellation between the two terms.
template <int F> struct LaneBlocks {
    uint32_t e[F == FMT_Q8_0 ? 2 : 1], o[F == FMT_Q8_0 ? 2 : 1];
    float de, dd, me, md;
    uint32_t qe, qo;                             // Q4_1: q0 of the even / odd block
};
__device__ __forceinline__ uint32_t q4_1_offset(float d, float m) {
    // any integer keeps the MMA exact; the nearest one to -m/d is what bounds
    // the two terms (an approximate quotient is enough)
    return static_cast<uint32_t>(min(max(__float2int_rn(__fdividef(-m, d)), 0), 15));
}
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
        b.dd = h_lo(r.w[1]);
        const float me = h_hi(r.w[0]), md = h_hi(r.w[1]);
        b.qe = q4_1_offset(b.de, me);
        b.qo = q4_1_offset(b.dd, md);
        b.me = fmaf(b.de, static_cast<float>(b.qe), me);
        b.md = fmaf(b.dd, static_cast<float>(b.qo), md);
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
// k-step (a0/a2 of this row), h[2], h[3] for the second.  q0: Q4_1 code
// offset (unused otherwise).
template <int F>
__device__ __forceinline__ void decode(const uint32_t (&wd)[F == FMT_Q8_0 ? 2 : 1], uint32_t h[4], uint32_t q0 = 0) {
    constexpr uint32_t kMagic = 0x64006400u;   // fp16 (1024, 1024)
    if constexpr (F == FMT_Q8_0) {
        constexpr uint32_t K = 0x64646464u, kOff = 0xE480E480u;   // -1152
        const uint32_t a = wd[0] ^ 0x80808080u, b = wd[1] ^ 0x80808080u;
        h[0] = hadd2(prmt(a, K, 0x4140), kOff);
        h[1] = hadd2(prmt(a, K, 0x4342), kOff);
        h[2] = hadd2(prmt(b, K, 0x4140), kOff);
        h[3] = hadd2(prmt(b, K, 0x4342), kOff);
    } else {
        // low nibbles: 1024 + q - (1024 + 8 | 1024 + q0); high nibbles (under
        // the magic as 1024 + 16 q): (1024 + 16 q) / 16 - (72 | 64 + q0).  In
        // fp16, -(1024 + q0) is 0xE400 | q0 and -(64 + q0) is 0xD400 | 16 q0.
        const uint32_t kLo = F == FMT_Q4_0 ? 0xE408E408u : 0xE400E400u | (q0 * 0x00010001u);
        const uint32_t kHi = F == FMT_Q4_0 ? 0xD480D480u : 0xD400D400u | ((q0 << 4) * 0x00010001u);
        constexpr uint32_t kSixteenth = 0x2C002C00u;                          // 1/16
        const uint32_t w = wd[0], w8 = wd[0] >> 8;
        h[0] = hadd2(and_or<0x000f000fu>(w, kMagic), kLo);
        h[1] = hadd2(and_or<0x000f000fu>(w8, kMagic), kLo);
        h[2] = hfma2(and_or<0x00f000f0u>(w, kMagic), kSixteenth, kHi);
        h[3] = hfma2(and_or<0x00f000f0u>(w8, kMagic), kSixteenth, kHi);
    }
}

// ------------------------------------------------------------ x staging
// Warp w stages, for the items it = kslot * batch + n (chunk ku_lo + kslot,
// batch column n; kslot < nch), the B fragments of its 2 PPW blocks of that
// chunk (pairs w + kCW j): lane f = l % LPI builds fragment (block X = f / 4,
// c = f % 4); the LPI-lane groups of the warp take consecutive items.  Per
// item the group finds the largest |x| of its 64 PPW values (as integer bit
// patterns, which also catches inf and nan), scales by 2^e, rounds to fp16,
// and flags the chunk when the fast path would lose more than fp16 rounding
// (see the file header): a non-finite value, or a nonzero value below 2^-14
// after scaling (found from the smallest nonzero magnitude); the caller
// clears the flags first.  x is read from global memory (L2) as coalesced
// 16-byte loads (an item is two runs of 64 consecutive values, one per block
// pair), converted in plain k order into a per-warp scratch in the partial-sum
// slots, and read back in the fragment order; with `arrive`, the warp arrives
// on barrier 2 once its first loads are in flight.
template <int F, bool ID>
__device__ __forceinline__ void stage_items(const SkParams &p, const SkCols &cc, int w, int lane, uint8_t *smem,
                                            const SkLayout &L, int ku_lo, int nch, bool arrive) {
    constexpr int LPI = 8 * PPW;                 // lanes per item
    constexpr int IPP = 32 / LPI;                // items per pass of the warp
    const int f = lane % LPI, hw = lane / LPI;
    const int blkX = f >> 2, c = f & 3;
    int off[4];
    piece_offsets<F>(blkX & 1, c, off);
    const int batch = p.batch;
    const int items = nch * batch;
    const int wit = p.ch * batch;                // item stride of a warp
    uint4 *xf = reinterpret_cast<uint4 *>(smem + L.xf) + static_cast<size_t>(w) * wit * (8 * PPW);
    float *us = reinterpret_cast<float *>(smem + L.us) + w * wit;
    int *wf = reinterpret_cast<int *>(smem + L.wf) + w * p.ch;
    float *xs = reinterpret_cast<float *>(smem + L.xs) + w * wit * 2 * PPW;
    // 512 bytes of this warp's in the partial-sum slots (idle until the units
    // start): the two items of a pass in plain k order, as fp16
    const uint32_t tmp = smem_u32(smem + L.pslot) + static_cast<uint32_t>(w) * 512u;
    // the lane's block (blkX) of its item inside the scratch
    const uint32_t tb = tmp + static_cast<uint32_t>(hw * 256 + (blkX >> 1) * 128 + (blkX & 1) * 64);
    constexpr int kIL = 4;                        // passes with loads in flight
    bool arrived = !arrive;
    for (int i0 = 0; i0 < items; i0 += IPP * kIL) {
        // v[t][sg]: values 4f .. 4f+3 of the item's segment sg (its blocks
        // 2w + 32 sg and 2w + 32 sg + 1, 64 consecutive values): the 16 lanes
        // of an item read each segment as one coalesced 256-byte run
        float4 v[kIL][2];
#pragma unroll
        for (int t = 0; t < kIL; ++t) {
            const int it = i0 + IPP * t + hw;
            const int ks = it < items ? it / batch : 0, n = it < items ? it - ks * batch : 0;
#pragma unroll
            for (int sg = 0; sg < 2; ++sg) {
                const int blk0 = (ku_lo + ks) * kUB + 2 * w + 32 * sg;
                // blocks past the row (the half last chunk) stage 0; both
                // blocks of a segment lie in the same half of the chunk
                const bool ld = it < items && blk0 * 32 < p.ncols;
                const float *src = p.x + col_x<ID>(p, cc, n) + static_cast<int64_t>(blk0) * 32 + 4 * f;
                v[t][sg] = ld ? __ldg(reinterpret_cast<const float4 *>(src)) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
        }
        if (!arrived) {
            xready_arrive();
            arrived = true;
        }
        // largest |x| bits, and smallest nonzero |x| bits minus one (zeros
        // wrap to the largest value and drop out of the minimum), per item;
        // the shuffle rounds of the group's passes are interleaved
        uint32_t mxs[kIL], mns[kIL];
#pragma unroll
        for (int t = 0; t < kIL; ++t) {
            const float vv[8] = {v[t][0].x, v[t][0].y, v[t][0].z, v[t][0].w, v[t][1].x, v[t][1].y, v[t][1].z, v[t][1].w};
            mxs[t] = 0u;
            mns[t] = 0xffffffffu;
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const uint32_t a = __float_as_uint(vv[h]) & 0x7fffffffu;
                mxs[t] = max(mxs[t], a);
                mns[t] = min(mns[t], a - 1u);
            }
        }
#pragma unroll
        for (int s = 1; s < LPI; s <<= 1) {
#pragma unroll
            for (int t = 0; t < kIL; ++t) {
                mxs[t] = max(mxs[t], __shfl_xor_sync(0xffffffffu, mxs[t], s));
                mns[t] = min(mns[t], __shfl_xor_sync(0xffffffffu, mns[t], s));
            }
        }
#pragma unroll
        for (int t = 0; t < kIL; ++t) {
            const int it0 = i0 + IPP * t;
            if (it0 >= items) break;                   // warp-uniform
            const int it = it0 + hw;
            const bool valid = it < items;
            const float vv[8] = {v[t][0].x, v[t][0].y, v[t][0].z, v[t][0].w, v[t][1].x, v[t][1].y, v[t][1].z, v[t][1].w};
            const uint32_t mx = mxs[t], mn1 = mns[t];
            const int be = static_cast<int>(mx >> 23);
            const int e = (mx == 0u || be >= 255) ? 0 : (be == 0 ? 120 : 136 - be);
            // a nonzero value is below 2^-14 after scaling by 2^e when its
            // magnitude is below 2^(be - 150): bits (be - 23) << 23 for be >= 24,
            // the subnormal 1 << (be - 1) below
            bool wide = be >= 255 || (be == 0 && mx != 0u);
            if (!wide && mn1 != 0xffffffffu && be >= 1) {
                const uint32_t thr = be >= 24 ? static_cast<uint32_t>(be - 23) << 23 : 1u << (be - 1);
                wide = mn1 + 1u < thr;
            }
            const float sc = pow2f(e);
            // scaled fp16 values in plain order to the scratch, then this
            // lane's fragment words (value pairs at off[h], off[h] + 1)
            sts64(tmp + static_cast<uint32_t>(hw * 256 + 8 * f), f16x2_rn(vv[0] * sc, vv[1] * sc),
                  f16x2_rn(vv[2] * sc, vv[3] * sc));
            sts64(tmp + static_cast<uint32_t>(hw * 256 + 128 + 8 * f), f16x2_rn(vv[4] * sc, vv[5] * sc),
                  f16x2_rn(vv[6] * sc, vv[7] * sc));
            __syncwarp();
            const uint32_t w0 = lds(tb + 2u * off[0]), w1 = lds(tb + 2u * off[1]);
            const uint32_t w2 = lds(tb + 2u * off[2]), w3 = lds(tb + 2u * off[3]);
            __syncwarp();                              // the next pass rewrites the scratch
            uint4 fr;
            if constexpr (F == FMT_Q8_0) {
                fr = make_uint4(w0, w1, w2, w3);
            } else {
                // (pa.x, pb.x) (pa.y, pb.y) (pc.x, pd.x) (pc.y, pd.y)
                fr = make_uint4(prmt(w0, w1, 0x5410u), prmt(w0, w1, 0x7632u), prmt(w2, w3, 0x5410u),
                                prmt(w2, w3, 0x7632u));
            }
            if (valid) {
                xf[it * (8 * PPW) + f] = fr;
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
                if (valid && c == 0) xs[it * 2 * PPW + blkX] = t4;
            }
        }
    }
    if (!arrived) xready_arrive();
    __syncwarp();
}

// ------------------------------------------------------------ one unit
// Per-lane word offsets (word i of pair slot q < sets, row g) inside a ring
// slot; row g + 8 is 512 bytes further, pair slot j at set j % sets plus
// (j / sets) * stride.
template <int F> struct LaneCtx {
    uint32_t off[SkPairs<F>::sets][PairWords<F>::NW];
    uint32_t sel;
};
template <int F> __device__ __forceinline__ uint32_t pair_word(const LaneCtx<F> &lc, int j, int i) {
    return lc.off[j % SkPairs<F>::sets][i] + static_cast<uint32_t>(j / SkPairs<F>::sets) * SkPairs<F>::stride;
}

// Fast path: the warp's PPW pair slots of the unit at sb (shared address).
// fb: shared address of this lane's fragment of block 0 for (chunk, its
// column); block X follows at + 64 X bytes.  xs0 / xs1 (Q4_1): shared
// addresses of the block sums for (chunk, n0) / (chunk, n1).
template <int F, bool B1>
__device__ __forceinline__ void unit_fast(uint32_t sb, const LaneCtx<F> &lc, uint32_t fb, uint32_t xs0,
                                          uint32_t xs1, float ak[4]) {
#pragma unroll
    for (int j = 0; j < PPW; ++j) {
        const uint4 fe = lds128(fb + (2 * j) * 64), fo = lds128(fb + (2 * j + 1) * 64);
        RowWords<F> r0, r8;
#pragma unroll
        for (int i = 0; i < PairWords<F>::NW; ++i) {
            const uint32_t a = sb + pair_word<F>(lc, j, i);
            r0.w[i] = lds(a);
            r8.w[i] = lds(a + 512);
        }
        const LaneBlocks<F> b0 = lane_blocks<F>(r0, lc.sel);
        const LaneBlocks<F> b8 = lane_blocks<F>(r8, lc.sel);
        uint32_t e0[4], e8[4], o0[4], o8[4];
        decode<F>(b0.e, e0, b0.qe);
        decode<F>(b8.e, e8, b8.qe);
        decode<F>(b0.o, o0, b0.qo);
        decode<F>(b8.o, o8, b8.qo);
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
__device__ __noinline__ AkOut unit_slow(uint32_t sb, const LaneCtx<F> lc, const float *x, const int64_t *xo,
                                        int ncols, int batch, int kb0, int w, int c, int n0, int n1) {
    AkOut out;
    out.v[0] = out.v[1] = out.v[2] = out.v[3] = 0.0f;
    for (int j = 0; j < PPW; ++j) {
        for (int h = 0; h < 2; ++h) {
            RowWords<F> r;
            for (int i = 0; i < PairWords<F>::NW; ++i) r.w[i] = lds(sb + pair_word<F>(lc, j, i) + 512u * h);
            const LaneBlocks<F> lb = lane_blocks<F>(r, lc.sel);
            for (int par = 0; par < 2; ++par) {
                const int blk = kb0 + 2 * (w + kCW * j) + par;
                if (blk * 32 >= ncols) continue;           // past the row: zero weights (TMA fill)
                int off[4];
                piece_offsets<F>(par, c, off);
                const float d = par ? lb.dd : lb.de;
                const float mm = par ? lb.md : lb.me;
                for (int n = 0; n < batch; ++n) {
                    const float *xb = x + (xo ? xo[n] : static_cast<int64_t>(n) * ncols) + static_cast<size_t>(blk) * 32;
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
                            val = F == FMT_Q4_0 ? nib - 8 : nib - static_cast<int>(par ? lb.qo : lb.qe);
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

__device__ __forceinline__ int range_lo(int i, int U, int G) {
    return static_cast<int>(static_cast<int64_t>(i) * U / G);
}

// Everything the consumer loop needs, gathered once (barriers by their
// 32-bit shared-memory addresses).
template <int F> struct ConsCtx {
    uint32_t fullA, emptyA, pfullA, pemptyA;
    volatile int *abort_flag;
    LaneCtx<F> lc;
    uint32_t ring, xfw, usw, xsw, pw;
    int u0, nunits, ku_lo, c, lane, wid, batch, n0, n1, NS;
};

// The consumer warps' loop over the CTA's units (SLOW: this warp has a
// flagged chunk, so every unit checks its chunk's flag and may take the exact
// fp32 path; the common instantiation carries neither the check nor the call).
// Per unit: wait for the weights, multiply, release the slot and add the
// result, scaled by the chunk's power of two, to the row group's sums; at
// the end of the CTA's part of a row group (every unit when k chunk major)
// leave the sums in the next partial slot.  Slots, barriers and their
// parities advance incrementally.
template <int F, bool B1, bool SLOW, bool ID>
__device__ __forceinline__ void consume(const SkParams &p, const SkCols &cc, const ConsCtx<F> &cx, const int *wfw) {
    constexpr uint32_t SLOT = sk_slot_bytes(F);
    constexpr int PS = SkPs<B1>::v;
    const LaneCtx<F> &lc = cx.lc;
    volatile int *abort_flag = cx.abort_flag;
    const int c = cx.c, lane = cx.lane, batch = cx.batch, n0 = cx.n0, n1 = cx.n1, g = lane >> 2;
    const int NS = cx.NS, ngr = p.ngr, nu = p.nu;
    const bool kmaj = p.kmaj != 0;
    const uint32_t share_b = static_cast<uint32_t>(RT * batch) * 4u;     // bytes of a warp's share of a sum
    const uint32_t item_b = static_cast<uint32_t>(batch) * 128u * PPW;   // fragment bytes of one chunk slot
    uint32_t sb = cx.ring, fA = cx.fullA, eA = cx.emptyA, phase = 0;     // ring slot s
    int s = 0;
    uint32_t pw = cx.pw, pfA = cx.pfullA, peA = cx.pemptyA, pph = 0;     // partial slot ps
    int ps = 0, nseg = 0;
    int ku, tg;
    if (kmaj) {
        ku = cx.u0 / ngr;
        tg = cx.u0 - ku * ngr;
    } else {
        tg = cx.u0 / nu;
        ku = cx.u0 - tg * nu;
    }
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int k = 0; k < cx.nunits; ++k) {
        // (every lane probes the same barrier in the same instruction: the
        // outcome is warp-uniform)
        if (!mbar_ready(fA, phase, p.probes, abort_flag)) {
            if (lane == 0) {
                *abort_flag = 1;
                atomicOr(p.err, ERRBIT_TIMEOUT);
            }
            return;
        }
        const int ks = ku - cx.ku_lo;
        float ak[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        float u0s = 1.0f, u1s = 1.0f;
        if (!SLOW || wfw[ks] == 0) {
            const uint32_t it = static_cast<uint32_t>(ks * batch);
            unit_fast<F, B1>(sb, lc, cx.xfw + static_cast<uint32_t>(ks) * item_b,
                             cx.xsw + (it + n0) * (8u * PPW), cx.xsw + (it + n1) * (8u * PPW), ak);
            u0s = ldsf(cx.usw + (it + n0) * 4u);
            if (!B1) u1s = ldsf(cx.usw + (it + n1) * 4u);
        } else if constexpr (SLOW) {
            const AkOut r = unit_slow<F, B1>(sb, lc, p.x, ID ? cc.xo : nullptr, p.ncols, batch, ku * kUB, cx.wid, c,
                                             n0, n1);
            ak[0] = r.v[0]; ak[1] = r.v[1]; ak[2] = r.v[2]; ak[3] = r.v[3];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_a(eA);
        if (++s == NS) {
            s = 0;
            phase ^= 1u;
            sb = cx.ring;
            fA = cx.fullA;
            eA = cx.emptyA;
        } else {
            sb += SLOT;
            fA += 8;
            eA += 8;
        }
        acc[0] = fmaf(ak[0], u0s, acc[0]);
        acc[2] = fmaf(ak[2], u0s, acc[2]);
        if (!B1) {
            acc[1] = fmaf(ak[1], u1s, acc[1]);
            acc[3] = fmaf(ak[3], u1s, acc[3]);
        }
        // next unit, and whether this one ends the CTA's part of its row group
        bool seg_end = k == cx.nunits - 1;
        if (kmaj) {
            seg_end = true;
            if (++tg == ngr) {
                tg = 0;
                ++ku;
            }
        } else if (++ku == nu) {
            seg_end = true;
            ku = 0;
            ++tg;
        }
        if (!seg_end) continue;
        // the partial slot is free once the reducer has read its previous use
        if (nseg >= PS && !mbar_ready(peA, pph, p.probes, abort_flag)) {
            if (lane == 0) {
                *abort_flag = 1;
                atomicOr(p.err, ERRBIT_TIMEOUT);
            }
            return;
        }
        const int ra = g, rb = g + 8;
        if (B1) {
            if (c == 0) {
                sts(pw + ra * 4u, acc[0]);
                sts(pw + rb * 4u, acc[2]);
            }
        } else {
            if (2 * c < batch) {
                sts(pw + (ra * batch + 2 * c) * 4u, acc[0]);
                sts(pw + (rb * batch + 2 * c) * 4u, acc[2]);
            }
            if (2 * c + 1 < batch) {
                sts(pw + (ra * batch + 2 * c + 1) * 4u, acc[1]);
                sts(pw + (rb * batch + 2 * c + 1) * 4u, acc[3]);
            }
        }
        acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
        __syncwarp();
        if (lane == 0) mbar_arrive_a(pfA);
        ++nseg;
        if (++ps == PS) {
            ps = 0;
            if (nseg > PS) pph ^= 1u;
            pw = cx.pw;
            pfA = cx.pfullA;
            peA = cx.pemptyA;
        } else {
            pw += kCW * share_b;
            pfA += 8;
            peA += 8;
        }
    }
}

// The CTA's sums ("segments"): row group major, one per row group the range
// touches; k chunk major, one per unit.
struct SegInfo {
    int first_tg;      // row group major: the first segment's group
    int nseg;
    bool partner;      // row group major: the first segment is a later part of a split group
    bool owner;        // row group major: the last segment is a split group this CTA owns
    int npart;         // its other CTAs
};

__device__ __forceinline__ int cta_of(int pos, int U, int G) {
    return static_cast<int>((static_cast<int64_t>(pos + 1) * G - 1) / U);
}

__device__ __forceinline__ SegInfo seg_info(const SkParams &p, int cta, int u0, int u1) {
    SegInfo si;
    if (p.kmaj) {
        si.first_tg = 0;
        si.nseg = u1 - u0;
        si.partner = si.owner = false;
        si.npart = 0;
        return si;
    }
    const int nu = p.nu;
    const int tgF = u0 / nu, tgL = (u1 - 1) / nu;
    si.first_tg = tgF;
    si.nseg = tgL - tgF + 1;
    si.partner = u0 % nu != 0;
    // the last group is split when this range does not hold all of it, and
    // owned when the range holds its first unit (then it continues past u1)
    const bool last_whole = u0 <= tgL * nu && u1 == tgL * nu + nu;
    si.owner = !last_whole && u0 <= tgL * nu;
    si.npart = si.owner ? cta_of(tgL * nu + nu - 1, p.U, p.G) - cta : 0;
    return si;
}

// A reducer warp: the segments q = r, r + kNR, ... of the CTA.  Sums the 16
// consumer warps' shares in warp order, then
//  - row group major: writes y for a whole group; publishes a partner part
//    (scratch slot of this CTA, release flag); for the owned split group adds
//    the partners' parts (fetched by the producer) in CTA order and writes y;
//  - k chunk major: writes y (one chunk) or stores the unit's partial for the
//    finishing CTAs.
template <bool B1, bool ID>
__device__ __forceinline__ void reduce_segments(const SkParams &p, const SkCols &cc, int r, int lane, int cta, int u0,
                                                const SegInfo &si, uint64_t *pfull, uint64_t *pempty,
                                                uint64_t *ppbar, const float *pslot, const float *pp,
                                                volatile int *abort_flag) {
    constexpr int PS = SkPs<B1>::v;
    const int nv = RT * p.batch, nu = p.nu, ngr = p.ngr, batch = p.batch;
    constexpr int kPer = (RT * (B1 ? 1 : QGEMV_MAX_BATCH) + 31) / 32;
    for (int q = r; q < si.nseg; q += kNR) {
        const int ps = q % PS;
        if (!mbar_wait_abortable(&pfull[ps], static_cast<uint32_t>(q / PS) & 1u, p.probes, abort_flag)) {
            if (lane == 0) {
                *abort_flag = 1;
                atomicOr(p.err, ERRBIT_TIMEOUT);
            }
            return;
        }
        const float *pb = pslot + static_cast<size_t>(ps) * kCW * nv;
        float vals[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int v = lane + 32 * i;
            float sum = 0.0f;
            if (v < nv) {
                sum = pb[v];
#pragma unroll 4
                for (int ww = 1; ww < kCW; ++ww) sum += pb[ww * nv + v];
            }
            vals[i] = sum;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&pempty[ps]);
        int tg;
        bool to_y = true;
        if (p.kmaj) {
            const int u = u0 + q;
            const int ku = u / ngr;
            tg = u - ku * ngr;
            if (nu > 1) {
                to_y = false;
                float *mine = p.part + (static_cast<size_t>(tg) * nu + ku) * nv;
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int v = lane + 32 * i;
                    if (v < nv) __stcg(mine + v, vals[i]);
                }
            }
        } else {
            tg = si.first_tg + q;
            if (q == 0 && si.partner) {
                // a later part of a split group: publish it for the owner
                to_y = false;
                float *mine = p.part + static_cast<size_t>(cta) * nv;
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int v = lane + 32 * i;
                    if (v < nv) __stcg(mine + v, vals[i]);
                }
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    st_release_u32(p.flag + cta, 1u);
                }
            } else if (q == si.nseg - 1 && si.owner) {
                if (!mbar_wait_abortable(ppbar, 0, p.probes, abort_flag)) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        atomicOr(p.err, ERRBIT_TIMEOUT);
                    }
                    return;
                }
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int v = lane + 32 * i;
                    if (v < nv) {
                        for (int j = 0; j < si.npart; ++j) vals[i] += pp[j * nv + v];
                    }
                }
            }
        }
        if (to_y) {
            const int row0 = tg * RT;
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const int v = lane + 32 * i;
                if (v < nv) {
                    const int rr = v / batch, n = v - rr * batch;
                    if (row0 + rr < p.nrows) p.y[col_y<ID>(p, cc, n) + row0 + rr] = vals[i];
                }
            }
        }
    }
}

// After every warp of the CTA is done (nu > 1): announce that this CTA's
// partials are stored; the last p.fin CTAs to announce wait for all G and
// sum their share of y in k order.  Runs with every thread of the CTA; `bc`
// is a shared word for broadcasts.
__device__ __forceinline__ void finish_split(const SkParams &p, int tid, volatile int *bc, volatile int *abort_flag) {
    const int G = p.G, M = p.fin;
    if (tid == 0) {
        __threadfence();                                  // this CTA's partials before the announcement
        const unsigned old = atomicAdd(p.sync, 1u);
        bc[0] = static_cast<int>(old) - (G - M);          // finisher index, < 0: none
    }
    cta_sync();
    const int j = bc[0];
    if (j < 0) return;
    if (tid == 0) {
        bool ok = false;
        unsigned ns = 32;
        for (unsigned i = 0; i < p.probes; ++i) {
            if (ld_acquire(p.sync) >= static_cast<unsigned>(G)) {
                ok = true;
                break;
            }
            __nanosleep(ns);
            if (ns < 256) ns <<= 1;
        }
        if (!ok) {
            *abort_flag = 1;
            atomicOr(p.err, ERRBIT_TIMEOUT);
        }
    }
    cta_sync();
    if (!*abort_flag) {
        const int nu = p.nu, batch = p.batch, nv = RT * batch;
        const int64_t T = static_cast<int64_t>(p.ngr) * nv;
        const int64_t o0 = T * j / M, o1 = T * (j + 1) / M;
        for (int64_t o = o0 + tid; o < o1; o += kThreads) {
            const int tg = static_cast<int>(o / nv), rem = static_cast<int>(o - static_cast<int64_t>(tg) * nv);
            const int rr = rem / batch, n = rem - rr * batch;
            const float *src = p.part + static_cast<size_t>(tg) * nu * nv + rem;
            float sum = 0.0f;
            for (int k0 = 0; k0 < nu; k0 += 8) {                // loads first, then the sums in k order
                float v[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) v[t] = k0 + t < nu ? __ldcg(src + static_cast<size_t>(k0 + t) * nv) : 0.0f;
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    if (k0 + t < nu) sum += v[t];
                }
            }
            const int row = tg * RT + rr;
            if (row < p.nrows) p.y[static_cast<int64_t>(n) * p.nrows + row] = sum;
        }
    }
    cta_sync();
    if (tid == 0) {
        // the last finisher puts the counters back for the next call (every
        // finisher has read p.sync[0] by now)
        if (atomicAdd(p.sync + 32, 1u) == static_cast<unsigned>(M - 1)) {
            p.sync[0] = 0u;
            p.sync[32] = 0u;
        }
    }
}

// ------------------------------------------------------------------ kernel
// The kernel's work for one problem.  ID: the expert-selected form -- the
// weights of expert `e` (4-D tensor map: expert outermost), columns gathered
// through cc, and each CTA's range cut at row-group boundaries (range of
// row groups [floor(i ngr / G), floor((i+1) ngr / G))), so that no row group
// is split between CTAs and no partial crosses CTAs.
template <int F, bool B1, bool ID>
__device__ __forceinline__ void sk_body(const CUtensorMap &tmap, const SkParams &p, const SkCols &cc, int e,
                                        uint8_t *smem) {
    constexpr uint32_t SLOT = sk_slot_bytes(F);
    constexpr int PS = SkPs<B1>::v;

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int ngr = p.ngr, nu = p.nu, U = p.U, G = p.G, NS = p.ns;
    const int cta = blockIdx.x;
    const int u0 = ID ? range_lo(cta, ngr, G) * nu : range_lo(cta, U, G);
    const int u1 = ID ? range_lo(cta + 1, ngr, G) * nu : range_lo(cta + 1, U, G);
    const int nunits = u1 - u0;
    // staged chunks: k chunk major, the one or two the range touches; row
    // group major, all of them
    const int ku_lo = p.kmaj ? u0 / ngr : 0;
    const int nch = p.kmaj ? (u1 - 1) / ngr - ku_lo + 1 : nu;
    const SegInfo si = seg_info(p, cta, u0, u1);
    const SkLayout L = sk_layout(F, p.ch, p.batch, NS, PS);
    const uint32_t ring = smem_u32(smem + L.ring);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + NS;
    uint64_t *pfull = empty + NS;
    uint64_t *pempty = pfull + PS;
    uint64_t *ppbar = pempty + PS;
    int *issued = reinterpret_cast<int *>(smem + L.issued);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.flag);
    const int nv = RT * p.batch;                 // values of one sum

    griddep_launch_dependents();

    // copies of units k = 0, 1, ... in order (producer lane 0): slot is_, unit (itg, iku)
    const uint64_t wpol = l2_evict_first();
    int is_ = 0, ik = 0, itg, iku;
    if (p.kmaj) {
        iku = u0 / ngr;
        itg = u0 - iku * ngr;
    } else {
        itg = u0 / nu;
        iku = u0 - itg * nu;
    }
    auto issue = [&]() {
        if (!(ik == 0 && p.withhold && cta == 0 && blockIdx.y == 0)) {       // (testing the timeout path)
            mbar_arrive_expect_tx(&full[is_], SLOT);
            if constexpr (ID) {
                tma_load_4d(ring + static_cast<uint32_t>(is_) * SLOT, &tmap, 0, itg * RT, iku * SkFmt<F>::BB, e,
                            &full[is_], wpol);
            } else {
                tma_load_3d(ring + static_cast<uint32_t>(is_) * SLOT, &tmap, 0, itg * RT, iku * SkFmt<F>::BB,
                            &full[is_], wpol);
            }
            issued[is_] += 1;
        }
        ++ik;
        if (++is_ == NS) is_ = 0;
        if (p.kmaj) {
            if (++itg == ngr) {
                itg = 0;
                ++iku;
            }
        } else if (++iku == nu) {
            iku = 0;
            ++itg;
        }
    };

    if (wid == kProd && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
            issued[s] = 0;
        }
        for (int q = 0; q < PS; ++q) {
            mbar_init(&pfull[q], kCW);
            mbar_init(&pempty[q], 1);
        }
        mbar_init(ppbar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    cta_sync();
    const int first = min(NS, nunits);
    const int ahead = min(first, p.pre);         // units copied before the loads of x
    if (wid == kProd) {
        // ------------------------------------------------ producer warp
        // (lane 0 issues the copies)
        if (lane == 0 && p.early) {
            while (ik < ahead) issue();
        }
        __syncwarp();
        griddep_wait();
        if (lane == 0 && !p.early) {
            while (ik < ahead) issue();
        }
        __syncwarp();
        xready_wait();
        if (lane == 0) {
            while (ik < first) issue();
            // refill each slot as soon as all consumer warps released it
            uint32_t eph = 0;                  // parity of the slot's release by its previous unit
            while (ik < nunits) {
                if (!mbar_ready(smem_u32(&empty[is_]), eph, p.probes, abort_flag)) {
                    atomicOr(p.err, ERRBIT_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                issue();
                if (is_ == 0) eph ^= 1u;
            }
        }
        __syncwarp();
        if (si.owner) {
            // the partners' parts of the owned split group, in CTA order
            float *pp = reinterpret_cast<float *>(smem + L.pp);
            for (int q = 0; q < si.npart && !*abort_flag; ++q) {
                const int i = cta + 1 + q;
                bool got = false;
                unsigned ns = 32;
                for (unsigned t = 0; t < p.probes; ++t) {
                    if (ld_acquire(p.flag + i) != 0u) {
                        got = true;
                        break;
                    }
                    __nanosleep(ns);
                    if (ns < 256) ns <<= 1;
                    if (*abort_flag) break;
                }
                if (!got) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        atomicOr(p.err, ERRBIT_TIMEOUT);
                    }
                    break;
                }
                const float *src = p.part + static_cast<size_t>(i) * nv;
                for (int v = lane; v < nv; v += 32) pp[q * nv + v] = __ldcg(src + v);
                __syncwarp();
                if (lane == 0) p.flag[i] = 0u;   // cleared for the next call (after this one completes)
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(ppbar);
        }
    } else if (wid >= kRed0) {
        // ------------------------------------------------ reducer warps
        griddep_wait();                         // y and the scratch: after the preceding kernel
        reduce_segments<B1, ID>(p, cc, wid - kRed0, lane, cta, u0, si, pfull, pempty, ppbar,
                            reinterpret_cast<const float *>(smem + L.pslot),
                            reinterpret_cast<const float *>(smem + L.pp), abort_flag);
    } else {
        // ------------------------------------------------ consumer warps
        griddep_wait();                         // x: after the preceding kernel
        int *wfw = reinterpret_cast<int *>(smem + L.wf) + wid * p.ch;
        for (int q = lane; q < p.ch; q += 32) wfw[q] = 0;
        __syncwarp();
        stage_items<F, ID>(p, cc, wid, lane, smem, L, ku_lo, nch, true);

        ConsCtx<F> cx;
        {
            int o[PairWords<F>::NW];
            PairWords<F>::offsets(c, o);
#pragma unroll
#pragma unroll
            for (int q = 0; q < SkPairs<F>::sets; ++q) {
#pragma unroll
                for (int i = 0; i < PairWords<F>::NW; ++i) cx.lc.off[q][i] = sk_off(SkFmt<F>::PB * (wid + kCW * q) + o[i], g);
            }
            cx.lc.sel = c == 3 ? 0x5432u : 0x3210u;
        }
        const int batch = B1 ? 1 : p.batch;
        const int wit = p.ch * p.batch;
        const int ncol = min(g, batch - 1);          // B columns past the batch repeat the last one
        cx.fullA = smem_u32(full);
        cx.emptyA = smem_u32(empty);
        cx.pfullA = smem_u32(pfull);
        cx.pemptyA = smem_u32(pempty);
        cx.abort_flag = abort_flag;
        cx.ring = ring;
        cx.xfw = smem_u32(smem + L.xf) + static_cast<uint32_t>((wid * wit + ncol) * 128 * PPW + c * 16);
        cx.usw = smem_u32(smem + L.us) + static_cast<uint32_t>(wid * wit * 4);
        cx.xsw = smem_u32(smem + L.xs) + static_cast<uint32_t>(wid * wit * 8 * PPW);
        cx.pw = smem_u32(smem + L.pslot) + static_cast<uint32_t>(wid * nv * 4);
        cx.u0 = u0;
        cx.nunits = nunits;
        cx.ku_lo = ku_lo;
        cx.c = c;
        cx.lane = lane;
        cx.wid = wid;
        cx.batch = batch;
        cx.n0 = min(2 * c, batch - 1);
        cx.n1 = min(2 * c + 1, batch - 1);
        cx.NS = NS;
        // a warp with a flagged chunk runs the loop that can take the exact path
        bool slow = false;
        for (int q = 0; q < nch; ++q) slow = slow || wfw[q] != 0;
        if (slow) consume<F, B1, true, ID>(p, cc, cx, wfw);
        else consume<F, B1, false, ID>(p, cc, cx, wfw);
        // nothing of the consumers is needed after their loop unless they
        // take part in the finishing sums: then they only announce that they
        // are done (no value stays live across the loop)
        if (!(p.kmaj && p.nu > 1)) {
            cta_arrive_all<kThreads>();
            return;
        }
    }
    cta_sync_all<kThreads>();
    if (*abort_flag && wid == kProd && lane == 0) {
        // a wait gave up: let every copy still in flight land before exiting
        for (int s = 0; s < NS; ++s) {
            if (issued[s] > 0) mbar_wait_bounded(&full[s], static_cast<uint32_t>(issued[s] - 1) & 1u, p.err);
        }
    }
    if (!ID && p.kmaj && nu > 1) finish_split(p, tid, abort_flag + 1, abort_flag);
}

template <int F, bool B1>
__global__ void __launch_bounds__(kThreads, 1)
gemv_sk_kernel(const __grid_constant__ CUtensorMap tmap, const SkParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    SkCols cc;
    sk_body<F, B1, false>(tmap, p, cc, 0, smem);
}

// ------------------------------------------------- expert-selected kernel
// Ring slots of a work unit of nb columns (entry nb - 1); everything else of
// the plan is common to all units.
struct SkIdParams {
    const int *ids;         // [batch] expert of each output column
    int batch;              // output columns, 1 .. kSkIdMaxBatch
    int n_expert;
    int x_group;            // column b reads activation row b / x_group
    int nbmax;              // columns of a unit, at most (<= QGEMV_MAX_BATCH)
    int ns[QGEMV_MAX_BATCH];
};
constexpr int kSkIdMaxBatch = 64;

// Work units as in the fixed-point expert kernel: the distinct valid experts
// of ids in order of first appearance, each cut into units of up to nbmax
// of its columns in column order; CTA (i, u) runs row groups i of unit u.
// The columns ride in the MMA's N dimension, so a unit of several columns
// costs little more than one.  CTAs past the last unit return at once; a
// column with an id outside [0, n_expert) is in no unit and sets
// ERRBIT_INDEX.
template <int F>
__global__ void __launch_bounds__(kThreads, 1)
gemv_sk_id_kernel(const __grid_constant__ CUtensorMap tmap, const SkParams p, const SkIdParams q) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    int *sid = reinterpret_cast<int *>(smem);                    // [kSkIdMaxBatch] ids
    int *snu = sid + kSkIdMaxBatch;                              // [kSkIdMaxBatch] units of a first column
    int *sinfo = snu + kSkIdMaxBatch;                            // expert, columns, column list
    const int tid = threadIdx.x;
    const int nbmax = q.nbmax;
    griddep_wait();                                              // ids, x and y: after the preceding kernel
    if (tid < 2 + QGEMV_MAX_BATCH) sinfo[tid] = 0;
    if (tid < q.batch) sid[tid] = q.ids[tid];
    cta_sync();
    int id = -1, cnt = 0, rank = 0, first = tid;
    bool valid = false;
    if (tid < q.batch) {
        id = sid[tid];
        valid = id >= 0 && id < q.n_expert;
        for (int s = 0; s < q.batch; ++s) {
            if (sid[s] == id) {
                ++cnt;
                if (s < tid) {
                    ++rank;
                    first = min(first, s);
                }
            }
        }
        snu[tid] = valid && rank == 0 ? (cnt + nbmax - 1) / nbmax : 0;
        if (!valid && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(p.err, ERRBIT_INDEX);
    }
    cta_sync();
    if (valid) {
        int u = rank / nbmax;
        for (int s = 0; s < first; ++s) u += snu[s];
        if (u == static_cast<int>(blockIdx.y)) {
            const int pos = rank % nbmax;
            sinfo[2 + pos] = tid;
            if (pos == 0) {
                sinfo[0] = id;
                sinfo[1] = min(nbmax, cnt - (rank / nbmax) * nbmax);
            }
        }
    }
    cta_sync();
    const int e = sinfo[0], nbu = sinfo[1];
    SkCols cc;
#pragma unroll
    for (int n = 0; n < QGEMV_MAX_BATCH; ++n) {
        const int col = n < nbu ? sinfo[2 + n] : 0;
        cc.xo[n] = static_cast<int64_t>(col / q.x_group) * p.ncols;
        cc.yo[n] = static_cast<int64_t>(col) * p.nrows;
    }
    cta_sync();                                                  // the scratch is free for the ring
    if (nbu == 0) return;
    SkParams pp = p;
    pp.batch = nbu;
    pp.ns = q.ns[nbu - 1];
    if (nbu == 1) sk_body<F, true, true>(tmap, pp, cc, e, smem);
    else sk_body<F, false, true>(tmap, pp, cc, e, smem);
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
    int64_t nrows = 0, rowbytes = 0, ne = 0;
    int nz = 0;
    CUtensorMap map;
};
constexpr int kMapCache = 32;
std::mutex g_map_mutex;
MapEntry g_maps[kMapCache];
int g_map_next = 0;
EncodeTiledFn g_encode = nullptr;

// ne > 0: a stack of ne matrices of nrows rows each, viewed 4-D with the
// expert outermost (stride nrows * rowbytes), so that rows past nrows of one
// expert read as zero too.
qgemv_status weight_map(const void *W, int64_t nrows, int64_t rowbytes, int nz, CUtensorMap *out, int64_t ne = 0) {
    std::lock_guard<std::mutex> lk(g_map_mutex);
    for (int i = 0; i < kMapCache; ++i) {
        const MapEntry &e = g_maps[i];
        if (e.ptr == W && e.nrows == nrows && e.rowbytes == rowbytes && e.nz == nz && e.ne == ne) {
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
    const cuuint64_t gdim[4] = {64u, static_cast<cuuint64_t>(nrows), static_cast<cuuint64_t>(rowbytes / 64),
                                static_cast<cuuint64_t>(ne > 0 ? ne : 1)};
    const cuuint64_t gstride[3] = {static_cast<cuuint64_t>(rowbytes), 64u, static_cast<cuuint64_t>(nrows * rowbytes)};
    const cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(RT), static_cast<cuuint32_t>(nz), 1u};
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    CUresult r = g_encode(&e.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, ne > 0 ? 4 : 3, const_cast<void *>(W), gdim,
                          gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        e.ptr = nullptr;
        set_last_error("cuTensorMapEncodeTiled(weights) failed (%d)", static_cast<int>(r));
        return QGEMV_ERR_CUDA;
    }
    e.ptr = W;
    e.nrows = nrows;
    e.rowbytes = rowbytes;
    e.ne = ne;
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
unsigned *g_sync_base[kMaxDev] = {nullptr};

qgemv_status scratch_for(int dev, cudaStream_t s, float **part, unsigned **flag, unsigned **sync) {
    std::lock_guard<std::mutex> lk(g_set_mutex);
    if (!g_part_base[dev]) {
        void *a = nullptr, *b = nullptr, *c = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&a, g_sk_part);
        if (e == cudaSuccess) e = cudaGetSymbolAddress(&b, g_sk_flag);
        if (e == cudaSuccess) e = cudaGetSymbolAddress(&c, g_sk_sync);
        if (e != cudaSuccess) {
            set_last_error("cudaGetSymbolAddress(GEMV scratch): %s", cudaGetErrorString(e));
            return QGEMV_ERR_CUDA;
        }
        g_part_base[dev] = static_cast<float *>(a);
        g_flag_base[dev] = static_cast<unsigned *>(b);
        g_sync_base[dev] = static_cast<unsigned *>(c);
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
    *part = g_part_base[dev] + static_cast<size_t>(set) * kSkPartFloats;
    *flag = g_flag_base[dev] + static_cast<size_t>(set) * kSkMaxG;
    *sync = g_sync_base[dev] + static_cast<size_t>(set) * kSkSyncWords;
    return QGEMV_OK;
}

struct SkPlan {
    int dev = -1, fmt = -1, batch = 0;
    int64_t nrows = 0, ncols = 0;
    int ns = 0, ps = 0, ch = 0, G = 0, kmaj = 0;
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

// Grid, ring and partial slots for a shape; G = 0 when the kernel does not
// take it (staged x or the scratch would not fit).
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
    const int64_t nu = (ncols + 2047) / 2048, ngr = (nrows + RT - 1) / RT, U = ngr * nu;
    const size_t budget = di.smem_optin;
    const uint32_t slot = sk_slot_bytes(F);
    const int ps = batch == 1 ? SkPs<true>::v : SkPs<false>::v;
    // ring slots next to a layout with ch chunk slots (0: not even three fit)
    auto slots_for = [&](int64_t ch) -> int {
        const SkLayout L0 = sk_layout(F, static_cast<int>(ch), batch, 0, ps);
        if (static_cast<size_t>(L0.total) + 1024 + 3u * (slot + 20) > budget) return 0;
        int ns = static_cast<int>((budget - 1024 - L0.total) / (slot + 20));
        if (ns > kMaxSlots) ns = kMaxSlots;
        while (ns > 0 && static_cast<size_t>(sk_layout(F, static_cast<int>(ch), batch, ns, ps).total) + 1024 > budget) --ns;
        return ns >= 3 ? ns : 0;
    };
    // row group major when the staged x of every chunk fits (<= 32 chunks):
    // every range holds >= ceil(nu / 4) units, so a group falls to <= 5 CTAs
    int64_t G = U / ((nu + 3) / 4);
    if (G > di.sm_count) G = di.sm_count;
    if (G > kSkMaxG) G = kSkMaxG;
    int ns = nu <= 32 && G >= 1 && G * RT * batch <= kSkPartFloats ? slots_for(nu) : 0;
    if (ns > 0) {
        pl.kmaj = 0;
        pl.ch = static_cast<int>(nu);
    } else {
        // k chunk major: the chunks the widest range touches
        G = U < di.sm_count ? U : di.sm_count;
        const bool scratch_ok = nu == 1 || ngr * nu * RT * batch <= kSkPartFloats;
        int64_t ch = 1;
        for (int64_t i = 0; i < G; ++i) {
            const int64_t a = i * U / G, b = (i + 1) * U / G;
            const int64_t span = (b - 1) / ngr - a / ngr + 1;
            if (span > ch) ch = span;
        }
        ns = G >= 1 && scratch_ok ? slots_for(ch) : 0;
        pl.kmaj = 1;
        pl.ch = static_cast<int>(ch);
    }
    if (ns > 0) {
        pl.ns = ns;
        pl.ps = ps;
        pl.G = static_cast<int>(G);
        pl.smem = static_cast<size_t>(sk_layout(F, pl.ch, batch, ns, ps).total) + 1024;
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
    if (ncols % 1024 != 0 || nrows < 1 || nrows > (1 << 28) || ncols > (1 << 24)) return QGEMV_OK;
    const int64_t nu = (ncols + 2047) / 2048, ngr = (nrows + RT - 1) / RT;
    if (ngr * nu > (int64_t(1) << 30)) return QGEMV_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return QGEMV_OK;
    SkPlan pl;
    if (!make_plan<F>(dev, nrows, ncols, batch, di, &pl)) return QGEMV_OK;
    SkParams p;
    p.x = x;
    p.y = y;
    p.err = err;
    qgemv_status st = scratch_for(dev, s, &p.part, &p.flag, &p.sync);
    if (st != QGEMV_OK) return st;
    p.nrows = static_cast<int>(nrows);
    p.ncols = static_cast<int>(ncols);
    p.batch = batch;
    p.nu = static_cast<int>(nu);
    p.ngr = static_cast<int>(ngr);
    p.U = static_cast<int>(ngr * nu);
    p.G = pl.G;
    p.ns = pl.ns;
    p.ch = pl.ch;
    p.kmaj = pl.kmaj;
    // finishing CTAs: enough for one pass of the CTA's threads over y
    {
        const int64_t outs = ngr * RT * batch;
        int64_t M = (outs + kThreads - 1) / kThreads;
        if (M > pl.G) M = pl.G;
        p.fin = static_cast<int>(M < 1 ? 1 : M);
    }
    p.early = g_opt_weights_static;
    // units copied before the loads of x: 4 when they may start before the
    // dependency wait (measured best of 2..12: more delays the x loads), else 2
    p.pre = p.early ? 4 : 2;
    p.probes = g_opt_wait_probes;
    p.withhold = g_opt_withhold_next;
    g_opt_withhold_next = 0;
    *taken = true;
    return batch == 1 ? launch_k<F, true>(pl, W, p, s, di) : launch_k<F, false>(pl, W, p, s, di);
}

template <int F>
bool set_id_smem_attr(int dev, size_t optin) {
    static bool done[kMaxDev] = {false};
    if (done[dev]) return true;
    if (cudaFuncSetAttribute(gemv_sk_id_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(optin)) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    done[dev] = true;
    return true;
}

// Ring slots of the row-group-major layout for nb columns (every chunk's x
// staged), 0 when not even three fit.
template <int F>
int id_slots(int64_t nu, int nb, const DevInfo &di) {
    const size_t budget = di.smem_optin;
    const uint32_t slot = sk_slot_bytes(F);
    const int ps = nb == 1 ? SkPs<true>::v : SkPs<false>::v;
    const SkLayout L0 = sk_layout(F, static_cast<int>(nu), nb, 0, ps);
    if (static_cast<size_t>(L0.total) + 1024 + 3u * (slot + 20) > budget) return 0;
    int ns = static_cast<int>((budget - 1024 - L0.total) / (slot + 20));
    if (ns > kMaxSlots) ns = kMaxSlots;
    while (ns > 0 && static_cast<size_t>(sk_layout(F, static_cast<int>(nu), nb, ns, ps).total) + 1024 > budget) --ns;
    return ns >= 3 ? ns : 0;
}

template <int F>
qgemv_status launch_sk_id_fmt(const void *W, int64_t n_expert, const int *ids, const float *x, int x_group,
                              float *y, int64_t nrows, int64_t ncols, int batch, cudaStream_t s, const DevInfo &di,
                              unsigned *err, bool *taken) {
    *taken = false;
    if (ncols % 1024 != 0 || nrows < 1 || nrows > (1 << 28) || ncols > (1 << 24) || batch > kSkIdMaxBatch)
        return QGEMV_OK;
    const int64_t nu = (ncols + 2047) / 2048, ngr = (nrows + RT - 1) / RT;
    if (nu > 32 || ngr * nu > (int64_t(1) << 30)) return QGEMV_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return QGEMV_OK;
    // the widest unit whose staged x (every chunk) fits beside a ring of three slots
    SkIdParams q = {};
    int nbmax = std::min(batch, QGEMV_MAX_BATCH);
    while (nbmax >= 1 && id_slots<F>(nu, nbmax, di) == 0) --nbmax;
    if (nbmax < 1) return QGEMV_OK;
    size_t smem = static_cast<size_t>((2 * kSkIdMaxBatch + 2 + QGEMV_MAX_BATCH) * 4) + 1024;
    for (int nb = 1; nb <= nbmax; ++nb) {
        q.ns[nb - 1] = id_slots<F>(nu, nb, di);
        if (q.ns[nb - 1] == 0) return QGEMV_OK;
        const int ps = nb == 1 ? SkPs<true>::v : SkPs<false>::v;
        smem = std::max(smem, static_cast<size_t>(sk_layout(F, static_cast<int>(nu), nb, q.ns[nb - 1], ps).total) + 1024);
    }
    // units: D distinct experts give D plus one for every further nbmax columns of an expert
    const int D = static_cast<int>(std::min<int64_t>(batch, n_expert));
    const int units = D + (batch - D) / nbmax;
    const int64_t G = std::max<int64_t>(1, std::min<int64_t>(ngr, di.sm_count / units));
    q.ids = ids;
    q.batch = batch;
    q.n_expert = static_cast<int>(std::min<int64_t>(n_expert, INT32_MAX));
    q.x_group = x_group;
    q.nbmax = nbmax;
    SkParams p = {};
    p.x = x;
    p.y = y;
    p.err = err;
    p.nrows = static_cast<int>(nrows);
    p.ncols = static_cast<int>(ncols);
    p.batch = 1;
    p.nu = static_cast<int>(nu);
    p.ngr = static_cast<int>(ngr);
    p.U = static_cast<int>(ngr * nu);
    p.G = static_cast<int>(G);
    p.kmaj = 0;
    p.ch = static_cast<int>(nu);
    p.fin = 1;
    p.early = 0;
    p.pre = 2;
    p.probes = g_opt_wait_probes;
    p.withhold = g_opt_withhold_next;
    if (!set_id_smem_attr<F>(dev, di.smem_optin)) {
        set_last_error("qgemv_id(tensor cores): cannot raise the shared-memory limit");
        return QGEMV_ERR_LAUNCH;
    }
    const int64_t rowbytes = ncols / 32 * block_bytes(F);
    CUtensorMap map;
    qgemv_status ms = weight_map(W, nrows, rowbytes, SkFmt<F>::BB, &map, n_expert);
    if (ms != QGEMV_OK) return ms;
    g_opt_withhold_next = 0;
    *taken = true;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(G), static_cast<unsigned>(units));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_sk_id_kernel<F>, map, p, q);
    if (e != cudaSuccess) {
        set_last_error("qgemv_id(tensor cores) launch: %s", cudaGetErrorString(e));
        return QGEMV_ERR_LAUNCH;
    }
    return check_launch("qgemv_id(tensor cores)");
}

}  // namespace

qgemv_status launch_gemv_sk_id(int fmt, const void *W, int64_t n_expert, const int *ids, const float *x,
                               int x_group, float *y, int64_t nrows, int64_t ncols, int batch, cudaStream_t s,
                               const DevInfo &di, unsigned *err, bool *taken) {
    switch (fmt) {
    case FMT_Q4_0:
        return launch_sk_id_fmt<FMT_Q4_0>(W, n_expert, ids, x, x_group, y, nrows, ncols, batch, s, di, err, taken);
    case FMT_Q4_1:
        return launch_sk_id_fmt<FMT_Q4_1>(W, n_expert, ids, x, x_group, y, nrows, ncols, batch, s, di, err, taken);
    case FMT_Q8_0:
        return launch_sk_id_fmt<FMT_Q8_0>(W, n_expert, ids, x, x_group, y, nrows, ncols, batch, s, di, err, taken);
    default:
        *taken = false;
        return QGEMV_OK;
    }
}

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

// Flags and counters of every scratch set of the current device back to zero
// (after a kernel gave up mid-call, a flag may still be raised or a counter
// hold a partial count).
void gemv_sk_reset_scratch() {
    void *b = nullptr;
    if (cudaGetSymbolAddress(&b, g_sk_flag) == cudaSuccess) {
        cudaMemset(b, 0, sizeof(unsigned) * kSkSets * kSkMaxG);
    }
    if (cudaGetSymbolAddress(&b, g_sk_sync) == cudaSuccess) {
        cudaMemset(b, 0, sizeof(unsigned) * kSkSets * kSkSyncWords);
    }
    cudaGetLastError();
}

}  // namespace qg
