// Tensor-core forward kernel of causal continuous attention for sm_103a:
// eq. (10)/(11) of Jianlin Su, "Continuous Softmax Attention" ("Assembly
// and Simplification"), bf16 inputs, d = 64 or 128, fp32 accumulation.
//
// Work split.  A work item is one 128-row query tile of one (b, h); it walks
// the key/value tiles up to its diagonal.  The grid is one persistent CTA per
// SM: CTA b starts with item b and its producer warp takes further items from
// a counter (heaviest query tiles first, heads grouped for L2), handing each
// to the other warps through a two-entry ring.  The K/V rings, the S buffers
// and the O accumulators count over all of the CTA's key tiles and carry on
// from one item to the next, so one item's epilogue overlaps the next item's
// first S products.  Warps:
//   0-7  softmax: warp w owns rows 32*(w%4).. (its TMEM lane quarter) and,
//        with h = w/4, the half h of the key columns of each S tile
//   8    TMA producer (lane 0; all lanes write the constant ones box once)
//   9    TMEM allocator and tcgen05.mma issuer (lane 0)
// Tensor memory (512 columns): S buffer 0 | S buffer 1 | O_0 | O_1.  S is
// double-buffered: the tensor core computes PV(j) and S(j+2) while the
// softmax works on S(j+1).  The two column halves are independent: each
// has its own running max, its own fp32 row sum and its own accumulator O_h
// (d + 16 columns), fed by its own PV product of 64 keys (P_h, bf16, over
// the half's own S columns, zero where the 64 keys reach into the other
// half).  They meet once per query tile, in the epilogue, where the two
// partial results are scaled to a common max and added.  Each V stage
// carries one more box holding a column of ones, so each PV product also
// accumulates, in column d of O_h, the row sum of exactly the bf16 P values
// it used.
//
// Key tiles and the halo.  b_{t,i} needs the logits of both neighbours of
// key i.  An S tile has NK columns (112 at d = 128, so that two S buffers
// and two accumulators fit; 128 at d = 64) and tiles start every NK - 2
// keys: column 0 and column NK-1 are halos whose weights belong to the
// neighbouring tiles, and every owned column 1..NK-2 has both neighbours in
// the tile.  Column c of tile j is position e = (NK-2) j + c - 1 of the
// extended sequence, whose position 0 is the sink pair and position i the
// i-th key.  Tile j starts at array row (NK-2) j - 2; TMA fills the rows -2
// and -1 with zeros, so the zero sink pair k_0 = v_0 = 0 is column 1 of tile
// 0 at no cost; the copy-first and given modes replace its logit (and, for
// given v_0, add w_0 * v_0 to the output at the end).
//
// The weights.  With the running max m (log2 units) and u = a*log2(e) - m,
// p = 2^u, each interval between neighbouring keys contributes
//   R = p_left * phi2(x)  to its left key and  L = p_right * phi2(-x)  to its
// right key (x the logit step), the regrouping of eq. (9); a key's weight
// e^{a+b-m} is L + R of its two intervals, one-sided at both ends.  R and L
// follow from the interval integral S = (p_right - p_left)/x by
// R = (S - p_left)/x and L = S - R, with a power series for small steps.
// All weights carry a common factor (ln 2)^2, which cancels in o and is
// removed from lse.  The arithmetic runs on pairs of lanes (f32x2): in a
// chunk of n keys, lane x takes key / interval i and lane y takes i + n/2.
//
// The running max of a half is the exact max of its columns in the query
// tile's first key tile; it is not raised per tile.  Weights may then exceed
// 1, which costs nothing in fp32 and bf16; a half-tile's bf16 P stays in
// registers until the half-tile is done, and only when a chunk's weights sum
// past 2^64 does the half take the exact max of its columns of the tile,
// rescale O_h, and compute the half-tile again.
//
// The template flag SHORT turns the kernel into the short-conv reading of
// eq. (13): b is replaced by its first-order term, so a key's weight is 2^z
// with z an affine combination of its own and its neighbours' logits
// (short_chunk) and no phi2 is formed.  SYM integrates over the symmetric
// interval [1/2, t + 1/2] instead (constant half-cells at both ends, no
// sink; cont_chunk).
//
// Every mbarrier wait is bounded in time; on expiry the kernel records
// CSA_ERR_TIMEOUT, every role skips its remaining work, the MMA issuer waits
// for its own MMAs, the producer waits for its own copies, and TMEM is
// freed.
#include <mutex>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "csa.h"
#include "csa_internal.h"
#include "csa_tc_common.cuh"

using namespace csa_tc;

namespace {

__device__ int g_tc_status;  // sticky status word of this file's kernels

constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr int kThreads = 32 * 10;
// -log((ln 2)^2): removes the common weight factor from lse
constexpr float kLseShift = 0.7330258411633287f;
// |X| below this (log2 units) takes the small-step coefficients.
constexpr float kTau = 0.0625f;
// the kernel's forms (template argument): interval weights, the short-conv
// reading, and the log-domain evaluation of the interval weights
constexpr int kTcExact = 0, kTcShort = 1, kTcLog = 2;
// A half-cell p/2 of the symmetric interval, times the common (ln 2)^2.
constexpr float kHalfCell = 0.5f * kLn2 * kLn2;
// A chunk whose weights sum past this raises its half's running max.
constexpr float kSumLimit = 18446744073709551616.0f;  // 2^64

template <int D>
struct TcCfg {
    static constexpr int kNK = D == 128 ? 112 : 128;  // keys (columns) per S tile
    static constexpr int kKS = kNK - 2;               // key-tile stride: owned columns
    static constexpr int kH0 = kNK / 2;               // keys of each column half
    static constexpr int kBoxes = D / 64;             // 64-column boxes per row
    static constexpr int kQBox = 128 * 128;           // 128 rows x 128 bytes
    static constexpr int kKBox = kNK * 128;           // NK rows x 128 bytes
    static constexpr int kQBytes = kBoxes * kQBox;
    static constexpr int kKBytes = kBoxes * kKBox;
    static constexpr int kVBytes = (kBoxes + 1) * kKBox;  // values + ones box
    static constexpr int kN = D + 16;                     // PV width
    static constexpr int kStagesK = D == 128 ? 2 : 3;
    static constexpr int kStagesV = D == 128 ? 2 : 3;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + kStagesK * kKBytes;
    static constexpr int kOffBar = kOffV + kStagesV * kVBytes;
    // barrier indices
    static constexpr int kBarQ = 0;
    static constexpr int kBarKFull = 1;
    static constexpr int kBarKEmpty = kBarKFull + kStagesK;
    static constexpr int kBarVFull = kBarKEmpty + kStagesK;
    static constexpr int kBarVEmpty = kBarVFull + kStagesV;
    static constexpr int kBarSFull = kBarVEmpty + kStagesV;  // [2] one per S buffer
    // [2 halves][2 S buffers]: a half may run up to two tiles ahead of the
    // other, so each half's arrivals alternate between two barriers (one
    // phase per two tiles) and none completes twice before it is consumed
    static constexpr int kBarPFull = kBarSFull + 2;
    // [2]: PV pair k completes a phase of barrier k % 2.  A wait by parity
    // is unambiguous only while the barrier's previous phase is complete;
    // with two barriers that phase is PV pair k-2, which every wait below
    // follows (the S wait of tile k covers every product issued before
    // S(k), PV pair k-2 among them).  One barrier would need PV pair k-1's
    // previous phase, k-2, at the epilogue, where nothing waited for it.
    static constexpr int kBarODone = kBarPFull + 4;
    static constexpr int kBarDrain = kBarODone + 2;
    static constexpr int kBarX = kBarDrain + 1;       // half-to-half exchange (epilogue)
    static constexpr int kBarQEmpty = kBarX + 1;      // an item's last S is done
    static constexpr int kBarQRead = kBarQEmpty + 1;  // its sink logits are read from Q
    static constexpr int kBarItemFull = kBarQRead + 1;      // [2] item ring
    static constexpr int kBarItemEmpty = kBarItemFull + 2;  // [2]
    static constexpr int kNumBars = kBarItemEmpty + 2;
    // misc: TMEM base, abort flag, then the item ring ([2][3] ints: bh, row0, n)
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    // the epilogue's exchange: [2 halves][128 rows][4] (max, sum, sink weight)
    static constexpr int kOffXFin = kOffMisc + 64;
    // d = 128: the output rows of each softmax warp (32 rows x 64 columns,
    // bf16, 128B-swizzled) staged for one TMA store per item
    static constexpr bool kTmaOut = D == 128;
    static constexpr int kOffOut = (kOffXFin + 2 * 128 * 4 * 4 + 1023) / 1024 * 1024;
    static constexpr int kOutBytes = kTmaOut ? 8 * 32 * 128 : 0;
    static constexpr int kSmemBytes = kOffOut + kOutBytes + 1024;  // + slack to align the base
    static_assert(kSmemBytes <= 227 * 1024, "shared memory per block");
    // TMEM columns: S buffer 0 | S buffer 1 | O_0 | O_1
    __device__ static constexpr uint32_t col_s(int b) { return (uint32_t)(kNK * b); }
    __device__ static constexpr uint32_t col_o(int h) { return (uint32_t)(2 * kNK + kN * h); }
    // P of half h: 64 keys (32 packed columns) over the half's own S columns
    __device__ static constexpr uint32_t col_p(int h) { return h ? (uint32_t)(kNK - 32) : 0u; }
    static_assert(2 * kNK + 2 * kN <= 512, "TMEM budget");
    static_assert(kH0 == 56 || kH0 == 64, "column halves of 56 or 64 keys");
};

struct TcParams {
    int B, H, T;
    int num_qtiles;
    int group;  // heads per scheduling group
    float k2;   // scale * log2(e)
    int mode;
    const __nv_bfloat16 *k0;
    const __nv_bfloat16 *v0;
    __nv_bfloat16 *out;
    float *lse;
    int num_items;  // query tiles: num_qtiles * B * H
    int slot;       // this launch's scheduling counters
    // test hook: the softmax threads of column half delay_half sleep
    // delay_ns before reading O in each epilogue (0: none)
    unsigned delay_ns;
    int delay_half;
};

// A work item is one query tile of one (b, h).  Heads go in groups whose K/V
// fit in L2 together; within a group the heaviest query tiles come first
// (longest-first keeps the tail short).
struct TcItem {
    int bh, row0, n;  // n: key tiles the query tile reads
};

template <int KS>
__device__ __forceinline__ TcItem tc_item(int item, const TcParams &p) {
    const int nq = p.num_qtiles, BH = p.B * p.H;
    const int grp = item / (p.group * nq);
    const int gsz = min(p.group, BH - grp * p.group);
    const int idx = item - grp * p.group * nq;
    TcItem w;
    w.bh = grp * p.group + idx % gsz;
    w.row0 = (nq - 1 - idx / gsz) * 128;
    w.n = (min(w.row0 + 127, p.T - 1) + 1) / KS + 1;
    return w;
}

// Persistent scheduling: one CTA per SM; CTA b starts with item b and takes
// the next one from a counter when it is about to need it.  Each launch draws
// one of kSchedSlots counter pairs (round robin on the host), and the last CTA
// of the launch to finish puts its pair back to zero.  The host orders each
// launch after the slot's previous launch (an event per slot), so two
// launches never use one counter at the same time.
constexpr int kSchedSlots = 64;
__device__ unsigned int g_sched_next[kSchedSlots];
__device__ unsigned int g_sched_done[kSchedSlots];

__device__ __forceinline__ bool wait_c(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    return wait_bar(bar, parity, abort_flag, &g_tc_status);
}

// mbarrier.try_wait with a suspend-time hint (100 us): a thread whose phase is
// not complete sleeps until it completes instead of polling.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(100000u)
        : "memory");
    return ok != 0;
}

// Bounded wait, as wait_c, on the sleeping try_wait.
__device__ __forceinline__ bool wait_s(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            *(volatile int *)&g_tc_status = kStatusTimeout;
            __threadfence();
            return false;
        }
    }
}

// ------------------------------------------------------------- TMEM access
// 32 lanes x 16 (8) consecutive 32-bit columns: thread i gets lane (base+i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}
// tcgen05.wait::ld naming the destination registers of the loads it waits
// for, so that no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_ld8(uint32_t (&r)[8]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7])
                 :
                 : "memory");
}

// K and V viewed as csa_tc_common's 3-D tensor {D, T, B*H}, with boxes of
// 64 columns x `rows` rows (the key-tile height).
inline bool encode_rows_map(CUtensorMap *map, const void *ptr, int BH, int T, int D, int rows) {
    auto fn = get_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)T * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult rc = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return rc == CUDA_SUCCESS;
}

// The output viewed as the same 3-D tensor {D, T, B*H}, with boxes of 64
// columns x 32 rows (one softmax warp's rows of one column half); rows past
// T are not written.
inline bool encode_out_map(CUtensorMap *map, void *ptr, int BH, int T, int D) {
    auto fn = get_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)T * D * 2};
    const cuuint32_t box[3] = {64, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult rc = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return rc == CUDA_SUCCESS;
}

// 3-D tiled TMA store of one box from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const void *desc, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];"
                 ::"l"(reinterpret_cast<uint64_t>(desc)), "r"(c0), "r"(c1), "r"(c2), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared-memory sources of this thread's committed stores have been read
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// this thread's committed stores have completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ------------------------------------------------------------- weights
// One interval's two end weights, times (ln 2)^2.  X = u_right - u_left in
// log2 units, p = 2^u, x = X ln2 the logit step.
// Closed form (|X| >= 1/16):
//     sig = (p1 - p0)/X = S ln2,  R = (sig - p0 ln2)/X,  L = sig ln2 - R.
// Its error, the independent rounding of the two exponentials divided by
// X^2, stays below 4e-4 relative.  For |X| < 1/16 the same three lines run
// with other coefficients, giving the trapezoid value of S and the
// first-order expansion of phi2:
//     sig = (p0 + p1) ln2/2,  R = (ln2)^2 (2 p0 + p1)/6,  L = (ln2)^2 (p0 + 2 p1)/6,
// which match p0 phi2(x) and p1 phi2(-x) to (x^2)/12 relative (< 1.6e-4).
// Both errors are below the 2^-9 rounding of the bf16 P these weights become.
// The kernel runs seg_weights2, the same operations on two intervals at
// once; this scalar form serves the test hook.
__device__ __forceinline__ void seg_weights(float X, float p0, float p1, float &R, float &L) {
    const float rx = rcp_approx(X);
    const bool small = fabsf(X) < kTau;
    const float a1 = small ? 1.0f : -1.0f;
    const float f1 = small ? 0.5f * kLn2 : rx;
    const float a2 = fmaf(a1, 0.75f * kLn2, -0.25f * kLn2);  // ln2/2 or -ln2
    const float f2 = small ? kLn2 / 3.0f : rx;
    const float sig = fmaf(p0, a1, p1) * f1;
    R = fmaf(p0, a2, sig) * f2;
    L = fmaf(sig, kLn2, -R);
}

// Two intervals (lanes x and y).  R: the left keys' shares; Ln: minus the
// right keys' shares (R - sig ln2, the same rounding as -L above).
__device__ __forceinline__ void seg_weights2(float2 X, float2 p0, float2 p1, float2 &R,
                                             float2 &Ln) {
    const float rxx = rcp_approx(X.x), rxy = rcp_approx(X.y);
    const bool sx = fabsf(X.x) < kTau, sy = fabsf(X.y) < kTau;
    const float2 a1 = make_float2(sx ? 1.0f : -1.0f, sy ? 1.0f : -1.0f);
    const float2 f1 = make_float2(sx ? 0.5f * kLn2 : rxx, sy ? 0.5f * kLn2 : rxy);
    const float2 f2 = make_float2(sx ? kLn2 / 3.0f : rxx, sy ? kLn2 / 3.0f : rxy);
    const float2 a2 = __ffma2_rn(a1, make_float2(0.75f * kLn2, 0.75f * kLn2),
                                 make_float2(-0.25f * kLn2, -0.25f * kLn2));
    const float2 sig = __fmul2_rn(__ffma2_rn(p0, a1, p1), f1);
    R = __fmul2_rn(__ffma2_rn(p0, a2, sig), f2);
    Ln = __ffma2_rn(sig, make_float2(-kLn2, -kLn2), R);
}

__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&r)[4]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}

// Per-row state of one softmax thread (one column half of one row).
struct RowState {
    float k2;      // scale * log2(e)
    float m;       // this half's running max of the logits, log2 units
    float l;       // fp32 sum of this half's weights (gives lse)
    float w_sink;  // weight of the given sink pair (k0, v0 supplied), half 0
    float s_sink;  // q . k0 of the given sink pair
    int mode;      // sink mode
};

// The weights of a chunk of NCK keys (16 or 8) of one half-row: the keys of
// columns cb..cb+NCK-1.  s[0..NCK]: their raw logits q.k and that of column
// cb+NCK.  Lnc: minus the L share key cb receives from interval (cb-1, cb);
// on return that of column cb+NCK.  EDGE_L / EDGE_R: the chunk is the first
// / last of its half, so that its first key may be the tile's left halo
// (halo_l), or the sink (sink: column 1 of the query tile's first key tile),
// and its last key the right halo (halo_r).  SYM: the symmetric interval
// [1/2, t + 1/2] with constant end half-cells: in the first tile the sink
// takes no weight and key 1's left share is its half-cell p_1/2; each row's
// last key (MASKED) adds its right half-cell p/2 (both times (ln 2)^2).
// Produces the bf16 P (pk, keys paired in order) and the keys' fp32 sum
// (csum); w1 is the weight of column cb+1 (the sink's, when sink).
template <int NCK, bool MASKED, bool SYM, bool EDGE_L, bool EDGE_R>
__device__ __forceinline__ void cont_chunk(const float (&s)[NCK + 1], const RowState &st, float nm,
                                           int cb, int c_last, bool halo_l, bool sink,
                                           bool halo_r, float &Lnc, uint32_t (&pk)[NCK / 2],
                                           float2 &csum, float &w1) {
    constexpr int NH = NCK / 2;
    float u[NCK + 1], p[NCK + 1];
#pragma unroll
    for (int i = 0; i <= NCK; ++i) {
        float sv = s[i];
        if (EDGE_L && !SYM && i == 1) {
            // the sink's logit: k_0 = k_1 (copy-first) or the given q.k0
            const float alt = st.mode == CSA_K0_GIVEN ? st.s_sink : s[2];
            sv = sink && st.mode != CSA_K0_ZERO ? alt : sv;
        }
        u[i] = fmaf(sv, st.k2, nm);
        p[i] = ex2_approx(u[i]);
    }
    float2 R[NH], Ln[NH];
#pragma unroll
    for (int k = 0; k < NH; ++k) {
        const float2 X = __ffma2_rn(make_float2(u[k], u[k + NH]), make_float2(-1.0f, -1.0f),
                                    make_float2(u[k + 1], u[k + NH + 1]));
        seg_weights2(X, make_float2(p[k], p[k + NH]), make_float2(p[k + 1], p[k + NH + 1]), R[k],
                     Ln[k]);
        if (MASKED) {
            // interval (c, c+1) exists for this row only if c+1 <= its last key
            const bool vx = cb + k + 1 <= c_last, vy = cb + k + NH + 1 <= c_last;
            R[k] = make_float2(vx ? R[k].x : 0.0f, vy ? R[k].y : 0.0f);
            Ln[k] = make_float2(vx ? Ln[k].x : 0.0f, vy ? Ln[k].y : 0.0f);
        }
    }
    if (EDGE_L) {
        // column 0 of the first tile is no position: no interval (0, 1)
        Ln[0].x = sink ? 0.0f : Ln[0].x;
        if (SYM) {
            R[1].x = sink ? 0.0f : R[1].x;
            Ln[1].x = sink ? -kHalfCell * p[2] : Ln[1].x;
        }
    }
    float2 W[NH];
    W[0] = __ffma2_rn(make_float2(Lnc, Ln[NH - 1].x), make_float2(-1.0f, -1.0f), R[0]);
#pragma unroll
    for (int k = 1; k < NH; ++k) W[k] = __ffma2_rn(Ln[k - 1], make_float2(-1.0f, -1.0f), R[k]);
    Lnc = Ln[NH - 1].y;
    if (SYM && MASKED) {
        // each row's last key adds its right half-cell p/2
#pragma unroll
        for (int k = 0; k < NH; ++k) {
            W[k].x = cb + k == c_last ? fmaf(kHalfCell, p[k], W[k].x) : W[k].x;
            W[k].y = cb + k + NH == c_last ? fmaf(kHalfCell, p[k + NH], W[k].y) : W[k].y;
        }
    }
    if (EDGE_L) W[0].x = halo_l ? 0.0f : W[0].x;
    if (EDGE_R) W[NH - 1].y = halo_r ? 0.0f : W[NH - 1].y;
    w1 = W[1].x;
    if (EDGE_L && !SYM) {
        // v_0 = v_1: the sink's weight lands on key 1; a given v_0's share
        // w_0 v_0 is added in fp32 at the end
        const bool copy = sink && st.mode == CSA_K0_COPY_FIRST;
        const bool given = sink && st.mode == CSA_K0_GIVEN;
        W[2].x = copy ? W[2].x + W[1].x : W[2].x;
        W[1].x = copy || given ? 0.0f : W[1].x;
    }
    float2 t = W[0];
#pragma unroll
    for (int k = 1; k < NH; ++k) t = __fadd2_rn(t, W[k]);
    csum = t;
#pragma unroll
    for (int m = 0; m < NH / 2; ++m) {
        pk[m] = pack_bf16x2(W[2 * m].x, W[2 * m + 1].x);
        pk[NH / 2 + m] = pack_bf16x2(W[2 * m].y, W[2 * m + 1].y);
    }
}

// The short-conv reading of eq. (13): a key's weight is 2^z, with z in log2
// units relative to the running max and b replaced by its first-order term:
//   inside the row   z = (4 u_c + u_{c-1} + u_{c+1}) / 6
//   one-sided ends   z = (2 u_c + u_nb) / 3 - 1   (the sink; each row's last key)
// (-1 is log2 of the 1/2 in log phi2(x) = -log 2 + x/3 + ...).  Every z is a
// convex combination of logits minus a constant, so the running max of the
// raw logits still bounds it.  Arguments as cont_chunk; ul is the u of
// column cb-1 on entry and that of column cb+NCK-1 on return.
template <int NCK, bool MASKED, bool EDGE_L, bool EDGE_R>
__device__ __forceinline__ void short_chunk(const float (&s)[NCK + 1], const RowState &st, float nm,
                                            int cb, int c_last, bool halo_l, bool sink,
                                            bool halo_r, float &ul, uint32_t (&pk)[NCK / 2],
                                            float2 &csum, float &w1) {
    constexpr int NH = NCK / 2;
    constexpr float kThird = 1.0f / 3.0f, kSixth = 1.0f / 6.0f;
    float u[NCK + 2];  // u[i + 1] is column cb + i
    u[0] = ul;
#pragma unroll
    for (int i = 0; i <= NCK; ++i) {
        float sv = s[i];
        if (EDGE_L && i == 1) {
            const float alt = st.mode == CSA_K0_GIVEN ? st.s_sink : s[2];
            sv = sink && st.mode != CSA_K0_ZERO ? alt : sv;
        }
        u[i + 1] = fmaf(sv, st.k2, nm);
    }
    ul = u[NCK];
    float2 W[NH];
#pragma unroll
    for (int k = 0; k < NH; ++k) {
        const float2 uc = make_float2(u[k + 1], u[k + NH + 1]);
        const float2 nbs =
            __fadd2_rn(make_float2(u[k], u[k + NH]), make_float2(u[k + 2], u[k + NH + 2]));
        const float2 z = __ffma2_rn(nbs, make_float2(kSixth, kSixth),
                                    __fmul2_rn(uc, make_float2(4.0f * kSixth, 4.0f * kSixth)));
        float zz[2] = {z.x, z.y};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int i = k + NH * hh;  // key cb + i
            if (EDGE_L && i == 1) {
                // the sink is a one-sided end (right neighbour only)
                zz[hh] = sink ? fmaf(u[i + 2], kThird, fmaf(2.0f * kThird, u[i + 1], -1.0f)) : zz[hh];
            }
            if (MASKED) {
                const int c = cb + i;
                const float zl = fmaf(u[i], kThird, fmaf(2.0f * kThird, u[i + 1], -1.0f));
                zz[hh] = c == c_last ? zl : zz[hh];
                zz[hh] = c <= c_last ? ex2_approx(zz[hh]) : 0.0f;
            } else {
                zz[hh] = ex2_approx(zz[hh]);
            }
        }
        W[k] = make_float2(zz[0], zz[1]);
    }
    if (EDGE_L) W[0].x = halo_l ? 0.0f : W[0].x;
    if (EDGE_R) W[NH - 1].y = halo_r ? 0.0f : W[NH - 1].y;
    w1 = W[1].x;
    if (EDGE_L) {
        const bool copy = sink && st.mode == CSA_K0_COPY_FIRST;
        const bool given = sink && st.mode == CSA_K0_GIVEN;
        W[2].x = copy ? W[2].x + W[1].x : W[2].x;
        W[1].x = copy || given ? 0.0f : W[1].x;
    }
    float2 t = W[0];
#pragma unroll
    for (int k = 1; k < NH; ++k) t = __fadd2_rn(t, W[k]);
    csum = t;
#pragma unroll
    for (int m = 0; m < NH / 2; ++m) {
        pk[m] = pack_bf16x2(W[2 * m].x, W[2 * m + 1].x);
        pk[NH / 2 + m] = pack_bf16x2(W[2 * m].y, W[2 * m + 1].y);
    }
}

__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2 phi2(x) and log2 phi2(-x) of one logit step x (natural units), from
// MUFU exp2/log2: |x| <= 1 from the power series of the integral definition
// (even and odd parts shared by both signs, seven terms: below 3e-6
// relative); |x| > 1 from e^{|x|} - 1 - |x| = e^{|x|} (1 - (1 + |x|) e^{-|x|})
// and e^{-|x|} - 1 + |x|, both free of cancellation there.
__device__ __forceinline__ void lg2_phi2_pm(float x, float &lp, float &lm) {
    const float ax = fabsf(x), x2 = x * x;
    const float ev = fmaf(x2, fmaf(x2, fmaf(x2, 1.0f / 40320.0f, 1.0f / 720.0f), 1.0f / 24.0f), 0.5f);
    const float od = x * fmaf(x2, fmaf(x2, 1.0f / 5040.0f, 1.0f / 120.0f), 1.0f / 6.0f);
    const float sp = lg2_approx(ev + od), sm = lg2_approx(ev - od);
    const float e = ex2_approx(-ax * kLog2e), l2ax = lg2_approx(ax);
    const float bpos = fmaf(ax, kLog2e, lg2_approx(fmaf(-(1.0f + ax), e, 1.0f))) - 2.0f * l2ax;
    const float bneg = lg2_approx(e - 1.0f + ax) - 2.0f * l2ax;
    const bool small = ax <= 1.0f, pos = x > 0.0f;
    lp = small ? sp : (pos ? bpos : bneg);
    lm = small ? sm : (pos ? bneg : bpos);
}

// The log-domain evaluation of the same weights, eq. (10)/(11) as written:
// a key's weight is 2^z, z = u + log2(phi2(a_{c-1} - a_c) + phi2(a_{c+1} - a_c))
// (u in log2 units relative to the running max), the two log2 phi2 added by
// a log-domain sum; one-sided at the sink (right neighbour only) and at each
// row's last key (left neighbour only).  These are cont_chunk's weights
// without the common (ln 2)^2 factor, formed with about nine MUFU
// operations per key where cont_chunk takes two.  Arguments as short_chunk.
template <int NCK, bool MASKED, bool EDGE_L, bool EDGE_R>
__device__ __forceinline__ void log_chunk(const float (&s)[NCK + 1], const RowState &st, float nm,
                                          int cb, int c_last, bool halo_l, bool sink, bool halo_r,
                                          float &ul, uint32_t (&pk)[NCK / 2], float2 &csum,
                                          float &w1) {
    float u[NCK + 2];  // u[i + 1] is column cb + i
    u[0] = ul;
#pragma unroll
    for (int i = 0; i <= NCK; ++i) {
        float sv = s[i];
        if (EDGE_L && i == 1) {
            const float alt = st.mode == CSA_K0_GIVEN ? st.s_sink : s[2];
            sv = sink && st.mode != CSA_K0_ZERO ? alt : sv;
        }
        u[i + 1] = fmaf(sv, st.k2, nm);
    }
    ul = u[NCK];
    // interval q joins columns cb + q - 1 and cb + q
    float lp[NCK + 1], lm[NCK + 1];
#pragma unroll
    for (int q = 0; q <= NCK; ++q) lg2_phi2_pm((u[q + 1] - u[q]) * kLn2, lp[q], lm[q]);
    float W[NCK];
#pragma unroll
    for (int i = 0; i < NCK; ++i) {
        const int c = cb + i;
        const float l = lm[i], r = lp[i + 1];  // phi2(a_{c-1} - a_c), phi2(a_{c+1} - a_c)
        const float hi = fmaxf(l, r), lo = fminf(l, r);
        float b = hi + lg2_approx(1.0f + ex2_approx(lo - hi));
        if (EDGE_L && i == 1) b = sink ? r : b;
        if (MASKED) b = c == c_last ? l : b;
        float w = ex2_approx(u[i + 1] + b);
        if (MASKED) w = c <= c_last ? w : 0.0f;
        W[i] = w;
    }
    if (EDGE_L) W[0] = halo_l ? 0.0f : W[0];
    if (EDGE_R) W[NCK - 1] = halo_r ? 0.0f : W[NCK - 1];
    w1 = W[1];
    if (EDGE_L) {
        const bool copy = sink && st.mode == CSA_K0_COPY_FIRST;
        const bool given = sink && st.mode == CSA_K0_GIVEN;
        W[2] = copy ? W[2] + W[1] : W[2];
        W[1] = copy || given ? 0.0f : W[1];
    }
    float2 t = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < NCK; i += 2) t = __fadd2_rn(t, make_float2(W[i], W[i + 1]));
    csum = t;
#pragma unroll
    for (int m = 0; m < NCK / 2; ++m) pk[m] = pack_bf16x2(W[2 * m], W[2 * m + 1]);
}

// Max of the valid scaled logits a*log2(e) of one half-row in the query
// tile's first key tile: the half's columns and the neighbour column its
// intervals reach (columns c0..c0+h0, c0 = h (h0 - 1)), read in one batch
// of TMEM loads.  Column 0 is no position there, column 1 is the sink (none
// in SYM).  -inf if the half holds none of the row's keys; it then holds
// none of them in any later tile either.
__device__ __forceinline__ float fmin3f(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

template <int H0, bool SYM>
__device__ __forceinline__ float first_tile_max(uint32_t tS, const RowState &st, int c0,
                                                int c_last) {
    static_assert(H0 == 56 || H0 == 64, "column halves of 56 or 64 keys");
    uint32_t a[32], b[H0 == 64 ? 32 : 16], e8[8], z[1];
    tmem_ld32(tS + c0, a);
    if constexpr (H0 == 64) {
        tmem_ld32(tS + c0 + 32, b);
#pragma unroll
        for (int i = 0; i < 8; ++i) e8[i] = 0u;  // unused at this width
    } else {
        tmem_ld16(tS + c0 + 32, b);
        tmem_ld8(tS + c0 + 48, e8);
    }
    tmem_ld1(tS + c0 + H0, z[0]);
    tmem_wait_ld_regs<32>(a);
    if constexpr (H0 == 64) {
        tmem_wait_ld_regs<32>(b);
    } else {
        tmem_wait_ld16(b);
        tmem_wait_ld8(e8);
    }
    tmem_wait_ld_regs<1>(z);
    auto val = [&](int i) {
        return __uint_as_float(i < 32 ? a[i & 31]
                                      : (i == H0 ? z[0]
                                                 : (H0 == 64 || i < 48 ? b[(i - 32) & 31]
                                                                       : e8[(i - 48) & 7])));
    };
    if (H0 == 56 && c_last >= c0 + H0) {
        // every column of the window from column 2 on is one of the row's
        // keys: the max (scale < 0: the min) of the raw logits, scaled once
        float hi, lo;
        auto scan = [&](auto first) {
            // columns first .. H0 in pairs (the last pair may repeat one)
            constexpr int F = decltype(first)::value;
            hi = lo = val(F);
#pragma unroll
            for (int i = F + 1; i <= H0; i += 2) {
                const float x = val(i), y = val(i + 1 <= H0 ? i + 1 : i);
                hi = fmax3f(hi, x, y);
                lo = fmin3f(lo, x, y);
            }
        };
        if (c0 == 0)
            scan(std::integral_constant<int, 2>{});
        else
            scan(std::integral_constant<int, 0>{});
        if (c0 == 0) {
            // column 1: the sink, a key unless copied (or no sink at all)
            const float v1 = st.mode == CSA_K0_GIVEN ? st.s_sink : val(1);
            const bool in = !SYM && st.mode != CSA_K0_COPY_FIRST;
            hi = in ? fmaxf(hi, v1) : hi;
            lo = in ? fminf(lo, v1) : lo;
        }
        return st.k2 >= 0.0f ? hi * st.k2 : lo * st.k2;
    }
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i <= H0; ++i) {
        const int col = c0 + i;
        float v = val(i);
        if (col == 1 && st.mode == CSA_K0_GIVEN) v = st.s_sink;
        // the copied sink duplicates column 2
        const bool skip = col == 0 || (col == 1 && (SYM || st.mode == CSA_K0_COPY_FIRST));
        m = !skip && col <= c_last ? fmaxf(m, v * st.k2) : m;
    }
    return m;
}

// Raises a half's running max when a chunk's weights came out too large (the
// whole warp calls it; lanes whose max does not move scale by 1).  The new
// max is the exact max of the valid logits the half's intervals reach in
// this tile (columns c0..c0+h0, still in S: P is written only once the
// half-tile is done); O_h, when it holds this item's earlier tiles, is
// scaled (after waiting for the previous PV) by the factor returned.
// Returns (factor, new max); the factor is 0 when that wait expired (the
// abort flag is then raised).
__device__ __noinline__ float2 raise_running_max(uint32_t tS, uint32_t tO, int c0, int h0,
                                                 int ncol_o, int c_last, float k2, float m,
                                                 bool rescale_o, uint32_t odone, uint32_t parity,
                                                 volatile int *abort_flag) {
    float mx = m;
#pragma unroll 1
    for (int o = 0; o <= h0; o += 8) {
        uint32_t t[8];
        tmem_ld8(tS + c0 + o, t);
        tmem_wait_ld8(t);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            mx = o + i <= h0 && c0 + o + i <= c_last ? fmaxf(mx, __uint_as_float(t[i]) * k2) : mx;
    }
    const float alpha = ex2_approx(m - mx);
    if (rescale_o) {
        if (!__all_sync(0xffffffffu, wait_c(odone, parity, abort_flag))) return make_float2(0.0f, mx);
        tc_fence_after();
#pragma unroll 1
        for (int o = 0; o < ncol_o; o += 16) {
            uint32_t t[16];
            tmem_ld16(tO + o, t);
            tmem_wait_ld16(t);
#pragma unroll
            for (int i = 0; i < 16; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
            tmem_st16(tO + o, t);
        }
        tmem_wait_st();
    }
    return make_float2(alpha, mx);
}

// One column half of one key tile for this thread's row: the weights of the
// half's keys (columns kb..kb+h0-1, kb = h h0), held as bf16 in registers,
// checked, then written as P_h over the half's own S columns (64 keys,
// zero beyond the half).  Returns false if a wait expired.
template <int D, int FORM, bool SYM, bool MASKED>
__device__ __forceinline__ bool half_tile(uint32_t tS, uint32_t tO, RowState &st, int h,
                                          int c_last, bool first, bool rescale_o, uint32_t odone,
                                          uint32_t parity, volatile int *abort_flag) {
    using C = TcCfg<D>;
    constexpr bool SHORT = FORM == kTcShort, LOGD = FORM == kTcLog;
    constexpr int NK = C::kNK, H0 = C::kH0, NL = H0 - 48;
    const int kb = h * H0;
    // two chunks: 32 keys, then the remaining NB2 (24 or 32)
    constexpr int NB2 = H0 - 32;
    uint32_t pkA[16], pkB[NB2 / 2];
    float2 tsum = make_float2(0.0f, 0.0f);
    float w1 = 0.0f;
    bool ok = true;
    for (int attempt = 0;; ++attempt) {
        // lg[0]: column kb-1 (0 for half 0), lg[1 + i]: column kb + i,
        // lg[h0 + 1]: column kb + h0 (NK-1 for half 1)
        float lg[H0 + 2];
        uint32_t r2[16], r3[NL], r4[1];
        {
            uint32_t t0[1], t1[32], t2[1];
            tmem_ld1(tS + (h ? kb - 1 : 0), t0[0]);
            tmem_ld32(tS + kb, t1);
            tmem_ld1(tS + kb + 32, t2[0]);
            tmem_wait_ld_regs<1>(t0);
            tmem_wait_ld_regs<32>(t1);
            tmem_wait_ld_regs<1>(t2);
            lg[0] = __uint_as_float(t0[0]);
#pragma unroll
            for (int i = 0; i < 32; ++i) lg[1 + i] = __uint_as_float(t1[i]);
            lg[33] = __uint_as_float(t2[0]);
            // the rest of the half, read while the first chunk is computed
            tmem_ld16(tS + kb + 32, r2);
            if constexpr (NL == 8)
                tmem_ld8(tS + kb + 48, r3);
            else
                tmem_ld16(tS + kb + 48, r3);
            tmem_ld1(tS + (h ? NK - 1 : H0), r4[0]);
        }
        const float nm = -st.m;
        // the share key kb receives from interval (kb-1, kb) (exact), or the
        // u of column kb-1 (short); for half 0, column 0 is a halo: unused
        float carry;
        if (SHORT || LOGD) {
            carry = fmaf(lg[0], st.k2, nm);
        } else {
            const float u0 = fmaf(lg[0], st.k2, nm), u1 = fmaf(lg[1], st.k2, nm);
            float R, L;
            seg_weights(u1 - u0, ex2_approx(u0), ex2_approx(u1), R, L);
            carry = (!MASKED || kb <= c_last) ? -L : 0.0f;
        }
        tsum = make_float2(0.0f, 0.0f);
        bool bad = false;
        auto chunk = [&](auto nck, auto edge_l, auto edge_r, int off, auto &pk) {
            constexpr int NC = decltype(nck)::value;
            constexpr bool EL = decltype(edge_l)::value, ER = decltype(edge_r)::value;
            float s[NC + 1];
#pragma unroll
            for (int i = 0; i <= NC; ++i) s[i] = lg[1 + off + i];
            float2 cs;
            float w1c;
            if (SHORT)
                short_chunk<NC, MASKED, EL, ER>(s, st, nm, kb + off, c_last, h == 0, first && h == 0,
                                                h == 1, carry, pk, cs, w1c);
            else if (LOGD)
                log_chunk<NC, MASKED, EL, ER>(s, st, nm, kb + off, c_last, h == 0, first && h == 0,
                                              h == 1, carry, pk, cs, w1c);
            else
                cont_chunk<NC, MASKED, SYM, EL, ER>(s, st, nm, kb + off, c_last, h == 0,
                                                   first && h == 0, h == 1, carry, pk, cs, w1c);
            if (EL) w1 = w1c;
            tsum = __fadd2_rn(tsum, cs);
            bad |= !(cs.x + cs.y < kSumLimit);
        };
        using T_ = std::true_type;
        using F_ = std::false_type;
        chunk(std::integral_constant<int, 32>{}, T_{}, F_{}, 0, pkA);
        tmem_wait_ld16(r2);
        if constexpr (NL == 8)
            tmem_wait_ld8(r3);
        else
            tmem_wait_ld16(r3);
        tmem_wait_ld_regs<1>(r4);
#pragma unroll
        for (int i = 1; i < 16; ++i) lg[33 + i] = __uint_as_float(r2[i]);
#pragma unroll
        for (int i = 0; i < NL; ++i) lg[49 + i] = __uint_as_float(r3[i]);
        lg[H0 + 1] = __uint_as_float(r4[0]);
        chunk(std::integral_constant<int, NB2>{}, F_{}, T_{}, 32, pkB);
        if (attempt > 0 || !__any_sync(0xffffffffu, bad)) break;
        // the weights outgrew the running max: raise it, rescale O_h, redo
        const float2 am = raise_running_max(tS, tO, kb - h, H0, C::kN, c_last, st.k2, st.m,
                                            rescale_o, odone, parity, abort_flag);
        if (*abort_flag) {
            ok = false;
            break;
        }
        st.l *= am.x;
        st.w_sink *= am.x;
        st.m = am.y;
    }
    if (!ok) return false;
    if (!SYM && first && h == 0 && st.mode == CSA_K0_GIVEN) {
        st.w_sink = w1;
        st.l += w1;
    }
    // P_h: 64 keys over the half's own S columns, zero where they reach
    // into the other half
    const uint32_t pb = tS + C::col_p(h);
    if constexpr (NL == 8) {
        const uint32_t rb = pb + (h ? 4u : 0u);
        uint32_t a8[8], a4[4];
#pragma unroll
        for (int i = 0; i < 8; ++i) a8[i] = pkB[i];
#pragma unroll
        for (int i = 0; i < 4; ++i) a4[i] = pkB[8 + i];
        tmem_st16(rb, pkA);
        tmem_st8(rb + 16, a8);
        tmem_st4(rb + 24, a4);
        const uint32_t z[4] = {0u, 0u, 0u, 0u};
        tmem_st4(pb + (h ? 0u : 28u), z);
    } else {
        uint32_t b16[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) b16[i] = pkB[i % (NB2 / 2)];
        tmem_st16(pb, pkA);
        tmem_st16(pb + 16, b16);
    }
    tmem_wait_st();
    st.l += tsum.x + tsum.y;
    return true;
}

template <int D, int FORM, bool SYM>
__global__ void __launch_bounds__(kThreads, 1)
    tc_forward_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_o, const TcParams p) {
    using C = TcCfg<D>;
    constexpr int NSK = C::kStagesK, NSV = C::kStagesV;
    constexpr int KS = C::kKS;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const uint32_t sQ = base + C::kOffQ, sK = base + C::kOffK, sV = base + C::kOffV;
    const uint32_t bars = base + C::kOffBar;
#define BAR(i) (bars + 8u * (uint32_t)(i))
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    // the item ring: query tiles taken by the producer, decoded, read by every role
    volatile int *item_ring = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = p.T;

    if (threadIdx.x == 0) {
        mbar_init(BAR(C::kBarQ), 1);
        for (int s = 0; s < NSK; ++s) {
            mbar_init(BAR(C::kBarKFull + s), 1);
            mbar_init(BAR(C::kBarKEmpty + s), 1);
        }
        for (int s = 0; s < NSV; ++s) {
            mbar_init(BAR(C::kBarVFull + s), 1);
            mbar_init(BAR(C::kBarVEmpty + s), 1);
        }
        mbar_init(BAR(C::kBarSFull + 0), 1);
        mbar_init(BAR(C::kBarSFull + 1), 1);
        for (int i = 0; i < 4; ++i) mbar_init(BAR(C::kBarPFull + i), 128);
        mbar_init(BAR(C::kBarODone + 0), 1);
        mbar_init(BAR(C::kBarODone + 1), 1);
        mbar_init(BAR(C::kBarDrain), 1);
        mbar_init(BAR(C::kBarX), 256);
        mbar_init(BAR(C::kBarQEmpty), 1);
        mbar_init(BAR(C::kBarQRead), 4);
        for (int s = 0; s < 2; ++s) {
            mbar_init(BAR(C::kBarItemFull + s), 1);
            mbar_init(BAR(C::kBarItemEmpty + s), 9);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpProducer) {
        // The ones box of every V stage: in swizzled row r (a key of the
        // tile), logical 16-byte chunk 0 holds (1, 0, .., 0) and chunk 1
        // zeros, so B columns d..d+15 of the PV products are (1, 0, .., 0).
        for (int s = 0; s < NSV; ++s) {
            uint8_t *ones = smem + C::kOffV + s * C::kVBytes + C::kKBytes;
            for (int r = lane; r < C::kNK; r += 32) {
                *reinterpret_cast<uint4 *>(ones + r * 128 + ((0 ^ (r & 7)) << 4)) =
                    make_uint4(0x3F80u, 0u, 0u, 0u);  // bf16 1.0 in element 0
                *reinterpret_cast<uint4 *>(ones + r * 128 + ((1 ^ (r & 7)) << 4)) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async_smem();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Item c of this CTA (c = 0, 1, ..) sits in ring slot c & 1; n = 0 marks the end.
    auto take_item = [&](int c, TcItem &w) -> bool {
        if (!wait_c(BAR(C::kBarItemFull + (c & 1)), (c >> 1) & 1, abort_flag)) return false;
        const volatile int *e = item_ring + 3 * (c & 1);
        w.bh = e[0];
        w.row0 = e[1];
        w.n = e[2];
        return true;
    };

    if (warp >= 8) {
      if (warp == kWarpProducer) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            if (C::kTmaOut) tma_prefetch_desc(&tm_o);
            int item = (int)blockIdx.x;
            int issued_q = 0, issued_k = 0, issued_v = 0;  // loads issued (K, V: tiles)
            bool ok = true;
            for (int c = 0; ok; ++c) {
                ok = wait_s(BAR(C::kBarItemEmpty + (c & 1)), ((c >> 1) & 1) ^ 1, abort_flag);
                if (!ok) break;
                const bool last = item >= p.num_items;
                TcItem w = {0, 0, 0};
                if (!last) w = tc_item<KS>(item, p);
                volatile int *e = item_ring + 3 * (c & 1);
                e[0] = w.bh;
                e[1] = w.row0;
                e[2] = w.n;
                mbar_arrive(BAR(C::kBarItemFull + (c & 1)));
                if (last) break;
                // Q is reloaded once the previous item's last S is done and,
                // with a given sink, its rows' sink logits have been read from
                // it (those reads follow the Q load they wait for, so QRead
                // cannot run a phase ahead of this wait)
                if (c > 0) {
                    ok = wait_s(BAR(C::kBarQEmpty), (c - 1) & 1, abort_flag) &&
                         (p.mode != CSA_K0_GIVEN || wait_s(BAR(C::kBarQRead), (c - 1) & 1, abort_flag));
                    if (!ok) break;
                }
                mbar_arrive_expect_tx(BAR(C::kBarQ), C::kQBytes);
                for (int cc = 0; cc < C::kBoxes; ++cc)
                    tma_load_3d(sQ + cc * C::kQBox, &tm_q, 64 * cc, w.row0, w.bh, BAR(C::kBarQ));
                issued_q = c + 1;
                for (int j = 0; j < w.n; ++j) {
                    const int krow = KS * j - 2;
                    const int g = issued_k;  // this CTA's key tile count
                    const int sk = g % NSK;
                    if (!(ok = wait_s(BAR(C::kBarKEmpty + sk), ((g / NSK) & 1) ^ 1, abort_flag))) break;
                    mbar_arrive_expect_tx(BAR(C::kBarKFull + sk), C::kKBytes);
                    for (int cc = 0; cc < C::kBoxes; ++cc)
                        tma_load_3d(sK + sk * C::kKBytes + cc * C::kKBox, &tm_k, 64 * cc, krow, w.bh,
                                    BAR(C::kBarKFull + sk));
                    issued_k = g + 1;
                    const int sv = g % NSV;
                    if (!(ok = wait_s(BAR(C::kBarVEmpty + sv), ((g / NSV) & 1) ^ 1, abort_flag))) break;
                    mbar_arrive_expect_tx(BAR(C::kBarVFull + sv), C::kKBytes);
                    for (int cc = 0; cc < C::kBoxes; ++cc)
                        tma_load_3d(sV + sv * C::kVBytes + cc * C::kKBox, &tm_v, 64 * cc, krow, w.bh,
                                    BAR(C::kBarVFull + sv));
                    issued_v = g + 1;
                }
                // the next item, taken when this CTA is about to need it
                item = (int)gridDim.x + (int)atomicAdd(&g_sched_next[p.slot], 1u);
            }
            // Let every copy this thread issued land before the block can exit.
            if (issued_q > 0) wait_bar_drain(BAR(C::kBarQ), (issued_q - 1) & 1, &g_tc_status);
            for (int j = max(0, issued_k - NSK); j < issued_k; ++j)
                wait_bar_drain(BAR(C::kBarKFull + j % NSK), (j / NSK) & 1, &g_tc_status);
            for (int j = max(0, issued_v - NSV); j < issued_v; ++j)
                wait_bar_drain(BAR(C::kBarVFull + j % NSV), (j / NSV) & 1, &g_tc_status);
        }
        __syncwarp();
      } else {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdescS = make_idesc(128, C::kNK, false);
            constexpr uint32_t kIdescO = make_idesc(128, C::kN, true);
            // One stream of key tiles over this CTA's items: within an item S
            // runs two tiles ahead of PV; the next item's first S wait until
            // this item's last PV is issued, since waiting for its Q must not
            // hold that PV (and the epilogue) back.  So S and PV are always
            // in the same item.
            int c = -1, n = 0;     // the current item and its key tiles
            int s_j = 0, p_j = 0;  // its S and PV issued
            int gs = 0, gp = 0;    // S and PV issued over all items
            // S(gs) = Q K^T into S buffer gs % 2; K tile gs is released once done
            auto issue_s = [&]() -> bool {
                if (!wait_s(BAR(C::kBarKFull + gs % NSK), (gs / NSK) & 1, abort_flag)) return false;
                tc_fence_after();
                const uint32_t kb = sK + (gs % NSK) * C::kKBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t qo = (kk >> 2) * C::kQBox + (kk & 3) * 32;
                    const uint32_t ko = (kk >> 2) * C::kKBox + (kk & 3) * 32;
                    tc_mma_ss(tmem + C::col_s(gs & 1), make_sdesc(sQ + qo, 16, 1024),
                              make_sdesc(kb + ko, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
                }
                tc_commit(BAR(C::kBarSFull + (gs & 1)));
                tc_commit(BAR(C::kBarKEmpty + gs % NSK));
                ++gs;
                if (++s_j == n) tc_commit(BAR(C::kBarQEmpty));  // the item's last S
                return true;
            };
            // the next item and its first two S (one if it has a single key
            // tile); n = 0 once there is none
            auto next_item = [&]() -> bool {
                TcItem w;
                if (!take_item(c + 1, w)) return false;
                mbar_arrive(BAR(C::kBarItemEmpty + ((c + 1) & 1)));
                ++c;
                s_j = p_j = 0;
                n = w.n;
                if (n == 0) return true;
                if (!wait_s(BAR(C::kBarQ), c & 1, abort_flag)) return false;
                return issue_s() && (n == 1 || issue_s());
            };
            bool ok = next_item();
            while (ok && n > 0) {
                const uint32_t vb = sV + (gp % NSV) * C::kVBytes;
                if (!(ok = wait_s(BAR(C::kBarVFull + gp % NSV), (gp / NSV) & 1, abort_flag))) break;
                tc_fence_after();
                // [O_h | rowsum] (+)= P_h [V | ones] over the 64 keys of half h,
                // P_h read from the TMEM of S buffer gp % 2
                for (int h = 0; h < 2 && ok; ++h) {
                    if (!(ok = wait_s(BAR(C::kBarPFull + 2 * h + (gp & 1)), (gp >> 1) & 1, abort_flag)))
                        break;
                    tc_fence_after();
                    const uint32_t row_b = h ? (uint32_t)(C::kNK - 64) * 128u : 0u;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_ts(tmem + C::col_o(h), tmem + C::col_s(gp & 1) + C::col_p(h) + 8 * kk,
                                  make_sdesc(vb + row_b + kk * 2048, C::kKBox, 1024), kIdescO,
                                  (p_j > 0 || kk > 0) ? 1u : 0u);
                }
                if (!ok) break;
                tc_commit(BAR(C::kBarODone + (gp & 1)));
                tc_commit(BAR(C::kBarVEmpty + gp % NSV));
                ++gp;
                ++p_j;
                // S(gp+1) overwrites the TMEM that PV(gp-1) read as P; both are
                // tcgen05.mma issued in order by this thread.
                if (s_j < n)
                    ok = issue_s();
                else if (p_j == n)
                    ok = next_item();
            }
            // every MMA this thread issued completes before the block exits
            tc_commit(BAR(C::kBarDrain));
            wait_bar_drain(BAR(C::kBarDrain), 0, &g_tc_status);
        }
        __syncwarp();
      }
    } else {
        // ------------------------------------------------------ softmax
        const int h = warp >> 2, wq = warp & 3;
        const int irow = wq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tO = tmem + lane_off + C::col_o(h);
        float *xfin = reinterpret_cast<float *>(smem + C::kOffXFin);
        const uint32_t xbar = BAR(C::kBarX);
        int g = 0;  // key tiles of this CTA done so far
        bool ok = true;
        for (int c = 0; ok; ++c) {
            TcItem w;
            ok = __all_sync(0xffffffffu, take_item(c, w));
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(C::kBarItemEmpty + (c & 1)));
            if (!ok || w.n == 0) break;
            const int bh = w.bh, row0 = w.row0, n = w.n;
            const int r = row0 + irow;
            // this item's first products overwrite O_0 and O_1, which every
            // softmax thread read in the previous item's epilogue (the second
            // phase of that item on the exchange barrier)
            if (c > 0) {
                ok = __all_sync(0xffffffffu, wait_c(xbar, 1, abort_flag));
                if (!ok) break;
            }
            RowState st;
            st.k2 = p.k2;
            st.m = -INFINITY;
            st.l = st.w_sink = st.s_sink = 0.0f;
            st.mode = p.mode;
            if (!SYM && h == 0 && p.mode == CSA_K0_GIVEN) {
                ok = __all_sync(0xffffffffu, wait_c(BAR(C::kBarQ), c & 1, abort_flag));
                if (!ok) break;
                // s_sink = q_r . k0[h], from this row of the swizzled Q tile
                const __nv_bfloat16 *k0h = p.k0 + (size_t)(bh % p.H) * D;
                float acc = 0.0f;
#pragma unroll
                for (int cc = 0; cc < C::kBoxes; ++cc) {
#pragma unroll
                    for (int kc = 0; kc < 8; ++kc) {
                        const uint8_t *src = smem + C::kOffQ + cc * C::kQBox + irow * 128 +
                                             ((kc ^ (irow & 7)) << 4);
                        const uint4 qv = *reinterpret_cast<const uint4 *>(src);
                        const __nv_bfloat16 *qb = reinterpret_cast<const __nv_bfloat16 *>(&qv);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            acc = fmaf(__bfloat162float(qb[e]),
                                       __bfloat162float(k0h[cc * 64 + kc * 8 + e]), acc);
                    }
                }
                st.s_sink = acc;
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(C::kBarQRead));
            }
            for (int j = 0; ok && j < n; ++j, ++g) {
                const uint32_t tS = tmem + lane_off + C::col_s(g & 1);
                ok = __all_sync(0xffffffffu,
                                wait_c(BAR(C::kBarSFull + (g & 1)), (g >> 1) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                // last valid column of this row, and whether the tile needs masks
                const int c_last = r + 2 - KS * j;
                const bool masked = KS * (j + 1) > row0 + 1;
                if (j == 0) st.m = first_tile_max<C::kH0, SYM>(tS, st, h * (C::kH0 - 1), c_last);
                // PV pair g-1, for a rescale of O_h
                const uint32_t odone = BAR(C::kBarODone + ((g - 1) & 1)), par = ((g - 1) >> 1) & 1;
                ok = masked ? half_tile<D, FORM, SYM, true>(tS, tO, st, h, c_last, j == 0, j > 0,
                                                             odone, par, abort_flag)
                            : half_tile<D, FORM, SYM, false>(tS, tO, st, h, c_last, j == 0, j > 0,
                                                              odone, par, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_before();
                mbar_arrive(BAR(C::kBarPFull + 2 * h + (g & 1)));
            }
            if (!ok) break;
            // the two halves meet: their maxima, sums and the given sink's weight
            float *mine = xfin + (h * 128 + irow) * 4;
            mine[0] = st.m;
            mine[1] = st.l;
            mine[2] = st.w_sink;
            mbar_arrive(xbar);
            // sleeping: the MMA thread is issuing this item's last PV meanwhile
            ok = __all_sync(0xffffffffu, wait_s(xbar, 0, abort_flag));
            if (!ok) break;
            const float *oth = xfin + ((h ^ 1) * 128 + irow) * 4;
            const float m0 = h ? oth[0] : st.m, m1 = h ? st.m : oth[0];
            const float l0 = h ? oth[1] : st.l, l1 = h ? st.l : oth[1];
            const float w_sink = h ? oth[2] : st.w_sink;  // in half 0's scale
            const float mx = fmaxf(m0, m1);
            const float a0 = ex2_approx(m0 - mx), a1 = ex2_approx(m1 - mx);
            // O holds this item's last PV pair, g-1, once it is done (the
            // next item's first PV waits for every softmax thread's reads of
            // O: the exchange barrier's second phase below)
            ok = __all_sync(0xffffffffu,
                            wait_s(BAR(C::kBarODone + ((g - 1) & 1)), ((g - 1) >> 1) & 1, abort_flag));
            if (!ok) break;
            if (p.delay_ns != 0u && h == p.delay_half) __nanosleep(p.delay_ns);
            tc_fence_after();
            const uint32_t tO0 = tmem + lane_off + C::col_o(0), tO1 = tmem + lane_off + C::col_o(1);
            // o is divided by the sum of exactly the bf16 weights that fed the
            // PV products (column d of each O_h) plus the given sink's fp32 weight
            uint32_t rs[2][1];
            tmem_ld1(tO0 + D, rs[0][0]);
            tmem_ld1(tO1 + D, rs[1][0]);
            tmem_wait_ld_regs<1>(rs[0]);
            tmem_wait_ld_regs<1>(rs[1]);
            const float den = fmaf(a0, __uint_as_float(rs[0][0]) + w_sink, a1 * __uint_as_float(rs[1][0]));
            const float inv_l = 1.0f / den;
            const bool store = r < T;
            __nv_bfloat16 *orow =
                p.out + ((size_t)bh * T + (size_t)(store ? r : 0)) * D + h * (D / 2);
            const __nv_bfloat16 *v0h = p.v0 + (size_t)(bh % p.H) * D + h * (D / 2);
            uint8_t *stage = smem + C::kOffOut + warp * 4096;
            if (C::kTmaOut) {
                // the previous item's store from this warp's stage has read it
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
            }
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                uint32_t o0[32], o1[32];
                tmem_ld32(tO0 + h * (D / 2) + 32 * cc, o0);
                tmem_ld32(tO1 + h * (D / 2) + 32 * cc, o1);
                tmem_wait_ld_regs<32>(o0);
                tmem_wait_ld_regs<32>(o1);
                float val[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    float xo = __uint_as_float(o0[e]);
                    if (!SYM && p.mode == CSA_K0_GIVEN)
                        xo = fmaf(w_sink, __bfloat162float(v0h[32 * cc + e]), xo);
                    val[e] = fmaf(a0, xo, a1 * __uint_as_float(o1[e])) * inv_l;
                }
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(val[2 * e], val[2 * e + 1]);
                if (C::kTmaOut) {
                    // this row's 16-byte chunks 4 cc .. 4 cc + 3 of the staged box
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        *reinterpret_cast<uint4 *>(stage + lane * 128 + (((4 * cc + e) ^ (lane & 7)) << 4)) =
                            make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                } else if (store) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * cc);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                }
            }
            // this thread's reads of O are done: the item's second phase on
            // the exchange barrier
            tc_fence_before();
            mbar_arrive(xbar);
            if (C::kTmaOut) {
                // one TMA store of the warp's 32 rows x 64 columns (rows past T
                // are not written; a box wholly past T is not issued)
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && row0 + 32 * wq < T) {
                    tma_store_3d(&tm_o, smem_u32(stage), h * (D / 2), row0 + 32 * wq, bh);
                    bulk_commit();
                }
            }
            if (store && h == 0 && p.lse)
                p.lse[(size_t)bh * T + r] =
                    (mx + log2f(fmaf(a0, l0, a1 * l1))) * kLn2 + (FORM == kTcExact ? kLseShift : 0.0f);
            tc_fence_before();
        }
        // the output stores are complete before the block exits
        if (C::kTmaOut && lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tmem, 512);
    // The last CTA to finish puts this launch's scheduling slot back to zero.
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&g_sched_done[p.slot], 1u) == gridDim.x - 1) {
            atomicExch(&g_sched_next[p.slot], 0u);
            atomicExch(&g_sched_done[p.slot], 0u);
        }
    }
#undef BAR
}

// ---------------------------------------------------------------- test kernels
__global__ void seg_eval_kernel(const float *u0, const float *u1, float *right, float *left, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float U0 = u0[i] * kLog2e, U1 = u1[i] * kLog2e;
    const float p0 = ex2_approx(U0), p1 = ex2_approx(U1);
    float R, L;
    seg_weights(U1 - U0, p0, p1, R, L);
    constexpr float kInvKappa = 2.0813689810056077f;  // 1 / (ln 2)^2
    right[i] = R * kInvKappa;
    left[i] = L * kInvKappa;
}

__global__ void selftest_wait_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // Nothing ever arrives on this barrier: the wait must give up.
        mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, &g_tc_status, limit_ns);
    }
    __syncthreads();
}

// ---------------------------------------------------------------- host side
// Scheduling slots of one device.  A launch takes the next slot round robin;
// the slot's event, recorded after its previous launch, orders the two, so a
// slot's counters are reset before they are used again whatever streams the
// launches run on.  (Stream capture skips the events: a captured graph keeps
// its slot, and its replays follow one another on their stream.)
struct SchedSlots {
    std::mutex m;
    unsigned next = 0;
    cudaEvent_t ev[kSchedSlots] = {};
};
constexpr int kMaxDevices = 64;
SchedSlots g_slots[kMaxDevices];

template <class Launch>
int launch_with_slot(int dev, cudaStream_t stream, Launch &&launch) {
    if (dev < 0 || dev >= kMaxDevices) return CSA_ERR_UNSUPPORTED;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return CSA_ERR_CUDA;
    SchedSlots &S = g_slots[dev];
    std::lock_guard<std::mutex> lock(S.m);
    const int slot = (int)(S.next++ % kSchedSlots);
    cudaEvent_t &ev = S.ev[slot];
    if (cap == cudaStreamCaptureStatusNone) {
        if (ev == nullptr) {
            if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
                ev = nullptr;
                return CSA_ERR_CUDA;
            }
        } else if (cudaStreamWaitEvent(stream, ev, 0) != cudaSuccess) {
            return CSA_ERR_CUDA;
        }
    }
    if (!launch(slot)) return CSA_ERR_CUDA;
    if (cap == cudaStreamCaptureStatusNone && cudaEventRecord(ev, stream) != cudaSuccess)
        return CSA_ERR_CUDA;
    return CSA_OK;
}

template <int D, int FORM, bool SYM>
int launch_tc(const void *q, const void *k, const void *v, const void *k0, const void *v0,
              void *out, float *lse, int B, int H, int T, float scale, int mode,
              cudaStream_t stream, unsigned delay_ns = 0u, int delay_half = 0) {
    using C = TcCfg<D>;
    const int BH = B * H;
    CUtensorMap mq, mk, mv, mo;
    if (!encode_qkv_map(&mq, q, BH, T, D) || !encode_rows_map(&mk, k, BH, T, D, C::kNK) ||
        !encode_rows_map(&mv, v, BH, T, D, C::kNK) || !encode_out_map(&mo, out, BH, T, D))
        return CSA_ERR_CUDA;
    TcParams prm;
    prm.B = B;
    prm.H = H;
    prm.T = T;
    prm.num_qtiles = (T + 127) / 128;
    prm.group = heads_per_group(BH, T, D);
    prm.k2 = scale * kLog2e;
    prm.mode = mode;
    prm.k0 = static_cast<const __nv_bfloat16 *>(k0);
    prm.v0 = static_cast<const __nv_bfloat16 *>(v0);
    prm.out = static_cast<__nv_bfloat16 *>(out);
    prm.lse = lse;
    prm.delay_ns = delay_ns;
    prm.delay_half = delay_half;
    const long long items = (long long)prm.num_qtiles * BH;
    if (items > 0x7fffffffLL) return CSA_ERR_UNSUPPORTED;
    prm.num_items = (int)items;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return CSA_ERR_CUDA;
    const unsigned grid = (unsigned)(items < sms ? items : sms);  // one CTA per SM
    auto kern = tc_forward_kernel<D, FORM, SYM>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
        return CSA_ERR_CUDA;
    return launch_with_slot(dev, stream, [&](int slot) {
        prm.slot = slot;
        kern<<<grid, kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, mo, prm);
        return cudaGetLastError() == cudaSuccess;
    });
}

}  // namespace

int csa_tc_forward(const void *q, const void *k, const void *v, const void *k0, const void *v0,
                   void *out, float *lse, int B, int H, int T, int d, float scale, int mode,
                   int form, cudaStream_t stream) {
#define CSA_TC_LAUNCH(DD, SC, SY) \
    return launch_tc<DD, SC, SY>(q, k, v, k0, v0, out, lse, B, H, T, scale, mode, stream)
    if (d != 64 && d != 128) return CSA_ERR_UNSUPPORTED;
    if (form == kFormShortConv) {
        if (d == 128) CSA_TC_LAUNCH(128, kTcShort, false);
        CSA_TC_LAUNCH(64, kTcShort, false);
    }
    if (form == kFormLogDomain) {
        if (d == 128) CSA_TC_LAUNCH(128, kTcLog, false);
        CSA_TC_LAUNCH(64, kTcLog, false);
    }
    if (form == kFormSymmetric) {  // no sink: mode is ignored
        mode = CSA_K0_ZERO;
        if (d == 128) CSA_TC_LAUNCH(128, kTcExact, true);
        CSA_TC_LAUNCH(64, kTcExact, true);
    }
    if (d == 128) CSA_TC_LAUNCH(128, kTcExact, false);
    CSA_TC_LAUNCH(64, kTcExact, false);
#undef CSA_TC_LAUNCH
}

int csa_tc_forward_delayed(const void *q, const void *k, const void *v, const void *k0,
                           const void *v0, void *out, float *lse, int B, int H, int T, int d,
                           float scale, int mode, unsigned delay_ns, int delay_half,
                           cudaStream_t stream) {
    if (d == 128)
        return launch_tc<128, kTcExact, false>(q, k, v, k0, v0, out, lse, B, H, T, scale, mode,
                                               stream, delay_ns, delay_half);
    if (d == 64)
        return launch_tc<64, kTcExact, false>(q, k, v, k0, v0, out, lse, B, H, T, scale, mode,
                                              stream, delay_ns, delay_half);
    return CSA_ERR_UNSUPPORTED;
}

cudaError_t csa_tc_segment_weights_eval(const float *u0, const float *u1, float *right,
                                        float *left, int n, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    seg_eval_kernel<<<(n + 255) / 256, 256, 0, stream>>>(u0, u1, right, left, n);
    return cudaGetLastError();
}

cudaError_t csa_tc_selftest_wait_timeout(unsigned timeout_us, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>((unsigned long long)timeout_us * 1000ull);
    return cudaGetLastError();
}

int csa_tc_take_status(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return CSA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_status, sizeof(int)) != cudaSuccess) return CSA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(int)) != cudaSuccess) return CSA_ERR_CUDA;
    return v;
}
