// Tensor-core forward kernel of causal continuous attention for sm_103a:
// eq. (10)/(11) of Jianlin Su, "Continuous Softmax Attention" ("Assembly
// and Simplification"), bf16 inputs, d = 64 or 128, fp32 accumulation.
//
// Work split.  A work item is one 128-row query tile of one (b, h); it walks
// the key/value tiles up to its diagonal.  The grid is one persistent CTA per
// SM: CTA b starts with item b and its producer warp takes further items from
// a counter (heaviest query tiles first, heads grouped for L2), handing each
// to the other warps through a two-entry ring.  The K/V rings, the S buffers
// and O count over all of the CTA's key tiles and carry on from one item to
// the next, so one item's epilogue overlaps the next item's first S products.
// Warps:
//   0-7  softmax: warp w owns rows 32*(w%4).. (its TMEM lane quarter) and,
//        with w/4, the column half 0..63 or 64..127 of S
//   8    TMA producer (lane 0; all lanes write the constant ones block once)
//   9    TMEM allocator and tcgen05.mma issuer (lane 0)
// Shared memory holds the Q tile, a K ring and a V ring of 128B-swizzled
// 64-column boxes written by TMA.  Each V stage has one more box holding a
// column of ones, so the PV product (N = d + 16) also accumulates, in O
// column d, the row sum of exactly the bf16 P values it used.
// Tensor memory (512 columns): S buffer 0 | S buffer 1 | O (d + 16 columns).
// S is double-buffered: the tensor core computes PV(j) and S(j+2) while the
// softmax works on S(j+1).  P (bf16) overwrites columns of its own S that
// are no longer read (0..31 and 80..111) and is the A operand of the PV
// product straight from TMEM.
//
// The halo for b.  b_{t,i} needs the logit of the key to the right of i.
// Key tiles are loaded at a stride of 127 rows: an S tile covers 128
// consecutive keys of the extended sequence (the sink first), its last
// column is the first key of the next tile, and that column's P is 0.  Tile
// j starts at array row 127*j - 1; for j = 0 this row is -1, which TMA fills
// with zeros: the zero sink pair k_0 = v_0 = 0 comes for free, and the
// copy-first and given modes only replace the first logit (and, for given
// v_0, add w_0 * v_0 to the output at the end).
//
// The weights.  With the running max m (log2 units) and u = a*log2(e) - m,
// p = 2^u, each interval between neighbouring keys contributes
//   R = p_left * phi2(x)  to its left key and  L = p_right * phi2(-x)  to its
// right key (x the logit step), the regrouping of eq. (9); a key's weight
// e^{a+b-m} is L + R of its two intervals, one-sided at both ends.  R and L
// follow from the interval integral S = (p_right - p_left)/x by
// R = (S - p_left)/x and L = S - R, with a power series for small steps.
// All weights carry a common factor (ln 2)^2, which cancels in o and is
// removed from lse.
//
// The template flag SHORT turns the kernel into the short-conv reading of
// eq. (13): b is replaced by its first-order term, so a key's weight is
// 2^z with z an affine combination of its own and its neighbours' logits
// (short_chunk) and no phi2 is formed.  SYM integrates over the symmetric
// interval [1/2, t + 1/2] instead (constant half-cells at both ends, no
// sink; cont_chunk).
//
// The two column halves of a row exchange their partial maxima, the L share
// that crosses into the next tile, and their final sums through shared
// memory, synchronised by an mbarrier.  Every mbarrier wait is bounded in
// time; on expiry the kernel records CSA_ERR_TIMEOUT, every role skips its
// remaining work, the MMA issuer waits for its own MMAs, the producer waits
// for its own copies, and TMEM is freed.
#include <mutex>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

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

template <int D>
struct TcCfg {
    static constexpr int kChunks = D / 64;  // 64-column boxes per tile
    static constexpr int kTileBytes = kChunks * kChunkBytes;
    static constexpr int kVStageBytes = kTileBytes + kChunkBytes;  // values + ones box
    static constexpr int kN = D + 16;                              // PV width
    static constexpr int kStagesK = D == 128 ? 2 : 3;
    static constexpr int kStagesV = D == 128 ? 2 : 3;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kTileBytes;
    static constexpr int kOffV = kOffK + kStagesK * kTileBytes;
    static constexpr int kOffBar = kOffV + kStagesV * kVStageBytes;
    // barrier indices
    static constexpr int kBarQ = 0;
    static constexpr int kBarKFull = 1;
    static constexpr int kBarKEmpty = kBarKFull + kStagesK;
    static constexpr int kBarVFull = kBarKEmpty + kStagesK;
    static constexpr int kBarVEmpty = kBarVFull + kStagesV;
    static constexpr int kBarSFull = kBarVEmpty + kStagesV;  // [2] one per S buffer
    static constexpr int kBarPFull = kBarSFull + 2;
    static constexpr int kBarODone = kBarPFull + 1;
    static constexpr int kBarDrain = kBarODone + 1;
    static constexpr int kBarX = kBarDrain + 1;  // half-to-half exchange
    static constexpr int kBarQEmpty = kBarX + 1;     // an item's last S is done
    static constexpr int kBarQRead = kBarQEmpty + 1;  // its sink logits are read from Q
    static constexpr int kBarItemFull = kBarQRead + 1;    // [2] item ring
    static constexpr int kBarItemEmpty = kBarItemFull + 2;  // [2]
    static constexpr int kNumBars = kBarItemEmpty + 2;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    // exchange buffers between the two column halves of the query tile:
    //   xmax   [2 slots][2 halves][128 rows]  partial row maxima
    //   xcarry [2 slots][128 rows]            L share carried to the next tile
    //   xfin   [2 halves][128 rows][2]        final fp32 sum, sink weight
    // misc: TMEM base, abort flag, then the item ring ([2][3] ints: bh, row0, n)
    static constexpr int kOffXMax = kOffMisc + 32;
    static constexpr int kOffXCarry = kOffXMax + 2 * 2 * 128 * 4;
    static constexpr int kOffXFin = kOffXCarry + 2 * 128 * 4;
    static constexpr int kSmemBytes = kOffXFin + 2 * 128 * 2 * 4 + 1024;  // + slack to align the base
    // TMEM columns: S buffer 0 | S buffer 1 | O
    __device__ static constexpr uint32_t col_s(int b) { return 128u * (uint32_t)b; }
    static constexpr uint32_t kColO = 256u;
};

struct TcParams {
    int B, H, T;
    int num_qtiles;
    int group;  // heads per scheduling group
    float k2;  // scale * log2(e)
    int mode;
    const __nv_bfloat16 *k0;
    const __nv_bfloat16 *v0;
    __nv_bfloat16 *out;
    float *lse;
    int num_items;  // query tiles: num_qtiles * B * H
    int slot;       // this launch's scheduling counters
};

// A work item is one query tile of one (b, h).  Heads go in groups whose K/V
// fit in L2 together; within a group the heaviest query tiles come first
// (longest-first keeps the tail short).
struct TcItem {
    int bh, row0, n;  // n: key tiles (127-row stride) the query tile reads
};

__device__ __forceinline__ TcItem tc_item(int item, const TcParams &p) {
    const int nq = p.num_qtiles, BH = p.B * p.H;
    const int grp = item / (p.group * nq);
    const int gsz = min(p.group, BH - grp * p.group);
    const int idx = item - grp * p.group * nq;
    TcItem w;
    w.bh = grp * p.group + idx % gsz;
    w.row0 = (nq - 1 - idx / gsz) * 128;
    w.n = (min(w.row0 + 127, p.T - 1) + 1) / 127 + 1;
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
// not complete sleeps until it completes instead of polling.  Used at the end
// of an item, where all softmax warps wait while the MMA thread issues and
// completes the item's last PV, so that their polling takes no issue slots
// from it.
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

// ------------------------------------------------------------- weights
// |X| below this (log2 units) takes the small-step coefficients.
constexpr float kTau = 0.0625f;

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

// One 32-column chunk of weights.  sv[0..32] are the raw logits q.k of
// columns cbase..cbase+32; Lc is the L share of column cbase coming from the
// left.  Produces w[0..31] (e^{a+b-m} * (ln2)^2), returns in Lc the L share
// of column cbase+32, and in L31 that of cbase+31.
// SYM, the symmetric interval [1/2, t + 1/2] with constant end half-cells:
// with first_cell (the chunk holding the sink and key 1) the sink takes no
// weight and key 1's left share is its half-cell p_1/2; each row's last key
// (MASKED) adds its right half-cell p/2 (both times (ln 2)^2).
template <bool MASKED, bool SYM>
__device__ __forceinline__ void cont_chunk(const float (&sv)[33], float k2, float nm, int cbase,
                                           int c_last, bool first_cell, float &Lc, float &L31,
                                           float (&w)[32]) {
    constexpr float kHalfCell = 0.5f * kLn2 * kLn2;
    float u[33], pe[33], L[33], R[32];
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const float2 t = __ffma2_rn(make_float2(sv[i], sv[i + 1]), make_float2(k2, k2),
                                    make_float2(nm, nm));
        u[i] = t.x;
        u[i + 1] = t.y;
    }
    u[32] = fmaf(sv[32], k2, nm);
#pragma unroll
    for (int i = 0; i < 33; ++i) pe[i] = ex2_approx(u[i]);
    L[0] = Lc;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        float Ri, Li;
        seg_weights(u[i + 1] - u[i], pe[i], pe[i + 1], Ri, Li);
        if (MASKED) {
            // interval (c, c+1) exists for this row only if c+1 <= its last key
            const bool seg_ok = cbase + i + 1 <= c_last;
            Ri = seg_ok ? Ri : 0.0f;
            Li = seg_ok ? Li : 0.0f;
        }
        if (SYM && i == 0 && first_cell) {
            Ri = 0.0f;                    // the sink is not part of [1/2, t + 1/2]
            Li = kHalfCell * pe[1];       // key 1's left half-cell
        }
        R[i] = Ri;
        L[i + 1] = Li;
    }
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const float2 t = __fadd2_rn(make_float2(L[i], L[i + 1]), make_float2(R[i], R[i + 1]));
        w[i] = t.x;
        w[i + 1] = t.y;
    }
    if (SYM && MASKED) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            w[i] = cbase + i == c_last ? fmaf(kHalfCell, pe[i], w[i]) : w[i];  // right half-cell
    }
    L31 = L[31];
    Lc = L[32];
}

// The short-conv reading of eq. (13): a key's weight is 2^z, with z in log2
// units relative to the running max and b replaced by its first-order term:
//   inside the row   z = (4 u_c + u_{c-1} + u_{c+1}) / 6
//   one-sided ends   z = (2 u_c + u_nb) / 3 - 1   (the sink; each row's last key)
// (-1 is log2 of the 1/2 in log phi2(x) = -log 2 + x/3 + ...).  Every z is a
// convex combination of logits minus a constant, so the running max of the
// raw logits still bounds it.  sv[0..32] are the raw logits of columns
// cbase..cbase+32, sl that of column cbase-1 (unused when first_end: the
// sink).  Produces w[0..31].
template <bool MASKED>
__device__ __forceinline__ void short_chunk(const float (&sv)[33], float sl, float k2, float nm,
                                            int cbase, int c_last, bool first_end,
                                            float (&w)[32]) {
    constexpr float kThird = 1.0f / 3.0f, kSixth = 1.0f / 6.0f;
    float u[34];
    u[0] = fmaf(sl, k2, nm);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const float2 t = __ffma2_rn(make_float2(sv[i], sv[i + 1]), make_float2(k2, k2),
                                    make_float2(nm, nm));
        u[i + 1] = t.x;
        u[i + 2] = t.y;
    }
    u[33] = fmaf(sv[32], k2, nm);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float ul = u[i], uc = u[i + 1], ur = u[i + 2];
        float z = fmaf(ul + ur, kSixth, 4.0f * kSixth * uc);
        if (i == 0 && first_end) z = fmaf(ur, kThird, fmaf(2.0f * kThird, uc, -1.0f));
        if (MASKED) {
            const int c = cbase + i;
            const float zl = fmaf(ul, kThird, fmaf(2.0f * kThird, uc, -1.0f));
            z = c == c_last ? zl : z;
            w[i] = c <= c_last ? ex2_approx(z) : 0.0f;
        } else {
            w[i] = ex2_approx(z);
        }
    }
}

// Per-row online-softmax state of one softmax thread.
struct RowState {
    float k2;      // scale * log2(e)
    float m_run;   // running max of the logits, log2 units
    float l_run;   // fp32 sum of this half's weights (gives lse)
    float w_sink;  // weight of the given sink pair (k0, v0 supplied)
    float s_sink;  // q . k0 of the given sink pair
};

// Pass 1 of a half tile: max of the raw logits over this warp's 64 columns
// (valid columns only; column 0 replaced by the sink logit if any).
template <bool MASKED>
__device__ __forceinline__ float half_max(const uint32_t (&a)[2][32], int half, int c_last,
                                          float s0) {
    float m[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) m[i] = -INFINITY;
#pragma unroll
    for (int c = 0; c < 64; c += 2) {
        const int col = 64 * half + c;
        float v0 = c == 0 ? s0 : __uint_as_float(a[c >> 5][c & 31]);
        float v1 = __uint_as_float(a[(c + 1) >> 5][(c + 1) & 31]);
        if (MASKED) {
            v0 = col <= c_last ? v0 : -INFINITY;
            v1 = col + 1 <= c_last ? v1 : -INFINITY;
        }
        m[(c >> 1) & 3] = fmax3f(m[(c >> 1) & 3], v0, v1);
    }
    return fmax3f(m[0], m[1], fmaxf(m[2], m[3]));
}

// TMEM column where the P of 32 keys of S (16 packed columns) is written:
// half 0's keys 0..63 go to columns 0..31 of S, half 1's keys 64..127 to
// 80..111: columns that by then only their own warp has read.
__device__ __forceinline__ uint32_t p_col(int k) { return k < 2 ? 16u * k : 80u + 16u * (k - 2); }

// Pass 2 of a half tile: weights of this warp's 64 keys, P written to TMEM,
// fp32 sum accumulated.  a: the half's 64 logits; nb: column 64 for half 0
// (right neighbour of its last key), column 63 for half 1 (left neighbour
// of its first key).  Lc enters as the L share of the half's first key
// coming from the left and leaves (half 1) as that of the halo key, the
// next tile's first key.
// SHORT: the short-conv reading of eq. (13) (short_chunk); Lc then carries
// raw logits instead of L shares: in, the logit of the column left of the
// half's first key (for half 0 of the first tile: none, the sink is an end);
// out (half 1), that of column 126, the left neighbour of the next tile's
// first key.  tile0: this is the first key tile (column 0 is the sink).
template <bool MASKED, bool SHORT, bool SYM>
__device__ __forceinline__ void half_weights(uint32_t tS, const uint32_t (&a)[2][32], uint32_t nb,
                                             RowState &st, int half, int c_last, int sink,
                                             bool tile0, float nm, float &Lc) {
    const float k2 = st.k2;
    if (SHORT && half == 1) Lc = __uint_as_float(nb);  // column 63
    if (!SHORT && half == 1) {
        // interval (63, 64) gives key 64 its share from the left
        const float u0 = fmaf(__uint_as_float(nb), k2, nm);
        const float u1 = fmaf(__uint_as_float(a[0][0]), k2, nm);
        float R, L;
        seg_weights(u1 - u0, ex2_approx(u0), ex2_approx(u1), R, L);
        Lc = (!MASKED || 64 <= c_last) ? L : 0.0f;
    }
    float2 lsum = make_float2(0.0f, 0.0f), ls2 = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        const int k = 2 * half + kk;
        float sv[33];
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[i] = __uint_as_float(a[kk][i]);
        if (kk == 0)
            sv[32] = __uint_as_float(a[1][0]);
        else
            sv[32] = half == 0 ? __uint_as_float(nb) : sv[31];  // column 64, or unused
        if (k == 0 && sink == 1) sv[0] = sv[1];       // k_0 = k_1
        if (k == 0 && sink == 2) sv[0] = st.s_sink;   // given k_0
        float w[32], L31;
        if (SHORT) {
            short_chunk<MASKED>(sv, Lc, k2, nm, 32 * k, c_last, k == 0 && tile0, w);
            L31 = sv[30];  // column 126 when k == 3
            Lc = sv[31];   // left neighbour of the next chunk
        } else {
            cont_chunk<MASKED, SYM>(sv, k2, nm, 32 * k, c_last, k == 0 && tile0, Lc, L31, w);
        }
        if (k == 3) {
            Lc = L31;  // carried to the next tile's first key
            w[31] = 0.0f;
        }
        if (k == 0 && sink == 1) {  // v_0 = v_1: the sink's weight lands on key 1
            w[1] += w[0];
            w[0] = 0.0f;
        }
        if (k == 0 && sink == 2) {  // w_0 * v0 is added in fp32 at the end
            st.w_sink = w[0];
            w[0] = 0.0f;
            st.l_run += st.w_sink;
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            pk[i >> 1] = pack_bf16x2(w[i], w[i + 1]);
            if ((i & 2) == 0)
                lsum = __fadd2_rn(lsum, make_float2(w[i], w[i + 1]));
            else
                ls2 = __fadd2_rn(ls2, make_float2(w[i], w[i + 1]));
        }
        tmem_st16(tS + p_col(k), pk);
    }
    tmem_wait_st();
    lsum = __fadd2_rn(lsum, ls2);
    st.l_run += lsum.x + lsum.y;
}

template <int D, bool SHORT, bool SYM>
__global__ void __launch_bounds__(kThreads, 1)
    tc_forward_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
    using C = TcCfg<D>;
    constexpr int NSK = C::kStagesK, NSV = C::kStagesV;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const uint32_t sQ = base + C::kOffQ, sK = base + C::kOffK, sV = base + C::kOffV;
    const uint32_t bars = base + C::kOffBar;
#define BAR(i) (bars + 8u * (uint32_t)(i))
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = p.T;
    // the item ring: query tiles taken by the producer, decoded, read by every role
    volatile int *item_ring = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 8);

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
        mbar_init(BAR(C::kBarPFull), 256);
        mbar_init(BAR(C::kBarODone), 1);
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
        // zeros, so B columns d..d+15 of the PV product are (1, 0, .., 0).
        for (int s = 0; s < NSV; ++s) {
            uint8_t *ones = smem + C::kOffV + s * C::kVStageBytes + C::kTileBytes;
            for (int r = lane; r < 128; r += 32) {
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
            int item = (int)blockIdx.x;
            int issued_q = 0, issued_k = 0, issued_v = 0;  // loads issued (K, V: tiles)
            bool ok = true;
            for (int c = 0; ok; ++c) {
                ok = wait_c(BAR(C::kBarItemEmpty + (c & 1)), ((c >> 1) & 1) ^ 1, abort_flag);
                if (!ok) break;
                const bool last = item >= p.num_items;
                TcItem w = {0, 0, 0};
                if (!last) w = tc_item(item, p);
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
                    ok = wait_c(BAR(C::kBarQEmpty), (c - 1) & 1, abort_flag) &&
                         (p.mode != 2 || wait_c(BAR(C::kBarQRead), (c - 1) & 1, abort_flag));
                    if (!ok) break;
                }
                mbar_arrive_expect_tx(BAR(C::kBarQ), C::kTileBytes);
                for (int cc = 0; cc < C::kChunks; ++cc)
                    tma_load_3d(sQ + cc * kChunkBytes, &tm_q, 64 * cc, w.row0, w.bh, BAR(C::kBarQ));
                issued_q = c + 1;
                for (int j = 0; j < w.n; ++j) {
                    const int krow = 127 * j - 1;
                    const int g = issued_k;  // this CTA's key tile count
                    const int sk = g % NSK;
                    if (!(ok = wait_c(BAR(C::kBarKEmpty + sk), ((g / NSK) & 1) ^ 1, abort_flag))) break;
                    mbar_arrive_expect_tx(BAR(C::kBarKFull + sk), C::kTileBytes);
                    for (int cc = 0; cc < C::kChunks; ++cc)
                        tma_load_3d(sK + sk * C::kTileBytes + cc * kChunkBytes, &tm_k, 64 * cc, krow,
                                    w.bh, BAR(C::kBarKFull + sk));
                    issued_k = g + 1;
                    const int sv = g % NSV;
                    if (!(ok = wait_c(BAR(C::kBarVEmpty + sv), ((g / NSV) & 1) ^ 1, abort_flag))) break;
                    mbar_arrive_expect_tx(BAR(C::kBarVFull + sv), C::kTileBytes);
                    for (int cc = 0; cc < C::kChunks; ++cc)
                        tma_load_3d(sV + sv * C::kVStageBytes + cc * kChunkBytes, &tm_v, 64 * cc,
                                    krow, w.bh, BAR(C::kBarVFull + sv));
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
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdescS = make_idesc(128, 128, false);
            constexpr uint32_t kIdescO = make_idesc(128, C::kN, true);
            // One stream of key tiles over this CTA's items: within an item S
            // runs two tiles ahead of PV; the next item's first S wait until
            // this item's last PV is issued, since waiting for its Q must not
            // hold that PV (and the epilogue) back.  So S and PV are always
            // in the same item.
            int c = -1, n = 0;    // the current item and its key tiles
            int s_j = 0, p_j = 0;  // its S and PV issued
            int gs = 0, gp = 0;    // S and PV issued over all items
            // S(gs) = Q K^T into S buffer gs % 2; K tile gs is released once done
            auto issue_s = [&]() -> bool {
                if (!wait_c(BAR(C::kBarKFull + gs % NSK), (gs / NSK) & 1, abort_flag)) return false;
                tc_fence_after();
                const uint32_t kb = sK + (gs % NSK) * C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                    tc_mma_ss(tmem + C::col_s(gs & 1), make_sdesc(sQ + off, 16, 1024),
                              make_sdesc(kb + off, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
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
                if (!wait_c(BAR(C::kBarQ), c & 1, abort_flag)) return false;
                return issue_s() && (n == 1 || issue_s());
            };
            bool ok = next_item();
            while (ok && n > 0) {
                if (!(ok = wait_c(BAR(C::kBarPFull), gp & 1, abort_flag))) break;
                tc_fence_after();
                // [O | rowsum] += P(gp) [V_gp | ones], P read from the TMEM of S buffer gp % 2
                if (!(ok = wait_c(BAR(C::kBarVFull + gp % NSV), (gp / NSV) & 1, abort_flag))) break;
                tc_fence_after();
                const uint32_t vb = sV + (gp % NSV) * C::kVStageBytes;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc_mma_ts(tmem + C::kColO, tmem + C::col_s(gp & 1) + p_col(kk >> 1) + (kk & 1) * 8,
                              make_sdesc(vb + kk * 2048, kChunkBytes, 1024), kIdescO,
                              (p_j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(BAR(C::kBarODone));
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
        const int half = warp >> 2, wq = warp & 3;
        const int irow = wq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tO = tmem + lane_off + C::kColO;
        float *xmax = reinterpret_cast<float *>(smem + C::kOffXMax);
        float *xcarry = reinterpret_cast<float *>(smem + C::kOffXCarry);
        float *xfin = reinterpret_cast<float *>(smem + C::kOffXFin);
        const uint32_t xbar = BAR(C::kBarX);
        uint32_t xe = 0;  // exchanges completed on xbar
        int g = 0;        // key tiles of this CTA done so far
        bool ok = true;
        while (ok) {
            // items done so far: one exchange per key tile, one more per item
            const int c = (int)xe - g;
            TcItem w;
            ok = __all_sync(0xffffffffu, take_item(c, w));
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(C::kBarItemEmpty + (c & 1)));
            if (!ok || w.n == 0) break;
            const int bh = w.bh, row0 = w.row0, n = w.n;
            const int r = row0 + irow;
            RowState st;
            st.k2 = p.k2;
            st.m_run = -INFINITY;
            st.l_run = st.w_sink = st.s_sink = 0.0f;
            if (half == 0) {
                if (p.mode == 2) {
                    ok = __all_sync(0xffffffffu, wait_c(BAR(C::kBarQ), c & 1, abort_flag));
                    if (!ok) break;
                    // s_sink = q_r . k0[h], from this row of the swizzled Q tile
                    const __nv_bfloat16 *k0h = p.k0 + (size_t)(bh % p.H) * D;
                    float acc = 0.0f;
#pragma unroll
                    for (int cc = 0; cc < C::kChunks; ++cc) {
#pragma unroll
                        for (int kc = 0; kc < 8; ++kc) {
                            const uint8_t *src = smem + C::kOffQ + cc * kChunkBytes + irow * 128 +
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
            }
            for (int j = 0; ok && j < n; ++j, ++g) {
                const uint32_t tS = tmem + lane_off + C::col_s(g & 1);
                ok = __all_sync(0xffffffffu,
                                wait_c(BAR(C::kBarSFull + (g & 1)), (g >> 1) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                // last valid column of this row, and whether the tile needs masks
                const int c_last = r + 1 - 127 * j;
                const bool masked = 127 * j + 127 > row0 + 1;
                const int sink = j == 0 ? p.mode : 0;
                // this half's 64 logits and its neighbour column (64 or 63)
                uint32_t a[2][32];
                uint32_t nb[1] = {0u};
                tmem_ld32(tS + 64 * half, a[0]);
                tmem_ld32(tS + 64 * half + 32, a[1]);
                tmem_ld1(tS + (half == 0 ? 64 : 63), nb[0]);
                tmem_wait_ld_regs<32>(a[0]);
                tmem_wait_ld_regs<32>(a[1]);
                tmem_wait_ld_regs<1>(nb);
                float s0 = __uint_as_float(a[0][0]);
                if (half == 0 && sink == 1) s0 = __uint_as_float(a[0][1]);
                if (half == 0 && sink == 2) s0 = st.s_sink;
                // the symmetric interval has no sink: its logit must not raise the max
                if (SYM && half == 0 && j == 0) s0 = -INFINITY;
                const float mine = masked ? half_max<true>(a, half, c_last, s0)
                                          : half_max<false>(a, half, c_last, s0);
                // exchange the partial maxima (and the carried L share) with the other half
                const int slot = xe & 1;
                xmax[(slot * 2 + half) * 128 + irow] = mine;
                mbar_arrive(xbar);
                ok = __all_sync(0xffffffffu, wait_c(xbar, xe & 1, abort_flag));
                ++xe;
                if (!ok) break;
                const float mx = fmaxf(mine, xmax[(slot * 2 + (half ^ 1)) * 128 + irow]);
                float Lc = 0.0f;
                if (half == 0 && j > 0) Lc = xcarry[slot * 128 + irow];
                const float mt = (!masked || c_last >= 0) ? mx * st.k2 : -INFINITY;
                float alpha = 1.0f;
                const bool grow = mt > st.m_run + 8.0f;
                if (grow) {
                    alpha = ex2_approx(st.m_run - mt);
                    st.m_run = mt;
                    st.l_run *= alpha;
                    st.w_sink *= alpha;
                    if (!SHORT) Lc *= alpha;  // SHORT carries a raw logit
                }
                const float nm = -st.m_run;
                if (masked)
                    half_weights<true, SHORT, SYM>(tS, a, nb[0], st, half, c_last, sink, j == 0, nm, Lc);
                else
                    half_weights<false, SHORT, SYM>(tS, a, nb[0], st, half, c_last, sink, j == 0, nm, Lc);
                if (half == 1) xcarry[(xe & 1) * 128 + irow] = Lc;
                // Rescale O (this half's value columns; half 1 also the row-sum
                // column) when the max moved, after PV of the previous tile finished.
                const bool need_o = grow && j > 0;
                if (__any_sync(0xffffffffu, need_o)) {
                    ok = __all_sync(0xffffffffu, wait_c(BAR(C::kBarODone), (g - 1) & 1, abort_flag));
                    if (!ok) break;
                    tc_fence_after();
                    const float s = need_o ? alpha : 1.0f;
#pragma unroll
                    for (int cc = 0; cc < D / 64; ++cc) {
                        uint32_t o[32];
                        const uint32_t ta = tO + half * (D / 2) + 32 * cc;
                        tmem_ld32(ta, o);
                        tmem_wait_ld_regs<32>(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * s);
                        tmem_st32(ta, o);
                    }
                    if (half == 1) {
                        uint32_t o[1];
                        tmem_ld1(tO + D, o[0]);
                        tmem_wait_ld_regs<1>(o);
                        o[0] = __float_as_uint(__uint_as_float(o[0]) * s);
                        tmem_st1(tO + D, o[0]);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                mbar_arrive(BAR(C::kBarPFull));
            }
            if (!ok) break;
            // combine the two halves' fp32 sums; the given sink's weight lives in half 0
            float *mine = xfin + (half * 128 + irow) * 2;
            mine[0] = st.l_run;
            mine[1] = st.w_sink;
            mbar_arrive(xbar);
            // sleeping: the MMA thread is issuing this item's last PV meanwhile
            ok = __all_sync(0xffffffffu, wait_s(xbar, xe & 1, abort_flag));
            ++xe;
            if (!ok) break;
            const float *oth = xfin + ((half ^ 1) * 128 + irow) * 2;
            const float l_run = st.l_run + oth[0];
            const float w_sink = half == 0 ? st.w_sink : oth[1];
            // O holds this item's last PV once it is done; the next item's
            // first PV waits for this thread's PFull arrival, after the reads
            ok = __all_sync(0xffffffffu, wait_s(BAR(C::kBarODone), (g - 1) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            // o is divided by the sum of exactly the bf16 weights that fed the
            // PV product (O column d) plus the given sink's fp32 weight
            uint32_t lb[1];
            tmem_ld1(tO + D, lb[0]);
            tmem_wait_ld_regs<1>(lb);
            const float inv_l = 1.0f / (__uint_as_float(lb[0]) + w_sink);
            const bool store = r < T;
            __nv_bfloat16 *orow =
                p.out + ((size_t)bh * T + (size_t)(store ? r : 0)) * D + half * (D / 2);
            const __nv_bfloat16 *v0h = p.v0 + (size_t)(bh % p.H) * D + half * (D / 2);
            uint32_t oc[D / 64][32];
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) tmem_ld32(tO + half * (D / 2) + 32 * cc, oc[cc]);
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) tmem_wait_ld_regs<32>(oc[cc]);
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                const uint32_t *o = oc[cc];
                float val[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    float x = __uint_as_float(o[e]);
                    if (p.mode == 2) x = fmaf(w_sink, __bfloat162float(v0h[32 * cc + e]), x);
                    val[e] = x * inv_l;
                }
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(val[2 * e], val[2 * e + 1]);
                if (store) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * cc);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                }
            }
            if (store && half == 0 && p.lse)
                p.lse[(size_t)bh * T + r] =
                    (st.m_run + log2f(l_run)) * kLn2 + (SHORT ? 0.0f : kLseShift);
            tc_fence_before();
        }
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

template <int D, bool SHORT, bool SYM>
int launch_tc(const void *q, const void *k, const void *v, const void *k0, const void *v0,
              void *out, float *lse, int B, int H, int T, float scale, int mode,
              cudaStream_t stream) {
    using C = TcCfg<D>;
    const int BH = B * H;
    CUtensorMap mq, mk, mv;
    if (!encode_qkv_map(&mq, q, BH, T, D) || !encode_qkv_map(&mk, k, BH, T, D) ||
        !encode_qkv_map(&mv, v, BH, T, D))
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
    const long long items = (long long)prm.num_qtiles * BH;
    if (items > 0x7fffffffLL) return CSA_ERR_UNSUPPORTED;
    prm.num_items = (int)items;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return CSA_ERR_CUDA;
    const unsigned grid = (unsigned)(items < sms ? items : sms);  // one CTA per SM
    auto kern = tc_forward_kernel<D, SHORT, SYM>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
        return CSA_ERR_CUDA;
    return launch_with_slot(dev, stream, [&](int slot) {
        prm.slot = slot;
        kern<<<grid, kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, prm);
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
        if (d == 128) CSA_TC_LAUNCH(128, true, false);
        CSA_TC_LAUNCH(64, true, false);
    }
    if (form == kFormSymmetric) {  // no sink: mode is ignored
        mode = CSA_K0_ZERO;
        if (d == 128) CSA_TC_LAUNCH(128, false, true);
        CSA_TC_LAUNCH(64, false, true);
    }
    if (d == 128) CSA_TC_LAUNCH(128, false, false);
    CSA_TC_LAUNCH(64, false, false);
#undef CSA_TC_LAUNCH
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
