// Tensor-core forward kernels for sm_103a (bf16 inputs, d = 64 or 128):
//  * continuous attention, eq. (10)/(11) of Jianlin Su, "Continuous Softmax
//    Attention" ("Assembly and Simplification");
//  * standard causal attention, eq. (12) of the same page ("Analysis of the
//    Result"), built from the same skeleton with b = 0 and no sink.
//
// Work split.  One CTA owns two 128-row query tiles of one (b, h) and walks
// the key/value tiles up to their diagonal.  Warps:
//   0-3  softmax warpgroup of query tile 0 (one thread = one query row)
//   4-7  softmax warpgroup of query tile 1
//   8    TMA producer (lane 0)
//   9    TMEM allocator and tcgen05.mma issuer (lane 0)
// Shared memory holds both Q tiles, a K ring and a V ring, all 128B-swizzled
// 64-column boxes written by TMA.  Tensor memory (512 columns) holds
// S0 | S1 | O0 | O1 in fp32; the bf16 P of a tile overwrites the first 64
// columns of its own S and feeds the PV product straight from TMEM.
//
// The continuous kernel's halo.  b_{t,i} needs the logit of the key to the
// right of i.  Key tiles are therefore loaded at a stride of 127 rows: an S
// tile covers 128 consecutive keys of the extended sequence (the sink
// first), its last column is the first key of the next tile, and that
// column's P is 0.  Tile j starts at array row 127*j - 1; for j = 0 this row
// is -1, which TMA fills with zeros: the zero sink pair k_0 = v_0 = 0 comes
// for free, and the copy-first and given modes only replace the first logit
// (and, for given v_0, add w_0 * v_0 to the output at the end).
//
// The weights.  With the running max m (log2 units) and u = a*log2(e) - m,
// p = 2^u, each interval between neighbouring keys contributes
//   R = p_left * phi2(x)  to its left key and  L = p_right * phi2(-x)  to its
// right key (x the logit step), which is the regrouping of eq. (9); a key's
// weight e^{a+b-m} is L + R of its two intervals, one-sided at both ends.
// R and L follow from the interval integral S = (p_right - p_left)/x by
// R = (S - p_left)/x and L = S - R, with a power series for small steps.
// All weights carry a common factor (ln 2)^2, which cancels in o and is
// removed from lse.
//
// Every mbarrier wait is bounded in time; on expiry the kernel records
// CSA_ERR_TIMEOUT, every role skips its remaining work, the MMA issuer waits
// for its own MMAs, the producer waits for its own copies, and TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "csa.h"
#include "csa_device.cuh"
#include "csa_internal.h"

using namespace csa_dev;

namespace {

__device__ int g_tc_status;  // sticky status word of this file's kernels

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
// Wait for PV(j) to complete before issuing S(j+1) into the TMEM it reads.
constexpr bool kWaitPvBeforeS = false;
constexpr int kThreads = 320;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.4426950408889634f;
// -log((ln 2)^2): removes the common weight factor from lse
constexpr float kLseShift = 0.7330258411633287f;

template <int D>
struct TcCfg {
    static constexpr int kChunks = D / 64;          // 64-column boxes per tile
    static constexpr int kChunkBytes = 128 * 128;   // 128 rows x 128 bytes
    static constexpr int kTileBytes = kChunks * kChunkBytes;
    static constexpr int kStagesK = D == 128 ? 2 : 3;
    static constexpr int kStagesV = D == 128 ? 2 : 3;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + 2 * kTileBytes;
    static constexpr int kOffV = kOffK + kStagesK * kTileBytes;
    static constexpr int kOffBar = kOffV + kStagesV * kTileBytes;
    // barrier indices
    static constexpr int kBarQ = 0;
    static constexpr int kBarKFull = 1;
    static constexpr int kBarKEmpty = kBarKFull + kStagesK;
    static constexpr int kBarVFull = kBarKEmpty + kStagesK;
    static constexpr int kBarVEmpty = kBarVFull + kStagesV;
    static constexpr int kBarSFull = kBarVEmpty + kStagesV;  // [2]
    static constexpr int kBarPFull = kBarSFull + 2;          // [2]
    static constexpr int kBarODone = kBarPFull + 2;          // [2]
    static constexpr int kBarDrain = kBarODone + 2;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base
    // TMEM columns: S0 | S1 | O0 | O1
    __device__ static constexpr uint32_t col_s(int qt) { return 128u * (uint32_t)qt; }
    __device__ static constexpr uint32_t col_o(int qt) { return 256u + (uint32_t)(D * qt); }
};

struct TcParams {
    int B, H, T;
    int num_pairs;
    float k2;  // scale * log2(e)
    int mode;
    const __nv_bfloat16 *k0;
    const __nv_bfloat16 *v0;
    __nv_bfloat16 *out;
    float *lse;
};

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, bf16 A
// and B, A K-major, B K-major or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;  // descriptor version for this architecture
    d |= 2ull << 61;  // 128-byte swizzle
    return d;
}

// One interval's two end weights (see the file comment), times (ln 2)^2.
// X = u_right - u_left in log2 units, p = 2^u, x = X ln2 the logit step.
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
    constexpr float kTau = 0.0625f;
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

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    return mbar_wait_bounded(bar, parity, abort_flag, &g_tc_status, kWaitLimitNs);
}

// Wait that ignores the abort flag: used only to let in-flight copies and
// MMAs finish before the block exits.
__device__ __forceinline__ void wait_bar_drain(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *(volatile int *)&g_tc_status = kStatusTimeout;
            return;
        }
    }
}

// Per-row online-softmax state of one softmax thread.
struct RowState {
    float k2;      // scale * log2(e)
    float m_run;   // running max of the logits, log2 units
    float l_run;   // fp32 sum of the weights (gives lse)
    float l_bf;    // sum of the weights as rounded to bf16 for PV (normalises o)
    float carry;   // L share of the next tile's first key (continuous kernel)
    float w_sink;  // weight of the given sink pair (k0, v0 supplied)
    float s_sink;  // q . k0 of the given sink pair
};

__device__ __forceinline__ float fmax3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ void tmem_ld1(uint32_t taddr, uint32_t &r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr) : "memory");
}

// tcgen05.wait::ld that also names the destination registers of the loads
// it waits for, so that no use of them can be scheduled before it.
template <int N>
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&r)[N]);
template <>
__device__ __forceinline__ void tmem_wait_ld_regs<32>(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}
template <>
__device__ __forceinline__ void tmem_wait_ld_regs<33>(uint32_t (&r)[33]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31]), "+r"(r[32])
                 :
                 : "memory");
}

// Issues the TMEM loads of S chunk k (32 columns, plus the next column for
// the continuous kernel's right neighbour); completed by tmem_wait_ld_regs.
template <bool CONT>
__device__ __forceinline__ void load_chunk(uint32_t tS, int k, uint32_t (&b)[33]) {
    tmem_ld32(tS + 32 * k, *reinterpret_cast<uint32_t(*)[32]>(&b[0]));
    if (CONT && k < 3) tmem_ld1(tS + 32 * k + 32, b[32]);
}

// One 32-column chunk of weights of the continuous kernel.  sv[0..32] are
// the raw logits q.k of columns cbase..cbase+32; Lc is the L share of column
// cbase coming from the left.  Produces w[0..31] (e^{a+b-m} * (ln2)^2),
// returns in Lc the L share of column cbase+32, and in L31 that of cbase+31.
template <bool MASKED>
__device__ __forceinline__ void cont_chunk(const float (&sv)[33], float k2, float nm, int cbase,
                                           int c_last, float &Lc, float &L31, float (&w)[32]) {
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
        R[i] = Ri;
        L[i + 1] = Li;
    }
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const float2 t = __fadd2_rn(make_float2(L[i], L[i + 1]), make_float2(R[i], R[i + 1]));
        w[i] = t.x;
        w[i + 1] = t.y;
    }
    L31 = L[31];
    Lc = L[32];
}

// Softmax of one S tile held in TMEM at tS for this thread's row: tile max,
// lazy rescale of the running state, weights, P (bf16) written back over the
// first 64 columns of S.  Returns whether the running max moved (alpha is
// then the factor the accumulated O must be scaled by).
template <bool CONT, bool MASKED>
__device__ __forceinline__ bool softmax_tile(uint32_t tS, RowState &st, int c_last, int sink,
                                             float &alpha) {
    // ---- pass 1: max over the valid columns
    float mx;
    {
        uint32_t sr[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + 32 * cc, sr[cc]);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_wait_ld_regs<32>(sr[cc]);
        float s0 = __uint_as_float(sr[0][0]);
        if (CONT && sink == 1) s0 = __uint_as_float(sr[0][1]);
        if (CONT && sink == 2) s0 = st.s_sink;
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
            float v0 = c == 0 ? s0 : __uint_as_float(sr[c >> 5][c & 31]);
            float v1 = __uint_as_float(sr[(c + 1) >> 5][(c + 1) & 31]);
            if (MASKED) {
                v0 = c <= c_last ? v0 : -INFINITY;
                v1 = c + 1 <= c_last ? v1 : -INFINITY;
            }
            a[(c >> 1) & 7] = fmax3f(a[(c >> 1) & 7], v0, v1);
        }
        mx = fmax3f(fmax3f(a[0], a[1], a[2]), fmax3f(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
    }
    const float mt = (!MASKED || c_last >= 0) ? mx * st.k2 : -INFINITY;
    alpha = 1.0f;
    const bool grow = mt > st.m_run + 8.0f;
    if (grow) {
        alpha = ex2_approx(st.m_run - mt);
        st.m_run = mt;
        st.l_run *= alpha;
        st.l_bf *= alpha;
        st.carry *= alpha;
        st.w_sink *= alpha;
    }
    const float nm = -st.m_run;
    const float k2 = st.k2;
    // ---- pass 2: weights, 32 columns at a time
    float2 lsum = make_float2(0.0f, 0.0f), bsum = make_float2(0.0f, 0.0f);
    float Lc = st.carry;
    auto chunk = [&](int k, uint32_t (&a)[33]) {
        float w[32];
        if (CONT) {
            float sv[33];
#pragma unroll
            for (int i = 0; i < 32; ++i) sv[i] = __uint_as_float(a[i]);
            sv[32] = k < 3 ? __uint_as_float(a[32]) : sv[31];
            if (k == 0 && sink == 1) sv[0] = sv[1];
            if (k == 0 && sink == 2) sv[0] = st.s_sink;
            float L31;
            cont_chunk<MASKED>(sv, k2, nm, 32 * k, c_last, Lc, L31, w);
            if (k == 3) {
                Lc = L31;  // L share of the halo key = next tile's first key
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
                st.l_bf += st.w_sink;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const float2 t = __ffma2_rn(make_float2(__uint_as_float(a[i]), __uint_as_float(a[i + 1])),
                                            make_float2(k2, k2), make_float2(nm, nm));
                w[i] = ex2_approx(t.x);
                w[i + 1] = ex2_approx(t.y);
            }
            if (MASKED) {
#pragma unroll
                for (int i = 0; i < 32; ++i) w[i] = 32 * k + i <= c_last ? w[i] : 0.0f;
            }
        }
        uint32_t pk[16];
        float2 ls2 = make_float2(0.0f, 0.0f), bs2 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            const uint32_t pr = pack_bf16x2(w[i], w[i + 1]);
            pk[i >> 1] = pr;
            if ((i & 2) == 0)
                lsum = __fadd2_rn(lsum, make_float2(w[i], w[i + 1]));
            else
                ls2 = __fadd2_rn(ls2, make_float2(w[i], w[i + 1]));
            if (CONT) {
                const float2 rb = make_float2(__uint_as_float(pr << 16), __uint_as_float(pr & 0xffff0000u));
                if ((i & 2) == 0)
                    bsum = __fadd2_rn(bsum, rb);
                else
                    bs2 = __fadd2_rn(bs2, rb);
            }
        }
        lsum = __fadd2_rn(lsum, ls2);
        if (CONT) bsum = __fadd2_rn(bsum, bs2);
        tmem_st16(tS + 16 * k, pk);
    };
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
        uint32_t b[33];
        b[32] = 0u;
        load_chunk<CONT>(tS, k, b);
        tmem_wait_ld_regs<33>(b);
        chunk(k, b);
    }
    tmem_wait_st();
    st.carry = Lc;
    st.l_run += lsum.x + lsum.y;
    if (CONT) st.l_bf += bsum.x + bsum.y;
    return grow;
}

template <int D, bool CONT>
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
    const int BH = p.B * p.H;
    const int bh = (int)(blockIdx.x % (unsigned)BH);
    const int pair = p.num_pairs - 1 - (int)(blockIdx.x / (unsigned)BH);
    const int T = p.T;
    int row0[2], ntiles[2];
#pragma unroll
    for (int qt = 0; qt < 2; ++qt) {
        row0[qt] = pair * 256 + qt * 128;
        if (row0[qt] >= T) {
            ntiles[qt] = 0;
        } else {
            const int rl = min(row0[qt] + 127, T - 1);
            ntiles[qt] = CONT ? (rl + 1) / 127 + 1 : rl / 128 + 1;
        }
    }
    const int nj = max(ntiles[0], ntiles[1]);

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
        for (int qt = 0; qt < 2; ++qt) {
            mbar_init(BAR(C::kBarSFull + qt), 1);
            mbar_init(BAR(C::kBarPFull + qt), 128);
            mbar_init(BAR(C::kBarODone + qt), 1);
        }
        mbar_init(BAR(C::kBarDrain), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 8) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0 && nj > 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            uint32_t qbytes = 0;
            for (int qt = 0; qt < 2; ++qt)
                if (ntiles[qt] > 0) qbytes += C::kTileBytes;
            mbar_arrive_expect_tx(BAR(C::kBarQ), qbytes);
            for (int qt = 0; qt < 2; ++qt)
                if (ntiles[qt] > 0)
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(sQ + qt * C::kTileBytes + c * C::kChunkBytes, &tm_q, 64 * c,
                                    row0[qt], bh, BAR(C::kBarQ));
            int issued_k = 0, issued_v = 0;
            for (int j = 0; j < nj; ++j) {
                const int krow = CONT ? 127 * j - 1 : 128 * j;
                const int sk = j % NSK;
                if (!wait_bar(BAR(C::kBarKEmpty + sk), ((j / NSK) & 1) ^ 1, abort_flag)) break;
                mbar_arrive_expect_tx(BAR(C::kBarKFull + sk), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sK + sk * C::kTileBytes + c * C::kChunkBytes, &tm_k, 64 * c, krow,
                                bh, BAR(C::kBarKFull + sk));
                issued_k = j + 1;
                const int sv = j % NSV;
                if (!wait_bar(BAR(C::kBarVEmpty + sv), ((j / NSV) & 1) ^ 1, abort_flag)) break;
                mbar_arrive_expect_tx(BAR(C::kBarVFull + sv), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sV + sv * C::kTileBytes + c * C::kChunkBytes, &tm_v, 64 * c, krow,
                                bh, BAR(C::kBarVFull + sv));
                issued_v = j + 1;
            }
            // Let every copy this thread issued land before the block can exit.
            wait_bar_drain(BAR(C::kBarQ), 0);
            for (int j = max(0, issued_k - NSK); j < issued_k; ++j)
                wait_bar_drain(BAR(C::kBarKFull + j % NSK), (j / NSK) & 1);
            for (int j = max(0, issued_v - NSV); j < issued_v; ++j)
                wait_bar_drain(BAR(C::kBarVFull + j % NSV), (j / NSV) & 1);
        }
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0 && nj > 0) {
            constexpr uint32_t kIdescS = make_idesc(128, 128, false);
            constexpr uint32_t kIdescO = make_idesc(128, D, true);
            bool ok = wait_bar(BAR(C::kBarQ), 0, abort_flag);
            tc_fence_after();
            int k_seen = -1, v_seen = -1;
            auto issue_s = [&](int qt, int j) -> bool {
                if (k_seen < j) {
                    if (!wait_bar(BAR(C::kBarKFull + j % NSK), (j / NSK) & 1, abort_flag))
                        return false;
                    k_seen = j;
                    tc_fence_after();
                }
                const uint32_t qb = sQ + qt * C::kTileBytes;
                const uint32_t kb = sK + (j % NSK) * C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
                    tc_mma_ss(tmem + C::col_s(qt), make_sdesc(qb + off, 16, 1024),
                              make_sdesc(kb + off, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
                }
                tc_commit(BAR(C::kBarSFull + qt));
                return true;
            };
            auto issue_pv = [&](int qt, int j) -> bool {
                if (v_seen < j) {
                    if (!wait_bar(BAR(C::kBarVFull + j % NSV), (j / NSV) & 1, abort_flag))
                        return false;
                    v_seen = j;
                    tc_fence_after();
                }
                const uint32_t vb = sV + (j % NSV) * C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc_mma_ts(tmem + C::col_o(qt), tmem + C::col_s(qt) + kk * 8,
                              make_sdesc(vb + kk * 2048, C::kChunkBytes, 1024), kIdescO,
                              (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(BAR(C::kBarODone + qt));
                return true;
            };
            // For each key tile j and query tile: wait P(j), PV(j), then S(j+1).
            // K tile j+1 is released after its S products, V tile j after its PV.
            for (int qt = 0; qt < 2 && ok; ++qt)
                if (ntiles[qt] > 0) ok = issue_s(qt, 0);
            if (ok) tc_commit(BAR(C::kBarKEmpty + 0));
            for (int j = 0; ok && j < nj; ++j) {
                for (int qt = 0; qt < 2; ++qt) {
                    if (j >= ntiles[qt]) continue;
                    if (!(ok = wait_bar(BAR(C::kBarPFull + qt), j & 1, abort_flag))) break;
                    tc_fence_after();
                    if (!(ok = issue_pv(qt, j))) break;
                    if (j + 1 < ntiles[qt]) {
                        // S(j+1) overwrites the TMEM that PV(j) reads as P; both
                        // are tcgen05.mma issued in order by this thread.
                        if (kWaitPvBeforeS) {
                            if (!(ok = wait_bar(BAR(C::kBarODone + qt), j & 1, abort_flag))) break;
                            tc_fence_after();
                        }
                        if (!(ok = issue_s(qt, j + 1))) break;
                    }
                }
                if (!ok) break;
                tc_commit(BAR(C::kBarVEmpty + j % NSV));
                if (j + 1 < nj) tc_commit(BAR(C::kBarKEmpty + (j + 1) % NSK));
            }
            // every MMA this thread issued completes before the block exits
            tc_commit(BAR(C::kBarDrain));
            wait_bar_drain(BAR(C::kBarDrain), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ softmax
        const int qt = warp >> 2, wq = warp & 3;
        const int n = ntiles[qt];
        const int irow = wq * 32 + lane;
        const int r = row0[qt] + irow;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + C::col_s(qt);
        const uint32_t tO = tmem + lane_off + C::col_o(qt);
        RowState st;
        st.k2 = p.k2;
        st.m_run = -INFINITY;
        st.l_run = st.l_bf = st.carry = st.w_sink = st.s_sink = 0.0f;
        bool ok = n > 0;
        if (CONT && ok && p.mode == 2) {
            ok = __all_sync(0xffffffffu, wait_bar(BAR(C::kBarQ), 0, abort_flag));
            if (ok) {
                // s_sink = q_r . k0[h], from this row of the swizzled Q tile
                const __nv_bfloat16 *k0h = p.k0 + (size_t)(bh % p.H) * D;
                float acc = 0.0f;
#pragma unroll
                for (int cc = 0; cc < C::kChunks; ++cc) {
#pragma unroll
                    for (int kc = 0; kc < 8; ++kc) {
                        const uint8_t *src = smem + C::kOffQ + qt * C::kTileBytes +
                                             cc * C::kChunkBytes + irow * 128 +
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
            }
        }
        for (int j = 0; ok && j < n; ++j) {
            ok = __all_sync(0xffffffffu, wait_bar(BAR(C::kBarSFull + qt), j & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            // last valid column of this row, and whether the tile needs masks
            const int c_last = CONT ? r + 1 - 127 * j : r - 128 * j;
            const bool masked = CONT ? (127 * j + 127 > row0[qt] + 1) : (128 * j + 127 > row0[qt]);
            const int sink = (CONT && j == 0) ? p.mode : 0;
            float alpha;
            bool grow;
            if (masked)
                grow = softmax_tile<CONT, true>(tS, st, c_last, sink, alpha);
            else
                grow = softmax_tile<CONT, false>(tS, st, c_last, sink, alpha);
            // Rescale O when this row's max moved (after PV(j-1) finished).
            const bool need_o = grow && j > 0;
            if (__any_sync(0xffffffffu, need_o)) {
                ok = __all_sync(0xffffffffu,
                                wait_bar(BAR(C::kBarODone + qt), (j - 1) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                const float a = need_o ? alpha : 1.0f;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * cc, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
                    tmem_st32(tO + 32 * cc, o);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(BAR(C::kBarPFull + qt));
        }
        if (ok && n > 0) {
            ok = __all_sync(0xffffffffu, wait_bar(BAR(C::kBarODone + qt), (n - 1) & 1, abort_flag));
            if (ok) {
                tc_fence_after();
                // the continuous kernel divides by the bf16-rounded weight sum that
                // fed the PV product; the standard one by the fp32 sum
                const float inv_l = 1.0f / (CONT ? st.l_bf : st.l_run);
                const bool store = r < T;
                __nv_bfloat16 *orow = p.out + ((size_t)bh * T + (size_t)(store ? r : 0)) * D;
                const __nv_bfloat16 *v0h = p.v0 + (size_t)(bh % p.H) * D;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * cc, o);
                    tmem_wait_ld();
                    float val[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        float x = __uint_as_float(o[e]);
                        if (CONT && p.mode == 2)
                            x = fmaf(st.w_sink, __bfloat162float(v0h[32 * cc + e]), x);
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
                if (store && p.lse)
                    p.lse[(size_t)bh * T + r] =
                        (st.m_run + log2f(st.l_run)) * kLn2 + (CONT ? kLseShift : 0.0f);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, 512);
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
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// [B*H, T, D] bf16 viewed as a 3-D tensor, boxes of 64 columns x 128 rows.
bool encode_qkv_map(CUtensorMap *map, const void *ptr, int BH, int T, int D) {
    auto fn = get_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)T * D * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult rc = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return rc == CUDA_SUCCESS;
}

template <int D, bool CONT>
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
    prm.num_pairs = (T + 255) / 256;
    prm.k2 = scale * kLog2e;
    prm.mode = mode;
    prm.k0 = static_cast<const __nv_bfloat16 *>(k0);
    prm.v0 = static_cast<const __nv_bfloat16 *>(v0);
    prm.out = static_cast<__nv_bfloat16 *>(out);
    prm.lse = lse;
    const long long grid = (long long)prm.num_pairs * BH;
    if (grid > 0x7fffffffLL) return CSA_ERR_UNSUPPORTED;
    auto kern = tc_forward_kernel<D, CONT>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
        return CSA_ERR_CUDA;
    kern<<<(unsigned)grid, kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, prm);
    return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

}  // namespace

int csa_tc_forward(const void *q, const void *k, const void *v, const void *k0, const void *v0,
                   void *out, float *lse, int B, int H, int T, int d, float scale, int mode,
                   bool continuous, cudaStream_t stream) {
    if (d == 128)
        return continuous ? launch_tc<128, true>(q, k, v, k0, v0, out, lse, B, H, T, scale, mode, stream)
                          : launch_tc<128, false>(q, k, v, k0, v0, out, lse, B, H, T, scale, mode, stream);
    if (d == 64)
        return continuous ? launch_tc<64, true>(q, k, v, k0, v0, out, lse, B, H, T, scale, mode, stream)
                          : launch_tc<64, false>(q, k, v, k0, v0, out, lse, B, H, T, scale, mode, stream);
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
