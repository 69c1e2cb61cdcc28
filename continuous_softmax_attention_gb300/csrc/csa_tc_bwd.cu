// Tensor-core backward kernel of causal continuous attention for sm_103a:
// the gradient of eq. (10)/(11) of Jianlin Su, "Continuous Softmax
// Attention" ("Assembly and Simplification"), bf16 inputs, d = 64 or 128.
//
// With p_i = e^{a_i - lse} (a_i = scale q.k_i), the interval between keys
// c and c+1 (natural step x) hands key c the share R = p_c phi2(x) and key
// c+1 the share L = p_{c+1} phi2(-x) of eq. (9), so P_c = L_c + R_c.  Their
// derivatives with respect to the two end logits combine, for each row, to
//     dL/da_c = P_c (dP_c - D) + F_c - F_{c+1},  F_c = k_c (dP_{c-1} - dP_c),
// where k_c = p_{c-1} phi2'(x) is the interval's flux coefficient,
// dP = dO . v and D = dO . o.  dS = scale dL/da, and
//     dV = P^T dO,  dK = dS^T Q,  dQ = dS K.
//
// Work split.  One CTA owns one key tile of one (b, h): 128 consecutive keys
// of the extended sequence (the sink first) at a stride of 126, so that its
// columns 1..126 are its own keys and columns 0 and 127 are the neighbours
// the stencil needs (for key tile 0, column 0 is the sink itself).  The CTA
// walks the 128-row query tiles from its diagonal to the end.  Per query
// tile the tensor core forms S = Q K^T and dP = dO V^T in TMEM; eight
// warps turn them into P and dS (bf16), written once to shared memory in the
// 128B-swizzled layout that serves as the MN-major A operand of
// dV += P^T dO and dK += dS^T Q and as the K-major A operand of
// dQ_part = dS K.  dV and dK accumulate in TMEM over the whole walk; dQ_part
// goes to TMEM (in the dP columns), is staged in fp32 where P and dS were
// once the MMAs reading them are done, and is added to an fp32 dq
// accumulator in global memory by TMA tensor reductions.  Per query tile the
// tensor core runs dP(j), S(j+1) as soon as S(j) and dP(j) have been read
// out of TMEM, then dV(j), dQ_part(j) and dK(j): after writing P and dS the
// elementwise warps wait for four products, not five.  Warps:
//   0-7  elementwise: warp w owns TMEM lanes 32*(w%4).. and the column half
//        w/4 (64 columns); they also stage dQ_part and run the final dK/dV
//        epilogue
//   8    TMA producer (the key tile once, then Q and dO per query tile; Q
//        double-buffered and fetched a tile ahead, dO as soon as dV has
//        released its buffer)
//   9    TMEM allocator and tcgen05.mma issuer
//   10   dQ reducer (TMA reductions of the staged dQ_part)
// Tensor memory: S | dP (then dQ_part) | dV | dK.
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

__device__ int g_bwd_status;  // sticky status word of this file's kernels

constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpReduce = 10;
constexpr int kThreads = 32 * 11;
constexpr int kKeyStride = 126;  // owned keys per key tile

// tcgen05.mma kind::f16 instruction descriptor with the major-ness of A and
// B chosen separately (fp32 accumulator, bf16 A and B).
__host__ __device__ constexpr uint32_t idesc_ab(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

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

// tcgen05.wait::ld naming the 17 registers it waits for, so that no use of
// them is scheduled before it.
__device__ __forceinline__ void wait_ld17(uint32_t (&r)[16], uint32_t &x) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(x)
                 :
                 : "memory");
}

// Tiled 3-D TMA reduction: adds one fp32 box from shared memory into global
// memory (elements outside the tensor are skipped).
__device__ __forceinline__ void tma_reduce_add_3d(uint32_t src, const void *desc, int c0, int c1,
                                                  int c2) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
        " [%0, {%1, %2, %3}], [%4];" ::"l"(reinterpret_cast<uint64_t>(desc)),
        "r"(c0), "r"(c1), "r"(c2), "r"(src)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared-memory sources of every committed reduction have been read
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// every committed reduction has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// A shared-memory descriptor with its low word (start address in 16-byte
// units, leading byte offset) kept apart, so that each constant offset of an
// unrolled loop costs one add: an operand inside the 227 KB of shared memory
// keeps its start address below 2^14 units, so the add never carries out of
// the field.  The single MMA-issuing thread shares its scheduler with two
// busy elementwise warps; every instruction it saves shortens its issue.
struct SDesc {
    uint32_t lo, hi;
    __device__ __forceinline__ uint64_t at(uint32_t off_bytes) const {
        return ((uint64_t)hi << 32) | (uint64_t)(lo + (off_bytes >> 4));
    }
};
__device__ __forceinline__ SDesc sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    const uint64_t d = make_sdesc(saddr, lbo, sbo);
    return {(uint32_t)d, (uint32_t)(d >> 32)};
}

template <int D>
struct BwCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kTileBytes = kChunks * kChunkBytes;  // [128 rows][D] bf16
    static constexpr int kStagesQ = 2;                        // Q: fetched a tile ahead
    static constexpr int kStagesG = D == 128 ? 1 : 2;         // dO
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kTileBytes;
    static constexpr int kOffQ = kOffV + kTileBytes;              // [stage]
    static constexpr int kOffG = kOffQ + kStagesQ * kTileBytes;   // [stage] dO
    static constexpr int kOffP = kOffG + kStagesG * kTileBytes;   // 2 boxes [128 q][64 keys]
    static constexpr int kOffS = kOffP + 2 * kChunkBytes;        // dS, same layout
    static constexpr int kOffBar = kOffS + 2 * kChunkBytes;
    static constexpr int kBarKV = 0;
    static constexpr int kBarQFull = 1;
    static constexpr int kBarQEmpty = kBarQFull + kStagesQ;
    static constexpr int kBarGFull = kBarQEmpty + kStagesQ;
    static constexpr int kBarGEmpty = kBarGFull + kStagesG;
    static constexpr int kBarSFull = kBarGEmpty + kStagesG;  // S and dP in TMEM
    static constexpr int kBarSRead = kBarSFull + 1;         // S and dP read out of TMEM
    static constexpr int kBarPReady = kBarSRead + 1;        // P, dS in shared memory
    static constexpr int kBarDqFull = kBarPReady + 1;       // dV, dQ_part MMAs done
    static constexpr int kBarDqRead = kBarDqFull + 1;       // dQ_part read out of TMEM
    static constexpr int kBarPFree = kBarDqRead + 1;       // dK done: P, dS no longer read
    // dQ_part staged (fp32): half 0's columns where P was, half 1's after them
    // (where dS was, at d = 128)
    static constexpr int kBarStageFull = kBarPFree + 1;     // [2], one per column half
    static constexpr int kBarStageFree = kBarStageFull + 2; // its reductions have read it
    static constexpr int kBarSEarly = kBarStageFree + 1;    // S(j+1) in TMEM (before dP(j+1))
    static constexpr int kBarDrain = kBarSEarly + 1;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base
    static_assert(kSmemBytes <= 227 * 1024, "shared memory per block");
    // the fp32 dQ_part, boxes of [128 rows][32 columns], fits where P and dS were
    static_assert(D / 32 * kChunkBytes <= 4 * kChunkBytes, "dQ staging");
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kColP = 128;
    static constexpr uint32_t kColV = 256;
    static constexpr uint32_t kColK = 256 + D;
};

struct BwParams {
    int B, H, T;
    int nq, nk;  // query tiles (128 rows), key tiles (126 keys)
    int group;   // heads per scheduling group
    float scale, k2;  // scale, scale * log2(e)
    int mode;
    const __nv_bfloat16 *k0, *v0;
    const float *lse, *Drow;  // [B*H*T]
    __nv_bfloat16 *dk, *dv;
    float *dk0, *dv0;
};

// mbarrier.try_wait with a suspend-time hint: a thread whose phase is not yet
// complete sleeps until it completes (or the hint elapses) instead of
// returning at once, so waiting roles take no issue slots from the
// elementwise warps that share their scheduler.
constexpr uint32_t kSuspendHintNs = 100000;
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// Bounded wait (2 s), as wait_bar, on the sleeping try_wait.
__device__ __forceinline__ bool wait_b(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            *(volatile int *)&g_bwd_status = kStatusTimeout;
            __threadfence();
            return false;
        }
    }
}

// One interval between a left key at u0 and a right key at u1 (log2 units,
// u = a log2(e) - lse log2(e), p = 2^u): R = p0 phi2(x), L = p1 phi2(-x)
// and the flux coefficient k = p0 phi2'(x), x = (u1 - u0) ln 2.
// Closed forms through the interval integral s = (p1 - p0)/x = p0 phi1(x):
//     R = (s - p0)/x,  L = s - R,  k = (s - 2R)/x,
// using phi2' = (phi1 - 2 phi2)/x and identity (7).  The independent
// rounding of p0 and p1 (2^-22 each) grows by up to 24/|x|^3 in k, so
// |x| < 0.35 takes series about the interval's midpoint instead: with
// h = x/2 and sig = p0 + p1 (= 2 e^c cosh h, c the mid logit),
//     s = sig tanh(h)/(2h)               = sig (1/2 - h^2/6 + ...),
//     k = sig (h cosh h - sinh h)/(4 h^3 cosh h) = sig (1/12 - h^2/30 + ...),
//     R = s/2 - h k,  L = s/2 + h k      (L - R = x k),
// even in h, so one term beyond the constant is enough: both sides of the
// switch stay below 2e-4 relative error, under the 2^-9 rounding of the
// bf16 P and dS.
__device__ __forceinline__ void interval(float u0, float u1, float p0, float p1, float &R,
                                         float &L, float &k) {
    const float h = (u1 - u0) * (0.5f * kLn2);
    const float rx = rcp_approx(h + h);
    const float s = (p1 - p0) * rx;
    const float Rc = (s - p0) * rx;
    const float kc = fmaf(-2.0f, Rc, s) * rx;
    const float sig = p0 + p1, hh = h * h;
    const float hs = sig * fmaf(hh, -1.0f / 12.0f, 0.25f);      // s/2
    const float ks = sig * fmaf(hh, -1.0f / 30.0f, 1.0f / 12.0f);
    const bool small = fabsf(h) < 0.175f;
    R = small ? fmaf(-h, ks, hs) : Rc;
    L = small ? fmaf(h, ks, hs) : s - Rc;
    k = small ? ks : kc;
}

// 16 columns [c0, c0+16) of this row: P and dS, given the raw logits sv[]
// and dP values gv[] of columns c0..c0+16 (the last one the right
// neighbour), the row's lse (log2 units) and D, and the L share and flux of
// column c0 from its left interval (Lc, Fc; updated to those of c0+16).
// MASKED (tiles that cross the diagonal or the end of the sequence): column
// c is a key of this row iff c <= c_last, and the interval (c, c+1) exists
// iff c + 1 <= c_last.  Always: the interval (127, 128) does not exist
// (last_chunk), and dS of columns owned by the neighbouring key tiles is 0
// for dQ (column 0 when zero_c0, column 127).
template <bool MASKED>
__device__ __forceinline__ void cols16(const float (&sv)[17], const float (&gv)[17], float k2,
                                       float lse2, float Dr, float scale, int c0, int c_last,
                                       bool zero_c0, bool last_chunk, float &Lc, float &Fc,
                                       uint32_t (&pP)[8], uint32_t (&pS)[8]) {
    float u[17], pe[17];
#pragma unroll
    for (int i = 0; i < 17; ++i) {
        u[i] = fmaf(sv[i], k2, -lse2);
        pe[i] = ex2_approx(u[i]);
    }
    float Pv[16], Sv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int c = c0 + i;
        float R, Ln, kf;
        interval(u[i], u[i + 1], pe[i], pe[i + 1], R, Ln, kf);
        float Fn = kf * (gv[i] - gv[i + 1]);
        bool seg = true, key = true;
        if (MASKED) {
            seg = c + 1 <= c_last;
            key = c <= c_last;
        }
        if (i == 15) seg = seg && !last_chunk;
        if (MASKED || i == 15) {
            R = seg ? R : 0.0f;
            Ln = seg ? Ln : 0.0f;
            Fn = seg ? Fn : 0.0f;
        }
        float P = Lc + R;
        float ds = scale * fmaf(P, gv[i] - Dr, Fc - Fn);
        if (MASKED) {
            P = key ? P : 0.0f;
            ds = key ? ds : 0.0f;
        }
        if (i == 0 && zero_c0) ds = 0.0f;
        if (i == 15 && last_chunk) ds = 0.0f;
        Pv[i] = P;
        Sv[i] = ds;
        Lc = Ln;
        Fc = Fn;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        pP[i] = pack_bf16x2(Pv[2 * i], Pv[2 * i + 1]);
        pS[i] = pack_bf16x2(Sv[2 * i], Sv[2 * i + 1]);
    }
}

// cols16 in two parts.  The first needs only the logits: P (masked) and
// the flux coefficient k of each column's right interval (zero where that
// interval does not exist), carrying the L share Lc across chunks.  The
// second adds dP: the fluxes F and dS, carrying Fc; it also packs P and dS.
template <bool MASKED>
__device__ __forceinline__ void cols16_s(const float (&sv)[17], float k2, float lse2, int c0,
                                         int c_last, bool last_chunk, float &Lc, float (&Pv)[16],
                                         float (&kv)[16]) {
    float u[17], pe[17];
#pragma unroll
    for (int i = 0; i < 17; ++i) {
        u[i] = fmaf(sv[i], k2, -lse2);
        pe[i] = ex2_approx(u[i]);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int c = c0 + i;
        float R, Ln, kf;
        interval(u[i], u[i + 1], pe[i], pe[i + 1], R, Ln, kf);
        bool seg = true, key = true;
        if (MASKED) {
            seg = c + 1 <= c_last;
            key = c <= c_last;
        }
        if (i == 15) seg = seg && !last_chunk;
        if (MASKED || i == 15) {
            R = seg ? R : 0.0f;
            Ln = seg ? Ln : 0.0f;
            kf = seg ? kf : 0.0f;
        }
        float P = Lc + R;
        if (MASKED) P = key ? P : 0.0f;
        Pv[i] = P;
        kv[i] = kf;
        Lc = Ln;
    }
}

template <bool MASKED>
__device__ __forceinline__ void cols16_d(const float (&gv)[17], const float (&Pv)[16],
                                         const float (&kv)[16], float Dr, float scale, int c0,
                                         int c_last, bool zero_c0, bool last_chunk, float &Fc,
                                         uint32_t (&pP)[8], uint32_t (&pS)[8]) {
    float Sv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float Fn = kv[i] * (gv[i] - gv[i + 1]);
        float ds = scale * fmaf(Pv[i], gv[i] - Dr, Fc - Fn);
        if (MASKED) ds = c0 + i <= c_last ? ds : 0.0f;
        if (i == 0 && zero_c0) ds = 0.0f;
        if (i == 15 && last_chunk) ds = 0.0f;
        Sv[i] = ds;
        Fc = Fn;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        pP[i] = pack_bf16x2(Pv[2 * i], Pv[2 * i + 1]);
        pS[i] = pack_bf16x2(Sv[2 * i], Sv[2 * i + 1]);
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    tc_backward_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_g,
                       const __grid_constant__ CUtensorMap tm_dq, const BwParams p) {
    using C = BwCfg<D>;
    constexpr int NQ = C::kStagesQ, NG = C::kStagesG;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const uint32_t sK = base + C::kOffK, sV = base + C::kOffV, sQ = base + C::kOffQ;
    const uint32_t sG = base + C::kOffG, sP = base + C::kOffP, sS = base + C::kOffS;
    const uint32_t bars = base + C::kOffBar;
#define BAR(i) (bars + 8u * (uint32_t)(i))
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Heads in groups whose Q and dO fit in L2 together; within a group the
    // longest walks (the first key tiles) go first.
    const int nk = p.nk, BH = p.B * p.H;
    const int grp = (int)(blockIdx.x / (unsigned)(p.group * nk));
    const int gsz = min(p.group, BH - grp * p.group);
    const int idx = (int)blockIdx.x - grp * p.group * nk;
    const int bh = grp * p.group + idx % gsz;
    const int kt = idx / gsz;
    const int T = p.T;
    const int krow0 = kKeyStride * kt - 1;          // array row of tile column 0
    const int q_first = (kKeyStride * kt) / 128;    // first query tile that sees an owned key
    const int nQ = p.nq - q_first;

    if (threadIdx.x == 0) {
        mbar_init(BAR(C::kBarKV), 1);
        for (int s = 0; s < NQ; ++s) {
            mbar_init(BAR(C::kBarQFull + s), 1);
            mbar_init(BAR(C::kBarQEmpty + s), 1);
        }
        for (int s = 0; s < NG; ++s) {
            mbar_init(BAR(C::kBarGFull + s), 1);
            mbar_init(BAR(C::kBarGEmpty + s), 1);
        }
        mbar_init(BAR(C::kBarSFull), 1);
        mbar_init(BAR(C::kBarSRead), 256);
        mbar_init(BAR(C::kBarPReady), 256);
        mbar_init(BAR(C::kBarDqFull), 1);
        mbar_init(BAR(C::kBarDqRead), 256);
        mbar_init(BAR(C::kBarPFree), 1);
        mbar_init(BAR(C::kBarStageFull), 128);
        mbar_init(BAR(C::kBarStageFull + 1), 128);
        mbar_init(BAR(C::kBarStageFree), 1);
        mbar_init(BAR(C::kBarSEarly), 1);
        mbar_init(BAR(C::kBarDrain), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kWarpProducer) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_g);
            mbar_arrive_expect_tx(BAR(C::kBarKV), 2 * C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_3d(sK + c * kChunkBytes, &tm_k, 64 * c, krow0, bh, BAR(C::kBarKV));
                tma_load_3d(sV + c * kChunkBytes, &tm_v, 64 * c, krow0, bh, BAR(C::kBarKV));
            }
            // Q of tile j goes out as soon as its stage is free (a tile ahead);
            // dO of tile j once dV(j-1) has released its buffer.
            int issued_q = 0, issued_g = 0;
            for (int j = 0; j < nQ; ++j) {
                const int qrow = 128 * (q_first + j);
                const int sq = j % NQ, sg = j % NG;
                if (!wait_b(BAR(C::kBarQEmpty + sq), ((j / NQ) & 1) ^ 1, abort_flag)) break;
                mbar_arrive_expect_tx(BAR(C::kBarQFull + sq), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sQ + sq * C::kTileBytes + c * kChunkBytes, &tm_q, 64 * c, qrow, bh,
                                BAR(C::kBarQFull + sq));
                issued_q = j + 1;
                if (!wait_b(BAR(C::kBarGEmpty + sg), ((j / NG) & 1) ^ 1, abort_flag)) break;
                mbar_arrive_expect_tx(BAR(C::kBarGFull + sg), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sG + sg * C::kTileBytes + c * kChunkBytes, &tm_g, 64 * c, qrow, bh,
                                BAR(C::kBarGFull + sg));
                issued_g = j + 1;
            }
            // Let every copy this thread issued land before the block can exit.
            wait_bar_drain(BAR(C::kBarKV), 0, &g_bwd_status);
            for (int j = max(0, issued_q - NQ); j < issued_q; ++j)
                wait_bar_drain(BAR(C::kBarQFull + j % NQ), (j / NQ) & 1, &g_bwd_status);
            for (int j = max(0, issued_g - NG); j < issued_g; ++j)
                wait_bar_drain(BAR(C::kBarGFull + j % NG), (j / NG) & 1, &g_bwd_status);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_ab(128, 128, false, false);  // S, dP
            constexpr uint32_t kIdKV = idesc_ab(128, D, true, true);     // dV, dK
            constexpr uint32_t kIdQ = idesc_ab(128, D, false, true);     // dQ_part
            bool ok = wait_b(BAR(C::kBarKV), 0, abort_flag);
            if (ok && kt == 0 && p.mode != 0) {
                // The sink is column 0 of key tile 0 (array row -1, read as
                // zeros): the copy-first mode takes key 1's row, the given
                // mode k0[h] and v0[h].  Rows r of a 128B-swizzled box keep
                // their 16-byte chunk c at position c ^ (r & 7).
                const size_t hoff = (size_t)(bh % p.H) * D;
                for (int c = 0; c < D / 8; ++c) {
                    uint8_t *k_row0 = smem + C::kOffK + (c >> 3) * kChunkBytes + ((c & 7) << 4);
                    uint8_t *v_row0 = smem + C::kOffV + (c >> 3) * kChunkBytes + ((c & 7) << 4);
                    uint4 kv, vv;
                    if (p.mode == 1) {
                        const int pos1 = ((c & 7) ^ 1) << 4;  // row 1
                        kv = *reinterpret_cast<const uint4 *>(smem + C::kOffK + (c >> 3) * kChunkBytes + 128 + pos1);
                        vv = *reinterpret_cast<const uint4 *>(smem + C::kOffV + (c >> 3) * kChunkBytes + 128 + pos1);
                    } else {
                        kv = *reinterpret_cast<const uint4 *>(p.k0 + hoff + 8 * c);
                        vv = *reinterpret_cast<const uint4 *>(p.v0 + hoff + 8 * c);
                    }
                    *reinterpret_cast<uint4 *>(k_row0) = kv;
                    *reinterpret_cast<uint4 *>(v_row0) = vv;
                }
                fence_proxy_async_smem();
            }
            tc_fence_after();
            // Per query tile j, in issue order: dP(j); S(j+1) once the
            // elementwise warps have read S(j) and dP(j) out of TMEM; then, once
            // P and dS are ready, dV(j) (frees dO's buffer), dQ_part(j) (read out
            // while the rest runs) and dK(j) (frees Q's stage and the P, dS
            // buffers).
            // the fixed operands' descriptors (K-major: LBO 16; MN-major: LBO
            // one 64-column box)
            const SDesc dK = sdesc(sK, 16, 1024), dV = sdesc(sV, 16, 1024);
            const SDesc dKmn = sdesc(sK, kChunkBytes, 1024);
            const SDesc dPmn = sdesc(sP, kChunkBytes, 1024), dSmn = sdesc(sS, kChunkBytes, 1024);
            const SDesc dS = sdesc(sS, 16, 1024);
            auto issue_s = [&](uint32_t qb) {
                const SDesc dQ = sdesc(qb, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                    tc_mma_ss(tmem + C::kColS, dQ.at(off), dK.at(off), kIdS, kk > 0 ? 1u : 0u);
                }
            };
            if (ok && (ok = wait_b(BAR(C::kBarQFull), 0, abort_flag))) {
                tc_fence_after();
                issue_s(sQ);
            }
            for (int j = 0; ok && j < nQ; ++j) {
                const int sq = j % NQ, sg = j % NG;
                const uint32_t qb = sQ + sq * C::kTileBytes, gb = sG + sg * C::kTileBytes;
                // dP overwrites the dQ_part columns of the previous tile
                if (j > 0 && !(ok = wait_b(BAR(C::kBarDqRead), (j - 1) & 1, abort_flag))) break;
                if (!(ok = wait_b(BAR(C::kBarGFull + sg), (j / NG) & 1, abort_flag))) break;
                tc_fence_after();
                const SDesc dG = sdesc(gb, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                    tc_mma_ss(tmem + C::kColP, dG.at(off), dV.at(off), kIdS, kk > 0 ? 1u : 0u);
                }
                tc_commit(BAR(C::kBarSFull));
                // S(j+1) as soon as the elementwise warps hold S(j) and dP(j) in registers
                if (j + 1 < nQ) {
                    const int sq1 = (j + 1) % NQ;
                    if (!(ok = wait_b(BAR(C::kBarSRead), j & 1, abort_flag))) break;
                    if (!(ok = wait_b(BAR(C::kBarQFull + sq1), ((j + 1) / NQ) & 1, abort_flag))) break;
                    tc_fence_after();
                    issue_s(sQ + sq1 * C::kTileBytes);
                    tc_commit(BAR(C::kBarSEarly));
                }
                if (!(ok = wait_b(BAR(C::kBarPReady), j & 1, abort_flag))) break;
                tc_fence_after();
                // dV += P^T dO and dK += dS^T Q: A = P^T / dS^T, MN-major (keys
                // contiguous, two 64-key boxes); B = dO / Q, MN-major; the
                // reduction runs over the 128 query rows, 16 per step.
                const SDesc dGmn = sdesc(gb, kChunkBytes, 1024), dQmn = sdesc(qb, kChunkBytes, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc_mma_ss(tmem + C::kColV, dPmn.at(kk * 2048), dGmn.at(kk * 2048), kIdKV,
                              (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(BAR(C::kBarGEmpty + sg));
                // dQ_part = dS K: A = dS K-major (reduction over the 128 keys),
                // B = the key tile, MN-major
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                    tc_mma_ss(tmem + C::kColP, dS.at(off), dKmn.at(kk * 2048), kIdQ, kk > 0 ? 1u : 0u);
                }
                tc_commit(BAR(C::kBarDqFull));
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc_mma_ss(tmem + C::kColK, dSmn.at(kk * 2048), dQmn.at(kk * 2048), kIdKV,
                              (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(BAR(C::kBarQEmpty + sq));
                tc_commit(BAR(C::kBarPFree));
            }
            // every MMA this thread issued completes before the block exits
            tc_commit(BAR(C::kBarDrain));
            wait_bar_drain(BAR(C::kBarDrain), 0, &g_bwd_status);
        }
        __syncwarp();
    } else if (warp == kWarpReduce) {
        // ------------------------------------------------------ dQ reducer
        // Adds each query tile's staged dQ_part into the fp32 accumulator
        // with TMA reductions and frees the staging area once they have read it.
        if (lane == 0) {
            tma_prefetch_desc(&tm_dq);
            bool ok = true;
            for (int j = 0; ok && j < nQ; ++j) {
                const int row0 = 128 * (q_first + j);
                // each column half's boxes as soon as that half has staged them
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (!(ok = wait_b(BAR(C::kBarStageFull + h), j & 1, abort_flag))) break;
#pragma unroll
                    for (int b = h * (D / 64); b < (h + 1) * (D / 64); ++b)
                        tma_reduce_add_3d(sP + b * kChunkBytes, &tm_dq, 32 * b, row0, bh);
                    bulk_commit();
                }
                if (!ok) break;
                bulk_wait_read_all();
                mbar_arrive(BAR(C::kBarStageFree));
            }
            bulk_wait_all();
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ elementwise
        const int half = warp >> 2, wq = warp & 3;
        const int irow = wq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + C::kColS, tD = tmem + lane_off + C::kColP;
        const float k2 = p.k2, scale = p.scale;
        const bool stage_in_ds = half * (D / 64) >= 2;  // this half's dQ boxes lie where dS was
        bool ok = true;
        // the row statistics of the first query tile; later ones are fetched
        // one tile ahead
        int r_next = 128 * q_first + irow;
        float lse_next = r_next < T ? p.lse[(size_t)bh * T + r_next] : 0.0f;
        float D_next = r_next < T ? p.Drow[(size_t)bh * T + r_next] : 0.0f;
        const int cb = 64 * half;
        // Chunk 0 (this half's first 16 columns) of a query tile, from S alone:
        // P, the flux coefficients of its intervals, the L share carried into
        // chunk 1 and, for half 1, the coefficient of the interval (63, 64)
        // entering it.  Computed during the previous tile's wait for its dV
        // and dQ_part products (S of this tile is in TMEM by then), or at the
        // start of the first tile.
        float P0[16], k0v[16], Lc1 = 0.0f, k63 = 0.0f;
        bool pre = false;
        auto chunk0_s = [&](float lse2c, int c_lastc, bool maskedc) {
            uint32_t a0[16], an0 = 0u, e0 = 0u, e1 = 0u;
            tmem_ld16(tS + cb, a0);
            tmem_ld1(tS + cb + 16, an0);
            if (half == 1) {
                tmem_ld1(tS + 63, e0);
                tmem_ld1(tS + 64, e1);
            }
            wait_ld17(a0, an0);
            asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(e0), "+r"(e1) : : "memory");
            float Lc = 0.0f;
            k63 = 0.0f;
            if (half == 1) {
                const float u0 = fmaf(__uint_as_float(e0), k2, -lse2c);
                const float u1 = fmaf(__uint_as_float(e1), k2, -lse2c);
                float R, L, kf;
                interval(u0, u1, ex2_approx(u0), ex2_approx(u1), R, L, kf);
                const bool seg = 64 <= c_lastc;
                Lc = seg ? L : 0.0f;
                k63 = seg ? kf : 0.0f;
            }
            float sv[17];
#pragma unroll
            for (int i = 0; i < 16; ++i) sv[i] = __uint_as_float(a0[i]);
            sv[16] = __uint_as_float(an0);
            if (maskedc)
                cols16_s<true>(sv, k2, lse2c, cb, c_lastc, false, Lc, P0, k0v);
            else
                cols16_s<false>(sv, k2, lse2c, cb, c_lastc, false, Lc, P0, k0v);
            Lc1 = Lc;
        };
        // last column of tile j that a row sees (its own key, position r + 1),
        // and whether the tile needs masks (some row stops before column 127)
        auto tile_clast = [&](int r) { return r < T ? min(r + 1 - kKeyStride * kt, 127) : -1; };
        auto tile_masked = [&](int row0) {
            return row0 + 1 - kKeyStride * kt < 127 || row0 + 127 >= T;
        };
        for (int j = 0; ok && j < nQ; ++j) {
            const int row0 = 128 * (q_first + j);
            const int r = row0 + irow;  // query row
            const bool rvalid = r < T;
            const float lse2 = rvalid ? lse_next * kLog2e : 0.0f;
            const float Dr = rvalid ? D_next : 0.0f;
            r_next = r + 128;
            if (j + 1 < nQ && r_next < T) {
                lse_next = p.lse[(size_t)bh * T + r_next];
                D_next = p.Drow[(size_t)bh * T + r_next];
            }
            const int c_last = tile_clast(r);
            const bool masked = tile_masked(row0);
            ok = __all_sync(0xffffffffu, wait_b(BAR(C::kBarSFull), j & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            if (!pre) chunk0_s(lse2, c_last, masked);
            pre = false;
            // this row's 16 keys from column c0 = 16-byte chunks ch, ch+1 of box c0/64
            auto store_pds = [&](int c0, const uint32_t (&qP)[8], const uint32_t (&qS)[8]) {
                const int box = c0 >> 6, ch = (c0 & 63) >> 3;
                uint8_t *prow = smem + C::kOffP + box * kChunkBytes + irow * 128;
                uint8_t *srow = smem + C::kOffS + box * kChunkBytes + irow * 128;
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int pos = ((ch + h2) ^ (irow & 7)) << 4;
                    *reinterpret_cast<uint4 *>(prow + pos) =
                        make_uint4(qP[4 * h2], qP[4 * h2 + 1], qP[4 * h2 + 2], qP[4 * h2 + 3]);
                    *reinterpret_cast<uint4 *>(srow + pos) =
                        make_uint4(qS[4 * h2], qS[4 * h2 + 1], qS[4 * h2 + 2], qS[4 * h2 + 3]);
                }
            };
            // dP of chunk 0 (and of half 1's entering interval); S and dP of
            // chunk 1, in flight while chunk 0 is finished
            uint32_t a[16], g[16], an[1] = {0u}, gn[1] = {0u};
            uint32_t g0[16], g0n = 0u, d0 = 0u, d1 = 0u;
            tmem_ld16(tD + cb, g0);
            tmem_ld1(tD + cb + 16, g0n);
            if (half == 1) {
                tmem_ld1(tD + 63, d0);
                tmem_ld1(tD + 64, d1);
            }
            wait_ld17(g0, g0n);
            asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(d0), "+r"(d1) : : "memory");
            tmem_ld16(tS + cb + 16, a);
            tmem_ld16(tD + cb + 16, g);
            tmem_ld1(tS + cb + 32, an[0]);
            tmem_ld1(tD + cb + 32, gn[0]);
            float Lc = Lc1;
            float Fc = half == 1 ? k63 * (__uint_as_float(d0) - __uint_as_float(d1)) : 0.0f;
            uint32_t hP[8], hS[8];  // chunk 0's P and dS
            {
                float gv[17];
#pragma unroll
                for (int i = 0; i < 16; ++i) gv[i] = __uint_as_float(g0[i]);
                gv[16] = __uint_as_float(g0n);
                const bool zero_c0 = cb == 0 && kt > 0;
                if (masked)
                    cols16_d<true>(gv, P0, k0v, Dr, scale, cb, c_last, zero_c0, false, Fc, hP, hS);
                else
                    cols16_d<false>(gv, P0, k0v, Dr, scale, cb, c_last, zero_c0, false, Fc, hP, hS);
            }
            // P and dS overwrite the previous tile's staged dQ_part: wait until
            // its reductions have read it (the MMAs reading the previous P
            // and dS finished before this tile's S and dP did).  At d = 128,
            // where those reductions take longest, chunk 0's P and dS are held
            // in registers and stored after chunk 1, so the wait comes later.
            constexpr int kFirstStore = D == 128 ? 1 : 0;
            if (kFirstStore == 0) {
                if (j > 0 &&
                    !__all_sync(0xffffffffu, wait_b(BAR(C::kBarStageFree), (j - 1) & 1, abort_flag))) {
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");  // chunk 1's loads
                    ok = false;
                    break;
                }
                store_pds(cb, hP, hS);
            }
#pragma unroll 1
            for (int kk = 1; kk < 4; ++kk) {
                const int c0 = cb + 16 * kk;
                wait_ld17(a, an[0]);
                wait_ld17(g, gn[0]);
                if (kk == 3) {  // every TMEM load of S and dP of this tile has landed
                    tc_fence_before();
                    mbar_arrive(BAR(C::kBarSRead));
                }
                float sv[17], gv[17];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    sv[i] = __uint_as_float(a[i]);
                    gv[i] = __uint_as_float(g[i]);
                }
                sv[16] = __uint_as_float(an[0]);
                gv[16] = __uint_as_float(gn[0]);
                if (kk < 3) {
                    tmem_ld16(tS + c0 + 16, a);
                    tmem_ld16(tD + c0 + 16, g);
                    if (c0 + 32 <= 127) {
                        tmem_ld1(tS + c0 + 32, an[0]);
                        tmem_ld1(tD + c0 + 32, gn[0]);
                    }
                }
                const bool last_chunk = c0 == 112;
                uint32_t pP[8], pS[8];
                if (masked)
                    cols16<true>(sv, gv, k2, lse2, Dr, scale, c0, c_last, false, last_chunk, Lc,
                                 Fc, pP, pS);
                else
                    cols16<false>(sv, gv, k2, lse2, Dr, scale, c0, c_last, false, last_chunk,
                                  Lc, Fc, pP, pS);
                if (kFirstStore == 1 && kk == 1) {
                    if (j > 0 &&
                        !__all_sync(0xffffffffu, wait_b(BAR(C::kBarStageFree), (j - 1) & 1, abort_flag))) {
                        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");  // the next chunk's loads
                        ok = false;
                        break;
                    }
                    store_pds(cb, hP, hS);
                }
                store_pds(c0, pP, pS);
            }
            if (!ok) break;
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(BAR(C::kBarPReady));
            // the next tile's chunk 0 from its S while dV and dQ_part run
            if (D == 128 && j + 1 < nQ) {
                ok = __all_sync(0xffffffffu, wait_b(BAR(C::kBarSEarly), j & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                const int r1 = r + 128;
                chunk0_s(r1 < T ? lse_next * kLog2e : 0.0f, tile_clast(r1), tile_masked(row0 + 128));
                pre = true;
            }
            // dQ_part of this query tile (in the dP columns): out of TMEM, which
            // frees the dP columns, then staged in fp32 where P and dS were, as
            // 128B-swizzled boxes of [128 rows][32 columns] for the reducer
            // warp's TMA reductions
            ok = __all_sync(0xffffffffu, wait_b(BAR(C::kBarDqFull), j & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            uint32_t o[D / 64][32];
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) tmem_ld32(tD + half * (D / 2) + 32 * cc, o[cc]);
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) tmem_wait_ld_regs<32>(o[cc]);
            tc_fence_before();
            mbar_arrive(BAR(C::kBarDqRead));
            // Boxes where P was are free once dV is done (DqFull covers it);
            // those where dS was (half 1 at d = 128) once dK, the last MMA
            // reading dS, is done.
            if (stage_in_ds) {
                ok = __all_sync(0xffffffffu, wait_b(BAR(C::kBarPFree), j & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
            }
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                uint8_t *srow = smem + C::kOffP + (half * (D / 64) + cc) * kChunkBytes + irow * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4 *>(srow + ((c ^ (irow & 7)) << 4)) =
                        make_uint4(o[cc][4 * c], o[cc][4 * c + 1], o[cc][4 * c + 2], o[cc][4 * c + 3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(BAR(C::kBarStageFull + half));
        }
        // the dK of the walk's last tile is complete before it is read out
        if (ok && !stage_in_ds) {
            ok = __all_sync(0xffffffffu, wait_b(BAR(C::kBarPFree), (nQ - 1) & 1, abort_flag));
            tc_fence_after();
        }
        if (ok) {
            // dV, dK of this tile's keys: TMEM lane = key row of the tile.
            // The last PFree wait covers every MMA of the walk.
            const int c = irow;
            const int arow = krow0 + c;
            const bool own = c >= 1 && c <= kKeyStride && arow < T;
            const int h = bh % p.H;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint32_t tcol = tmem + lane_off + (which ? C::kColK : C::kColV) + half * (D / 2);
                __nv_bfloat16 *outp = which ? p.dk : p.dv;
                float *sinkp = which ? p.dk0 : p.dv0;
#pragma unroll
                for (int cc = 0; cc < D / 64; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tcol + 32 * cc, o);
                    tmem_wait_ld_regs<32>(o);
                    float val[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) val[e] = __uint_as_float(o[e]);
                    const int col0 = half * (D / 2) + 32 * cc;
                    if (kt == 0 && wq == 0) {
                        // the sink (row 0): its own gradient, or key 1's share
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const float sinkv = __shfl_sync(0xffffffffu, val[e], 0);
                            if (p.mode == 1 && c == 1) val[e] += sinkv;
                        }
                        if (p.mode == 2 && c == 0) {
#pragma unroll
                            for (int e = 0; e < 32; ++e) atomicAdd(sinkp + (size_t)h * D + col0 + e, val[e]);
                        }
                    }
                    if (own) {
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(val[2 * e], val[2 * e + 1]);
                        uint4 *dstp = reinterpret_cast<uint4 *>(outp + ((size_t)bh * T + arow) * D + col0);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dstp[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tmem, 512);
#undef BAR
}

// D_t = dO_t . o_t for every row (one warp per row), and dq (bf16) from its
// fp32 accumulator.
template <int D>
__global__ void row_dot_kernel(const __nv_bfloat16 *g, const __nv_bfloat16 *o, float *Drow,
                               long long rows) {
    const long long w = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (w >= rows) return;
    const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(g + w * D);
    const __nv_bfloat162 *o2 = reinterpret_cast<const __nv_bfloat162 *>(o + w * D);
    float s = 0.0f;
#pragma unroll
    for (int i = lane; i < D / 2; i += 32) {
        const float2 a = __bfloat1622float2(g2[i]), b = __bfloat1622float2(o2[i]);
        s = fmaf(a.x, b.x, fmaf(a.y, b.y, s));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) Drow[w] = s;
}

__global__ void to_bf16_kernel(const float *a, __nv_bfloat16 *out, long long n4) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n4) return;
    const float4 v = reinterpret_cast<const float4 *>(a)[i];
    uint2 pk;
    pk.x = pack_bf16x2(v.x, v.y);
    pk.y = pack_bf16x2(v.z, v.w);
    reinterpret_cast<uint2 *>(out)[i] = pk;
}

// The fp32 dq accumulator [B*H, T, D] viewed as {D, T, B*H}, boxes of 32
// columns x 128 rows (128 bytes per row, 128B swizzle); rows outside [0, T)
// of a head are skipped by the reductions.
bool encode_acc_map(CUtensorMap *map, float *ptr, int BH, int T, int D) {
    auto fn = get_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)T * D * 4};
    const cuuint32_t box[3] = {32, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
int launch_bwd(const void *q, const void *k, const void *v, const void *k0, const void *v0,
               const void *o, const float *lse, const void *dout, void *dq, void *dk, void *dv,
               float *dk0, float *dv0, void *scratch, int B, int H, int T, float scale, int mode,
               cudaStream_t stream) {
    using C = BwCfg<D>;
    const int BH = B * H;
    const long long rows = (long long)BH * T;
    float *dq_acc = static_cast<float *>(scratch);
    float *Drow = dq_acc + rows * D;
    CUtensorMap mq, mk, mv, mg, mdq;
    if (!encode_qkv_map(&mq, q, BH, T, D) || !encode_qkv_map(&mk, k, BH, T, D) ||
        !encode_qkv_map(&mv, v, BH, T, D) || !encode_qkv_map(&mg, dout, BH, T, D) ||
        !encode_acc_map(&mdq, dq_acc, BH, T, D))
        return CSA_ERR_CUDA;
    if (cudaMemsetAsync(dq_acc, 0, sizeof(float) * (size_t)rows * D, stream) != cudaSuccess)
        return CSA_ERR_CUDA;
    if (mode == 2 && (cudaMemsetAsync(dk0, 0, sizeof(float) * (size_t)H * D, stream) != cudaSuccess ||
                      cudaMemsetAsync(dv0, 0, sizeof(float) * (size_t)H * D, stream) != cudaSuccess))
        return CSA_ERR_CUDA;
    row_dot_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(dout), static_cast<const __nv_bfloat16 *>(o), Drow, rows);
    BwParams prm;
    prm.B = B;
    prm.H = H;
    prm.T = T;
    prm.nq = (T + 127) / 128;
    prm.nk = (T + kKeyStride - 1) / kKeyStride;
    // Q and dO of a head are read by all of its key tiles: as many heads per
    // group as keep those within 64 MiB.
    prm.group = heads_per_group(BH, T, D);
    prm.scale = scale;
    prm.k2 = scale * kLog2e;
    prm.mode = mode;
    prm.k0 = static_cast<const __nv_bfloat16 *>(k0);
    prm.v0 = static_cast<const __nv_bfloat16 *>(v0);
    prm.lse = lse;
    prm.Drow = Drow;
    prm.dk = static_cast<__nv_bfloat16 *>(dk);
    prm.dv = static_cast<__nv_bfloat16 *>(dv);
    prm.dk0 = dk0;
    prm.dv0 = dv0;
    const long long grid = (long long)prm.nk * BH;
    if (grid > 0x7fffffffLL) return CSA_ERR_UNSUPPORTED;
    auto kern = tc_backward_kernel<D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
        return CSA_ERR_CUDA;
    kern<<<(unsigned)grid, kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, mg, mdq, prm);
    const long long n4 = rows * D / 4;
    to_bf16_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, stream>>>(
        dq_acc, static_cast<__nv_bfloat16 *>(dq), n4);
    return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

}  // namespace

long long csa_tc_backward_scratch_bytes(int B, int H, int T, int d) {
    return (long long)B * H * T * ((long long)d + 1) * (long long)sizeof(float);
}

int csa_tc_backward(const void *q, const void *k, const void *v, const void *k0, const void *v0,
                    const void *o, const float *lse, const void *dout, void *dq, void *dk,
                    void *dv, float *dk0, float *dv0, void *scratch, int B, int H, int T, int d,
                    float scale, int mode, cudaStream_t stream) {
    if (d == 128)
        return launch_bwd<128>(q, k, v, k0, v0, o, lse, dout, dq, dk, dv, dk0, dv0, scratch, B, H,
                               T, scale, mode, stream);
    if (d == 64)
        return launch_bwd<64>(q, k, v, k0, v0, o, lse, dout, dq, dk, dv, dk0, dv0, scratch, B, H, T,
                              scale, mode, stream);
    return CSA_ERR_UNSUPPORTED;
}

int csa_tc_backward_take_status(void) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_bwd_status, sizeof(int)) != cudaSuccess) return CSA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(int)) != cudaSuccess) return CSA_ERR_CUDA;
    return v;
}
