// Decode step of causal continuous softmax attention: for every sequence b
// and head h, the query of the newest token against the sink and the n_b
// cached keys and values.  This is eq. (10)/(11) of "Continuous Softmax
// Attention" ("Assembly and Simplification") for the single row t = n_b.
//
// The step reads every cached key and value once and does about two flops
// per byte read, so it is bound by HBM bandwidth and runs on CUDA cores.
// The key positions 0..n (0 is the sink k_0, position i >= 1 is cache row
// i - 1) are cut into chunks of C positions (126 at d = 128, 254 at d = 64,
// 110 at d = 256).  One CTA per (b, h, chunk):
//   1. stages the chunk's keys plus one halo key on each side (the correction
//      b of a key needs both neighbours' logits, eq. (10)) and the chunk's
//      values, with two bulk asynchronous copies on separate barriers, so
//      that the values still load while steps 2 and 3 run;
//   2. forms the logits, in log2 units, two keys per group of d/8 lanes;
//   3. forms each key's weight e^{a+b} relative to the chunk's own maximum m:
//      for a key with logit a and a neighbour at a + x, the neighbour's
//      interval contributes e^{a-m} phi2(x) (eq. (9));
//   4. writes the partial sums l = sum w and o = sum w v, with m.
// A second kernel merges the chunks of each (b, h): with M the largest m,
// o = sum_c 2^{m_c-M} o_c / sum_c 2^{m_c-M} l_c and lse = (M + log2 L) ln 2.
// It is launched as a programmatic dependent of the first, so that its launch
// overlaps the first kernel's tail; it waits for the partials before reading.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "csa.h"
#include "csa_device.cuh"
#include "csa_internal.h"

namespace {

using namespace csa_dev;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMergeThreads = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.4426950408889634f;

__device__ int g_dec_status;  // sticky status word of this file's kernels

// Untiled bulk copy of `bytes` contiguous bytes from global to shared memory,
// completing on `bar`.  Both addresses 16-byte aligned, bytes a multiple of
// 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

template <int D>
struct DecCfg {
    // keys staged: the chunk and a halo key each side (32 KiB, three CTAs per
    // SM; at d = 256, 56 KiB and two CTAs per SM, which measured faster than
    // 32 KiB chunks of only 62 positions)
    static constexpr int KRows = D == 256 ? 112 : 16384 / D;
    static constexpr int C = KRows - 2;      // positions per chunk
    static constexpr int LPK = D / 8;        // lanes per key, 16 bytes (8 columns) each
    static constexpr int NGrp = kThreads / LPK;  // lane groups in the block
    static constexpr int kOffK = 0;              // keys; later the value partials [NGrp][D] floats
    static constexpr int kOffV = kOffK + KRows * D * 2;
    static constexpr int kOffA = kOffV + C * D * 2;   // logits, [KRows] floats
    static constexpr int kOffW = kOffA + KRows * 4;   // weights, [C] floats
    static constexpr int kOffWarp = kOffW + C * 4;    // block reductions, [2][kWarps] floats
    static constexpr int kOffBar = (kOffWarp + 2 * kWarps * 4 + 15) / 16 * 16;
    static constexpr int kSmemBytes = kOffBar + 32;  // two mbarriers and the abort flag
    static_assert(kOffV % 16 == 0 && kOffA % 16 == 0, "bulk copy destinations 16-byte aligned");
    static_assert(NGrp * D * 4 <= KRows * D * 2, "value partials fit in the key buffer");
    static_assert(KRows % (2 * NGrp) == 0, "the logit loop has no idle lanes");
    static_assert(kSmemBytes <= (D == 256 ? 113 : 75) * 1024, "three CTAs per SM (two at d = 256)");
};

struct DecParams {
    const __nv_bfloat16 *q, *k, *v, *k0, *v0;
    const int *seqlens;
    float *part_o;   // [B*H][S][D]: unnormalised partial outputs
    float *part_ml;  // [B*H][S][2]: chunk maximum (log2 units), chunk weight sum
    __nv_bfloat16 *out;  // o in bf16, or
    float *out_f32;      // o in fp32 (a range's partial output)
    float *lse;
    int B, H, T, S;
    int rows;      // cache rows per (b, h) in k, v: T, or a shard's rows
    int row_base;  // cache row held in row 0 of k, v
    int pos_lo, pos_hi;  // owned positions [pos_lo, pos_hi): 0, T + 1 for a whole row
    float qscale;  // scale * log2(e): logits come out in log2 units
    int mode;
};

__device__ __forceinline__ void unpack8(const uint4 &raw, float (&f)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// acc + q.k over the two bf16 pairs of a word each, with the bf16 operands
// widened exactly inside the fused multiply-add (one rounding per step).
__device__ __forceinline__ float fma_bf16x2(uint32_t q, uint32_t k, float acc) {
    asm("{\n\t.reg .b16 ql, qh, kl, kh;\n\t"
        "mov.b32 {ql, qh}, %1;\n\t"
        "mov.b32 {kl, kh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, ql, kl, %0;\n\t"
        "fma.rn.f32.bf16 %0, qh, kh, %0;\n\t}"
        : "+f"(acc)
        : "r"(q), "r"(k));
    return acc;
}

__device__ __forceinline__ float dot8(const uint4 &q, const uint4 &k) {
    float acc = 0.f;
    acc = fma_bf16x2(q.x, k.x, acc);
    acc = fma_bf16x2(q.y, k.y, acc);
    acc = fma_bf16x2(q.z, k.z, acc);
    acc = fma_bf16x2(q.w, k.w, acc);
    return acc;
}

// e^{u} phi2(x) for a key at u (log2 units, u <= 0) whose neighbour is at
// u + x2 = un (log2 units); x = x2 ln 2 is the natural-log gap and
// pc = 2^u.  phi2(x) = (e^x - 1 - x)/x^2 ("Preliminaries", eq. (6)).
//   |x| < 1: pc * sum_{j=0..9} x^j/(j+2)!  (truncation below 3e-9 relative);
//   x <= 20: pc * (e^x - 1 - x)/x^2, with e^x = 2^{x2};
//   x > 20:  (2^{un} - pc (1 + x))/x^2, since pc e^x = 2^{un} <= 1 while e^x
//            alone could overflow.
// All three are evaluated and one is selected (no divergent branches); the
// unselected ones may be inf or NaN.
__device__ __forceinline__ float side_weight(float x2, float un, float pc) {
    const float x = x2 * kLn2;
    float s = 2.505210838544172e-08f;           // 1/11!
    s = fmaf(s, x, 2.755731922398589e-07f);     // 1/10!
    s = fmaf(s, x, 2.755731922398589e-06f);     // 1/9!
    s = fmaf(s, x, 2.48015873015873e-05f);      // 1/8!
    s = fmaf(s, x, 1.984126984126984e-04f);     // 1/7!
    s = fmaf(s, x, 1.388888888888889e-03f);     // 1/6!
    s = fmaf(s, x, 8.333333333333333e-03f);     // 1/5!
    s = fmaf(s, x, 4.166666666666667e-02f);     // 1/4!
    s = fmaf(s, x, 1.666666666666667e-01f);     // 1/3!
    s = fmaf(s, x, 0.5f);                       // 1/2!
    const float num = x > 20.0f ? ex2_approx(un) - pc * (1.0f + x)
                                : pc * (ex2_approx(x2) - 1.0f - x);
    const float direct = num * rcp_approx(x * x);
    return fabsf(x) < 1.0f ? pc * s : direct;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// After an expired wait: keeps the block, and so its shared memory, alive
// (for at most one more wait limit per barrier) until its copies have landed.
__device__ __forceinline__ void drain(int tid, uint32_t bar_k, uint32_t bar_v) {
    if (tid != 0) return;
    const uint32_t bars[2] = {bar_k, bar_v};
    for (int i = 0; i < 2; ++i) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bars[i], 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads) decode_chunk_kernel(const DecParams p) {
    using Cf = DecCfg<D>;
    constexpr int C = Cf::C;
    extern __shared__ __align__(128) uint8_t smem[];
    __nv_bfloat16 *ks = reinterpret_cast<__nv_bfloat16 *>(smem + Cf::kOffK);
    __nv_bfloat16 *vs = reinterpret_cast<__nv_bfloat16 *>(smem + Cf::kOffV);
    float *as = reinterpret_cast<float *>(smem + Cf::kOffA);
    float *ws = reinterpret_cast<float *>(smem + Cf::kOffW);
    float *red = reinterpret_cast<float *>(smem + Cf::kOffK);  // after the logits
    float *wred = reinterpret_cast<float *>(smem + Cf::kOffWarp);
    const uint32_t bar_k = smem_u32(smem + Cf::kOffBar);      // keys landed
    const uint32_t bar_v = smem_u32(smem + Cf::kOffBar + 8);  // values landed
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cf::kOffBar + 16);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bh = blockIdx.x / p.S, chunk = blockIdx.x - bh * p.S;
    const int b = bh / p.H, h = bh - b * p.H;
    const int n = p.seqlens ? p.seqlens[b] : p.T;
    const int P0 = p.pos_lo + chunk * C;
    if (n < 1 || n > p.T || P0 > n) return;  // no position of this chunk exists
    const int P1 = min(min(P0 + C, p.pos_hi), n + 1);  // owned positions [P0, P1)
    const int own = P1 - P0;
    const int kp_lo = max(P0 - 1, 1), kp_hi = min(P1, n);  // cached keys staged
    const int vp_lo = max(P0, 1);                          // cached values staged: [vp_lo, P1)
    // position pos >= 1 is cache row pos - 1, held in row pos - 1 - row_base
    const long long head = (long long)bh * p.rows - p.row_base;
    // Shared-memory slot of position pos: keys pos - P0 + 1, values pos - P0.

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bar_k, 1);
        mbar_init(bar_v, 1);
        fence_mbar_init();
        const uint32_t kbytes = (uint32_t)(kp_hi - kp_lo + 1) * D * 2;
        const uint32_t vbytes = (uint32_t)(P1 - vp_lo) * D * 2;
        mbar_arrive_expect_tx(bar_k, kbytes);
        bulk_load(smem_u32(ks + (kp_lo - P0 + 1) * D), p.k + (head + kp_lo - 1) * D, kbytes, bar_k);
        mbar_arrive_expect_tx(bar_v, vbytes);
        bulk_load(smem_u32(vs + (vp_lo - P0) * D), p.v + (head + vp_lo - 1) * D, vbytes, bar_v);
    }

    constexpr int LPK = Cf::LPK, NGrp = Cf::NGrp;
    const int c8 = lane % LPK;  // this lane's 8 columns of a row
    const int grp = tid / LPK;  // this lane's group
    const uint4 qraw = reinterpret_cast<const uint4 *>(p.q + (size_t)bh * D)[c8];

    __syncthreads();  // barriers initialised
    // The values keep loading while the logits and weights are formed.
    if (!mbar_wait_bounded(bar_k, 0, abort_flag, &g_dec_status, kWaitLimitNs)) {
        drain(tid, bar_k, bar_v);
        return;
    }

    // Logits of the staged positions [kp_lo - 1 or the sink, kp_hi]: each
    // lane group takes two rows per step, ra and rb = ra + NGrp.  Rows
    // outside that range hold stale data; their logits are never read.
    const int r_lo = (P0 == 0) ? 1 : 0, r_hi = kp_hi - P0 + 1;
#pragma unroll 1
    for (int base = 0; base < Cf::KRows; base += 2 * NGrp) {
        if (base > r_hi) break;  // block-uniform
        const int ra = base + grp, rb = ra + NGrp;
        uint4 ka = reinterpret_cast<const uint4 *>(ks + ra * D)[c8];
        const uint4 kb = reinterpret_cast<const uint4 *>(ks + rb * D)[c8];
        if (P0 == 0 && ra == 1) {  // the sink, position 0
            if (p.mode == CSA_K0_GIVEN)
                ka = reinterpret_cast<const uint4 *>(p.k0 + (size_t)h * D)[c8];
            else if (p.mode == CSA_K0_COPY_FIRST)
                ka = reinterpret_cast<const uint4 *>(ks + 2 * D)[c8];  // position 1
            else
                ka = make_uint4(0u, 0u, 0u, 0u);
        }
        const float pa = dot8(qraw, ka), pb = dot8(qraw, kb);
        // Reduce-scatter over the group: the lower half ends with row ra's
        // sum, the upper half with row rb's.
        const bool upper = (c8 & (LPK / 2)) != 0;
        float keep = upper ? pb : pa;
        keep += __shfl_xor_sync(0xffffffffu, upper ? pa : pb, LPK / 2);
#pragma unroll
        for (int off = LPK / 4; off > 0; off >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, off);
        if (c8 == 0) as[ra] = keep * p.qscale;
        if (c8 == LPK / 2) as[rb] = keep * p.qscale;
    }
    __syncthreads();

    // Chunk maximum over every staged logit (halo included, so that every
    // 2^{u} below is at most 1).
    float mx = -INFINITY;
    for (int r = r_lo + tid; r <= r_hi; r += kThreads) mx = fmaxf(mx, as[r]);
    mx = warp_max(mx);
    if (lane == 0) wred[warp] = mx;
    __syncthreads();
    mx = wred[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i) mx = fmaxf(mx, wred[i]);

    // Weights of the owned positions: the interval to the left (absent for
    // the sink) and the interval to the right (absent for position n).
    float lsum = 0.f;
    for (int i = tid; i < own; i += kThreads) {
        const int r = i + 1, pos = P0 + i;
        const float ar = as[r];
        const float u = ar - mx;
        const float pc = ex2_approx(u);
        float w = 0.f;
        if (pos >= 1) w += side_weight(as[r - 1] - ar, as[r - 1] - mx, pc);
        if (pos + 1 <= n) w += side_weight(as[r + 1] - ar, as[r + 1] - mx, pc);
        ws[i] = w;
        lsum += w;
    }
    lsum = warp_sum(lsum);
    if (lane == 0) wred[kWarps + warp] = lsum;
    if (!mbar_wait_bounded(bar_v, 0, abort_flag, &g_dec_status, kWaitLimitNs)) {
        drain(tid, bar_k, bar_v);
        return;
    }
    // The sink's value in slot 0 (chunk 0 only).
    if (P0 == 0 && tid < D / 8) {
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (p.mode == CSA_K0_GIVEN)
            val = reinterpret_cast<const uint4 *>(p.v0 + (size_t)h * D)[tid];
        else if (p.mode == CSA_K0_COPY_FIRST)
            val = reinterpret_cast<const uint4 *>(vs + D)[tid];
        reinterpret_cast<uint4 *>(vs)[tid] = val;
    }
    __syncthreads();
    lsum = 0.f;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) lsum += wred[kWarps + i];

    // o = sum_i w_i v_i: each lane group takes every NGrp-th key, 8 columns
    // per lane, two keys per step into two accumulator sets; the groups'
    // partials meet in the (now unused) key buffer.
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    float acc2[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc2[j] = 0.f;
    int i = grp;
    for (; i + NGrp < own; i += 2 * NGrp) {
        const float w = ws[i], w2 = ws[i + NGrp];
        const uint4 r1 = reinterpret_cast<const uint4 *>(vs + i * D)[c8];
        const uint4 r2 = reinterpret_cast<const uint4 *>(vs + (i + NGrp) * D)[c8];
        float vf[8], vf2[8];
        unpack8(r1, vf);
        unpack8(r2, vf2);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            acc[j] = fmaf(w, vf[j], acc[j]);
            acc2[j] = fmaf(w2, vf2[j], acc2[j]);
        }
    }
    if (i < own) {
        const float w = ws[i];
        float vf[8];
        unpack8(reinterpret_cast<const uint4 *>(vs + i * D)[c8], vf);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = fmaf(w, vf[j], acc[j]);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] += acc2[j];
    float4 *dst = reinterpret_cast<float4 *>(red + grp * D + 8 * c8);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    __syncthreads();
    const size_t slot = (size_t)bh * p.S + chunk;
    float *po = p.part_o + slot * D;
    for (int col = tid; col < D; col += kThreads) {
        float s = 0.f;
#pragma unroll
        for (int gg = 0; gg < NGrp; ++gg) s += red[gg * D + col];
        po[col] = s;
    }
    if (tid == 0) {
        p.part_ml[2 * slot] = mx;
        p.part_ml[2 * slot + 1] = lsum;
    }
}

// One block per (b, h).  The chunk maxima reduce to M across the block; the
// chunk factors 2^{m_c - M} go to shared memory a tile at a time, and each
// output column sums its chunks' partials (kParts threads per column, loads
// coalesced across columns).
template <int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const DecParams p) {
    constexpr int C = DecCfg<D>::C;
    constexpr int kParts = kMergeThreads / D, kTile = 1024, kMW = kMergeThreads / 32;
    __shared__ float fac[kTile];
    __shared__ float red[2][kMW];
    __shared__ float part[kParts][D];
    const int bh = blockIdx.x, b = bh / p.H, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = p.seqlens ? p.seqlens[b] : p.T;
    // launched as a programmatic dependent of the chunk kernel: wait until its
    // partials are complete and visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    auto store = [&](int col, float val) {
        if (p.out_f32)
            p.out_f32[(size_t)bh * D + col] = val;
        else
            p.out[(size_t)bh * D + col] = __float2bfloat16_rn(val);
    };
    if (n < 1 || n > p.T) {  // a length outside [1, T]: NaN result, status word set
        for (int col = tid; col < D; col += kMergeThreads) store(col, NAN);
        if (tid == 0) {
            if (p.lse) p.lse[bh] = NAN;
            atomicCAS(&g_dec_status, 0, CSA_ERR_INVALID_ARG);
        }
        return;
    }
    if (p.pos_lo > n) {  // a range past this sequence's end: an empty partial
        for (int col = tid; col < D; col += kMergeThreads) store(col, 0.0f);
        if (tid == 0 && p.lse) p.lse[bh] = -INFINITY;
        return;
    }
    // chunks holding the owned positions [pos_lo, min(pos_hi, n + 1))
    const int nch = (min(p.pos_hi, n + 1) - p.pos_lo + C - 1) / C;
    const float *ml = p.part_ml + (size_t)bh * p.S * 2;
    const float *po = p.part_o + (size_t)bh * p.S * D;
    float M = -INFINITY;
    for (int c = tid; c < nch; c += kMergeThreads) M = fmaxf(M, ml[2 * c]);
    M = warp_max(M);
    if (lane == 0) red[0][warp] = M;
    __syncthreads();
    M = red[0][0];
#pragma unroll
    for (int i = 1; i < kMW; ++i) M = fmaxf(M, red[0][i]);
    const int col = tid % D, prt = tid / D;
    float acc = 0.f, L = 0.f;
    for (int t0 = 0; t0 < nch; t0 += kTile) {
        const int tn = min(kTile, nch - t0);
        for (int c = tid; c < tn; c += kMergeThreads) {
            const float f = ex2_approx(ml[2 * (t0 + c)] - M);
            fac[c] = f;
            L = fmaf(ml[2 * (t0 + c) + 1], f, L);
        }
        __syncthreads();
        const float *pt = po + (size_t)t0 * D + col;
#pragma unroll 4
        for (int c = prt; c < tn; c += kParts) acc = fmaf(pt[(size_t)c * D], fac[c], acc);
        __syncthreads();
    }
    L = warp_sum(L);
    if (lane == 0) red[1][warp] = L;
    part[prt][col] = acc;
    __syncthreads();
    L = 0.f;
#pragma unroll
    for (int i = 0; i < kMW; ++i) L += red[1][i];
    if (prt == 0) {
        float s = acc;
#pragma unroll
        for (int i = 1; i < kParts; ++i) s += part[i][col];
        store(col, s * (1.0f / L));
    }
    if (tid == 0 && p.lse) p.lse[bh] = (M + log2f(L)) * kLn2;
}

// Merge of R partial results of the same rows, one per range of positions
// (eq. (11) restricted to the range's keys): with L the largest lse_r,
//     o = sum_r e^{lse_r - L} o_r / sum_r e^{lse_r - L},
//     lse = L + log sum_r e^{lse_r - L};
// an empty range (lse_r = -inf) weighs nothing.  One warp per row.
__global__ void __launch_bounds__(256) merge_ranges_kernel(const float *o_parts,
                                                           const float *lse_parts, int R,
                                                           long long rows, int d,
                                                           __nv_bfloat16 *out, float *lse) {
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float L = -INFINITY;
    for (int r = 0; r < R; ++r) L = fmaxf(L, lse_parts[(long long)r * rows + row]);
    float den = 0.0f;
    for (int r = 0; r < R; ++r) den += ex2_approx((lse_parts[(long long)r * rows + row] - L) * kLog2e);
    const float inv = 1.0f / den;
    for (int col = lane; col < d; col += 32) {
        float num = 0.0f;
        for (int r = 0; r < R; ++r) {
            const float w = ex2_approx((lse_parts[(long long)r * rows + row] - L) * kLog2e);
            num = fmaf(w, o_parts[((long long)r * rows + row) * d + col], num);
        }
        out[row * d + col] = __float2bfloat16_rn(num * inv);
    }
    if (lane == 0 && lse) lse[row] = L + logf(den);
}

template <int D>
int launch_decode(DecParams p, cudaStream_t stream) {
    using Cf = DecCfg<D>;
    p.S = (p.pos_hi - p.pos_lo + Cf::C - 1) / Cf::C;  // chunks of the owned positions
    const long long BH = (long long)p.B * p.H;
    const long long grid = BH * p.S;
    if (grid > 0x7fffffffLL || BH > 0x7fffffffLL) return CSA_ERR_UNSUPPORTED;
    auto kern = decode_chunk_kernel<D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::kSmemBytes) !=
        cudaSuccess)
        return CSA_ERR_CUDA;
    kern<<<(unsigned)grid, kThreads, Cf::kSmemBytes, stream>>>(p);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)BH);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_merge_kernel<D>, p) != cudaSuccess) return CSA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

int chunk_positions(int d) { return d == 64 ? DecCfg<64>::C : d == 128 ? DecCfg<128>::C : DecCfg<256>::C; }

}  // namespace

namespace {
// Scratch bytes for the positions [pos_lo, pos_hi) of B*H rows (positions
// counted in 64 bits: pos_hi = T + 1 for the whole cache), or -1.
long long range_scratch_bytes(long long B, long long H, long long pos_lo, long long pos_hi, int d) {
    if (B < 0 || H < 0 || pos_lo < 0 || pos_hi < pos_lo || !(d == 64 || d == 128 || d == 256))
        return -1;
    const long long C = chunk_positions(d);
    const long long S = (pos_hi - pos_lo + C - 1) / C;
    // B, H < 2^31 and S < 2^31: B*H*S < 2^93 could overflow; sizes beyond
    // 2^62 bytes are reported as unsupported (-1)
    const long double bytes = (long double)B * H * S * (d + 2) * (long double)sizeof(float);
    if (bytes > 4.0e18L) return -1;
    return B * H * S * (d + 2) * (long long)sizeof(float);
}
}  // namespace

long long csa_decode_scratch_bytes(int B, int H, int T, int d) {
    return range_scratch_bytes(B, H, 0, (long long)T + 1, d);
}

long long csa_decode_range_scratch_bytes(int B, int H, int pos_lo, int pos_hi, int d) {
    return range_scratch_bytes(B, H, pos_lo, pos_hi, d);
}

namespace {

int run_range(const void *q, const void *k, const void *v, const void *k0, const void *v0,
              const int *seqlens, void *out, float *out_f32, float *lse, void *scratch, int B,
              int H, int T, int d, float scale, int mode, int pos_lo, int pos_hi,
              cudaStream_t stream) {
    DecParams p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.v = static_cast<const __nv_bfloat16 *>(v);
    p.k0 = static_cast<const __nv_bfloat16 *>(k0);
    p.v0 = static_cast<const __nv_bfloat16 *>(v0);
    p.seqlens = seqlens;
    const int C = chunk_positions(d);
    const long long S = ((long long)pos_hi - pos_lo + C - 1) / C;
    p.part_o = static_cast<float *>(scratch);
    p.part_ml = p.part_o + (long long)B * H * S * d;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.out_f32 = out_f32;
    p.lse = lse;
    p.B = B;
    p.H = H;
    p.T = T;
    p.S = (int)S;
    // a range's shard holds cache rows [max(pos_lo - 2, 0), min(pos_hi, T)): its
    // positions and the neighbour on each side
    p.row_base = pos_lo >= 2 ? pos_lo - 2 : 0;
    p.rows = min(pos_hi, T) - p.row_base;
    p.pos_lo = pos_lo;
    p.pos_hi = pos_hi;
    p.qscale = scale * kLog2e;
    p.mode = mode;
    if (d == 128) return launch_decode<128>(p, stream);
    if (d == 64) return launch_decode<64>(p, stream);
    if (d == 256) return launch_decode<256>(p, stream);
    return CSA_ERR_UNSUPPORTED;
}

}  // namespace

int csa_decode_run(const void *q, const void *k_cache, const void *v_cache, const void *k0,
                   const void *v0, const int *seqlens, void *out, float *lse, void *scratch, int B,
                   int H, int T, int d, float scale, int mode, cudaStream_t stream) {
    return run_range(q, k_cache, v_cache, k0, v0, seqlens, out, nullptr, lse, scratch, B, H, T, d,
                     scale, mode, 0, T + 1, stream);
}

int csa_decode_merge_ranges_run(const float *o_parts, const float *lse_parts, int R, int B, int H,
                                int d, void *out, float *lse, cudaStream_t stream) {
    const long long rows = (long long)B * H;
    const long long blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL) return CSA_ERR_UNSUPPORTED;
    merge_ranges_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        o_parts, lse_parts, R, rows, d, static_cast<__nv_bfloat16 *>(out), lse);
    return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

int csa_decode_range_run(const void *q, const void *k_shard, const void *v_shard, const void *k0,
                         const void *v0, const int *seqlens, float *out, float *lse,
                         void *scratch, int B, int H, int T, int d, float scale, int mode,
                         int pos_lo, int pos_hi, cudaStream_t stream) {
    return run_range(q, k_shard, v_shard, k0, v0, seqlens, nullptr, out, lse, scratch, B, H, T, d,
                     scale, mode, pos_lo, pos_hi, stream);
}

int csa_decode_take_status(void) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_dec_status, sizeof(int)) != cudaSuccess) return CSA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_dec_status, &zero, sizeof(int)) != cudaSuccess) return CSA_ERR_CUDA;
    return v;
}
