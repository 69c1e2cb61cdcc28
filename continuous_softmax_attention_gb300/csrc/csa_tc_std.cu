// Tensor-core forward kernel for standard causal softmax attention, eq. (12)
// of Jianlin Su, "Continuous Softmax Attention" ("Analysis of the Result"):
// o_t = sum_{i<=t} e^{a_{t,i}} v_i / sum_{i<=t} e^{a_{t,i}}, a = scale q.k;
// the same as softmax(Q K^T scale + M) V with the causal mask M of
// "Attention, from the softmax up" ("The one line").  bf16 in/out, d = 64
// or 128, fp32 accumulation; the in-build comparator of the continuous
// kernel.
//
// Work split.  One CTA owns two 128-row query tiles of one (b, h) and walks
// the 128-row key/value tiles up to their diagonal.  Warps:
//   0-3  softmax of query tile 0 (one thread = one query row)
//   4-7  softmax of query tile 1
//   8    TMA producer (lane 0)
//   9    TMEM allocator and tcgen05.mma issuer (lane 0)
// Tensor memory: S0 | S1 | O0 | O1 (fp32); the bf16 P overwrites the first
// 64 columns of its S and is the A operand of the PV product.  While one
// query tile's softmax runs, the tensor core works on the other tile's PV
// and next S.  The softmax takes the tile max with a 3-input max tree,
// moves the running max lazily (only when it would rise by more than 8 in
// log2 units, so weights stay <= 2^8), and rescales O in TMEM when it does.
// Waits are bounded in time like those of the continuous kernel.
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

__device__ int g_std_status;  // sticky status word of this file's kernel

constexpr int kThreads = 320;

template <int D>
struct StdCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kTileBytes = kChunks * kChunkBytes;
    static constexpr int kStagesK = D == 128 ? 2 : 3;
    static constexpr int kStagesV = D == 128 ? 2 : 3;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + 2 * kTileBytes;
    static constexpr int kOffV = kOffK + kStagesK * kTileBytes;
    static constexpr int kOffBar = kOffV + kStagesV * kTileBytes;
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
    __device__ static constexpr uint32_t col_s(int qt) { return 128u * (uint32_t)qt; }
    __device__ static constexpr uint32_t col_o(int qt) { return 256u + (uint32_t)(D * qt); }
};

struct StdParams {
    int B, H, T;
    int num_pairs;
    int group;  // heads per scheduling group
    float k2;  // scale * log2(e)
    __nv_bfloat16 *out;
    float *lse;
};

__device__ __forceinline__ bool wait_s(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    return wait_bar(bar, parity, abort_flag, &g_std_status);
}

__device__ __forceinline__ float fmin3f(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Softmax of one S tile at tS for this thread's row.  Returns whether the
// running max moved (alpha is then the factor O must be scaled by).  NEG:
// the scale is negative, so the largest scaled logit is the smallest q.k.
template <bool MASKED, bool NEG>
__device__ __forceinline__ bool std_tile(uint32_t tS, float k2, int c_last, float &m_run,
                                         float &l_run, float &alpha) {
    float mx;
    {
        uint32_t sr[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + 32 * cc, sr[cc]);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_wait_ld_regs<32>(sr[cc]);
        constexpr float kNone = NEG ? INFINITY : -INFINITY;
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = kNone;
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
            float v0 = __uint_as_float(sr[c >> 5][c & 31]);
            float v1 = __uint_as_float(sr[(c + 1) >> 5][(c + 1) & 31]);
            if (MASKED) {
                v0 = c <= c_last ? v0 : kNone;
                v1 = c + 1 <= c_last ? v1 : kNone;
            }
            a[(c >> 1) & 7] = NEG ? fmin3f(a[(c >> 1) & 7], v0, v1) : fmax3f(a[(c >> 1) & 7], v0, v1);
        }
        if (NEG)
            mx = fmin3f(fmin3f(a[0], a[1], a[2]), fmin3f(a[3], a[4], a[5]), fminf(a[6], a[7]));
        else
            mx = fmax3f(fmax3f(a[0], a[1], a[2]), fmax3f(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
    }
    const float mt = (!MASKED || c_last >= 0) ? mx * k2 : -INFINITY;
    alpha = 1.0f;
    const bool grow = mt > m_run + 8.0f;
    if (grow) {
        alpha = ex2_approx(m_run - mt);
        m_run = mt;
        l_run *= alpha;
    }
    const float nm = -m_run;
    float2 lsum = make_float2(0.0f, 0.0f), ls2 = make_float2(0.0f, 0.0f);
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
        uint32_t a[32];
        tmem_ld32(tS + 32 * k, a);
        tmem_wait_ld_regs<32>(a);
        float w[32];
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
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            pk[i >> 1] = pack_bf16x2(w[i], w[i + 1]);
            if ((i & 2) == 0)
                lsum = __fadd2_rn(lsum, make_float2(w[i], w[i + 1]));
            else
                ls2 = __fadd2_rn(ls2, make_float2(w[i], w[i + 1]));
        }
        tmem_st16(tS + 16 * k, pk);
    }
    tmem_wait_st();
    lsum = __fadd2_rn(lsum, ls2);
    l_run += lsum.x + lsum.y;
    return grow;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    std_forward_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const StdParams p) {
    using C = StdCfg<D>;
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
    // Heads go in groups whose K/V fit in L2 together; within a group the
    // heaviest query tiles go first (longest-first keeps the tail short).
    const int nq = p.num_pairs, BH = p.B * p.H;
    const int grp = (int)(blockIdx.x / (unsigned)(p.group * nq));
    const int gsz = min(p.group, BH - grp * p.group);
    const int idx = (int)blockIdx.x - grp * p.group * nq;
    const int bh = grp * p.group + idx % gsz;
    const int pair = nq - 1 - idx / gsz;
    const int T = p.T;
    int row0[2], ntiles[2];
#pragma unroll
    for (int qt = 0; qt < 2; ++qt) {
        row0[qt] = pair * 256 + qt * 128;
        ntiles[qt] = row0[qt] >= T ? 0 : min(row0[qt] + 127, T - 1) / 128 + 1;
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
                        tma_load_3d(sQ + qt * C::kTileBytes + c * kChunkBytes, &tm_q, 64 * c,
                                    row0[qt], bh, BAR(C::kBarQ));
            int issued_k = 0, issued_v = 0;
            for (int j = 0; j < nj; ++j) {
                const int sk = j % NSK;
                if (!wait_s(BAR(C::kBarKEmpty + sk), ((j / NSK) & 1) ^ 1, abort_flag)) break;
                mbar_arrive_expect_tx(BAR(C::kBarKFull + sk), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sK + sk * C::kTileBytes + c * kChunkBytes, &tm_k, 64 * c, 128 * j,
                                bh, BAR(C::kBarKFull + sk));
                issued_k = j + 1;
                const int sv = j % NSV;
                if (!wait_s(BAR(C::kBarVEmpty + sv), ((j / NSV) & 1) ^ 1, abort_flag)) break;
                mbar_arrive_expect_tx(BAR(C::kBarVFull + sv), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sV + sv * C::kTileBytes + c * kChunkBytes, &tm_v, 64 * c, 128 * j,
                                bh, BAR(C::kBarVFull + sv));
                issued_v = j + 1;
            }
            wait_bar_drain(BAR(C::kBarQ), 0, &g_std_status);
            for (int j = max(0, issued_k - NSK); j < issued_k; ++j)
                wait_bar_drain(BAR(C::kBarKFull + j % NSK), (j / NSK) & 1, &g_std_status);
            for (int j = max(0, issued_v - NSV); j < issued_v; ++j)
                wait_bar_drain(BAR(C::kBarVFull + j % NSV), (j / NSV) & 1, &g_std_status);
        }
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0 && nj > 0) {
            constexpr uint32_t kIdescS = make_idesc(128, 128, false);
            constexpr uint32_t kIdescO = make_idesc(128, D, true);
            bool ok = wait_s(BAR(C::kBarQ), 0, abort_flag);
            tc_fence_after();
            int k_seen = -1, v_seen = -1;
            auto issue_s = [&](int qt, int j) -> bool {
                if (k_seen < j) {
                    if (!wait_s(BAR(C::kBarKFull + j % NSK), (j / NSK) & 1, abort_flag)) return false;
                    k_seen = j;
                    tc_fence_after();
                }
                const uint32_t qb = sQ + qt * C::kTileBytes;
                const uint32_t kb = sK + (j % NSK) * C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                    tc_mma_ss(tmem + C::col_s(qt), make_sdesc(qb + off, 16, 1024),
                              make_sdesc(kb + off, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
                }
                tc_commit(BAR(C::kBarSFull + qt));
                return true;
            };
            auto issue_pv = [&](int qt, int j) -> bool {
                if (v_seen < j) {
                    if (!wait_s(BAR(C::kBarVFull + j % NSV), (j / NSV) & 1, abort_flag)) return false;
                    v_seen = j;
                    tc_fence_after();
                }
                const uint32_t vb = sV + (j % NSV) * C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc_mma_ts(tmem + C::col_o(qt), tmem + C::col_s(qt) + kk * 8,
                              make_sdesc(vb + kk * 2048, kChunkBytes, 1024), kIdescO,
                              (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(BAR(C::kBarODone + qt));
                return true;
            };
            for (int qt = 0; qt < 2 && ok; ++qt)
                if (ntiles[qt] > 0) ok = issue_s(qt, 0);
            if (ok) tc_commit(BAR(C::kBarKEmpty + 0));
            for (int j = 0; ok && j < nj; ++j) {
                for (int qt = 0; qt < 2; ++qt) {
                    if (j >= ntiles[qt]) continue;
                    if (!(ok = wait_s(BAR(C::kBarPFull + qt), j & 1, abort_flag))) break;
                    tc_fence_after();
                    if (!(ok = issue_pv(qt, j))) break;
                    // S(j+1) overwrites the TMEM that PV(j) reads as P; both are
                    // tcgen05.mma issued in order by this thread.
                    if (j + 1 < ntiles[qt] && !(ok = issue_s(qt, j + 1))) break;
                }
                if (!ok) break;
                tc_commit(BAR(C::kBarVEmpty + j % NSV));
                if (j + 1 < nj) tc_commit(BAR(C::kBarKEmpty + (j + 1) % NSK));
            }
            tc_commit(BAR(C::kBarDrain));
            wait_bar_drain(BAR(C::kBarDrain), 0, &g_std_status);
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
        float m_run = -INFINITY, l_run = 0.0f;
        bool ok = n > 0;
        for (int j = 0; ok && j < n; ++j) {
            ok = __all_sync(0xffffffffu, wait_s(BAR(C::kBarSFull + qt), j & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            const int c_last = r - 128 * j;
            float alpha;
            const bool masked = 128 * j + 127 > row0[qt];
            const bool grow =
                p.k2 < 0.0f
                    ? (masked ? std_tile<true, true>(tS, p.k2, c_last, m_run, l_run, alpha)
                              : std_tile<false, true>(tS, p.k2, c_last, m_run, l_run, alpha))
                    : (masked ? std_tile<true, false>(tS, p.k2, c_last, m_run, l_run, alpha)
                              : std_tile<false, false>(tS, p.k2, c_last, m_run, l_run, alpha));
            const bool need_o = grow && j > 0;
            if (__any_sync(0xffffffffu, need_o)) {
                ok = __all_sync(0xffffffffu, wait_s(BAR(C::kBarODone + qt), (j - 1) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                const float a = need_o ? alpha : 1.0f;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * cc, o);
                    tmem_wait_ld_regs<32>(o);
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
            ok = __all_sync(0xffffffffu, wait_s(BAR(C::kBarODone + qt), (n - 1) & 1, abort_flag));
            if (ok) {
                tc_fence_after();
                const float inv_l = 1.0f / l_run;
                const bool store = r < T;
                __nv_bfloat16 *orow = p.out + ((size_t)bh * T + (size_t)(store ? r : 0)) * D;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * cc, o);
                    tmem_wait_ld_regs<32>(o);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l,
                                            __uint_as_float(o[2 * e + 1]) * inv_l);
                    if (store) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * cc);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                    }
                }
                if (store && p.lse) p.lse[(size_t)bh * T + r] = (m_run + log2f(l_run)) * kLn2;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, 512);
#undef BAR
}

template <int D>
int launch_std(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
               int T, float scale, cudaStream_t stream) {
    using C = StdCfg<D>;
    const int BH = B * H;
    CUtensorMap mq, mk, mv;
    if (!encode_qkv_map(&mq, q, BH, T, D) || !encode_qkv_map(&mk, k, BH, T, D) ||
        !encode_qkv_map(&mv, v, BH, T, D))
        return CSA_ERR_CUDA;
    StdParams prm;
    prm.B = B;
    prm.H = H;
    prm.T = T;
    prm.num_pairs = (T + 255) / 256;
    prm.group = heads_per_group(BH, T, D);
    prm.k2 = scale * kLog2e;
    prm.out = static_cast<__nv_bfloat16 *>(out);
    prm.lse = lse;
    const long long grid = (long long)prm.num_pairs * BH;
    if (grid > 0x7fffffffLL) return CSA_ERR_UNSUPPORTED;
    auto kern = std_forward_kernel<D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
        return CSA_ERR_CUDA;
    kern<<<(unsigned)grid, kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, prm);
    return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

}  // namespace

int csa_tc_std_forward(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                       int H, int T, int d, float scale, cudaStream_t stream) {
    if (d == 128) return launch_std<128>(q, k, v, out, lse, B, H, T, scale, stream);
    if (d == 64) return launch_std<64>(q, k, v, out, lse, B, H, T, scale, stream);
    return CSA_ERR_UNSUPPORTED;
}

int csa_tc_std_take_status(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return CSA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_std_status, sizeof(int)) != cudaSuccess) return CSA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_std_status, &zero, sizeof(int)) != cudaSuccess) return CSA_ERR_CUDA;
    return v;
}
