// Decode step of causal continuous softmax attention: for every sequence b
// and head h, the query of the newest token against the sink and the n_b
// cached keys and values.  This is eq. (10)/(11) of "Continuous Softmax
// Attention" ("Assembly and Simplification") for the single row t = n_b.
//
// The step reads every cached key and value once and does about two flops
// per byte read, so it is bound by HBM bandwidth and runs on CUDA cores.
// The key positions 0..n (0 is the sink k_0, position i >= 1 is cache row
// i - 1) are cut into chunks of C positions.  One CTA per (b, h, chunk):
//   1. stages the chunk's keys plus one halo key on each side (the correction
//      b of a key needs both neighbours' logits, eq. (10)) and the chunk's
//      values, with two bulk asynchronous copies;
//   2. forms the logits, in log2 units, one key per group of d/8 lanes;
//   3. forms each key's weight e^{a+b} relative to the chunk's own maximum m:
//      for a key with logit a and a neighbour at a + x, the neighbour's
//      interval contributes e^{a-m} phi2(x) (eq. (9));
//   4. writes the partial sums l = sum w and o = sum w v, with m.
// A second kernel merges the chunks of each (b, h): with M the largest m,
// o = sum_c 2^{m_c-M} o_c / sum_c 2^{m_c-M} l_c and lse = (M + log2 L) ln 2.
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
constexpr int kMergeThreads = 128;
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
    static constexpr int C = 16384 / D;     // positions per chunk: 32 KiB of values
    static constexpr int KRows = C + 2;      // keys staged: the chunk and a halo key each side
    static constexpr int LPK = D / 8;        // lanes per key in the logit loop (16 B each)
    static constexpr int KPW = 32 / LPK;     // keys per warp per step of that loop
    static constexpr int CP = D / 2;         // column pairs of a value row
    static constexpr int G = kThreads / CP;  // key groups in the value loop
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + KRows * D * 2;
    static constexpr int kOffA = kOffV + C * D * 2;       // logits, [KRows] floats
    static constexpr int kOffW = kOffA + KRows * 4;       // weights, [C] floats
    static constexpr int kOffRed = kOffW + C * 4;         // value partials, [G][D] floats
    static constexpr int kOffWarp = kOffRed + G * D * 4;  // block reductions, [2][kWarps]
    static constexpr int kOffBar = (kOffWarp + 2 * kWarps * 4 + 15) / 16 * 16;
    static constexpr int kSmemBytes = kOffBar + 16;
    static_assert(kOffV % 16 == 0 && kOffA % 16 == 0, "bulk copy destinations 16-byte aligned");
    static_assert(kSmemBytes <= 75 * 1024, "three CTAs per SM");
};

struct DecParams {
    const __nv_bfloat16 *q, *k, *v, *k0, *v0;
    const int *seqlens;
    float *part_o;   // [B*H][S][D]: unnormalised partial outputs
    float *part_ml;  // [B*H][S][2]: chunk maximum (log2 units), chunk weight sum
    __nv_bfloat16 *out;
    float *lse;
    int B, H, T, S;
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

__device__ __forceinline__ float dot8(const float (&q)[8], const uint4 &raw) {
    float kf[8];
    unpack8(raw, kf);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = fmaf(q[i], kf[i], acc);
    return acc;
}

// e^{u} phi2(x) for a key at u (log2 units, u <= 0) whose neighbour is at
// u + x2 = un (log2 units); x = x2 ln 2 is the natural-log gap and
// pc = 2^u.  phi2(x) = (e^x - 1 - x)/x^2 ("Preliminaries", eq. (6)).
//   |x| < 1: pc * sum_{j=0..9} x^j/(j+2)!  (truncation below 3e-9 relative);
//   x <= 20: pc * (e^x - 1 - x)/x^2, with e^x = 2^{x2};
//   x > 20:  (2^{un} - pc (1 + x))/x^2, since pc e^x = 2^{un} <= 1 while e^x
//            alone could overflow.
__device__ __forceinline__ float side_weight(float x2, float un, float pc) {
    const float x = x2 * kLn2;
    if (fabsf(x) < 1.0f) {
        float s = 2.505210838544172e-08f;       // 1/11!
        s = fmaf(s, x, 2.755731922398589e-07f);  // 1/10!
        s = fmaf(s, x, 2.755731922398589e-06f);  // 1/9!
        s = fmaf(s, x, 2.48015873015873e-05f);   // 1/8!
        s = fmaf(s, x, 1.984126984126984e-04f);  // 1/7!
        s = fmaf(s, x, 1.388888888888889e-03f);  // 1/6!
        s = fmaf(s, x, 8.333333333333333e-03f);  // 1/5!
        s = fmaf(s, x, 4.166666666666667e-02f);  // 1/4!
        s = fmaf(s, x, 1.666666666666667e-01f);  // 1/3!
        s = fmaf(s, x, 0.5f);                    // 1/2!
        return pc * s;
    }
    if (x <= 20.0f) return pc * ((ex2_approx(x2) - 1.0f - x) / (x * x));
    return (ex2_approx(un) - pc * (1.0f + x)) / (x * x);
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

template <int D>
__global__ void __launch_bounds__(kThreads) decode_chunk_kernel(const DecParams p) {
    using Cf = DecCfg<D>;
    constexpr int C = Cf::C;
    extern __shared__ __align__(128) uint8_t smem[];
    __nv_bfloat16 *ks = reinterpret_cast<__nv_bfloat16 *>(smem + Cf::kOffK);
    __nv_bfloat16 *vs = reinterpret_cast<__nv_bfloat16 *>(smem + Cf::kOffV);
    float *as = reinterpret_cast<float *>(smem + Cf::kOffA);
    float *ws = reinterpret_cast<float *>(smem + Cf::kOffW);
    float *red = reinterpret_cast<float *>(smem + Cf::kOffRed);
    float *wred = reinterpret_cast<float *>(smem + Cf::kOffWarp);
    const uint32_t bar = smem_u32(smem + Cf::kOffBar);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cf::kOffBar + 8);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bh = blockIdx.x / p.S, chunk = blockIdx.x - bh * p.S;
    const int b = bh / p.H, h = bh - b * p.H;
    const int n = p.seqlens ? p.seqlens[b] : p.T;
    const int P0 = chunk * C;
    if (n < 1 || n > p.T || P0 > n) return;  // no position of this chunk exists
    const int P1 = min(P0 + C, n + 1);        // owned positions [P0, P1)
    const int own = P1 - P0;
    const int kp_lo = max(P0 - 1, 1), kp_hi = min(P1, n);  // cached keys staged
    const int vp_lo = max(P0, 1);                          // cached values staged: [vp_lo, P1)
    const size_t head = (size_t)bh * p.T;
    // Shared-memory slot of position pos: keys pos - P0 + 1, values pos - P0.

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bar, 1);
        fence_mbar_init();
        const uint32_t kbytes = (uint32_t)(kp_hi - kp_lo + 1) * D * 2;
        const uint32_t vbytes = (uint32_t)(P1 - vp_lo) * D * 2;
        mbar_arrive_expect_tx(bar, kbytes + vbytes);
        bulk_load(smem_u32(ks + (kp_lo - P0 + 1) * D), p.k + (head + kp_lo - 1) * D, kbytes, bar);
        bulk_load(smem_u32(vs + (vp_lo - P0) * D), p.v + (head + vp_lo - 1) * D, vbytes, bar);
    }

    const int c8 = lane % Cf::LPK;  // this lane's 8 columns of a key
    float qf[8];
    unpack8(reinterpret_cast<const uint4 *>(p.q + (size_t)bh * D)[c8], qf);
#pragma unroll
    for (int i = 0; i < 8; ++i) qf[i] *= p.qscale;

    __syncthreads();  // barrier initialised
    if (!mbar_wait_bounded(bar, 0, abort_flag, &g_dec_status, kWaitLimitNs)) {
        // Keep the block (and its shared memory) alive until the copies land.
        if (tid == 0 && !mbar_try_wait(bar, 0)) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
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

    // Logits of the staged positions [kp_lo - 1 or the sink, kp_hi].
    const int r_lo = (P0 == 0) ? 1 : 0, r_hi = kp_hi - P0 + 1;
    const int grp = warp * Cf::KPW + lane / Cf::LPK;
    for (int base = r_lo; base <= r_hi; base += kWarps * Cf::KPW) {
        const int r = base + grp;
        float acc = 0.f;
        if (r <= r_hi) {
            const int pos = r + P0 - 1;
            uint4 raw = make_uint4(0u, 0u, 0u, 0u);
            if (pos > 0)
                raw = reinterpret_cast<const uint4 *>(ks + r * D)[c8];
            else if (p.mode == CSA_K0_GIVEN)
                raw = reinterpret_cast<const uint4 *>(p.k0 + (size_t)h * D)[c8];
            else if (p.mode == CSA_K0_COPY_FIRST)
                raw = reinterpret_cast<const uint4 *>(ks + 2 * D)[c8];  // position 1
            acc = dot8(qf, raw);
        }
#pragma unroll
        for (int off = Cf::LPK / 2; off > 0; off >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (r <= r_hi && c8 == 0) as[r] = acc;
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
    __syncthreads();
    lsum = 0.f;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) lsum += wred[kWarps + i];

    // o = sum_i w_i v_i: G groups of keys, a column pair per thread.
    const int cp = tid % Cf::CP, g = tid / Cf::CP;
    float o0 = 0.f, o1 = 0.f;
    for (int i = g; i < own; i += Cf::G) {
        const float w = ws[i];
        const float2 vf =
            __bfloat1622float2(reinterpret_cast<const __nv_bfloat162 *>(vs + i * D)[cp]);
        o0 = fmaf(w, vf.x, o0);
        o1 = fmaf(w, vf.y, o1);
    }
    reinterpret_cast<float2 *>(red + g * D)[cp] = make_float2(o0, o1);
    __syncthreads();
    const size_t slot = (size_t)bh * p.S + chunk;
    float *po = p.part_o + slot * D;
    for (int col = tid; col < D; col += kThreads) {
        float s = 0.f;
#pragma unroll
        for (int gg = 0; gg < Cf::G; ++gg) s += red[gg * D + col];
        po[col] = s;
    }
    if (tid == 0) {
        p.part_ml[2 * slot] = mx;
        p.part_ml[2 * slot + 1] = lsum;
    }
}

template <int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const DecParams p) {
    constexpr int C = DecCfg<D>::C;
    const int bh = blockIdx.x, b = bh / p.H, tid = threadIdx.x;
    const int n = p.seqlens ? p.seqlens[b] : p.T;
    __nv_bfloat16 *out = p.out + (size_t)bh * D;
    if (n < 1 || n > p.T) {  // a length outside [1, T]: NaN result, status word set
        for (int col = tid; col < D; col += kMergeThreads) out[col] = __float2bfloat16_rn(NAN);
        if (tid == 0) {
            if (p.lse) p.lse[bh] = NAN;
            atomicCAS(&g_dec_status, 0, CSA_ERR_INVALID_ARG);
        }
        return;
    }
    const int nch = n / C + 1;  // chunks holding positions 0..n
    const float *ml = p.part_ml + (size_t)bh * p.S * 2;
    const float *po = p.part_o + (size_t)bh * p.S * D;
    float M = -INFINITY;
    for (int c = 0; c < nch; ++c) M = fmaxf(M, ml[2 * c]);
    float L = 0.f;
    for (int c = 0; c < nch; ++c) L = fmaf(ml[2 * c + 1], ex2_approx(ml[2 * c] - M), L);
    const float inv = 1.0f / L;
    for (int col = tid; col < D; col += kMergeThreads) {
        float acc = 0.f;
        for (int c = 0; c < nch; ++c) acc = fmaf(po[(size_t)c * D + col], ex2_approx(ml[2 * c] - M), acc);
        out[col] = __float2bfloat16_rn(acc * inv);
    }
    if (tid == 0 && p.lse) p.lse[bh] = (M + log2f(L)) * kLn2;
}

template <int D>
int launch_decode(DecParams p, cudaStream_t stream) {
    using Cf = DecCfg<D>;
    p.S = p.T / Cf::C + 1;
    const long long BH = (long long)p.B * p.H;
    const long long grid = BH * p.S;
    if (grid > 0x7fffffffLL || BH > 0x7fffffffLL) return CSA_ERR_UNSUPPORTED;
    auto kern = decode_chunk_kernel<D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::kSmemBytes) !=
        cudaSuccess)
        return CSA_ERR_CUDA;
    kern<<<(unsigned)grid, kThreads, Cf::kSmemBytes, stream>>>(p);
    decode_merge_kernel<D><<<(unsigned)BH, kMergeThreads, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

int chunk_positions(int d) { return d == 64 ? DecCfg<64>::C : d == 128 ? DecCfg<128>::C : DecCfg<256>::C; }

}  // namespace

long long csa_decode_scratch_bytes(int B, int H, int T, int d) {
    if (B < 0 || H < 0 || T < 0 || !(d == 64 || d == 128 || d == 256)) return -1;
    const long long S = (long long)T / chunk_positions(d) + 1;
    return (long long)B * H * S * (d + 2) * (long long)sizeof(float);
}

int csa_decode_run(const void *q, const void *k_cache, const void *v_cache, const void *k0,
                   const void *v0, const int *seqlens, void *out, float *lse, void *scratch, int B,
                   int H, int T, int d, float scale, int mode, cudaStream_t stream) {
    DecParams p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k_cache);
    p.v = static_cast<const __nv_bfloat16 *>(v_cache);
    p.k0 = static_cast<const __nv_bfloat16 *>(k0);
    p.v0 = static_cast<const __nv_bfloat16 *>(v0);
    p.seqlens = seqlens;
    const long long S = (long long)T / chunk_positions(d) + 1;
    p.part_o = static_cast<float *>(scratch);
    p.part_ml = p.part_o + (long long)B * H * S * d;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.lse = lse;
    p.B = B;
    p.H = H;
    p.T = T;
    p.S = (int)S;
    p.qscale = scale * kLog2e;
    p.mode = mode;
    if (d == 128) return launch_decode<128>(p, stream);
    if (d == 64) return launch_decode<64>(p, stream);
    if (d == 256) return launch_decode<256>(p, stream);
    return CSA_ERR_UNSUPPORTED;
}

// Scratch of csa_decode_noalloc: a file-scope device array, so that the
// entry point allocates nothing.  Its address is looked up once per device.
static __device__ __align__(256) float g_noalloc_scratch[CSA_DECODE_NOALLOC_SCRATCH_BYTES / 4];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_addr[kMaxDevices];
}  // namespace

int csa_decode_noalloc_scratch(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CSA_ERR_NO_DEVICE;
    if (dev < 0 || dev >= kMaxDevices) return CSA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        // dev is the current device here, so the address is that device's copy.
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return CSA_ERR_CUDA;
        g_noalloc_addr[dev] = p;
    }
    *addr = g_noalloc_addr[dev];
    return CSA_OK;
}

int csa_decode_take_status(void) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_dec_status, sizeof(int)) != cudaSuccess) return CSA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_dec_status, &zero, sizeof(int)) != cudaSuccess) return CSA_ERR_CUDA;
    return v;
}
