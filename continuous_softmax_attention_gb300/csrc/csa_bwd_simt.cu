// Backward pass of causal continuous softmax attention on CUDA cores, for
// fp32 inputs and for bf16 inputs whose head dimension the tensor-core
// kernel does not cover.
//
// Gradient of eq. (10)/(11) of Jianlin Su, "Continuous Softmax Attention"
// ("Assembly and Simplification").  With p_i = e^{a_i - lse}, the interval
// between keys i-1 and i (logit step x = a_i - a_{i-1}) hands its left key
// R = p_{i-1} phi2(x) and its right key L = p_i phi2(-x) (eq. (9)), so that
// P_i = L_i + R_i.  Differentiating the two shares with respect to their
// end logits gives, for one row with upstream gradient dO:
//     da_i = P_i (dP_i - D) + F_i - F_{i+1},
//     F_i  = c_i (dP_{i-1} - dP_i),   c_i = p_{i-1} phi2'(x) = p_i phi2'(-x),
// with dP_i = dO . v_i, D = dO . o and F = 0 past either end of the row:
// the share of an interval moves along it as its end logits move, so each
// interval passes a flux between its two keys.  Then dq = scale sum da_i k_i,
// dk_i += scale da_i q, dv_i += P_i dO.
//
// One warp per query row walks its keys in order (lanes split the head
// dimension), writes dq directly and adds its dk, dv contributions into
// fp32 accumulators with atomics; a second kernel converts them.  This
// path is for small problems and for cross-checking; its atomics make it
// slow at long sequence lengths.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "csa_internal.h"

namespace {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f32(float *p, float x) { *p = x; }
__device__ __forceinline__ void from_f32(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// The interval between a left key at logit al and a right key at ar, for a
// row with normaliser lse: its share R of the left key, its share L of the
// right key and the flux coefficient c = p_l phi2'(x), x = ar - al.
// phi2'(x) = ((x - 2) e^x + x + 2)/x^3 is the derivative of eq. (6)'s phi2.
// Every form is written around the larger end, p = e^{max(al, ar) - lse},
// with m = e^{-|x|} <= 1, so nothing overflows and the two ends stay
// consistent; |x| < 1 uses the power series of the integral definitions,
// phi2 = sum x^n/(n+2)!, phi2' = sum (n+1) x^n/(n+3)!.
struct Interval {
    float R, L, c;
};

__device__ __forceinline__ float series_phi2(float x) {
    // sum_{n=0}^{12} x^n / (n+2)!, Horner from n = 12 (1/14!) down
    float s = 1.0f / 87178291200.0f;
    const float inv[11] = {1.0f / 6227020800.0f, 1.0f / 479001600.0f, 1.0f / 39916800.0f,
                           1.0f / 3628800.0f,    1.0f / 362880.0f,    1.0f / 40320.0f,
                           1.0f / 5040.0f,       1.0f / 720.0f,       1.0f / 120.0f,
                           1.0f / 24.0f,         1.0f / 6.0f};
#pragma unroll
    for (int i = 0; i < 11; ++i) s = fmaf(s, x, inv[i]);
    return fmaf(s, x, 0.5f);
}

__device__ __forceinline__ float series_dphi2(float x) {
    // sum_{n=0}^{11} (n+1) x^n / (n+3)!, Horner from n = 11 (12/14!) down
    float s = 12.0f / 87178291200.0f;
    const float c[10] = {11.0f / 6227020800.0f, 10.0f / 479001600.0f, 9.0f / 39916800.0f,
                         8.0f / 3628800.0f,     7.0f / 362880.0f,     6.0f / 40320.0f,
                         5.0f / 5040.0f,        4.0f / 720.0f,        3.0f / 120.0f,
                         2.0f / 24.0f};
#pragma unroll
    for (int i = 0; i < 10; ++i) s = fmaf(s, x, c[i]);
    return fmaf(s, x, 1.0f / 6.0f);
}

__device__ Interval interval(float al, float ar, float lse) {
    const float x = ar - al;
    const float p = expf(fmaxf(al, ar) - lse);
    const float m = expf(-fabsf(x));
    Interval s;
    if (fabsf(x) < 1.0f) {
        const float pl = x >= 0.0f ? p * m : p, pr = x >= 0.0f ? p : p * m;
        s.R = pl * series_phi2(x);
        s.L = pr * series_phi2(-x);
        s.c = pl * series_dphi2(x);
    } else if (x > 0.0f) {  // p = p_r, p_l = p m
        const float x2 = x * x;
        s.R = p * (1.0f - (1.0f + x) * m) / x2;
        s.L = p * (m - 1.0f + x) / x2;
        s.c = p * ((x - 2.0f) + (x + 2.0f) * m) / (x2 * x);
    } else {  // p = p_l, p_r = p m
        const float x2 = x * x;
        s.R = p * (m - 1.0f - x) / x2;
        s.L = p * (1.0f - (1.0f - x) * m) / x2;
        s.c = p * ((x - 2.0f) * m + x + 2.0f) / (x2 * x);
    }
    return s;
}

template <typename Tin, int NPL>
struct Row {
    const Tin *k, *v, *k0, *v0;
    int T, d, mode, h, lane;
    long long bh;
    __device__ const Tin *key(int i) const {
        if (i >= 1) return k + ((size_t)bh * T + (size_t)(i - 1)) * d;
        if (mode == 1) return k + (size_t)bh * T * d;
        if (mode == 2) return k0 + (size_t)h * d;
        return nullptr;
    }
    __device__ const Tin *val(int i) const {
        if (i >= 1) return v + ((size_t)bh * T + (size_t)(i - 1)) * d;
        if (mode == 1) return v + (size_t)bh * T * d;
        if (mode == 2) return v0 + (size_t)h * d;
        return nullptr;
    }
    __device__ void load(const Tin *p, float (&x)[NPL]) const {
#pragma unroll
        for (int j = 0; j < NPL; ++j) {
            const int c = lane + 32 * j;
            x[j] = (p && c < d) ? to_f32(p[c]) : 0.0f;
        }
    }
};

template <int NPL>
__device__ __forceinline__ float dot(const float (&a)[NPL], const float (&b)[NPL]) {
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < NPL; ++j) s = fmaf(a[j], b[j], s);
    return warp_sum(s);
}

// Gradient contributions of key i of the extended sequence (0 = the sink)
// with weight P and logit gradient da.
template <typename Tin, int NPL>
__device__ __forceinline__ void add_key_grads(const Row<Tin, NPL> &rw, int i, float P, float ds,
                                              const float (&qv)[NPL], const float (&gv)[NPL],
                                              float *dk_acc, float *dv_acc, float (&sk)[NPL],
                                              float (&sv)[NPL]) {
    if (i >= 1) {
        float *dk = dk_acc + ((size_t)rw.bh * rw.T + (size_t)(i - 1)) * rw.d;
        float *dv = dv_acc + ((size_t)rw.bh * rw.T + (size_t)(i - 1)) * rw.d;
#pragma unroll
        for (int j = 0; j < NPL; ++j) {
            const int c = rw.lane + 32 * j;
            if (c < rw.d) {
                atomicAdd(dk + c, ds * qv[j]);
                atomicAdd(dv + c, P * gv[j]);
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < NPL; ++j) {
            sk[j] = ds * qv[j];
            sv[j] = P * gv[j];
        }
    }
}

template <typename Tin, int NPL>
__global__ void __launch_bounds__(256) simt_backward_kernel(
    const Tin *q, const Tin *k, const Tin *v, const Tin *k0, const Tin *v0, const Tin *o,
    const float *lse, const Tin *dout, Tin *dq, float *dk_acc, float *dv_acc, float *dk0,
    float *dv0, int B, int H, int T, int d, float scale, int mode) {
    const long long BH = (long long)B * H;
    const long long gw = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (gw >= BH * T) return;
    const int r = T - 1 - (int)(gw / BH);  // longest rows first
    Row<Tin, NPL> rw;
    rw.k = k; rw.v = v; rw.k0 = k0; rw.v0 = v0;
    rw.T = T; rw.d = d; rw.mode = mode;
    rw.bh = gw % BH;
    rw.h = (int)(rw.bh % H);
    rw.lane = threadIdx.x & 31;
    const size_t row = (size_t)rw.bh * T + (size_t)r;
    float qv[NPL], gv[NPL], ov[NPL], kc[NPL], kp[NPL], vv[NPL], dqv[NPL], sk[NPL], sv[NPL];
    rw.load(q + row * d, qv);
    rw.load(dout + row * d, gv);
    rw.load(o + row * d, ov);
#pragma unroll
    for (int j = 0; j < NPL; ++j) dqv[j] = sk[j] = sv[j] = 0.0f;
    const float D = dot(gv, ov);
    const float ls = lse[row];
    const int t = r + 1;

    // key 0 (the sink)
    rw.load(rw.key(0), kp);
    rw.load(rw.val(0), vv);
    float a_p = scale * dot(qv, kp), g_p = dot(gv, vv);
    float L_p = 0.0f, F_p = 0.0f;  // key i-1's left share and the flux into it
    for (int i = 1; i <= t; ++i) {
        rw.load(rw.key(i), kc);
        rw.load(rw.val(i), vv);
        const float a = scale * dot(qv, kc), g = dot(gv, vv);
        const Interval s = interval(a_p, a, ls);
        const float F = s.c * (g_p - g);
        // key i-1 is complete: both of its intervals are known
        const float P = L_p + s.R;
        const float ds = scale * (P * (g_p - D) + F_p - F);
#pragma unroll
        for (int j = 0; j < NPL; ++j) dqv[j] = fmaf(ds, kp[j], dqv[j]);
        add_key_grads(rw, i - 1, P, ds, qv, gv, dk_acc, dv_acc, sk, sv);
        L_p = s.L;
        F_p = F;
        a_p = a;
        g_p = g;
#pragma unroll
        for (int j = 0; j < NPL; ++j) kp[j] = kc[j];
    }
    {  // key t: only its left interval
        const float P = L_p;
        const float ds = scale * (P * (g_p - D) + F_p);
#pragma unroll
        for (int j = 0; j < NPL; ++j) dqv[j] = fmaf(ds, kp[j], dqv[j]);
        add_key_grads(rw, t, P, ds, qv, gv, dk_acc, dv_acc, sk, sv);
    }
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
        const int c = rw.lane + 32 * j;
        if (c < d) from_f32(dq + row * d + c, dqv[j]);
    }
    // the sink: trainable (mode 2), or array key 0 (mode 1), or constant
    if (mode == 0) return;
    float *tk = mode == 2 ? dk0 + (size_t)rw.h * d : dk_acc + (size_t)rw.bh * T * d;
    float *tv = mode == 2 ? dv0 + (size_t)rw.h * d : dv_acc + (size_t)rw.bh * T * d;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
        const int c = rw.lane + 32 * j;
        if (c < d) {
            atomicAdd(tk + c, sk[j]);
            atomicAdd(tv + c, sv[j]);
        }
    }
}

template <typename Tout>
__global__ void convert_kernel(const float *a, Tout *out, long long n) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) from_f32(out + i, a[i]);
}

template <typename Tin, int NPL>
cudaError_t launch_bwd(const Tin *q, const Tin *k, const Tin *v, const Tin *k0, const Tin *v0,
                       const Tin *o, const float *lse, const Tin *dout, Tin *dq, Tin *dk, Tin *dv,
                       float *dk0, float *dv0, float *ws, int B, int H, int T, int d, float scale,
                       int mode, cudaStream_t stream) {
    const long long n = (long long)B * H * T * d;
    float *dk_acc = ws, *dv_acc = ws + n;
    cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(float) * 2 * (size_t)n, stream);
    if (e != cudaSuccess) return e;
    if (mode == 2) {
        if ((e = cudaMemsetAsync(dk0, 0, sizeof(float) * (size_t)H * d, stream)) != cudaSuccess ||
            (e = cudaMemsetAsync(dv0, 0, sizeof(float) * (size_t)H * d, stream)) != cudaSuccess)
            return e;
    }
    const long long rows = (long long)B * H * T;
    simt_backward_kernel<Tin, NPL><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
        q, k, v, k0, v0, o, lse, dout, dq, dk_acc, dv_acc, dk0, dv0, B, H, T, d, scale, mode);
    const unsigned blocks = (unsigned)((n + 255) / 256);
    convert_kernel<Tin><<<blocks, 256, 0, stream>>>(dk_acc, dk, n);
    convert_kernel<Tin><<<blocks, 256, 0, stream>>>(dv_acc, dv, n);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_bwd_any(const Tin *q, const Tin *k, const Tin *v, const Tin *k0, const Tin *v0,
                           const Tin *o, const float *lse, const Tin *dout, Tin *dq, Tin *dk,
                           Tin *dv, float *dk0, float *dv0, float *ws, int B, int H, int T, int d,
                           float scale, int mode, cudaStream_t stream) {
#define CSA_BWD_LAUNCH(N)                                                                       \
    return launch_bwd<Tin, N>(q, k, v, k0, v0, o, lse, dout, dq, dk, dv, dk0, dv0, ws, B, H, T, \
                              d, scale, mode, stream)
    if (d <= 32) CSA_BWD_LAUNCH(1);
    if (d <= 64) CSA_BWD_LAUNCH(2);
    if (d <= 128) CSA_BWD_LAUNCH(4);
    CSA_BWD_LAUNCH(8);
#undef CSA_BWD_LAUNCH
}

}  // namespace

long long csa_simt_backward_scratch_bytes(int B, int H, int T, int d) {
    return 2LL * B * H * T * d * (long long)sizeof(float);
}

cudaError_t csa_simt_backward_f32(const float *q, const float *k, const float *v, const float *k0,
                                  const float *v0, const float *o, const float *lse,
                                  const float *dout, float *dq, float *dk, float *dv, float *dk0,
                                  float *dv0, void *scratch, int B, int H, int T, int d,
                                  float scale, int mode, cudaStream_t stream) {
    return launch_bwd_any<float>(q, k, v, k0, v0, o, lse, dout, dq, dk, dv, dk0, dv0,
                                 static_cast<float *>(scratch), B, H, T, d, scale, mode, stream);
}

cudaError_t csa_simt_backward_bf16(const void *q, const void *k, const void *v, const void *k0,
                                   const void *v0, const void *o, const float *lse,
                                   const void *dout, void *dq, void *dk, void *dv, float *dk0,
                                   float *dv0, void *scratch, int B, int H, int T, int d,
                                   float scale, int mode, cudaStream_t stream) {
    using bf = __nv_bfloat16;
    return launch_bwd_any<bf>(
        static_cast<const bf *>(q), static_cast<const bf *>(k), static_cast<const bf *>(v),
        static_cast<const bf *>(k0), static_cast<const bf *>(v0), static_cast<const bf *>(o), lse,
        static_cast<const bf *>(dout), static_cast<bf *>(dq), static_cast<bf *>(dk),
        static_cast<bf *>(dv), dk0, dv0, static_cast<float *>(scratch), B, H, T, d, scale, mode,
        stream);
}
