// CUDA-core kernels: continuous attention (eq. (10)/(11) of Jianlin Su,
// "Continuous Softmax Attention"), its short-conv reading (b replaced by the
// first-order term of eq. (13)) and standard causal attention (eq. (12)),
// for fp32 inputs and for bf16 inputs whose head dimension the tensor-core
// kernel does not cover.
//
// One warp owns one query row.  Lanes split the head dimension (element
// c = lane + 32*j), a key's logit is a warp-wide sum, and the row walks its
// keys in order with a one-key lookahead, because b_{t,i} needs the logits of
// both neighbours.  The correction is formed in the log domain:
//     z_i = a_i + log(phi2(a_{i-1} - a_i) + phi2(a_{i+1} - a_i))
// with a stable log phi2 and logaddexp, and z enters an online softmax
// (running max and sum, the running output rescaled when the max grows).
// Everything is fp32 with accurate (non-intrinsic) exp/log.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "csa_internal.h"

namespace {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f32(float *p, float x) { *p = x; }
__device__ __forceinline__ void from_f32(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// log phi2(x), phi2(x) = (e^x - 1 - x)/x^2 (eq. (6)), in fp32.
//  |x| <= 1 : log(1/2) + log1p(sum_{n>=1} 2 x^n / (n+2)!), the power series
//             of the integral definition; ten terms leave < 4e-10 at |x| = 1.
//  x > 1    : log phi2 = x + log1p(-(1+x) e^{-x}) - 2 log x   (no overflow)
//  x < -1   : log phi2 = log(e^x - 1 - x) - 2 log(-x), with e^x - 1 computed
//             by expm1f.
__device__ __forceinline__ float log_phi2_f32(float x) {
    const float ax = fabsf(x);
    if (ax <= 1.0f) {
        // 2/(n+2)! for n = 10 .. 1
        float s = 2.0f / 479001600.0f;
        s = fmaf(s, x, 2.0f / 39916800.0f);
        s = fmaf(s, x, 2.0f / 3628800.0f);
        s = fmaf(s, x, 2.0f / 362880.0f);
        s = fmaf(s, x, 2.0f / 40320.0f);
        s = fmaf(s, x, 2.0f / 5040.0f);
        s = fmaf(s, x, 2.0f / 720.0f);
        s = fmaf(s, x, 2.0f / 120.0f);
        s = fmaf(s, x, 2.0f / 24.0f);
        s = fmaf(s, x, 2.0f / 6.0f);
        s = s * x;
        return log1pf(s) - 0.69314718055994531f;
    }
    if (x > 0.0f) return x + log1pf(-(1.0f + x) * expf(-x)) - 2.0f * logf(x);
    return logf(expm1f(x) - x) - 2.0f * logf(-x);
}

__device__ __forceinline__ float logaddexp_f32(float a, float b) {
    const float hi = fmaxf(a, b), lo = fminf(a, b);
    return hi + log1pf(expf(lo - hi));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Online softmax state of one row, distributed over the warp: every lane
// holds the same m, l and its own NPL output elements.
template <int NPL>
struct RowAcc {
    float m = -INFINITY, l = 0.0f;
    float acc[NPL];
    __device__ RowAcc() {
#pragma unroll
        for (int j = 0; j < NPL; ++j) acc[j] = 0.0f;
    }
    __device__ void add(float z, const float (&v)[NPL]) {
        if (z > m) {
            const float a = expf(m - z);  // 0 when m = -inf
#pragma unroll
            for (int j = 0; j < NPL; ++j) acc[j] = fmaf(acc[j], a, v[j]);
            l = fmaf(l, a, 1.0f);
            m = z;
        } else {
            const float w = expf(z - m);
#pragma unroll
            for (int j = 0; j < NPL; ++j) acc[j] = fmaf(w, v[j], acc[j]);
            l += w;
        }
    }
};

template <typename Tin, int NPL>
struct RowIO {
    const Tin *q, *k, *v, *k0, *v0;
    int T, d, mode;
    long long bh;
    int h;
    int lane;
    float qv[NPL];

    // Key/value row i of the extended sequence: 0 = the sink, i >= 1 = array
    // row i - 1.  Returns nullptr for the all-zero sink.
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
    __device__ float logit(const Tin *kr, float scale) const {
        float s = 0.0f;
        if (kr) {
#pragma unroll
            for (int j = 0; j < NPL; ++j) {
                const int c = lane + 32 * j;
                if (c < d) s = fmaf(qv[j], to_f32(kr[c]), s);
            }
        }
        return scale * warp_sum(s);
    }
    __device__ void load_val(const Tin *vr, float (&out)[NPL]) const {
#pragma unroll
        for (int j = 0; j < NPL; ++j) {
            const int c = lane + 32 * j;
            out[j] = (vr && c < d) ? to_f32(vr[c]) : 0.0f;
        }
    }
};

// grid: one warp per (b, h, row); rows handed out longest first.
// FORM: 0 eq. (10)/(11), 1 the short-conv reading of eq. (13), 2 eq. (12),
// 3 the symmetric interval [1/2, t + 1/2] (constant end half-cells, no sink).
template <typename Tin, int NPL, int FORM>
__global__ void __launch_bounds__(256) simt_forward_kernel(const Tin *q, const Tin *k,
                                                           const Tin *v, const Tin *k0,
                                                           const Tin *v0, Tin *out, float *lse,
                                                           int B, int H, int T, int d, float scale,
                                                           int mode) {
    const long long BH = (long long)B * H;
    const long long gw = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (gw >= BH * T) return;
    const int r = T - 1 - (int)(gw / BH);
    RowIO<Tin, NPL> io;
    io.q = q; io.k = k; io.v = v; io.k0 = k0; io.v0 = v0;
    io.T = T; io.d = d; io.mode = mode;
    io.bh = gw % BH;
    io.h = (int)(io.bh % H);
    io.lane = threadIdx.x & 31;
    const Tin *qr = q + ((size_t)io.bh * T + (size_t)r) * d;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
        const int c = io.lane + 32 * j;
        io.qv[j] = c < d ? to_f32(qr[c]) : 0.0f;
    }
    RowAcc<NPL> acc;
    float vv[NPL];
    const int t = r + 1;  // the page's token index
    if (FORM != 2) {
        // keys i = 0..t with b from eq. (10), or its first-order term
        float a_prev = 0.0f;
        float a_cur = io.logit(io.key(0), scale);
        float a_next = io.logit(io.key(1), scale);
        for (int i = 0; i <= t; ++i) {
            float b;
            if (FORM == 3) {
                // e^{b_i} = (i == 1 ? 1/2 : phi2(a_{i-1} - a_i)) + (i == t ? 1/2 : phi2(a_{i+1} - a_i));
                // the sink takes no part
                constexpr float kLogHalf = -0.69314718055994531f;
                if (i == 0) {
                    a_prev = a_cur;
                    a_cur = a_next;
                    if (i + 2 <= t) a_next = io.logit(io.key(i + 2), scale);
                    continue;
                }
                const float lb = i == 1 ? kLogHalf : log_phi2_f32(a_prev - a_cur);
                const float rb = i == t ? kLogHalf : log_phi2_f32(a_next - a_cur);
                b = logaddexp_f32(lb, rb);
            } else if (FORM == 1) {
                // log phi2(x) = -log 2 + x/3 + ..; log(phi2(x) + phi2(y)) = (x + y)/6 + ..
                constexpr float kLn2f = 0.69314718055994531f;
                if (i == 0)
                    b = (a_next - a_cur) * (1.0f / 3.0f) - kLn2f;
                else if (i == t)
                    b = (a_prev - a_cur) * (1.0f / 3.0f) - kLn2f;
                else
                    b = (a_prev + a_next - 2.0f * a_cur) * (1.0f / 6.0f);
            } else if (i == 0) {
                b = log_phi2_f32(a_next - a_cur);
            } else if (i == t) {
                b = log_phi2_f32(a_prev - a_cur);
            } else {
                b = logaddexp_f32(log_phi2_f32(a_prev - a_cur), log_phi2_f32(a_next - a_cur));
            }
            io.load_val(io.val(i), vv);
            acc.add(a_cur + b, vv);
            a_prev = a_cur;
            a_cur = a_next;
            if (i + 2 <= t) a_next = io.logit(io.key(i + 2), scale);
        }
    } else {
        // eq. (12): keys i = 1..t, no correction, no sink
        for (int i = 1; i <= t; ++i) {
            const float a = io.logit(io.key(i), scale);
            io.load_val(io.val(i), vv);
            acc.add(a, vv);
        }
    }
    const float inv = 1.0f / acc.l;
    Tin *orow = out + ((size_t)io.bh * T + (size_t)r) * d;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
        const int c = io.lane + 32 * j;
        if (c < d) from_f32(orow + c, acc.acc[j] * inv);
    }
    if (lse && io.lane == 0) lse[(size_t)io.bh * T + (size_t)r] = acc.m + logf(acc.l);
}

__global__ void logphi2_eval_kernel(const float *x, float *y, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) y[i] = log_phi2_f32(x[i]);
}

template <typename Tin, int FORM, int NPL>
cudaError_t launch_npl(const Tin *q, const Tin *k, const Tin *v, const Tin *k0, const Tin *v0,
                       Tin *out, float *lse, int B, int H, int T, int d, float scale, int mode,
                       cudaStream_t stream) {
    const long long rows = (long long)B * H * T;
    const int threads = 256;
    const long long blocks = (rows + 7) / 8;
    simt_forward_kernel<Tin, NPL, FORM><<<(unsigned)blocks, threads, 0, stream>>>(
        q, k, v, k0, v0, out, lse, B, H, T, d, scale, mode);
    return cudaGetLastError();
}

template <typename Tin, int FORM>
cudaError_t launch_any(const Tin *q, const Tin *k, const Tin *v, const Tin *k0, const Tin *v0,
                       Tin *out, float *lse, int B, int H, int T, int d, float scale, int mode,
                       cudaStream_t stream) {
    if (d <= 32) return launch_npl<Tin, FORM, 1>(q, k, v, k0, v0, out, lse, B, H, T, d, scale, mode, stream);
    if (d <= 64) return launch_npl<Tin, FORM, 2>(q, k, v, k0, v0, out, lse, B, H, T, d, scale, mode, stream);
    if (d <= 128) return launch_npl<Tin, FORM, 4>(q, k, v, k0, v0, out, lse, B, H, T, d, scale, mode, stream);
    return launch_npl<Tin, FORM, 8>(q, k, v, k0, v0, out, lse, B, H, T, d, scale, mode, stream);
}

}  // namespace

cudaError_t csa_simt_forward_f32(const float *q, const float *k, const float *v, const float *k0,
                                 const float *v0, float *out, float *lse, int B, int H, int T,
                                 int d, float scale, int mode, int form,
                                 cudaStream_t stream) {
    if (form == 0)
        return launch_any<float, 0>(q, k, v, k0, v0, out, lse, B, H, T, d, scale, mode, stream);
    if (form == 1)
        return launch_any<float, 1>(q, k, v, k0, v0, out, lse, B, H, T, d, scale, mode, stream);
    if (form == 3)
        return launch_any<float, 3>(q, k, v, k0, v0, out, lse, B, H, T, d, scale, 0, stream);
    return launch_any<float, 2>(q, k, v, k0, v0, out, lse, B, H, T, d, scale, mode, stream);
}

cudaError_t csa_simt_forward_bf16(const void *q, const void *k, const void *v, const void *k0,
                                  const void *v0, void *out, float *lse, int B, int H, int T,
                                  int d, float scale, int mode, int form,
                                  cudaStream_t stream) {
    using bf = __nv_bfloat16;
    const bf *q_ = static_cast<const bf *>(q), *k_ = static_cast<const bf *>(k);
    const bf *v_ = static_cast<const bf *>(v), *k0_ = static_cast<const bf *>(k0);
    const bf *v0_ = static_cast<const bf *>(v0);
    bf *o_ = static_cast<bf *>(out);
    if (form == 0)
        return launch_any<bf, 0>(q_, k_, v_, k0_, v0_, o_, lse, B, H, T, d, scale, mode, stream);
    if (form == 1)
        return launch_any<bf, 1>(q_, k_, v_, k0_, v0_, o_, lse, B, H, T, d, scale, mode, stream);
    if (form == 3)
        return launch_any<bf, 3>(q_, k_, v_, k0_, v0_, o_, lse, B, H, T, d, scale, 0, stream);
    return launch_any<bf, 2>(q_, k_, v_, k0_, v0_, o_, lse, B, H, T, d, scale, mode, stream);
}

cudaError_t csa_simt_logphi2_eval(const float *x, float *y, int n, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    logphi2_eval_kernel<<<(n + 255) / 256, 256, 0, stream>>>(x, y, n);
    return cudaGetLastError();
}
