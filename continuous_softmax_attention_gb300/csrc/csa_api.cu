// C ABI of libcsa.so (declared in include/csa.h): argument validation and
// dispatch to the CUDA-core and tensor-core kernels.  No allocation, no
// host synchronisation on the compute entry points.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "csa.h"
#include "csa_internal.h"

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Common checks of the attention entry points.  Returns CSA_OK, or the
// error code; *empty is set when there is nothing to compute.
int check_common(const void *q, const void *k, const void *v, const void *k0, const void *v0,
                 const void *out, int B, int H, int T, int d, float scale, int mode, bool use_sink,
                 bool *empty) {
    *empty = false;
    if (B < 0 || H < 0 || T < 0 || d < 1) return CSA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return CSA_ERR_INVALID_ARG;
    if (use_sink && (mode < CSA_K0_ZERO || mode > CSA_K0_GIVEN)) return CSA_ERR_INVALID_ARG;
    if ((long long)B * H * T == 0) {
        *empty = true;
        return CSA_OK;
    }
    if (!q || !k || !v || !out) return CSA_ERR_INVALID_ARG;
    if (use_sink && mode == CSA_K0_GIVEN && (!k0 || !v0)) return CSA_ERR_INVALID_ARG;
    if ((long long)B * H > 0x7fffffffLL || (long long)B * H * T > (1LL << 40))
        return CSA_ERR_UNSUPPORTED;
    return CSA_OK;
}

int device_ok() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CSA_ERR_NO_DEVICE;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return CSA_ERR_NO_DEVICE;
    // The binary carries sm_103a code only.
    if (major != 10 || minor != 3) return CSA_ERR_NO_DEVICE;
    return CSA_OK;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

int forward_bf16(const void *q, const void *k, const void *v, const void *k0, const void *v0,
                 void *out, float *lse, int B, int H, int T, int d, float scale, int mode,
                 int form, csa_stream_t stream) {
    const bool continuous = form != kFormStd;
    bool empty;
    int rc = check_common(q, k, v, k0, v0, out, B, H, T, d, scale, mode, continuous, &empty);
    if (rc != CSA_OK || empty) return rc;
    if (d > 256) return CSA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
        (lse && !aligned(lse, 4)))
        return CSA_ERR_ALIGNMENT;
    if (continuous && mode == CSA_K0_GIVEN && (!aligned(k0, 2) || !aligned(v0, 2)))
        return CSA_ERR_ALIGNMENT;
    if ((rc = device_ok()) != CSA_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (d == 64 || d == 128) {
        if (continuous)
            return csa_tc_forward(q, k, v, k0, v0, out, lse, B, H, T, d, scale, mode, form, s);
        return csa_tc_std_forward(q, k, v, out, lse, B, H, T, d, scale, s);
    }
    // the CUDA-core kernel forms b in the log domain in its exact form
    return from_cuda(csa_simt_forward_bf16(q, k, v, k0, v0, out, lse, B, H, T, d, scale, mode,
                                           form == kFormLogDomain ? kFormExact : form, s));
}

int forward_f32(const float *q, const float *k, const float *v, const float *k0, const float *v0,
                float *out, float *lse, int B, int H, int T, int d, float scale, int mode,
                int form, csa_stream_t stream) {
    const bool continuous = form != kFormStd;
    bool empty;
    int rc = check_common(q, k, v, k0, v0, out, B, H, T, d, scale, mode, continuous, &empty);
    if (rc != CSA_OK || empty) return rc;
    if (d > 256) return CSA_ERR_UNSUPPORTED;
    if (!aligned(q, 4) || !aligned(k, 4) || !aligned(v, 4) || !aligned(out, 4) ||
        (lse && !aligned(lse, 4)))
        return CSA_ERR_ALIGNMENT;
    if ((rc = device_ok()) != CSA_OK) return rc;
    return from_cuda(csa_simt_forward_f32(q, k, v, k0, v0, out, lse, B, H, T, d, scale, mode,
                                          form, reinterpret_cast<cudaStream_t>(stream)));
}

// The checks of the decode step's arguments other than its workspace, in
// csa_decode's order.  Returns CSA_OK, or the error code; *empty is set when
// there is nothing to compute (B*H == 0).  On CSA_OK, *need holds the scratch
// bytes the sizes take.
int decode_check(const void *q, const void *k_cache, const void *v_cache, const void *k0,
                 const void *v0, const int *seqlens, const void *out, const float *lse, int B,
                 int H, int T, int d, float scale, int mode, bool *empty, long long *need) {
    *empty = false;
    if (B < 0 || H < 0 || T < 0 || d < 1) return CSA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return CSA_ERR_INVALID_ARG;
    if (mode < CSA_K0_ZERO || mode > CSA_K0_GIVEN) return CSA_ERR_INVALID_ARG;
    if (!(d == 64 || d == 128 || d == 256)) return CSA_ERR_UNSUPPORTED;
    if ((long long)B * H == 0) {
        *empty = true;
        return CSA_OK;
    }
    if (T == 0) return CSA_ERR_INVALID_ARG;  // the newest token's own key is in the cache
    if (T == INT_MAX) return CSA_ERR_UNSUPPORTED;  // positions 0..T must fit an int
    if (!q || !k_cache || !v_cache || !out) return CSA_ERR_INVALID_ARG;
    if (mode == CSA_K0_GIVEN && (!k0 || !v0)) return CSA_ERR_INVALID_ARG;
    if ((long long)B * H * T > (1LL << 40)) return CSA_ERR_UNSUPPORTED;
    *need = csa_decode_scratch_bytes(B, H, T, d);
    if (*need < 0) return CSA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        (lse && !aligned(lse, 4)) || (seqlens && !aligned(seqlens, 4)))
        return CSA_ERR_ALIGNMENT;
    if (mode == CSA_K0_GIVEN && (!aligned(k0, 16) || !aligned(v0, 16))) return CSA_ERR_ALIGNMENT;
    return CSA_OK;
}

int decode_bf16(const void *q, const void *k_cache, const void *v_cache, const void *k0,
                const void *v0, const int *seqlens, void *out, float *lse, void *workspace,
                long long workspace_bytes, int B, int H, int T, int d, float scale, int mode,
                csa_stream_t stream) {
    bool empty;
    long long need = 0;
    int rc = decode_check(q, k_cache, v_cache, k0, v0, seqlens, out, lse, B, H, T, d, scale, mode,
                          &empty, &need);
    if (rc != CSA_OK || empty) return rc;
    if (!workspace || workspace_bytes < need) return CSA_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return CSA_ERR_ALIGNMENT;
    if ((rc = device_ok()) != CSA_OK) return rc;
    return csa_decode_run(q, k_cache, v_cache, k0, v0, seqlens, out, lse, workspace, B, H, T, d,
                          scale, mode, reinterpret_cast<cudaStream_t>(stream));
}

int decode_range_bf16(const void *q, const void *k_shard, const void *v_shard, const void *k0,
                      const void *v0, const int *seqlens, float *out, float *lse,
                      void *workspace, long long workspace_bytes, int B, int H, int T, int d,
                      float scale, int mode, int pos_lo, int pos_hi, csa_stream_t stream) {
    if (B < 0 || H < 0 || T < 0 || d < 1) return CSA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return CSA_ERR_INVALID_ARG;
    if (mode < CSA_K0_ZERO || mode > CSA_K0_GIVEN) return CSA_ERR_INVALID_ARG;
    if (!(d == 64 || d == 128 || d == 256)) return CSA_ERR_UNSUPPORTED;
    // positions 0..T exist; a range may not start right after the sink
    if (pos_lo < 0 || pos_lo == 1 || pos_hi <= pos_lo || (long long)pos_hi > (long long)T + 1)
        return CSA_ERR_INVALID_ARG;
    if ((long long)B * H == 0) return CSA_OK;
    if (T == 0) return CSA_ERR_INVALID_ARG;
    if (!q || !k_shard || !v_shard || !out || !lse || !workspace) return CSA_ERR_INVALID_ARG;
    if (mode == CSA_K0_GIVEN && (!k0 || !v0)) return CSA_ERR_INVALID_ARG;
    if ((long long)B * H * T > (1LL << 40)) return CSA_ERR_UNSUPPORTED;
    const long long need = csa_decode_range_scratch_bytes(B, H, pos_lo, pos_hi, d);
    if (need < 0) return CSA_ERR_UNSUPPORTED;
    if (workspace_bytes < need) return CSA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_shard, 16) || !aligned(v_shard, 16) || !aligned(out, 16) ||
        !aligned(workspace, 16) || !aligned(lse, 4) || (seqlens && !aligned(seqlens, 4)))
        return CSA_ERR_ALIGNMENT;
    if (mode == CSA_K0_GIVEN && (!aligned(k0, 16) || !aligned(v0, 16))) return CSA_ERR_ALIGNMENT;
    int rc = device_ok();
    if (rc != CSA_OK) return rc;
    return csa_decode_range_run(q, k_shard, v_shard, k0, v0, seqlens, out, lse, workspace, B, H, T,
                                d, scale, mode, pos_lo, pos_hi,
                                reinterpret_cast<cudaStream_t>(stream));
}

long long backward_scratch_bytes(int B, int H, int T, int d) {
    if (B < 0 || H < 0 || T < 0 || d < 1 || d > 256) return -1;
    const long long a = csa_simt_backward_scratch_bytes(B, H, T, d);
    const long long b = csa_tc_backward_scratch_bytes(B, H, T, d);
    return a > b ? a : b;
}

int backward_any(const void *q, const void *k, const void *v, const void *k0, const void *v0,
                 const void *out, const float *lse, const void *dout, void *dq, void *dk,
                 void *dv, float *dk0, float *dv0, void *workspace, long long workspace_bytes,
                 int B, int H, int T, int d, float scale, int mode, bool bf16,
                 csa_stream_t stream) {
    bool empty;
    int rc = check_common(q, k, v, k0, v0, out, B, H, T, d, scale, mode, true, &empty);
    if (rc != CSA_OK) return rc;
    if (empty) {
        // nothing to differentiate; the sink gradients are zero
        if (mode == CSA_K0_GIVEN && (long long)H * d > 0) {
            if (!dk0 || !dv0) return CSA_ERR_INVALID_ARG;
            if ((rc = device_ok()) != CSA_OK) return rc;
            cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
            if (cudaMemsetAsync(dk0, 0, sizeof(float) * (size_t)H * d, s) != cudaSuccess ||
                cudaMemsetAsync(dv0, 0, sizeof(float) * (size_t)H * d, s) != cudaSuccess)
                return CSA_ERR_CUDA;
        }
        return CSA_OK;
    }
    if (!lse || !dout || !dq || !dk || !dv || !workspace) return CSA_ERR_INVALID_ARG;
    if (mode == CSA_K0_GIVEN && (!dk0 || !dv0)) return CSA_ERR_INVALID_ARG;
    if (d > 256) return CSA_ERR_UNSUPPORTED;
    const long long need = backward_scratch_bytes(B, H, T, d);
    if (need < 0) return CSA_ERR_UNSUPPORTED;
    if (workspace_bytes < need) return CSA_ERR_INVALID_ARG;
    const uintptr_t al = bf16 ? 2 : 4;
    if (!aligned(q, al) || !aligned(k, al) || !aligned(v, al) || !aligned(out, al) ||
        !aligned(dout, al) || !aligned(dq, al) || !aligned(dk, al) || !aligned(dv, al) ||
        !aligned(lse, 4) || !aligned(workspace, 16) ||
        (mode == CSA_K0_GIVEN && (!aligned(k0, al) || !aligned(v0, al) || !aligned(dk0, 4) ||
                                  !aligned(dv0, 4))))
        return CSA_ERR_ALIGNMENT;
    if ((rc = device_ok()) != CSA_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool tc_aligned = aligned(q, 16) && aligned(k, 16) && aligned(v, 16) &&
                            aligned(out, 16) && aligned(dout, 16) && aligned(dq, 16) &&
                            aligned(dk, 16) && aligned(dv, 16) &&
                            (mode != CSA_K0_GIVEN || (aligned(k0, 16) && aligned(v0, 16)));
    if (bf16 && (d == 64 || d == 128) && tc_aligned)
        return csa_tc_backward(q, k, v, k0, v0, out, lse, dout, dq, dk, dv, dk0, dv0, workspace,
                               B, H, T, d, scale, mode, s);
    if (bf16)
        return from_cuda(csa_simt_backward_bf16(q, k, v, k0, v0, out, lse, dout, dq, dk, dv, dk0,
                                                dv0, workspace, B, H, T, d, scale, mode, s));
    return from_cuda(csa_simt_backward_f32(
        static_cast<const float *>(q), static_cast<const float *>(k),
        static_cast<const float *>(v), static_cast<const float *>(k0),
        static_cast<const float *>(v0), static_cast<const float *>(out), lse,
        static_cast<const float *>(dout), static_cast<float *>(dq), static_cast<float *>(dk),
        static_cast<float *>(dv), dk0, dv0, workspace, B, H, T, d, scale, mode, s));
}

}  // namespace

extern "C" {

long long csa_backward_workspace_bytes(int B, int H, int T, int d) {
    return backward_scratch_bytes(B, H, T, d);
}

int csa_backward(const void *q, const void *k, const void *v, const void *k0, const void *v0,
                 const void *out, const float *lse, const void *dout, void *dq, void *dk,
                 void *dv, float *dk0, float *dv0, void *workspace, long long workspace_bytes,
                 int B, int H, int T, int d, float scale, int k0_mode, csa_stream_t stream) {
    return backward_any(q, k, v, k0, v0, out, lse, dout, dq, dk, dv, dk0, dv0, workspace,
                        workspace_bytes, B, H, T, d, scale, k0_mode, true, stream);
}

int csa_backward_f32(const float *q, const float *k, const float *v, const float *k0,
                     const float *v0, const float *out, const float *lse, const float *dout,
                     float *dq, float *dk, float *dv, float *dk0, float *dv0, void *workspace,
                     long long workspace_bytes, int B, int H, int T, int d, float scale,
                     int k0_mode, csa_stream_t stream) {
    return backward_any(q, k, v, k0, v0, out, lse, dout, dq, dk, dv, dk0, dv0, workspace,
                        workspace_bytes, B, H, T, d, scale, k0_mode, false, stream);
}

long long csa_forward_host_workspace_bytes(int B, int H, int T, int d) {
    if (d > 256) return -1;
    return csa_host_scratch_bytes(B, H, T, d);
}

int csa_forward_host_ex(const void *q, const void *k, const void *v, const void *k0,
                        const void *v0, void *out, float *lse, void *workspace,
                        long long workspace_bytes, int B, int H, int T, int d, float scale,
                        int k0_mode, int heads_per_chunk, unsigned flags, csa_stream_t stream,
                        csa_stream_t stream_h2d, csa_stream_t stream_d2h) {
    if (flags & ~CSA_HOST_NO_ENTRY_WAIT) return CSA_ERR_INVALID_ARG;
    bool empty;
    int rc = check_common(q, k, v, k0, v0, out, B, H, T, d, scale, k0_mode, true, &empty);
    if (rc != CSA_OK || empty) return rc;
    if (d > 256) return CSA_ERR_UNSUPPORTED;
    if (heads_per_chunk < 1 || heads_per_chunk > H || H % heads_per_chunk != 0)
        return CSA_ERR_INVALID_ARG;
    if (!workspace) return CSA_ERR_INVALID_ARG;
    const long long need = csa_host_scratch_bytes(B, H, T, d);
    if (need < 0 || workspace_bytes < need) return CSA_ERR_INVALID_ARG;
    if (!aligned(workspace, 256) || (lse && !aligned(lse, 4))) return CSA_ERR_ALIGNMENT;
    if (k0_mode == CSA_K0_GIVEN && (!aligned(k0, 2) || !aligned(v0, 2))) return CSA_ERR_ALIGNMENT;
    if ((rc = device_ok()) != CSA_OK) return rc;
    return csa_host_forward(q, k, v, k0, v0, out, lse, workspace, B, H, T, d, scale, k0_mode,
                            heads_per_chunk, !(flags & CSA_HOST_NO_ENTRY_WAIT),
                            reinterpret_cast<cudaStream_t>(stream),
                            reinterpret_cast<cudaStream_t>(stream_h2d),
                            reinterpret_cast<cudaStream_t>(stream_d2h));
}

int csa_forward_host(const void *q, const void *k, const void *v, const void *k0, const void *v0,
                     void *out, float *lse, void *workspace, long long workspace_bytes, int B,
                     int H, int T, int d, float scale, int k0_mode, int heads_per_chunk,
                     csa_stream_t stream, csa_stream_t stream_h2d, csa_stream_t stream_d2h) {
    return csa_forward_host_ex(q, k, v, k0, v0, out, lse, workspace, workspace_bytes, B, H, T, d,
                               scale, k0_mode, heads_per_chunk, 0u, stream, stream_h2d,
                               stream_d2h);
}

long long csa_decode_range_workspace_bytes(int B, int H, int pos_lo, int pos_hi, int d) {
    return csa_decode_range_scratch_bytes(B, H, pos_lo, pos_hi, d);
}

int csa_decode_range(const void *q, const void *k_shard, const void *v_shard, const void *k0,
                     const void *v0, const int *seqlens, float *out, float *lse, void *workspace,
                     long long workspace_bytes, int B, int H, int T, int d, float scale,
                     int k0_mode, int pos_lo, int pos_hi, csa_stream_t stream) {
    return decode_range_bf16(q, k_shard, v_shard, k0, v0, seqlens, out, lse, workspace,
                             workspace_bytes, B, H, T, d, scale, k0_mode, pos_lo, pos_hi, stream);
}

int csa_decode_merge_ranges(const float *o_parts, const float *lse_parts, int R, int B, int H,
                            int d, void *out, float *lse, csa_stream_t stream) {
    if (R < 1 || B < 0 || H < 0 || d < 1 || d > 256) return CSA_ERR_INVALID_ARG;
    if ((long long)B * H == 0) return CSA_OK;
    if (!o_parts || !lse_parts || !out) return CSA_ERR_INVALID_ARG;
    if ((long long)R * B * H * d > (1LL << 40)) return CSA_ERR_UNSUPPORTED;
    if (!aligned(o_parts, 4) || !aligned(lse_parts, 4) || !aligned(out, 2) || (lse && !aligned(lse, 4)))
        return CSA_ERR_ALIGNMENT;
    int rc = device_ok();
    if (rc != CSA_OK) return rc;
    return csa_decode_merge_ranges_run(o_parts, lse_parts, R, B, H, d, out, lse,
                                       reinterpret_cast<cudaStream_t>(stream));
}

long long csa_decode_workspace_bytes(int B, int H, int T, int d) {
    return csa_decode_scratch_bytes(B, H, T, d);
}

int csa_decode(const void *q, const void *k_cache, const void *v_cache, const void *k0,
               const void *v0, const int *seqlens, void *out, float *lse, void *workspace,
               long long workspace_bytes, int B, int H, int T, int d, float scale, int k0_mode,
               csa_stream_t stream) {
    return decode_bf16(q, k_cache, v_cache, k0, v0, seqlens, out, lse, workspace,
                       workspace_bytes, B, H, T, d, scale, k0_mode, stream);
}

int csa_forward(const void *q, const void *k, const void *v, const void *k0, const void *v0,
                void *out, float *lse, int B, int H, int T, int d, float scale, int k0_mode,
                csa_stream_t stream) {
    return forward_bf16(q, k, v, k0, v0, out, lse, B, H, T, d, scale, k0_mode, kFormExact, stream);
}

int csa_forward_short_conv(const void *q, const void *k, const void *v, const void *k0,
                           const void *v0, void *out, float *lse, int B, int H, int T, int d,
                           float scale, int k0_mode, csa_stream_t stream) {
    return forward_bf16(q, k, v, k0, v0, out, lse, B, H, T, d, scale, k0_mode, kFormShortConv,
                        stream);
}

int csa_forward_logdomain(const void *q, const void *k, const void *v, const void *k0,
                          const void *v0, void *out, float *lse, int B, int H, int T, int d,
                          float scale, int k0_mode, csa_stream_t stream) {
    return forward_bf16(q, k, v, k0, v0, out, lse, B, H, T, d, scale, k0_mode, kFormLogDomain,
                        stream);
}

int csa_forward_symmetric(const void *q, const void *k, const void *v, void *out, float *lse,
                          int B, int H, int T, int d, float scale, csa_stream_t stream) {
    return forward_bf16(q, k, v, nullptr, nullptr, out, lse, B, H, T, d, scale, CSA_K0_ZERO,
                        kFormSymmetric, stream);
}

int csa_forward_symmetric_f32(const float *q, const float *k, const float *v, float *out,
                              float *lse, int B, int H, int T, int d, float scale,
                              csa_stream_t stream) {
    return forward_f32(q, k, v, nullptr, nullptr, out, lse, B, H, T, d, scale, CSA_K0_ZERO,
                       kFormSymmetric, stream);
}

int csa_forward_short_conv_f32(const float *q, const float *k, const float *v, const float *k0,
                               const float *v0, float *out, float *lse, int B, int H, int T,
                               int d, float scale, int k0_mode, csa_stream_t stream) {
    return forward_f32(q, k, v, k0, v0, out, lse, B, H, T, d, scale, k0_mode, kFormShortConv,
                       stream);
}

int csa_forward_f32(const float *q, const float *k, const float *v, const float *k0,
                    const float *v0, float *out, float *lse, int B, int H, int T, int d,
                    float scale, int k0_mode, csa_stream_t stream) {
    return forward_f32(q, k, v, k0, v0, out, lse, B, H, T, d, scale, k0_mode, kFormExact, stream);
}

int csa_std_forward(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                    int H, int T, int d, float scale, csa_stream_t stream) {
    return forward_bf16(q, k, v, nullptr, nullptr, out, lse, B, H, T, d, scale, CSA_K0_ZERO,
                        kFormStd, stream);
}

int csa_std_forward_f32(const float *q, const float *k, const float *v, float *out, float *lse,
                        int B, int H, int T, int d, float scale, csa_stream_t stream) {
    return forward_f32(q, k, v, nullptr, nullptr, out, lse, B, H, T, d, scale, CSA_K0_ZERO,
                       kFormStd, stream);
}

int csa_logphi2_eval(const float *x, float *y, int n, csa_stream_t stream) {
    if (n < 0) return CSA_ERR_INVALID_ARG;
    if (n == 0) return CSA_OK;
    if (!x || !y) return CSA_ERR_INVALID_ARG;
    int rc = device_ok();
    if (rc != CSA_OK) return rc;
    return from_cuda(csa_simt_logphi2_eval(x, y, n, reinterpret_cast<cudaStream_t>(stream)));
}

int csa_segment_weights_eval(const float *u0, const float *u1, float *right, float *left, int n,
                             csa_stream_t stream) {
    if (n < 0) return CSA_ERR_INVALID_ARG;
    if (n == 0) return CSA_OK;
    if (!u0 || !u1 || !right || !left) return CSA_ERR_INVALID_ARG;
    int rc = device_ok();
    if (rc != CSA_OK) return rc;
    return from_cuda(csa_tc_segment_weights_eval(u0, u1, right, left, n,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

int csa_device_status(void) {
    int rc = device_ok();
    if (rc != CSA_OK) return rc;
    const int a = csa_tc_take_status();
    const int b = csa_tc_std_take_status();
    const int c = csa_decode_take_status();
    const int e = csa_tc_backward_take_status();
    return a != CSA_OK ? a : b != CSA_OK ? b : c != CSA_OK ? c : e;
}

int csa_selftest_wait_timeout(unsigned timeout_us, csa_stream_t stream) {
    if (timeout_us < 1 || timeout_us > 1000000u) return CSA_ERR_INVALID_ARG;
    int rc = device_ok();
    if (rc != CSA_OK) return rc;
    return from_cuda(csa_tc_selftest_wait_timeout(timeout_us, reinterpret_cast<cudaStream_t>(stream)));
}

int csa_selftest_forward_delay(const void *q, const void *k, const void *v, const void *k0,
                               const void *v0, void *out, float *lse, int B, int H, int T, int d,
                               float scale, int k0_mode, unsigned delay_ns, int delay_half,
                               csa_stream_t stream) {
    if (delay_ns > 1000000u || (delay_half != 0 && delay_half != 1)) return CSA_ERR_INVALID_ARG;
    bool empty;
    int rc = check_common(q, k, v, k0, v0, out, B, H, T, d, scale, k0_mode, true, &empty);
    if (rc != CSA_OK || empty) return rc;
    if (d != 64 && d != 128) return CSA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
        (lse && !aligned(lse, 4)))
        return CSA_ERR_ALIGNMENT;
    if (k0_mode == CSA_K0_GIVEN && (!aligned(k0, 2) || !aligned(v0, 2))) return CSA_ERR_ALIGNMENT;
    if ((rc = device_ok()) != CSA_OK) return rc;
    return csa_tc_forward_delayed(q, k, v, k0, v0, out, lse, B, H, T, d, scale, k0_mode, delay_ns,
                                  delay_half, reinterpret_cast<cudaStream_t>(stream));
}

int csa_decode_noalloc(const void *q, const void *k_cache, const void *v_cache, const void *k0,
                       const void *v0, const int *seqlens, void *out, float *lse, int B, int H,
                       int T, int d, float scale, int k0_mode, csa_stream_t stream) {
    // csa_decode's checks first, in its order; then the scratch capacity
    bool empty;
    long long need = 0;
    int rc = decode_check(q, k_cache, v_cache, k0, v0, seqlens, out, lse, B, H, T, d, scale,
                          k0_mode, &empty, &need);
    if (rc != CSA_OK || empty) return rc;
    if (need > (long long)CSA_DECODE_NOALLOC_SCRATCH_BYTES) return CSA_ERR_UNSUPPORTED;
    if ((rc = device_ok()) != CSA_OK) return rc;
    void *scratch = nullptr;
    if ((rc = csa_decode_noalloc_scratch(&scratch)) != CSA_OK) return rc;
    return csa_decode_run(q, k_cache, v_cache, k0, v0, seqlens, out, lse, scratch, B, H, T, d,
                          scale, k0_mode, reinterpret_cast<cudaStream_t>(stream));
}

const char *csa_status_string(int status) {
    switch (status) {
        case CSA_OK: return "ok";
        case CSA_ERR_INVALID_ARG: return "invalid argument";
        case CSA_ERR_UNSUPPORTED: return "unsupported shape or value";
        case CSA_ERR_ALIGNMENT: return "misaligned pointer";
        case CSA_ERR_CUDA: return "CUDA runtime error";
        case CSA_ERR_TIMEOUT: return "device-side wait timed out";
        case CSA_ERR_NO_DEVICE: return "no sm_103 device is current";
        default: return "unknown status";
    }
}

int csa_abi_version(void) { return CSA_ABI_VERSION; }

}  // extern "C"
