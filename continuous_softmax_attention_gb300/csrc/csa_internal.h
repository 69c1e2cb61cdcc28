// Launchers shared between the kernel translation units and the C ABI.
// Arguments are validated by the C ABI before any of these is called.
#pragma once

#include <cuda_runtime.h>

// Forms of the forward pass: eq. (10)/(11), the short-conv reading of
// eq. (13) (b replaced by its first-order term), eq. (12), eq. (2) over
// the symmetric interval [1/2, t + 1/2] (constant end half-cells, no sink),
// and eq. (10)/(11) evaluated in the log domain (z = a + b, then e^z).
enum { kFormExact = 0, kFormShortConv = 1, kFormStd = 2, kFormSymmetric = 3, kFormLogDomain = 4 };

// CUDA-core kernels (csa_simt.cu).
cudaError_t csa_simt_forward_f32(const float *q, const float *k, const float *v, const float *k0,
                                 const float *v0, float *out, float *lse, int B, int H, int T,
                                 int d, float scale, int mode, int form, cudaStream_t stream);
cudaError_t csa_simt_forward_bf16(const void *q, const void *k, const void *v, const void *k0,
                                  const void *v0, void *out, float *lse, int B, int H, int T,
                                  int d, float scale, int mode, int form, cudaStream_t stream);
cudaError_t csa_simt_logphi2_eval(const float *x, float *y, int n, cudaStream_t stream);

// Tensor-core kernels, d in {64, 128}, bf16.  Return a CSA_* status code
// (CSA_OK on success).  Continuous attention, form kFormExact,
// kFormShortConv, kFormSymmetric or kFormLogDomain (csa_tc.cu):
int csa_tc_forward(const void *q, const void *k, const void *v, const void *k0, const void *v0,
                   void *out, float *lse, int B, int H, int T, int d, float scale, int mode,
                   int form, cudaStream_t stream);
// The exact form with a planted delay in the epilogue (test hook): the
// softmax threads of column half delay_half sleep delay_ns before reading O.
int csa_tc_forward_delayed(const void *q, const void *k, const void *v, const void *k0,
                           const void *v0, void *out, float *lse, int B, int H, int T, int d,
                           float scale, int mode, unsigned delay_ns, int delay_half,
                           cudaStream_t stream);
// Standard causal attention, eq. (12) (csa_tc_std.cu):
int csa_tc_std_forward(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                       int H, int T, int d, float scale, cudaStream_t stream);
cudaError_t csa_tc_segment_weights_eval(const float *u0, const float *u1, float *right,
                                        float *left, int n, cudaStream_t stream);
cudaError_t csa_tc_selftest_wait_timeout(unsigned timeout_us, cudaStream_t stream);
// Read and clear the device status words of csa_tc.cu / csa_tc_std.cu on
// the current device.
int csa_tc_take_status(void);
int csa_tc_std_take_status(void);

// Decode step (csa_decode.cu), bf16, d in {64, 128, 256}.  Scratch holds
// the per-chunk partials; csa_decode_scratch_bytes gives its size (-1 for an
// unsupported d or a negative size).
long long csa_decode_scratch_bytes(int B, int H, int T, int d);
int csa_decode_run(const void *q, const void *k_cache, const void *v_cache, const void *k0,
                   const void *v0, const int *seqlens, void *out, float *lse, void *scratch, int B,
                   int H, int T, int d, float scale, int mode, cudaStream_t stream);
// The same for the owned positions [pos_lo, pos_hi) of each row only, from a
// cache shard holding rows [max(pos_lo - 2, 0), min(pos_hi, T)); o in fp32.
long long csa_decode_range_scratch_bytes(int B, int H, int pos_lo, int pos_hi, int d);
int csa_decode_range_run(const void *q, const void *k_shard, const void *v_shard, const void *k0,
                         const void *v0, const int *seqlens, float *out, float *lse,
                         void *scratch, int B, int H, int T, int d, float scale, int mode,
                         int pos_lo, int pos_hi, cudaStream_t stream);
// lse-weighted merge of R such partials ([R][B*H][d] and [R][B*H], fp32)
// into o (bf16) and lse.
int csa_decode_merge_ranges_run(const float *o_parts, const float *lse_parts, int R, int B, int H,
                                int d, void *out, float *lse, cudaStream_t stream);
int csa_decode_take_status(void);
// Address of the file-scope scratch array of csa_decode_noalloc on the
// current device (looked up once per device).
int csa_decode_noalloc_scratch(void **addr);

// Backward pass on CUDA cores (csa_bwd_simt.cu), any d <= 256.  scratch
// holds csa_simt_backward_scratch_bytes bytes (fp32 dk, dv accumulators).
long long csa_simt_backward_scratch_bytes(int B, int H, int T, int d);
cudaError_t csa_simt_backward_f32(const float *q, const float *k, const float *v, const float *k0,
                                  const float *v0, const float *o, const float *lse,
                                  const float *dout, float *dq, float *dk, float *dv, float *dk0,
                                  float *dv0, void *scratch, int B, int H, int T, int d,
                                  float scale, int mode, cudaStream_t stream);
cudaError_t csa_simt_backward_bf16(const void *q, const void *k, const void *v, const void *k0,
                                   const void *v0, const void *o, const float *lse,
                                   const void *dout, void *dq, void *dk, void *dv, float *dk0,
                                   float *dv0, void *scratch, int B, int H, int T, int d,
                                   float scale, int mode, cudaStream_t stream);

// Backward pass on the tensor cores (csa_tc_bwd.cu), bf16, d in {64, 128},
// all tensors 16-byte aligned.  scratch: csa_tc_backward_scratch_bytes bytes
// (fp32 dq accumulator and the per-row D = dout . out).  Returns a CSA_*
// status code.
long long csa_tc_backward_scratch_bytes(int B, int H, int T, int d);
int csa_tc_backward(const void *q, const void *k, const void *v, const void *k0, const void *v0,
                    const void *o, const float *lse, const void *dout, void *dq, void *dk,
                    void *dv, float *dk0, float *dv0, void *scratch, int B, int H, int T, int d,
                    float scale, int mode, cudaStream_t stream);
int csa_tc_backward_take_status(void);

// End-to-end forward from host buffers (csa_host.cu), pipelined over chunks
// of heads_per_chunk heads on three streams.  entry_wait: the copies wait for
// the work already queued on s_compute (false: the caller orders calls that
// share a workspace).
long long csa_host_scratch_bytes(int B, int H, int T, int d);
int csa_host_forward(const void *q_h, const void *k_h, const void *v_h, const void *k0,
                     const void *v0, void *out_h, float *lse_h, void *scratch, int B, int H, int T,
                     int d, float scale, int mode, int heads_per_chunk, bool entry_wait,
                     cudaStream_t s_compute, cudaStream_t s_h2d, cudaStream_t s_d2h);
