/*
 * csa.h - C ABI of libcsa.so: forward pass of causal Continuous Softmax
 * Attention on one NVIDIA GB300 (sm_103a).
 *
 * The method: Jianlin Su, "Continuous Softmax Attention" (Scientific Spaces
 * #11980).  Attention over the causal prefix is made continuous by linear
 * interpolation of keys and values between integer positions (eq. (2), (3));
 * the integrals close (eq. (4)-(7)) and reduce to a softmax over corrected
 * logits (eq. (10), (11)):
 *
 *     a_{t,i} = scale * q_t . k_i                       i = 0..t
 *     e^{b_{t,0}} = phi2(a_{t,1} - a_{t,0})
 *     e^{b_{t,i}} = phi2(a_{t,i-1} - a_{t,i}) + phi2(a_{t,i+1} - a_{t,i})
 *     e^{b_{t,t}} = phi2(a_{t,t-1} - a_{t,t})
 *     o_t = sum_i e^{a+b} v_i / sum_i e^{a+b},   phi2(x) = (e^x - 1 - x)/x^2
 *
 * with an extra sink pair k_0, v_0 (section "Analysis of the Result": zero,
 * a copy of the first token, or trainable).
 *
 * Common conventions for every attention entry point below
 * ---------------------------------------------------------
 *  Layout     q, k, v, out: contiguous row-major [B, H, T, d]; token r of the
 *             arrays (0-based) is the page's t = r + 1, array key j is the
 *             page's k_{j+1}.  k0, v0: contiguous [H, d] (one sink pair per
 *             head, shared across the batch).  lse: contiguous float [B, H, T].
 *  Memory     every pointer is DEVICE memory owned by the caller; the library
 *             allocates nothing and keeps no pointer after the call returns.
 *             out and lse must not overlap any input.
 *  Scheduling the tensor-core forward kernels (csa_forward, its short-conv and
 *             symmetric forms, and the kernels csa_forward_host launches)
 *             run one CTA per SM and take query tiles from a counter in the
 *             library's device image: 64 counter slots per device, drawn in
 *             turn.  Each slot has one CUDA event, created on first use and
 *             kept for the life of the process; a launch's stream waits on
 *             its slot's event (the slot's previous launch), so calls on any
 *             streams never share a counter.  Under stream capture the event
 *             is left out: a captured graph keeps the slot it drew, so a
 *             replay must not run at the same time as another replay of the
 *             same graph, nor as a later call that draws the same slot (every
 *             64th forward call on the device).
 *  Stream     the work is enqueued on `stream` (a cudaStream_t; NULL = the
 *             legacy default stream) and the call returns without waiting.
 *             Outputs are valid once the stream reaches that point.
 *  Scale      logits are scale * q.k; the correction b is formed on the
 *             scaled logits.  scale must be finite.
 *  lse        natural-log normaliser: lse_t = log sum_i e^{a_{t,i}+b_{t,i}},
 *             which equals log of eq. (2)'s denominator integral.  May be
 *             NULL when not wanted.
 *  Empty      B, H or T equal to 0 is a valid empty problem: CSA_OK, nothing
 *             is launched.
 *  Errors     the return value is CSA_OK (0) or one of the negative codes
 *             below.  Argument errors are detected on the host before any
 *             launch, and nothing is enqueued.  CSA_ERR_CUDA reports a launch
 *             failure (cudaGetLastError); asynchronous kernel faults surface,
 *             as usual in CUDA, on the next synchronising call.  Device-side
 *             bounded waits that expire set a sticky status word readable
 *             with csa_device_status().
 */
#ifndef CSA_H_
#define CSA_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle type as cudaStream_t / CUstream. */
typedef struct CUstream_st *csa_stream_t;

/* Choice of the extra pair k_0, v_0 ("Analysis of the Result", last
 * paragraph: all zeros; k_0 = k_1, v_0 = v_1; or trainable). */
typedef enum {
    CSA_K0_ZERO = 0,       /* k_0 = v_0 = 0 (the page's experiments)       */
    CSA_K0_COPY_FIRST = 1, /* k_0 = k_1, v_0 = v_1 of the same (b, h)       */
    CSA_K0_GIVEN = 2       /* k0, v0 supplied per head, [H, d]              */
} csa_k0_mode;

enum {
    CSA_OK = 0,
    CSA_ERR_INVALID_ARG = -1, /* NULL pointer, negative size, d < 1,
                                 non-finite scale, bad mode, k0/v0 NULL in
                                 CSA_K0_GIVEN                                 */
    CSA_ERR_UNSUPPORTED = -2, /* shape or value outside what a kernel
                                 supports (see each entry point)              */
    CSA_ERR_ALIGNMENT = -3,   /* a pointer is not aligned as required         */
    CSA_ERR_CUDA = -4,        /* a CUDA runtime call or launch failed         */
    CSA_ERR_TIMEOUT = -5,     /* a device-side bounded wait expired           */
    CSA_ERR_NO_DEVICE = -6    /* no usable sm_103 device is current           */
};

/*
 * csa_forward - continuous attention, bf16 inputs, tensor-core path.
 *   Defines: eq. (10)/(11) of "Continuous Softmax Attention" ("Assembly and
 *   Simplification"), which equals eq. (2) ("Problem Statement").
 *   q, k, v, k0, v0: bf16 (__nv_bfloat16); out: bf16; lse: float.
 *   Accumulation and the correction b are computed in fp32.
 *   d = 64 or 128 runs the tcgen05/TMA kernel; any other 1 <= d <= 256 runs
 *   the CUDA-core kernel.  d > 256: CSA_ERR_UNSUPPORTED.  Any finite scale,
 *   of either sign, on both kernels.
 *   q, k, v, out must be 16-byte aligned (CSA_ERR_ALIGNMENT otherwise).
 *   k0, v0 are read only in CSA_K0_GIVEN mode and may be NULL otherwise.
 */
int csa_forward(const void *q, const void *k, const void *v, const void *k0, const void *v0,
                void *out, float *lse, int B, int H, int T, int d, float scale, int k0_mode,
                csa_stream_t stream);

/*
 * csa_forward_f32 - continuous attention, fp32 inputs and outputs, computed
 *   in fp32 on CUDA cores (no TF32), with b formed in the log domain by a
 *   stable log phi2 (series near 0, logarithmic form for large |x|, combined
 *   by logaddexp).  Same definition and conventions as csa_forward;
 *   1 <= d <= 256.  All pointers 4-byte aligned.
 */
int csa_forward_f32(const float *q, const float *k, const float *v, const float *k0,
                    const float *v0, float *out, float *lse, int B, int H, int T, int d,
                    float scale, int k0_mode, csa_stream_t stream);

/*
 * csa_forward_host - csa_forward from HOST buffers, end to end: copies q, k,
 *   v to the device, runs the forward pass and copies out and lse back,
 *   overlapping the copies of one chunk of heads with the kernel of another
 *   (the (b, h) problems are independent).  Same definition, result and
 *   d rules as csa_forward.
 *   q, k, v, out: HOST bf16 [B, H, T, d]; lse: HOST float [B, H, T] or NULL.
 *   They should be page-locked (cudaHostAlloc / cudaHostRegister): pageable
 *   memory is still correct but the copies then do not overlap.  The host
 *   inputs must stay unchanged, and out/lse must not be read, until the work
 *   completes on `stream`.
 *   k0, v0: DEVICE bf16 [H, d] (CSA_K0_GIVEN only).
 *   workspace: DEVICE scratch of at least csa_forward_host_workspace_bytes
 *   (B, H, T, d) bytes, 256-byte aligned (device copies of q, k, v, out,
 *   lse).
 *   heads_per_chunk: heads per pipeline chunk; must divide H.
 *   stream runs the kernels; stream_h2d and stream_d2h the two copy
 *   directions (they may equal stream, at the cost of the overlap).  All
 *   work of the call is complete once `stream` reaches the point after it.
 *   Errors as csa_forward, plus CSA_ERR_INVALID_ARG for a heads_per_chunk
 *   that does not divide H or a workspace too small.
 */
int csa_forward_host(const void *q, const void *k, const void *v, const void *k0, const void *v0,
                     void *out, float *lse, void *workspace, long long workspace_bytes, int B,
                     int H, int T, int d, float scale, int k0_mode, int heads_per_chunk,
                     csa_stream_t stream, csa_stream_t stream_h2d, csa_stream_t stream_d2h);

/*
 * csa_forward_host_ex - csa_forward_host with flags (the pages have no
 *   counterpart).  flags = 0 is csa_forward_host.  CSA_HOST_NO_ENTRY_WAIT:
 *   the host-to-device copies do not wait for the work already queued on
 *   `stream`, so that a call's copies in can overlap the previous call's
 *   kernels and copies out.  The caller then orders the calls that share a
 *   workspace itself: a call's copies in must not start before the previous
 *   call on the same workspace has completed on `stream` (for instance: two
 *   workspaces used alternately, each call recording an event on `stream`
 *   after it, and stream_h2d waiting for the event of the call before last).
 *   Unknown flag bits: CSA_ERR_INVALID_ARG.  Otherwise as csa_forward_host.
 */
#define CSA_HOST_NO_ENTRY_WAIT 1u
int csa_forward_host_ex(const void *q, const void *k, const void *v, const void *k0,
                        const void *v0, void *out, float *lse, void *workspace,
                        long long workspace_bytes, int B, int H, int T, int d, float scale,
                        int k0_mode, int heads_per_chunk, unsigned flags, csa_stream_t stream,
                        csa_stream_t stream_h2d, csa_stream_t stream_d2h);

/* csa_forward_host_workspace_bytes - device workspace csa_forward_host needs
 * (host only), or -1 for a negative size or d outside 1..256. */
long long csa_forward_host_workspace_bytes(int B, int H, int T, int d);

/*
 * csa_forward_short_conv - the short-conv reading of eq. (13) ("Analysis of
 *   the Result" of "Continuous Softmax Attention"): the correction b is
 *   replaced by its first-order Taylor term, which the page likens to a
 *   short convolution over the attention logits:
 *       b_{t,i} = (a_{t,i-1} + a_{t,i+1} - 2 a_{t,i}) / 6      1 <= i <= t-1
 *       b_{t,0} = -log 2 + (a_{t,1} - a_{t,0}) / 3
 *       b_{t,t} = -log 2 + (a_{t,t-1} - a_{t,t}) / 3
 *   (the ends from log phi2(x) = -log 2 + x/3 + O(x^2)); o and lse as in
 *   eq. (11).  It agrees with csa_forward to second order in the logit
 *   steps and forms no phi2, so it runs faster.  Same arguments, layout,
 *   alignment, d rules, sink modes and errors as csa_forward.
 */
int csa_forward_short_conv(const void *q, const void *k, const void *v, const void *k0,
                           const void *v0, void *out, float *lse, int B, int H, int T, int d,
                           float scale, int k0_mode, csa_stream_t stream);

/*
 * csa_forward_logdomain - csa_forward with the weights formed as eq. (10)
 *   and (11) of "Continuous Softmax Attention" ("Assembly and
 *   Simplification") write them: per key, z = a + b with
 *   b = log(phi2(a_{i-1} - a_i) + phi2(a_{i+1} - a_i)) (one-sided at the
 *   sink and at the row's own key) from log phi2 of each logit step, added
 *   in the log domain, and then e^{z - m}.  The same result as csa_forward
 *   (which forms each key's weight from the two interval shares of eq. (9)
 *   with one exponential and one reciprocal) within the bf16 rounding of
 *   the weights; it takes about nine special-function operations per
 *   (query, key) pair where csa_forward takes two, and is kept as the
 *   reference evaluation of that step.  Same arguments, layout, alignment,
 *   d rules (d other than 64 and 128 runs the CUDA-core kernel, which
 *   forms b this way too), sink modes and errors as csa_forward.
 */
int csa_forward_logdomain(const void *q, const void *k, const void *v, const void *k0,
                          const void *v0, void *out, float *lse, int B, int H, int T, int d,
                          float scale, int k0_mode, csa_stream_t stream);

/* csa_forward_short_conv_f32 - the same in fp32 on CUDA cores, 1 <= d <= 256. */
int csa_forward_short_conv_f32(const float *q, const float *k, const float *v, const float *k0,
                               const float *v0, float *out, float *lse, int B, int H, int T,
                               int d, float scale, int k0_mode, csa_stream_t stream);

/*
 * csa_forward_symmetric - continuous attention over the symmetric interval
 *   [1/2, t + 1/2] that the original Continuum Attention paper uses (cited in
 *   "Problem Statement" of "Continuous Softmax Attention"; eq. (2) with that
 *   interval).  Inside [1, t] keys and values follow eq. (3); the end
 *   half-cells [1/2, 1] and [t, t + 1/2] hold k_1, v_1 and k_t, v_t constant
 *   (a causal row has no k_{t+1}), so there is no sink.  As weights:
 *       e^{b_{t,1}} = 1/2 + phi2(a_{t,2} - a_{t,1}),
 *       e^{b_{t,t}} = phi2(a_{t,t-1} - a_{t,t}) + 1/2,
 *       interior keys as eq. (10); t = 1 gives o_1 = v_1.
 *   lse_t = log of the denominator integral over [1/2, t + 1/2].  bf16; same
 *   layout, alignment and d rules as csa_forward (no k0, v0, mode).
 */
int csa_forward_symmetric(const void *q, const void *k, const void *v, void *out, float *lse,
                          int B, int H, int T, int d, float scale, csa_stream_t stream);

/* csa_forward_symmetric_f32 - the same in fp32 on CUDA cores, 1 <= d <= 256. */
int csa_forward_symmetric_f32(const float *q, const float *k, const float *v, float *out,
                              float *lse, int B, int H, int T, int d, float scale,
                              csa_stream_t stream);

/*
 * csa_std_forward - standard causal softmax attention (b = 0, no sink),
 *   bf16 inputs, tensor-core path.
 *   Defines: eq. (12) of "Continuous Softmax Attention" ("Analysis of the
 *   Result"), the same as softmax(q k^T * scale + M) v with the causal mask M
 *   of "Attention, from the softmax up" ("The one line").
 *   lse_t = log sum_{i=1}^t e^{a_{t,i}}.  Same layout, alignment and d rules
 *   as csa_forward.
 */
int csa_std_forward(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                    int H, int T, int d, float scale, csa_stream_t stream);

/* csa_std_forward_f32 - eq. (12) in fp32 on CUDA cores; 1 <= d <= 256. */
int csa_std_forward_f32(const float *q, const float *k, const float *v, float *out, float *lse,
                        int B, int H, int T, int d, float scale, csa_stream_t stream);

/*
 * csa_backward - gradients of the continuous forward pass (csa_forward) for
 *   an upstream gradient dout = dL/d(out): dq, dk, dv and, in CSA_K0_GIVEN
 *   mode, the gradients of the trainable sink pair.
 *   Defines: the derivative of eq. (10)/(11) of "Continuous Softmax
 *   Attention" ("Assembly and Simplification"); the pages train models with
 *   the method ("Simple Experiments") but do not write this step out.  With
 *   p_i = e^{a_i - lse}, P_i the attention weight e^{a_i + b_i - lse},
 *   dP_i = dout . v_i and D = dout . out, for every row
 *       dL/da_i = P_i (dP_i - D) + F_i - F_{i+1},
 *       F_i = c_i (dP_{i-1} - dP_i),  c_i = p_{i-1} phi2'(a_i - a_{i-1}),
 *   (F = 0 past both ends of the row; phi2' is the derivative of eq. (6)'s
 *   phi2), and dq = scale sum_i dL/da_i k_i, dk_i += scale dL/da_i q,
 *   dv_i += P_i dout.
 *   q, k, v, out, dout: bf16 [B, H, T, d] (out from csa_forward);
 *   lse: float [B, H, T] from csa_forward (required);
 *   dq, dk, dv: bf16 [B, H, T, d], overwritten;
 *   k0, v0: bf16 [H, d] (CSA_K0_GIVEN only); dk0, dv0: float [H, d], the
 *   gradients of the sink pair summed over the batch and the rows
 *   (CSA_K0_GIVEN only; may be NULL otherwise).  In CSA_K0_COPY_FIRST the
 *   sink's gradient is added to key 0's; in CSA_K0_ZERO the sink is a
 *   constant.
 *   workspace: DEVICE scratch of at least csa_backward_workspace_bytes(B, H,
 *   T, d) bytes, 16-byte aligned, contents on entry irrelevant.  Concurrent
 *   calls need distinct workspaces.
 *   1 <= d <= 256 (CSA_ERR_UNSUPPORTED otherwise).  Tensors 2-byte aligned,
 *   lse, dk0, dv0 4-byte aligned.  Empty problems (B, H or T = 0) are
 *   CSA_OK; in CSA_K0_GIVEN mode dk0 and dv0 are then zeroed.  Atomic
 *   accumulation makes the low bits of dk, dv, dk0, dv0 depend on the order
 *   in which the hardware completes them.
 */
int csa_backward(const void *q, const void *k, const void *v, const void *k0, const void *v0,
                 const void *out, const float *lse, const void *dout, void *dq, void *dk,
                 void *dv, float *dk0, float *dv0, void *workspace, long long workspace_bytes,
                 int B, int H, int T, int d, float scale, int k0_mode, csa_stream_t stream);

/* csa_backward_f32 - the same in fp32 throughout (CUDA cores, no TF32); all
 * tensors 4-byte aligned. */
int csa_backward_f32(const float *q, const float *k, const float *v, const float *k0,
                     const float *v0, const float *out, const float *lse, const float *dout,
                     float *dq, float *dk, float *dv, float *dk0, float *dv0, void *workspace,
                     long long workspace_bytes, int B, int H, int T, int d, float scale,
                     int k0_mode, csa_stream_t stream);

/* csa_backward_workspace_bytes - workspace bytes csa_backward and
 * csa_backward_f32 need (host only), or -1 for a negative size or d outside
 * 1..256. */
long long csa_backward_workspace_bytes(int B, int H, int T, int d);

/*
 * csa_decode - one decode step: for every sequence b and head h, the output
 *   of the newest token, position t = n_b, against the sink and the n_b
 *   cached keys and values.
 *   Defines: eq. (10)/(11) of "Continuous Softmax Attention" ("Assembly and
 *   Simplification") for the single row t = n_b; the result equals row
 *   n_b - 1 of csa_forward run on the first n_b tokens, except that the
 *   weights stay in fp32 (they are not rounded to bf16 for a tensor core).
 *   q:         bf16 [B, H, d], the newest token's query of each sequence.
 *   k_cache, v_cache: bf16 [B, H, T, d]; T is the capacity.  Sequence b uses
 *              rows 0 .. n_b - 1, the last being the newest token's own key
 *              and value.
 *   k0, v0:    bf16 [H, d], read in CSA_K0_GIVEN mode only.  In
 *              CSA_K0_COPY_FIRST the sink is row 0 of the cache.
 *   seqlens:   DEVICE int32 [B] with n_b, or NULL for n_b = T for every b.
 *              A length outside [1, T] is not detectable on the host: that
 *              sequence's out and lse are set to NaN and the sticky status
 *              word (csa_device_status) records CSA_ERR_INVALID_ARG.
 *   out:       bf16 [B, H, d]; lse: float [B, H] natural log, or NULL.
 *   workspace: DEVICE scratch of at least csa_decode_workspace_bytes(B, H,
 *              T, d) bytes owned by the caller (16-byte aligned); its
 *              contents on entry do not matter and are overwritten.  Calls
 *              that run concurrently must use distinct workspaces.
 *   d must be 64, 128 or 256 (CSA_ERR_UNSUPPORTED otherwise).  q, k_cache,
 *   v_cache, out, workspace (and k0, v0 in GIVEN mode) must be 16-byte
 *   aligned.  B * H == 0: CSA_OK, nothing launched.  T == 0 with B * H > 0:
 *   CSA_ERR_INVALID_ARG (the newest token's key must be in the cache).
 *   workspace_bytes smaller than needed: CSA_ERR_INVALID_ARG.
 *   Computed on CUDA cores in fp32 (the step is bound by reading the cache):
 *   the positions 0..n_b are split into chunks, each chunk's partial sums
 *   are formed against its own maximum and merged by log-sum-exp.
 */
int csa_decode(const void *q, const void *k_cache, const void *v_cache, const void *k0,
               const void *v0, const int *seqlens, void *out, float *lse, void *workspace,
               long long workspace_bytes, int B, int H, int T, int d, float scale, int k0_mode,
               csa_stream_t stream);

/*
 * csa_decode_noalloc - csa_decode without a caller workspace.  The method's
 *   pages have no counterpart to this entry point: it is a convenience of
 *   this library for callers that cannot hand over scratch memory.
 *   Same arguments and result as csa_decode, minus workspace and
 *   workspace_bytes.  The chunk partials go to a fixed scratch array of
 *   CSA_DECODE_NOALLOC_SCRATCH_BYTES bytes that lives in the library's device
 *   image (one per device); the call allocates no memory of any kind.  Each
 *   call writes every partial it reads, so nothing in the array needs to
 *   start at zero.
 *   Memory: the array is CSA_DECODE_NOALLOC_SCRATCH_BYTES (64 MiB) of device
 *   memory on each device that loads it, held until the process exits.  It
 *   sits in a module of its own: with lazy module loading (the CUDA
 *   default) only processes that call csa_decode_noalloc hold it.
 *   Set-up: the first call on a device, and the first call after a device
 *   reset (a new context), looks the scratch address up with
 *   cudaGetSymbolAddress (that device must be current): make that call
 *   before any stream capture begins.
 *   Checks: csa_decode's argument checks run first, in its order and with
 *   its error codes; a size that passes them but whose scratch need exceeds
 *   the capacity then gives CSA_ERR_UNSUPPORTED, before anything is
 *   launched.
 *   Concurrency: every call on a device shares that one scratch array, so
 *   calls that can overlap on the device (different streams, or several host
 *   threads) race and corrupt each other's results.  Serialise them, e.g. on
 *   one stream, or use csa_decode with distinct workspaces.
 */
#define CSA_DECODE_NOALLOC_SCRATCH_BYTES (64u << 20)
int csa_decode_noalloc(const void *q, const void *k_cache, const void *v_cache, const void *k0,
                       const void *v0, const int *seqlens, void *out, float *lse, int B, int H,
                       int T, int d, float scale, int k0_mode, csa_stream_t stream);

/*
 * csa_decode_workspace_bytes - bytes of workspace csa_decode needs for these
 *   sizes (host only, no device needed), or -1 for a negative size, a d
 *   other than 64, 128, 256, or a size beyond 2^62 bytes.
 */
long long csa_decode_workspace_bytes(int B, int H, int T, int d);

/*
 * csa_decode_range - the decode step restricted to the positions [pos_lo,
 *   pos_hi) of every row (position 0 is the sink, position i >= 1 is cache
 *   row i - 1), for a KV cache whose time axis is split across devices
 *   (context parallelism).  The pages have no counterpart; it is eq. (11)
 *   ("Assembly and Simplification" of "Continuous Softmax Attention")
 *   summed over the owned positions only, each position's weight e^{a+b}
 *   still taking its correction b from both neighbours (eq. (10)), so that
 *   merging the ranges of a partition of [0, n] with csa_decode_merge_ranges
 *   gives csa_decode's result.
 *   q: DEVICE bf16 [B, H, d]; seqlens, k0, v0, scale, k0_mode, T and d as
 *   csa_decode (T is the capacity of the whole cache, 1 <= n_b <= T).
 *   k_shard, v_shard: DEVICE bf16 [B, H, rows, d] holding the cache rows
 *   [max(pos_lo - 2, 0), min(pos_hi, T)), rows = min(pos_hi, T) -
 *   max(pos_lo - 2, 0): the owned positions and one neighbour on each side.
 *   0 <= pos_lo < pos_hi <= T + 1 and pos_lo != 1 (a range cannot start
 *   right after the sink); otherwise CSA_ERR_INVALID_ARG.
 *   out: DEVICE fp32 [B, H, d], the range's normalised output o_r;
 *   lse: DEVICE fp32 [B, H] (required), log of the range's weight sum.  A
 *   row whose length n_b < pos_lo has no owned position: o_r = 0 and
 *   lse_r = -inf.
 *   workspace: DEVICE scratch of csa_decode_range_workspace_bytes(B, H,
 *   pos_lo, pos_hi, d) bytes, 16-byte aligned.  Tensors 16-byte aligned,
 *   lse and seqlens 4-byte aligned.  Errors as csa_decode.
 */
int csa_decode_range(const void *q, const void *k_shard, const void *v_shard, const void *k0,
                     const void *v0, const int *seqlens, float *out, float *lse, void *workspace,
                     long long workspace_bytes, int B, int H, int T, int d, float scale,
                     int k0_mode, int pos_lo, int pos_hi, csa_stream_t stream);

/* csa_decode_range_workspace_bytes - workspace bytes csa_decode_range needs
 * (host only), or -1 for a negative size, pos_hi < pos_lo or d outside
 * {64, 128, 256}. */
long long csa_decode_range_workspace_bytes(int B, int H, int pos_lo, int pos_hi, int d);

/*
 * csa_decode_merge_ranges - merges R partial results of the same rows (from
 *   csa_decode_range over ranges that partition each row's positions):
 *       o = sum_r e^{lse_r - L} o_r / sum_r e^{lse_r - L},
 *       lse = L + log sum_r e^{lse_r - L},   L = max_r lse_r;
 *   an empty range (lse_r = -inf) weighs nothing.  The pages have no
 *   counterpart: this is the one exchange step of context parallelism.
 *   o_parts: DEVICE fp32 [R, B, H, d]; lse_parts: DEVICE fp32 [R, B, H];
 *   out: DEVICE bf16 [B, H, d]; lse: DEVICE fp32 [B, H] or NULL.
 *   R >= 1, 1 <= d <= 256; CSA_ERR_INVALID_ARG otherwise.
 */
int csa_decode_merge_ranges(const float *o_parts, const float *lse_parts, int R, int B, int H,
                            int d, void *out, float *lse, csa_stream_t stream);

/*
 * csa_logphi2_eval - y[i] = log phi2(x[i]) with the library's fp32 device
 *   function (phi2 of eq. (6), "Preliminaries").  x, y: device float arrays
 *   of n elements (n >= 0).  A test hook for the numerics of b.
 */
int csa_logphi2_eval(const float *x, float *y, int n, csa_stream_t stream);

/*
 * csa_segment_weights_eval - the tensor-core kernel's fp32 evaluation of
 *   one interval's two end weights, for tests.  For each i, with
 *   x = u1[i] - u0[i] in natural-log units and p = e^{u}:
 *       right[i] = p0 * phi2(x)    (the share of interval (u0,u1) that eq. (9)
 *       left[i]  = p1 * phi2(-x)    moves onto its left and right key)
 *   u0, u1: device float arrays (u <= 0 expected, as after subtracting a
 *   running max); right, left: device float outputs; n >= 0.
 */
int csa_segment_weights_eval(const float *u0, const float *u1, float *right, float *left, int n,
                             csa_stream_t stream);

/*
 * csa_device_status - reads and clears the library's sticky device status
 *   words of the current device: CSA_OK; CSA_ERR_TIMEOUT if a kernel's
 *   bounded wait expired since the last read (that kernel then skipped the
 *   rest of its work and its outputs are undefined); CSA_ERR_INVALID_ARG if
 *   csa_decode met a sequence length outside [1, T].  Synchronises the
 *   device.  Returns CSA_ERR_CUDA if the read itself fails.
 */
int csa_device_status(void);

/*
 * csa_selftest_wait_timeout - launches one block whose thread waits on an
 *   mbarrier that nothing ever completes, with a time limit of timeout_us
 *   microseconds (1..10^6).  The wait gives up, the kernel records
 *   CSA_ERR_TIMEOUT in the status word and returns normally; the context
 *   stays usable.  Exercises the bounded-wait path of the kernels without
 *   any fault.
 */
int csa_selftest_wait_timeout(unsigned timeout_us, csa_stream_t stream);

/*
 * csa_selftest_forward_delay - csa_forward's exact form (the tensor-core
 *   kernel, bf16, d in {64, 128}; arguments, layout, ownership and checks as
 *   csa_forward) with a delay planted in every epilogue: the softmax threads
 *   of column half delay_half (0 or 1) sleep delay_ns nanoseconds (at most
 *   10^6) after the item's last PV product is done and before they read the
 *   two accumulators O_0 and O_1.  Meanwhile the other half's threads run
 *   ahead into the CTA's next query tile, whose first PV product overwrites
 *   O_0 and O_1 ("Assembly and Simplification", eq. (10): the numerator and
 *   denominator sums per query row).  The kernel orders that product after
 *   every thread's reads, so the output and lse must equal csa_forward's bit
 *   for bit whatever the delay.  CSA_ERR_INVALID_ARG for a delay or half out
 *   of range.  A test hook: it only slows the kernel down.
 */
int csa_selftest_forward_delay(const void *q, const void *k, const void *v, const void *k0,
                               const void *v0, void *out, float *lse, int B, int H, int T, int d,
                               float scale, int k0_mode, unsigned delay_ns, int delay_half,
                               csa_stream_t stream);

/* Human-readable text for a status code (never NULL, static storage). */
const char *csa_status_string(int status);

/* ABI version of this header (bumped on incompatible change). */
int csa_abi_version(void);
#define CSA_ABI_VERSION 1

#ifdef __cplusplus
}
#endif
#endif /* CSA_H_ */
