// End-to-end forward pass from host buffers (csa_forward_host in csa.h):
// the (b, h) problems are independent, so they go through in chunks of
// heads, and the copies of one chunk overlap the kernel of another:
//   h2d stream      copy q, k, v of chunk c           -> event in[c]
//   compute stream  wait in[c]; forward kernel on c   -> event done[c]
//   d2h stream      wait done[c]; copy out, lse of c  -> event back[c]
// and the compute stream finally waits for the last copy back, so the
// whole call is complete once the compute stream reaches that point.  One
// cudaMemcpyAsync per tensor and chunk.
#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "csa.h"
#include "csa_internal.h"

namespace {

struct Events {
    std::vector<cudaEvent_t> ev;
    ~Events() {
        for (cudaEvent_t e : ev) cudaEventDestroy(e);  // released once complete
    }
    cudaEvent_t make() {
        cudaEvent_t e = nullptr;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
        ev.push_back(e);
        return e;
    }
};

}  // namespace

long long csa_host_scratch_bytes(int B, int H, int T, int d) {
    if (B < 0 || H < 0 || T < 0 || d < 1) return -1;
    const long long rows = (long long)B * H * T;
    const long long tensor = (rows * d * 2 + 255) / 256 * 256;  // bf16, 256-byte aligned pieces
    const long long lse = (rows * 4 + 255) / 256 * 256;
    return 4 * tensor + lse;  // q, k, v, out and lse on the device
}

int csa_host_forward(const void *q_h, const void *k_h, const void *v_h, const void *k0,
                     const void *v0, void *out_h, float *lse_h, void *scratch, int B, int H, int T,
                     int d, float scale, int mode, int heads_per_chunk, bool entry_wait,
                     cudaStream_t s_compute, cudaStream_t s_h2d, cudaStream_t s_d2h) {
    const long long rows = (long long)B * H * T;
    const long long tensor = (rows * d * 2 + 255) / 256 * 256;
    uint8_t *base = static_cast<uint8_t *>(scratch);
    uint8_t *q_d = base, *k_d = base + tensor, *v_d = base + 2 * tensor, *o_d = base + 3 * tensor;
    float *l_d = reinterpret_cast<float *>(base + 4 * tensor);
    const size_t chunk_rows = (size_t)heads_per_chunk * T;
    const size_t chunk_bytes = chunk_rows * d * 2;
    const int chunks_per_b = H / heads_per_chunk;
    Events evs;
    // The copies of this call must not overtake work still queued on the
    // compute stream (a previous call reading the same device buffers),
    // unless the caller orders calls that share a workspace itself.
    if (entry_wait) {
        cudaEvent_t start = evs.make();
        if (!start || cudaEventRecord(start, s_compute) != cudaSuccess ||
            cudaStreamWaitEvent(s_h2d, start, 0) != cudaSuccess ||
            cudaStreamWaitEvent(s_d2h, start, 0) != cudaSuccess)
            return CSA_ERR_CUDA;
    }
    cudaEvent_t last_back = nullptr;
    for (int b = 0; b < B; ++b) {
        for (int c = 0; c < chunks_per_b; ++c) {
            const int h0 = c * heads_per_chunk;
            const size_t row0 = ((size_t)b * H + h0) * T;  // first row of the chunk
            const size_t off = row0 * d * 2;
            cudaEvent_t in = evs.make(), done = evs.make(), back = evs.make();
            if (!in || !done || !back) return CSA_ERR_CUDA;
            const uint8_t *qh = static_cast<const uint8_t *>(q_h) + off;
            const uint8_t *kh = static_cast<const uint8_t *>(k_h) + off;
            const uint8_t *vh = static_cast<const uint8_t *>(v_h) + off;
            if (cudaMemcpyAsync(q_d + off, qh, chunk_bytes, cudaMemcpyHostToDevice, s_h2d) != cudaSuccess ||
                cudaMemcpyAsync(k_d + off, kh, chunk_bytes, cudaMemcpyHostToDevice, s_h2d) != cudaSuccess ||
                cudaMemcpyAsync(v_d + off, vh, chunk_bytes, cudaMemcpyHostToDevice, s_h2d) != cudaSuccess ||
                cudaEventRecord(in, s_h2d) != cudaSuccess ||
                cudaStreamWaitEvent(s_compute, in, 0) != cudaSuccess)
                return CSA_ERR_CUDA;
            const void *k0c = k0 ? static_cast<const uint8_t *>(k0) + (size_t)h0 * d * 2 : nullptr;
            const void *v0c = v0 ? static_cast<const uint8_t *>(v0) + (size_t)h0 * d * 2 : nullptr;
            float *lse_c = l_d + row0;
            int rc;
            if (d == 64 || d == 128)
                rc = csa_tc_forward(q_d + off, k_d + off, v_d + off, k0c, v0c, o_d + off, lse_c, 1,
                                    heads_per_chunk, T, d, scale, mode, kFormExact, s_compute);
            else
                rc = csa_simt_forward_bf16(q_d + off, k_d + off, v_d + off, k0c, v0c, o_d + off,
                                           lse_c, 1, heads_per_chunk, T, d, scale, mode,
                                           kFormExact, s_compute) == cudaSuccess
                         ? CSA_OK
                         : CSA_ERR_CUDA;
            if (rc != CSA_OK) return rc;
            if (cudaEventRecord(done, s_compute) != cudaSuccess ||
                cudaStreamWaitEvent(s_d2h, done, 0) != cudaSuccess ||
                cudaMemcpyAsync(static_cast<uint8_t *>(out_h) + off, o_d + off, chunk_bytes,
                                cudaMemcpyDeviceToHost, s_d2h) != cudaSuccess)
                return CSA_ERR_CUDA;
            if (lse_h && cudaMemcpyAsync(lse_h + row0, lse_c, chunk_rows * 4,
                                         cudaMemcpyDeviceToHost, s_d2h) != cudaSuccess)
                return CSA_ERR_CUDA;
            if (cudaEventRecord(back, s_d2h) != cudaSuccess) return CSA_ERR_CUDA;
            last_back = back;
        }
    }
    if (last_back && cudaStreamWaitEvent(s_compute, last_back, 0) != cudaSuccess)
        return CSA_ERR_CUDA;
    return CSA_OK;
}
