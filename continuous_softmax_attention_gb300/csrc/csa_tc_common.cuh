// Pieces shared by the two tensor-core kernels (csa_tc.cu: continuous
// attention, csa_tc_std.cu: standard attention): tcgen05 instruction and
// shared-memory descriptors, TMEM load helpers, bounded mbarrier waits that
// report into a caller-chosen status word, and the host-side TMA tensor
// maps.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "csa_device.cuh"

namespace csa_tc {

using namespace csa_dev;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kChunkBytes = 128 * 128;  // one 64-column x 128-row box, 128B swizzled

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, bf16 A
// and B, A K-major, B K-major or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;  // descriptor version for this architecture
    d |= 2ull << 61;  // 128-byte swizzle
    return d;
}

__device__ __forceinline__ float fmax3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ void tmem_ld1(uint32_t taddr, uint32_t &r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr) : "memory");
}

// tcgen05.wait::ld that also names the destination registers of the loads
// it waits for, so that no use of them can be scheduled before it.
template <int N>
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&r)[N]);
template <>
__device__ __forceinline__ void tmem_wait_ld_regs<1>(uint32_t (&r)[1]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]) : : "memory");
}
template <>
__device__ __forceinline__ void tmem_wait_ld_regs<32>(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         int *status) {
    return mbar_wait_bounded(bar, parity, abort_flag, status, kWaitLimitNs);
}

// Wait that ignores the abort flag: used only to let in-flight copies and
// MMAs finish before the block exits.
__device__ __forceinline__ void wait_bar_drain(uint32_t bar, uint32_t parity, int *status) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *(volatile int *)status = kStatusTimeout;
            return;
        }
    }
}

// ---------------------------------------------------------------- host side
// Heads per scheduling group: as many as keep the group's K and V (bf16)
// within 64 MiB, half of L2, so that they are read from HBM about once.
inline int heads_per_group(int BH, int T, int D) {
    const long long per_head = 2LL * T * D * 2;
    long long g = (64LL << 20) / (per_head > 0 ? per_head : 1);
    if (g < 1) g = 1;
    if (g > BH) g = BH;
    return (int)g;
}

inline PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// [B*H, T, D] bf16 viewed as a 3-D tensor {D, T, B*H}, boxes of 64 columns x
// 128 rows.  Rows outside [0, T) of a head read as zeros.
inline bool encode_qkv_map(CUtensorMap *map, const void *ptr, int BH, int T, int D) {
    auto fn = get_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)T * D * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult rc = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return rc == CUDA_SUCCESS;
}

}  // namespace csa_tc
