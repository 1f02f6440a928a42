// Warp-specialised streaming pipeline shared by the decode and MoE kernels:
// one producer thread fills a ring of shared-memory stages with bulk /
// tensor-map copies tracked by mbarriers; consumer warps release stages.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "tp_internal.h"

namespace tpk {

constexpr int kStages = 4;                 // ring depth
constexpr int kConsumers = 256;            // eight consumer warps
constexpr int kStreamThreads = kConsumers + 32;
constexpr int kBoxK = 256;                 // reduction elements per tensor-map box
constexpr int kBoxBytes = kBoxK * 32 * 2;  // one box: 32 rows x 256 bf16 = 16 KB
constexpr int kXBoxBytes = kBoxK * kTMax * 2;   // activation box: 8 token rows x 256 bf16 = 4 KB
constexpr int kGemvStageBytes = 2 * kBoxBytes + kXBoxBytes;
constexpr int kGemvStages = 3;             // projection ring depth (96 KB)
constexpr int kAttnStageBytes = 16384;     // one contiguous run of K or V rows
constexpr int kCtrlBytes = 128;            // barriers and flags at the start of shared memory

struct Ring {
    uint64_t* full;
    uint64_t* empty;
    volatile int* abort;
    unsigned* s_flag;
};

__device__ __forceinline__ Ring ring_setup(unsigned char* smem, int stages = kStages) {
    Ring R;
    R.full = reinterpret_cast<uint64_t*>(smem);
    R.empty = R.full + kStages;
    R.abort = reinterpret_cast<volatile int*>(smem + 16 * kStages);
    R.s_flag = reinterpret_cast<unsigned*>(smem + 16 * kStages + 4);
    if (threadIdx.x == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(&R.full[i], 1);
            mbar_init(&R.empty[i], kConsumers / 32);
        }
        *R.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    return R;
}

// After an aborted wait the producer must not leave copies writing into
// shared memory of an exited CTA: wait (bounded) for every stage issued.
__device__ __forceinline__ void producer_drain(const Ring& R, uint32_t issued, int stages = kStages) {
    volatile int no_abort = 0;
    const uint32_t first = issued > (uint32_t)stages ? issued - stages : 0u;
    for (uint32_t k = first; k < issued; ++k) mbar_wait(&R.full[k % stages], (k / stages) & 1, &no_abort, nullptr);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_keep(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 3-D tiled loads (the decode step's 128-byte-swizzled stage boxes).
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* tm, int x, int y, int z, uint64_t* bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_keep(void* dst, const CUtensorMap* tm, int x, int y, int z,
                                                 uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace tpk
