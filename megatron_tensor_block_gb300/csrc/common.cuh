// Device helpers shared by the kernels: storage-type conversion, streaming
// loads, the bf16 tensor-core fragment MMA, status reporting.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tp_block.h"

namespace tpk {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------- types

template <typename T> struct Stor;
template <> struct Stor<float> {
    static __device__ __forceinline__ float load(const float* p) { return *p; }
    static __device__ __forceinline__ void store(float* p, float v) { *p = v; }
};
template <> struct Stor<bf16> {
    static __device__ __forceinline__ float load(const bf16* p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ void store(bf16* p, float v) { *p = __float2bfloat16_rn(v); }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
    float2 r;
    r.x = __uint_as_float(u << 16);
    r.y = __uint_as_float(u & 0xFFFF0000u);
    return r;
}

// ---------------------------------------------------------------- loads

// 16-byte read-only streaming load: no L1 allocation, 256-byte L2 prefetch.
// Used for weights and KV, which every launch reads exactly once.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// 16-byte load that bypasses L1 (sees other CTAs' writes made visible by a
// fence), for partial sums written earlier in the same launch.
__device__ __forceinline__ float4 ld_cg_f4(const float* p) {
    return __ldcg(reinterpret_cast<const float4*>(p));
}

// ---------------------------------------------------------------- MMA

// D += A * B for one m16n8k16 bf16 tile with fp32 accumulation.
// Fragment ownership (lane = 4*g + t): a0 = (row g, k 2t..2t+1),
// a1 = (row g+8, k 2t..), a2 = (row g, k 2t+8..), a3 = (row g+8, k 2t+8..);
// b0 = (k 2t..2t+1, col g), b1 = (k 2t+8.., col g);
// c0,c1 = (row g, cols 2t, 2t+1), c2,c3 = (row g+8, cols 2t, 2t+1).
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- status

// First device-detected error wins; the host reads it with
// tp_get_device_status.
__device__ __forceinline__ void set_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Completion counting for "the last CTA of a group reduces": every CTA of
// the group has stored its partial; returns true in the CTA that arrived
// last, which then reads all partials (through L2) in a fixed order. The
// last CTA also resets the counter, so it is zero again after the launch.
// No CTA ever waits for another.
__device__ __forceinline__ bool arrive_last(unsigned* counter, unsigned n_in_group) {
    __shared__ unsigned s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned old = atomicAdd(counter, 1u);
        s_last = (old == n_in_group - 1) ? 1u : 0u;
        if (s_last) *counter = 0u;
    }
    __syncthreads();
    if (s_last) __threadfence();
    return s_last != 0;
}

}  // namespace tpk

// ---------------------------------------------------------------- async copy pipeline

namespace tpk {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// 2^x on the special-function unit: PTX ex2.approx.ftz.f32 (relative error
// near 2^-22; results below the normal range flush to zero, -inf gives 0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

constexpr uint64_t kWaitLimitNs = 1000000000ull;   // every device-side wait gives up after 1 s

// Waits for the phase of `bar` with parity `parity` to complete. Gives up
// after kWaitLimitNs or when another thread of the CTA has given up
// (*abort != 0); then records TP_ERR_TIMEOUT and returns false. Callers keep
// executing the same barriers either way, so a CTA never deadlocks.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            set_status(status, TP_ERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Bulk asynchronous copy global -> shared, completion counted in bytes on `bar`.
// Both addresses 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Programmatic dependent launch: wait for the preceding kernel's completion
// (and visibility of its writes) / allow the next kernel to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Barrier among the first `n` threads (consumer warps) only.
__device__ __forceinline__ void consumer_sync(int n) { asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory"); }

// arrive_last for kernels whose barrier covers only the consumer threads.
// The barrier orders the CTA's partial-sum stores before thread 0's fence,
// which (being cumulative) publishes them device-wide before its atomic.
__device__ __forceinline__ bool arrive_last_consumers(unsigned* counter, unsigned n_in_group, int nthreads,
                                                      unsigned* s_flag) {
    consumer_sync(nthreads);
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned old = atomicAdd(counter, 1u);
        const unsigned last = (old == n_in_group - 1) ? 1u : 0u;
        if (last) {
            *counter = 0u;
            __threadfence();
        }
        *s_flag = last;
    }
    consumer_sync(nthreads);
    return *reinterpret_cast<volatile unsigned*>(s_flag) != 0;
}

}  // namespace tpk
