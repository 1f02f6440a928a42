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
