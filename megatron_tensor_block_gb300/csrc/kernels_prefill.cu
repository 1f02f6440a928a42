// Prefill-regime projections on the fifth-generation tensor cores.
//
// C[M, N] = A[M, K] * B[N, K]^T with bf16 operands and fp32 accumulation in
// tensor memory. One CTA computes a 128 x 256 tile:
//   warp 0   TMA producer: 128-byte-swizzled K-major boxes of A (128 x 64) and
//            B (256 x 64) into a 4-stage shared-memory ring (mbarriers);
//   warp 1   allocates tensor memory and issues tcgen05.mma (128 x 256 x 16,
//            four per 64-wide stage) from one thread; each stage is released
//            by tcgen05.commit when its MMAs complete;
//   warps 2-5 epilogue: tcgen05.ld of the accumulator (one token row per
//            thread, 32 columns at a time) and the store.
// Every wait is bounded; tensor memory is freed on every path.
#include <cuda.h>

#include <cstring>

#include "common.cuh"
#include "stream.cuh"
#include "tcgen05.cuh"
#include "tp_internal.h"

namespace tpk {

constexpr int kTcBM = 128, kTcBN = 256, kTcBK = 64;
constexpr int kTcStages = 4;
constexpr int kTcABytes = kTcBM * kTcBK * 2;            // 16 KB
constexpr int kTcBBytes = kTcBN * kTcBK * 2;            // 32 KB
constexpr int kTcStageBytes = kTcABytes + kTcBBytes;
constexpr int kTcThreads = 192;
constexpr int kTcSmem = 1024 + kTcStages * kTcStageBytes;

struct TcGemmArgs {
    CUtensorMap ta;       // A [M, K], boxes 64 x 128, 128-byte swizzle
    CUtensorMap tb;       // B [N, K], boxes 64 x 256, 128-byte swizzle
    float* C;             // [M, N]
    int M, N, K;
    int* status;
};

__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_plain_kernel(const __grid_constant__ TcGemmArgs g) {
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kTcStages;
    uint64_t* accum = empty + kTcStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    unsigned char* stages = smem + 1024;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kTcBM, n0 = blockIdx.y * kTcBN;
    const int nk = g.K / kTcBK;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kTcStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(accum, 1);
        *abort_flag = (smem_u32(stages) & 1023u) ? 1 : 0;
        if (*abort_flag) set_status(g.status, TP_ERR_ALIGN);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0 && !*abort_flag) {
            int kb = 0;
            for (; kb < nk; ++kb) {
                const int s = kb % kTcStages;
                if (!mbar_wait(&empty[s], ((kb / kTcStages) & 1) ^ 1, abort_flag, g.status)) break;
                mbar_arrive_expect_tx(&full[s], kTcStageBytes);
                unsigned char* st = stages + s * kTcStageBytes;
                tma_load_2d_keep(st, &g.ta, kb * kTcBK, m0, &full[s]);
                tma_load_2d_keep(st + kTcABytes, &g.tb, kb * kTcBK, n0, &full[s]);
            }
            // no copy may still be landing when the CTA exits
            volatile int no_abort = 0;
            for (int k = kb > kTcStages ? kb - kTcStages : 0; k < kb; ++k)
                mbar_wait(&full[k % kTcStages], (k / kTcStages) & 1, &no_abort, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kTcBM, kTcBN);
            bool ok = !*abort_flag;
            for (int kb = 0; kb < nk && ok; ++kb) {
                const int s = kb % kTcStages;
                if (!mbar_wait(&full[s], (kb / kTcStages) & 1, abort_flag, g.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_u32(stages + s * kTcStageBytes), b0 = a0 + kTcABytes;
#pragma unroll
                for (int k = 0; k < kTcBK / 16; ++k)
                    tc_mma(tmem, smem_desc_sw128(a0 + k * 32), smem_desc_sw128(b0 + k * 32), idesc,
                           (kb | k) != 0);
                tc_commit(smem_u32(&empty[s]));
            }
            tc_commit(smem_u32(accum));       // fires when every issued MMA has completed
        }
    } else {
        // epilogue warps 2..5 -> tensor-memory lane quarters 2,3,0,1
        const int q = warp & 3;
        const bool ok = mbar_wait(accum, 0, abort_flag, g.status);
        tc_fence_after();
        const int row = m0 + 32 * q + lane;
        for (int c = 0; c < kTcBN / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + c * 32, v);
            tmem_wait_ld();
            if (ok && row < g.M) {
                float* dst = g.C + (size_t)row * g.N + n0 + c * 32;
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    *reinterpret_cast<float4*>(dst + i) = make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                                      __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        volatile int no_abort = 0;                   // every MMA has retired before the columns are freed
        mbar_wait(accum, 0, &no_abort, nullptr);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 256);
        tmem_relinquish();
    }
}

cudaError_t launch_tc_gemm_plain(const void* A, const void* B, float* C, int M, int N, int K, int* status,
                                 cudaStream_t s) {
    TcGemmArgs g;
    memset(&g, 0, sizeof g);
    cudaError_t e = tensor_map_2d(A, K, M, kTcBK, kTcBM, 1, &g.ta);
    if (e == cudaSuccess) e = tensor_map_2d(B, K, N, kTcBK, kTcBN, 1, &g.tb);
    if (e != cudaSuccess) return e;
    g.C = C;
    g.M = M;
    g.N = N;
    g.K = K;
    g.status = status;
    static bool set = false;
    if (!set) {
        e = cudaFuncSetAttribute(tc_gemm_plain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
        if (e != cudaSuccess) return e;
        set = true;
    }
    dim3 grid(M / kTcBM, N / kTcBN);
    tc_gemm_plain_kernel<<<grid, kTcThreads, kTcSmem, s>>>(g);
    return cudaGetLastError();
}

}  // namespace tpk
