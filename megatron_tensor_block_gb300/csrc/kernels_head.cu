// Logits of the final hidden state over the vocab-parallel head.
//
// "Gather tensor-parallel sharded parameters on read in a trace" (Change):
// the head is split by vocabulary rows, padded to a multiple of 64 x tp with
// the padding rows at the tail of the last shard, and the gather drops rows
// >= org_vocab. "Multi-GPU & Multi-Node" (How tensor parallelism works): the
// norm before it is replicated. So
//
//   logits[t][v] = (sum_k bf16(x[t][k] * gamma[k]) * W[v][k]) / rms(x[t]),   v < org_vocab,
//
// with row v of the stacked shards (shard v / rows_per_shard). Every shard's
// rows are column-parallel logits; writing only v < org_vocab is the gather.
//
// GB300 design: an HBM-bound GEMV over the whole head (272 MB for a
// Qwen2.5-0.5B-shaped vocabulary). Each CTA streams a contiguous range of
// rows through a ring of stages with 1-D bulk copies (a stage crossing a
// shard boundary takes two); one warp per row reads it along its length
// (512 contiguous bytes per warp access, no bank conflicts), with the bf16
// operand rows of all tokens from shared memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tp_internal.h"

namespace tpk {

namespace {

constexpr int kHW = 8;                      // consumer warps
constexpr int kHCT = kHW * 32;

__device__ __forceinline__ float hbf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float hbf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float hdot8(const uint4 w, const uint4 x, float s) {
    s = fmaf(hbf_lo(w.x), hbf_lo(x.x), s);
    s = fmaf(hbf_hi(w.x), hbf_hi(x.x), s);
    s = fmaf(hbf_lo(w.y), hbf_lo(x.y), s);
    s = fmaf(hbf_hi(w.y), hbf_hi(x.y), s);
    s = fmaf(hbf_lo(w.z), hbf_lo(x.z), s);
    s = fmaf(hbf_hi(w.z), hbf_hi(x.z), s);
    s = fmaf(hbf_lo(w.w), hbf_lo(x.w), s);
    s = fmaf(hbf_hi(w.w), hbf_hi(x.w), s);
    return s;
}

__global__ void __launch_bounds__(kHeadThreads, 3) lm_head_kernel(const __grid_constant__ HeadArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kHeadMaxStages;
    volatile int* abort = reinterpret_cast<volatile int*>(empty + kHeadMaxStages);
    float* rinv = reinterpret_cast<float*>(smem + 320);                    // [8]
    bf16* xs = reinterpret_cast<bf16*>(smem + 512);                        // [T][H]
    unsigned char* ring = smem + A.ring_off;                               // [ns][rs][H] bf16
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = A.H, rs = A.rs, ns = A.ns;
    const long total = (long)A.N * A.rows_s;
    const long g0 = (long)blockIdx.x * A.rpc, g1 = min(g0 + A.rpc, total);
    const int nst = g0 < g1 ? (int)((g1 - g0 + rs - 1) / rs) : 0;
    if (tid == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kHW);
        }
        *abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_trigger();
    if (warp == kHW) {                                  // producer: the head does not depend on the preceding kernel
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            const size_t row_bytes = (size_t)H * 2;
            int s = 0;
            for (; s < nst; ++s) {
                const int sl = s % ns;
                if (s >= ns && !mbar_wait(&empty[sl], (s / ns - 1) & 1, abort, A.status)) break;
                const long r0 = g0 + (long)s * rs, r1 = min(r0 + rs, g1);
                mbar_arrive_expect_tx(&full[sl], (uint32_t)((r1 - r0) * row_bytes));
                unsigned char* dst = ring + (size_t)sl * rs * row_bytes;
                long r = r0;
                while (r < r1) {                        // at most two pieces: the stage may cross a shard boundary
                    const int sh = (int)(r / A.rows_s);
                    const long local = r - (long)sh * A.rows_s;
                    const long n = min(r1 - r, (long)A.rows_s - local);
                    bulk_g2s(dst + (size_t)(r - r0) * row_bytes,
                             static_cast<const unsigned char*>(A.W[sh]) + (size_t)local * row_bytes,
                             (uint32_t)(n * row_bytes), &full[sl], pol);
                    r += n;
                }
            }
            // every copy issued has landed before this thread leaves; bounded
            volatile int no_abort = 0;
            for (int q = s > ns ? s - ns : 0; q < s; ++q) mbar_wait(&full[q % ns], (q / ns) & 1, &no_abort, nullptr);
        }
        return;
    }
    pdl_wait();                                         // the hidden state comes from the preceding kernel
    const int T = A.T;
    // operand rows bf16(x * gamma) and 1/rms per token
    for (int i = tid; i < T * H / 2; i += kHCT) {
        const int e = 2 * i, t = e / H, k = e - t * H;
        const float2 xv = *reinterpret_cast<const float2*>(A.x + (size_t)t * H + k);
        const float2 gv = __ldg(reinterpret_cast<const float2*>(A.gamma + k));
        *reinterpret_cast<uint32_t*>(xs + (size_t)t * H + k) = pack_bf16x2(xv.x * gv.x, xv.y * gv.y);
    }
    if (warp < T) {
        float a = 0.f;
        for (int k = lane; k < H; k += 32) {
            const float v = A.x[(size_t)warp * H + k];
            a = fmaf(v, v, a);
        }
        a = warp_sum(a);
        if (lane == 0) rinv[warp] = 1.0f / sqrtf(a * (1.0f / (float)H) + A.eps);
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kHCT) : "memory");
    const size_t row_bytes = (size_t)H * 2;
    const int nu = H / 8;                               // 16-byte units per row
    for (int s = 0; s < nst; ++s) {
        const int sl = s % ns;
        mbar_wait(&full[sl], (s / ns) & 1, abort, A.status);
        const long r0 = g0 + (long)s * rs;
        const int nr = (int)min((long)rs, g1 - r0);
        const unsigned char* st = ring + (size_t)sl * rs * row_bytes;
        for (int rr = warp; rr < nr; rr += kHW) {
            const long v = r0 + rr;                     // row of the stacked, padded head = logit column
            const unsigned char* wr = st + (size_t)rr * row_bytes;
            for (int t = 0; t < T; ++t) {
                const bf16* xr = xs + (size_t)t * H;
                float acc = 0.f;
#pragma unroll 4
                for (int u = lane; u < nu; u += 32)
                    acc = hdot8(*reinterpret_cast<const uint4*>(wr + 16 * u),
                                *reinterpret_cast<const uint4*>(xr + 8 * u), acc);
                acc = warp_sum(acc);
                if (lane == t && v < A.org_vocab) A.logits[(size_t)t * A.org_vocab + v] = acc * rinv[t];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[sl]);
    }
}

}  // namespace

// Several CTAs per SM, each with its own copy stream, keep more of HBM busy
// than one CTA with a deep ring (measured on the Qwen-shaped head: 16-row
// stages at 1, 2 and 3 CTAs per SM read at 0.49, 0.73 and 0.81 of the copy
// peak): take the most CTAs per SM (up to 3) that still leave two stages each.
size_t head_smem(HeadArgs& a, int smem_max) {
    a.rs = a.H <= 1024 ? 16 : (a.H <= 2048 ? 8 : 4);
    const size_t stage = (size_t)a.rs * a.H * 2;
    const size_t fixed = 512 + (size_t)kTMax * a.H * 2;
    a.ring_off = (int)((fixed + 127) & ~(size_t)127);
    for (a.cps = 3; a.cps >= 1; --a.cps) {
        const long budget = (long)smem_max / a.cps - (a.cps > 1 ? 2048 : 0);   // room for the per-CTA reserve
        long ns = (budget - a.ring_off) / (long)stage;
        if (ns > kHeadMaxStages) ns = kHeadMaxStages;
        a.ns = (int)ns;
        if (a.ns >= 2 || a.cps == 1) break;
    }
    return (size_t)a.ring_off + (size_t)a.ns * stage;
}

cudaError_t launch_lm_head(const HeadArgs& a, size_t smem, cudaStream_t s) {
    static size_t configured = 0;
    if (smem > configured) {
        cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(lm_head_kernel),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    HeadArgs A = a;
    void* args[] = {&A};
    return launch_pdl(reinterpret_cast<const void*>(lm_head_kernel), args, a.grid, smem, s, kHeadThreads);
}

}  // namespace tpk
