// MoE feed-forward block ("Multi-GPU & Multi-Node", Supported architectures:
// the router is replicated; each shard holds 1/tp of every expert's weights --
// expert slicing, balanced whichever experts a token picks -- or, with expert
// parallelism, 1/tp of the experts whole). Decode-sized token counts, bf16
// weights, fp32 accumulation.
//
//   route   : softmax top-k per token (chosen by logit, ties to the lower id),
//             weights renormalised over the chosen experts
//   bucket  : stable counting sort of the (token, choice) slots by expert
//   prep    : per token, x_t * gamma_r (bf16) into each of its slots' rows, 1/rms per slot
//   gate/up : per shard and expert it holds, grouped GEMM on the tensor cores
//             (tcgen05) over the expert's slots, SwiGLU epilogue
//   down    : per shard and expert it holds, the same grouped GEMM -> slot outputs
//   combine : y_t = x_t + sum_r ( sum_j w_tj * o[r][slot(t, j)] ), j then r; with
//             expert parallelism shard r's sum keeps the choices of its experts
#include <cuda.h>

#include <cstring>

#include "common.cuh"
#include "stream.cuh"
#include "tcgen05.cuh"
#include "tp_internal.h"

namespace tpk {

// Expert GEMMs (tcgen05): weight tiles of 128 rows are the MMA's A operand,
// a pass of at most kMtN of the expert's slots its N dimension.
constexpr int kMtN = 32;                          // slots per pass (MMA N: 16 or 32)
constexpr int kMtKB = 2;                          // K-blocks of 64 elements per stage
constexpr int kMtA = 128 * 64 * 2;                // one K-block of a weight tile: 16 KB
constexpr int kMtB = kMtN * 64 * 2;               // one K-block of a pass's slots: 4 KB
constexpr int kMtStage = kMtKB * (kMtA + kMtB);   // 40 KB
constexpr int kMtStages = 4;
constexpr int kMtThreads = 192;                   // copy warp, MMA warp, four read-back warps
constexpr int kMtCols = 2 * kMtN;                 // tensor-memory columns: two accumulator buffers
constexpr int kMaxExperts = 256;         // router
constexpr int kMaxBucketExperts = 64;    // bucketing (per-warp count table)

struct MoeArgs {
    CUtensorMap tw[TP_MAX_SHARDS];   // weights of the launch (egu or ed), 128-byte-swizzled boxes 64 x 16 (gate/up)
                                     // or 64 x 128 (down)
    CUtensorMap tx[TP_MAX_SHARDS];   // activations in slot order (xs or act), 128-byte-swizzled boxes 64 x 8
    MoeParams p;
    int down;                        // 0: gate/up, 1: down
};

// ---------------------------------------------------------------- route

// One token per warp: the chosen experts and their renormalised weights.
__device__ __forceinline__ void moe_route_token(const MoeParams& p, int t, int lane) {
    const float* lg = p.logits + (size_t)t * p.E;
    constexpr int kPer = kMaxExperts / 32;
    float v[kPer];
    bool taken[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int e = lane + 32 * q;
        v[q] = e < p.E ? lg[e] : -INFINITY;
        taken[q] = e >= p.E;
    }
    int sel[8];
    float sl[8];
    for (int j = 0; j < p.top_k; ++j) {
        float best = -INFINITY;
        int bi = 0x7fffffff;
        #pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int e = lane + 32 * q;
            if (!taken[q] && (v[q] > best || (v[q] == best && e < bi))) {
                best = v[q];
                bi = e;
            }
        }
        // warp arg-max, ties to the lower expert id
        for (int o = 16; o > 0; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ob > best || (ob == best && oi < bi)) {
                best = ob;
                bi = oi;
            }
        }
#pragma unroll
        for (int q = 0; q < kPer; ++q)
            if (lane + 32 * q == bi) taken[q] = true;
        sel[j] = bi;
        sl[j] = best;
    }
    if (lane == 0) {
        // softmax restricted to the chosen experts == renormalised top-k softmax
        float den = 0.f;
        for (int j = 0; j < p.top_k; ++j) den += expf(sl[j] - sl[0]);
        for (int j = 0; j < p.top_k; ++j) {
            p.ids[t * p.top_k + j] = sel[j];
            p.wts[t * p.top_k + j] = expf(sl[j] - sl[0]) / den;
        }
    }
}

__global__ void __launch_bounds__(256) moe_route_kernel(const MoeParams p) {
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t < p.T) moe_route_token(p, t, threadIdx.x & 31);
}

// ---------------------------------------------------------------- bucket (one CTA, 1024 threads)

__global__ void __launch_bounds__(1024) moe_bucket_kernel(const MoeParams p) {
    pdl_trigger();
    pdl_wait();
    __shared__ int cnt[kMaxExperts];
    __shared__ int base[kMaxExperts];
    __shared__ int wcnt[32][kMaxBucketExperts];    // per-warp counts of a 1024-slot chunk
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = p.T * p.top_k, E = p.E;
    for (int e = tid; e < E; e += 1024) cnt[e] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += 1024) atomicAdd(&cnt[p.ids[i]], 1);
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int e = 0; e < E; ++e) {
            base[e] = run;
            p.offsets[e] = run;
            run += cnt[e];
        }
        p.offsets[E] = run;
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int c0 = 0; c0 < n; c0 += 1024) {
        for (int q = tid; q < 32 * E; q += 1024) wcnt[q / E][q % E] = 0;
        __syncthreads();
        const int i = c0 + tid;
        const int e = i < n ? p.ids[i] : -1;
        const unsigned same = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(same & lt);
        if (e >= 0 && rank == 0) wcnt[warp][e] = __popc(same);
        __syncthreads();
        if (tid < E) {                       // exclusive prefix over warps, in warp order
            int run = 0;
            for (int w = 0; w < 32; ++w) {
                const int c = wcnt[w][tid];
                wcnt[w][tid] = run;
                run += c;
            }
            cnt[tid] = run;                  // this chunk's count of expert tid
        }
        __syncthreads();
        if (e >= 0) {
            const int pos = base[e] + wcnt[warp][e] + rank;
            p.perm[pos] = i;
            p.slot_of[i] = pos;
        }
        __syncthreads();
        if (tid < E) base[tid] += cnt[tid];
        __syncthreads();
    }
}

// ---------------------------------------------------------------- prep (one CTA per slot)

__global__ void __launch_bounds__(256) moe_prep_kernel(const MoeParams p) {
    pdl_trigger();
    pdl_wait();
    __shared__ float wsum[8];
    __shared__ int s_slot[8];
    const int t = blockIdx.x, tid = threadIdx.x, K = p.top_k, nslot = p.T * K;
    if (tid < K) s_slot[tid] = p.slot_of[t * K + tid];
    __syncthreads();
    // one CTA per token: its sum of squares once, x * gamma_r written to each of its slots' rows
    const float* x = p.x + (size_t)t * p.H;
    float a = 0.f;
    for (int k = tid * 4; k < p.H; k += 1024) {
        const float4 v = *reinterpret_cast<const float4*>(x + k);
        a = fmaf(v.x, v.x, a);
        a = fmaf(v.y, v.y, a);
        a = fmaf(v.z, v.z, a);
        a = fmaf(v.w, v.w, a);
        for (int r = 0; r < p.xs_copies; ++r) {
            const float4 g = *reinterpret_cast<const float4*>(p.gamma[r] + k);
            uint2 pk;
            pk.x = pack_bf16x2(v.x * g.x, v.y * g.y);
            pk.y = pack_bf16x2(v.z * g.z, v.w * g.w);
            for (int j = 0; j < K; ++j) {
                const size_t row = (size_t)r * nslot + s_slot[j];
                *reinterpret_cast<uint2*>(reinterpret_cast<bf16*>(p.xs) + row * p.H + k) = pk;
            }
        }
    }
    a = warp_sum(a);
    if ((tid & 31) == 0) wsum[tid >> 5] = a;
    __syncthreads();
    if (tid < K) {
        float ss = 0.f;
        for (int w = 0; w < 8; ++w) ss += wsum[w];
        p.rinv[s_slot[tid]] = 1.0f / sqrtf(ss / (float)p.H + p.eps);
    }
}

// ---------------------------------------------------------------- expert GEMMs
//
// Unit = (shard r, expert it holds, tile of 128 weight rows). Down: 128 rows of
// the expert's [H][Fs] slice, K = Fs. Gate/up: 64 gate rows and the matching 64
// up rows, K = H, interleaved in 16-row groups (gate rows 16q.., then up rows
// 16q..), so that tensor-memory lane quarter q holds 16 gate rows in lanes 0-15
// and their up rows in lanes 16-31 and SwiGLU pairs them with one shuffle.
//
// The weight tile is the A operand of tcgen05.mma (M = 128, one row per
// tensor-memory lane); the expert's slots, in passes of at most kMtN, are the
// B operand (N = the pass rounded up to 16). The slots arrive in boxes of 8
// rows; B rows past the pass's last box hold whatever the stage held before,
// and the accumulator columns they produce are dropped (a column of the
// product depends on its own B row only). fp32 accumulators live in tensor memory, in two
// buffers, so that one unit's read-back overlaps the next unit's MMAs.
//   warp 0, one thread: TMA copies, two K-blocks of 64 per stage, a ring of
//           four stages (weights evict-first: read once)
//   warp 1, one thread: the MMAs of a stage, then a commit that frees it
//   warps 2-5: read lane quarter (warp % 4) of the accumulator back; down
//           stores each slot's 128 outputs (fp32 partial of shard r), gate/up
//           applies 1/rms and SwiGLU and stores the bf16 activations
// Every wait is bounded; a CTA that gives up sets the status, lets its copies
// land, waits for its MMAs and frees its tensor memory before it exits.

struct MoeUnit {
    int r, le, tb, off, cnt;
};
__device__ __forceinline__ MoeUnit moe_unit(const MoeParams& p, const int* s_off, int tiles, int u) {
    MoeUnit m;
    m.tb = u % tiles;
    m.le = (u / tiles) % p.El;
    m.r = u / (tiles * p.El);
    const int e = p.ep ? m.r * p.El + m.le : m.le;   // global expert id (slot buckets)
    m.off = s_off[e];
    m.cnt = s_off[e + 1] - m.off;
    return m;
}

// DOWN: the expert down projection (else gate/up + SwiGLU), one instantiation
// each so that neither epilogue shapes the other's code.
template <bool DOWN>
__global__ void __launch_bounds__(kMtThreads, 1) moe_gemm_kernel(const __grid_constant__ MoeArgs A) {
    const MoeParams& p = A.p;
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kMtStages;
    uint64_t* acc_full = empty + kMtStages;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* done = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    unsigned char* ring = smem + 1024;                  // swizzled boxes need 1024-byte alignment
    int* s_off = reinterpret_cast<int*>(ring + kMtStages * kMtStage);   // [E+1]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int i = 0; i < kMtStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 4);                // one arrival per read-back warp
        }
        mbar_init(done, 1);
        *abort_flag = (smem_u32(ring) & 1023u) ? 1 : 0;
        if (*abort_flag) set_status(p.status, TP_ERR_ALIGN);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kMtCols);
    pdl_wait();                                         // routing, slot rows and activations of earlier kernels
    for (int i = tid; i <= p.E; i += kMtThreads) s_off[i] = p.offsets[i];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int nslot = p.T * p.top_k;
    const int K = DOWN ? p.Fs : p.H;
    const int tiles = DOWN ? p.H / 128 : p.Fs / 64;
    const int nst = K / (64 * kMtKB);                   // stages per pass
    const int U = p.N * p.El * tiles;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            uint32_t it = 0;
            bool ok = !*abort_flag;
            for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
                const MoeUnit m = moe_unit(p, s_off, tiles, u);
                const int row0 = DOWN ? m.le * p.H + m.tb * 128 : m.le * 2 * p.Fs + m.tb * 64;
                for (int ps = 0; ps < m.cnt && ok; ps += kMtN) {
                    const int nb = (min(kMtN, m.cnt - ps) + 7) / 8;     // 8-slot boxes of the pass
                    for (int st = 0; st < nst; ++st, ++it) {
                        const int s = it % kMtStages;
                        if (!mbar_wait(&empty[s], ((it / kMtStages) & 1) ^ 1, abort_flag, p.status)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[s], (uint32_t)(kMtKB * (kMtA + nb * 1024)));
                        unsigned char* sa = ring + s * kMtStage;
                        unsigned char* sb = sa + kMtKB * kMtA;
                        for (int kb = 0; kb < kMtKB; ++kb) {
                            const int x = (st * kMtKB + kb) * 64;
                            if (DOWN) {
                                tma_load_2d(sa + kb * kMtA, &A.tw[m.r], x, row0, &full[s], pol);
                            } else {
                                // 16-row groups: gate rows 16q.., then up rows 16q.. (2 KB each)
                                for (int q = 0; q < 4; ++q) {
                                    tma_load_2d(sa + kb * kMtA + q * 4096, &A.tw[m.r], x, row0 + 16 * q, &full[s], pol);
                                    tma_load_2d(sa + kb * kMtA + q * 4096 + 2048, &A.tw[m.r], x, row0 + p.Fs + 16 * q,
                                                &full[s], pol);
                                }
                            }
                            for (int i = 0; i < nb; ++i)
                                tma_load_2d_keep(sb + kb * kMtB + i * 1024, &A.tx[m.r], x, m.off + ps + 8 * i, &full[s]);
                        }
                    }
                }
            }
            pdl_trigger();
            // no copy may still be landing when the CTA exits
            volatile int no_abort = 0;
            for (uint32_t k = it > (uint32_t)kMtStages ? it - kMtStages : 0u; k < it; ++k)
                mbar_wait(&full[k % kMtStages], (k / kMtStages) & 1, &no_abort, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t it = 0, acc_i = 0;
            bool ok = !*abort_flag;
            for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
                const MoeUnit m = moe_unit(p, s_off, tiles, u);
                for (int ps = 0; ps < m.cnt && ok; ps += kMtN, ++acc_i) {
                    const int n16 = (min(kMtN, m.cnt - ps) + 15) & ~15;
                    const uint32_t idesc = idesc_bf16(128, n16);
                    const int buf = acc_i & 1;
                    if (!mbar_wait(&acc_empty[buf], ((acc_i >> 1) & 1) ^ 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)(buf * kMtN);
                    for (int st = 0; st < nst; ++st, ++it) {
                        const int s = it % kMtStages;
                        if (!mbar_wait(&full[s], (it / kMtStages) & 1, abort_flag, p.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a0 = smem_u32(ring + s * kMtStage), b0 = a0 + kMtKB * kMtA;
#pragma unroll
                        for (int kb = 0; kb < kMtKB; ++kb)
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                tc_mma(d, smem_desc_sw128(a0 + kb * kMtA + k * 32), smem_desc_sw128(b0 + kb * kMtB + k * 32),
                                       idesc, (st | kb | k) != 0);
                        tc_commit(smem_u32(&empty[s]));
                    }
                    if (ok) tc_commit(smem_u32(&acc_full[buf]));
                }
            }
            tc_commit(smem_u32(done));                  // fires when every issued MMA has completed
        }
    } else {
        const int q = warp & 3;                         // tensor-memory lane quarter of this warp
        uint32_t acc_i = 0;
        bool ok = !*abort_flag;
        for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
            const MoeUnit m = moe_unit(p, s_off, tiles, u);
            for (int ps = 0; ps < m.cnt && ok; ps += kMtN, ++acc_i) {
                const int n = min(kMtN, m.cnt - ps), buf = acc_i & 1;
                if (!mbar_wait(&acc_full[buf], (acc_i >> 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * kMtN), v);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[buf]);    // the buffer may take the next unit
                const size_t slot0 = (size_t)m.r * nslot + m.off + ps;
                if (DOWN) {
                    // lane = output row 128 tb + 32 q + lane; 32 lanes store 128 consecutive bytes per slot
                    float* o = p.o + slot0 * p.H + m.tb * 128 + 32 * q + lane;
#pragma unroll
                    for (int c = 0; c < kMtN; ++c)
                        if (c < n) o[(size_t)c * p.H] = __uint_as_float(v[c]);
                } else {
                    // lanes 0-15: gate rows j = 64 tb + 16 q + lane; lanes 16-31: the same rows' up values
                    const float rl = lane < n ? p.rinv[m.off + ps + lane] : 0.f;
                    bf16* act = reinterpret_cast<bf16*>(p.act) + slot0 * p.Fs + m.tb * 64 + 16 * q + lane;
#pragma unroll
                    for (int c = 0; c < kMtN; ++c) {
                        const float rv = __shfl_sync(0xffffffffu, rl, c);
                        const float upv = __shfl_down_sync(0xffffffffu, __uint_as_float(v[c]), 16);
                        if (c < n && lane < 16) {
                            const float gt = __uint_as_float(v[c]) * rv, up = upv * rv;
                            act[(size_t)c * p.Fs] = __float2bfloat16_rn(gt / (1.0f + expf(-gt)) * up);
                        }
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        volatile int no_abort = 0;                      // every MMA has retired before the columns are freed
        mbar_wait(done, 0, &no_abort, nullptr);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kMtCols);
        tmem_relinquish();
    }
}

// ---------------------------------------------------------------- combine
//
// y_t = x_t + sum over shards r (rank order) of sum over the token's choices j
// (descending logit) of w_tj * o[r][slot(t, j)]. One CTA per (token, 512-column
// block), one float4 column group per thread. The token's slots and weights
// are staged in shared memory once; the (r, j) terms are walked in that order
// in batches of 16 whose loads are all issued before any is summed, so a
// thread waits about one memory round trip per batch.
constexpr int kCombineCols = 512, kCombineBatch = 16;

__global__ void __launch_bounds__(kCombineCols / 4) moe_combine_kernel(const MoeParams p) {
    __shared__ int s_slot[8];
    __shared__ int s_owner[8];
    __shared__ float s_w[8];
    pdl_trigger();
    pdl_wait();
    const int nhb = (p.H + kCombineCols - 1) / kCombineCols;
    const int t = blockIdx.x / nhb, h = (blockIdx.x - t * nhb) * kCombineCols + threadIdx.x * 4;
    const int nslot = p.T * p.top_k, K = p.top_k, nterm = p.N * K;
    if (threadIdx.x < K) {
        const int f = t * K + threadIdx.x;
        s_slot[threadIdx.x] = p.slot_of[f];
        s_w[threadIdx.x] = p.wts[f];
        s_owner[threadIdx.x] = p.ep ? p.ids[f] / p.El : -1;   // -1: every shard holds a slice
    }
    __syncthreads();
    if (h >= p.H) return;
    const float* o = p.o + h;
    float4 total = make_float4(0.f, 0.f, 0.f, 0.f), acc = total;
    int r0 = 0, j0 = 0;                                 // the batch's first term
    #pragma unroll 1
    for (int b0 = 0; b0 < nterm; b0 += kCombineBatch) {
        float4 v[kCombineBatch];
        int r = r0, j = j0;
#pragma unroll
        for (int u = 0; u < kCombineBatch; ++u) {
            if (b0 + u < nterm && (s_owner[j] < 0 || s_owner[j] == r))
                v[u] = *reinterpret_cast<const float4*>(o + ((size_t)r * nslot + s_slot[j]) * p.H);
            if (++j == K) { j = 0; ++r; }
        }
        r = r0;
        j = j0;
#pragma unroll
        for (int u = 0; u < kCombineBatch; ++u) {
            if (b0 + u < nterm) {
                if (j == 0 && r > 0) {                  // shard r-1 done: ((p0 + p1) + p2) + ...
                    if (r == 1) total = acc;
                    else { total.x += acc.x; total.y += acc.y; total.z += acc.z; total.w += acc.w; }
                    acc = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if (s_owner[j] < 0 || s_owner[j] == r) {
                    const float w = s_w[j];
                    acc.x = fmaf(w, v[u].x, acc.x);
                    acc.y = fmaf(w, v[u].y, acc.y);
                    acc.z = fmaf(w, v[u].z, acc.z);
                    acc.w = fmaf(w, v[u].w, acc.w);
                }
            }
            if (++j == K) { j = 0; ++r; }
        }
        r0 = r;
        j0 = j;
    }
    if (p.N == 1) total = acc;
    else { total.x += acc.x; total.y += acc.y; total.z += acc.z; total.w += acc.w; }
    const float4 xv = *reinterpret_cast<const float4*>(p.x + (size_t)t * p.H + h);
    *reinterpret_cast<float4*>(p.y + (size_t)t * p.H + h) =
        make_float4(xv.x + total.x, xv.y + total.y, xv.z + total.z, xv.w + total.w);
}

// ---------------------------------------------------------------- launch sequence

static size_t moe_gemm_smem(int E) { return 1024 + (size_t)kMtStages * kMtStage + (size_t)(E + 1) * 4 + 16; }

static cudaError_t launch_small(const void* fn, void* arg, int grid, int threads, cudaStream_t s) {
    void* args[] = {arg};
    return launch_pdl(fn, args, grid, 0, s, threads);
}

cudaError_t launch_moe(const MoeParams& p, cudaStream_t s, cudaEvent_t const* marks, int n_marks) {
    MoeParams q = p;
    auto mark = [&](int i) {
        if (i < n_marks && marks[i]) cudaEventRecord(marks[i], s);
    };
    mark(0);
    // one normalised copy of the slots' activations when every shard shares the gamma
    q.xs_copies = p.N;
    bool same = true;
    for (int r = 1; r < p.N; ++r) same = same && p.gamma[r] == p.gamma[0];
    if (same) q.xs_copies = 1;
    cudaError_t e = launch_small(reinterpret_cast<const void*>(moe_route_kernel), &q, (p.T + 7) / 8, 256, s);
    if (e == cudaSuccess) e = launch_small(reinterpret_cast<const void*>(moe_bucket_kernel), &q, 1, 1024, s);
    if (e == cudaSuccess) e = launch_small(reinterpret_cast<const void*>(moe_prep_kernel), &q, p.T, 256, s);
    if (e != cudaSuccess) return e;
    mark(1);
    // the expert GEMMs take K in stages of 128 and weight tiles of 128 rows
    if (p.H % 128 || p.Fs % 128 || p.E > kMaxBucketExperts) return cudaErrorInvalidValue;
    const size_t smem = moe_gemm_smem(p.E);
    static int set_bytes = -1;
    if ((int)smem > set_bytes) {
        e = cudaFuncSetAttribute(moe_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(moe_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        set_bytes = (int)smem;
    }
    const long nslot = (long)p.T * p.top_k;
    for (int down = 0; down < 2; ++down) {
        MoeArgs A;
        memset(&A, 0, sizeof A);
        A.p = q;
        A.down = down;
        for (int r = 0; r < p.N; ++r) {
            if (down) {
                e = tensor_map_2d(p.ed[r], p.Fs, (long)p.El * p.H, 64, 128, 1, &A.tw[r]);
                if (e == cudaSuccess)
                    e = tensor_map_2d(static_cast<const bf16*>(p.act) + (size_t)r * nslot * p.Fs, p.Fs, nslot, 64, 8, 1,
                                      &A.tx[r]);
            } else {
                e = tensor_map_2d(p.egu[r], p.H, (long)p.El * 2 * p.Fs, 64, 16, 1, &A.tw[r]);
                if (e == cudaSuccess)
                    e = tensor_map_2d(static_cast<const bf16*>(p.xs) + (size_t)(q.xs_copies > 1 ? r : 0) * nslot * p.H,
                                      p.H, nslot, 64, 8, 1, &A.tx[r]);
            }
            if (e != cudaSuccess) return e;
        }
        const int U = p.N * p.El * (down ? p.H / 128 : p.Fs / 64);
        void* args[] = {&A};
        const void* fn = down ? reinterpret_cast<const void*>(moe_gemm_kernel<true>)
                              : reinterpret_cast<const void*>(moe_gemm_kernel<false>);
        e = launch_pdl(fn, args, U < kSMs ? U : kSMs, smem, s, kMtThreads);
        if (e != cudaSuccess) return e;
        mark(2 + down);
    }
    e = launch_small(reinterpret_cast<const void*>(moe_combine_kernel), &q,
                     p.T * ((p.H + kCombineCols - 1) / kCombineCols), kCombineCols / 4, s);
    mark(4);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace tpk
