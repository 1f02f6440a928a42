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
//   gate/up : per shard and expert it holds, streaming grouped GEMM over the
//             expert's slots, SwiGLU epilogue
//   down    : per shard and expert it holds, streaming grouped GEMM -> slot outputs
//   combine : y_t = x_t + sum_r ( sum_j w_tj * o[r][slot(t, j)] ), j then r; with
//             expert parallelism shard r's sum keeps the choices of its experts
#include <cuda.h>

#include <cstring>

#include "common.cuh"
#include "stream.cuh"
#include "tp_internal.h"

namespace tpk {

constexpr int kMoeTokPass = 32;                        // slots per pass of a unit (4 MMA column groups)
constexpr int kMoeGroups = kMoeTokPass / 8;
constexpr int kMoeXBytes = kMoeGroups * kBoxK * 8 * 2; // 4 activation boxes of 8 rows x 256
constexpr int kMoeStageBytes = 2 * kBoxBytes + kMoeXBytes;
constexpr int kMoeStages = 4;
constexpr int kMoeTG = 4;                // down projection with one stage per tile: tiles per unit
constexpr int kMoeTS = kMoeTokPass + 1;  // tile row stride in shared memory (column reads free of bank conflicts)
constexpr int kMaxExperts = 256;         // router
constexpr int kMaxBucketExperts = 64;    // bucketing (per-warp count table)

struct MoeArgs {
    CUtensorMap tw[TP_MAX_SHARDS];   // weights of the launch (egu or ed), 128-byte-swizzled boxes of 32 rows x 256
    CUtensorMap tx[TP_MAX_SHARDS];   // activations in slot order (xs or act), swizzled boxes of 8 rows x 256
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

// ---------------------------------------------------------------- grouped streaming GEMM
//
// Unit = (shard r, expert e, group of tiles of 64 rows). Gate/up: rows are 32
// gate + the matching 32 up rows of the expert's shard slice, K = H, one tile
// per unit. Down: 64 rows of H, K = Fs; when Fs fits one stage, a unit takes
// kMoeTG tiles of the same expert, whose activation boxes arrive with the first
// stage only and stay in registers for the rest. The expert's slots are
// processed in passes of 32 (four 8-column MMA groups).

// DOWN: the expert down projection (else gate/up + SwiGLU), one instantiation
// each so that neither epilogue shapes the other's code.
template <bool DOWN>
__global__ void __launch_bounds__(kStreamThreads, 1) moe_gemm_kernel(const __grid_constant__ MoeArgs A) {
    const MoeParams& p = A.p;
    extern __shared__ __align__(1024) unsigned char smem[];
    const Ring R = ring_setup(smem, kMoeStages);
    unsigned char* ring = smem + 1024;                  // swizzled boxes need 1024-byte alignment
    float* tile = reinterpret_cast<float*>(ring + kMoeStages * kMoeStageBytes);   // [2][64][kMoeTS]
    int* s_off = reinterpret_cast<int*>(tile + 2 * kTileRows * kMoeTS);           // [E+1]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr bool down = DOWN;
    const int nslot = p.T * p.top_k;
    const int tiles = down ? p.H / kTileRows : (2 * p.Fs) / kTileRows;
    const int K = down ? p.Fs : p.H;
    const int spu = (K + kBoxK - 1) / kBoxK;
    const int TG = (down && spu == 1) ? kMoeTG : 1;     // tiles per unit sharing the activation boxes
    const int ngrp = (tiles + TG - 1) / TG;
    const int U = p.N * p.El * ngrp;                   // units: (shard, expert it holds, tile group)

    if (warp == kConsumers / 32) {                     // ---- producer
        if (lane == 0) {
            pdl_wait();                                // routing and activations come from earlier kernels
            const uint64_t pol = l2_evict_first_policy();
            uint32_t it = 0;
            bool ok = (smem_u32(ring) & 1023u) == 0;
            if (!ok) {
                *R.abort = 1;
                set_status(p.status, TP_ERR_ALIGN);
            }
            for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
                const int tg = u % ngrp, le = (u / ngrp) % p.El, r = u / (ngrp * p.El);
                const int e = p.ep ? r * p.El + le : le;     // global expert id (slot buckets)
                const int ntg = min(TG, tiles - tg * TG);
                const int off = p.offsets[e], cnt = p.offsets[e + 1] - off;
                for (int ps = 0; ps < cnt && ok; ps += kMoeTokPass) {
                    const int ng = min(kMoeGroups, (cnt - ps + 7) / 8);
                    for (int i = 0; i < ntg && ok; ++i) {
                        const int tb = tg * TG + i;
                        int rowa, rowb;
                        if (down) {
                            rowa = le * p.H + tb * kTileRows;
                            rowb = rowa + 32;
                        } else {
                            rowa = le * 2 * p.Fs + tb * 32;
                            rowb = rowa + p.Fs;
                        }
                        const int nx = (TG == 1 || i == 0) ? ng : 0;    // activation boxes of this stage
                        for (int st = 0; st < spu; ++st, ++it) {
                            const int sl = it % kMoeStages;
                            if (!mbar_wait(&R.empty[sl], ((it / kMoeStages) & 1) ^ 1, R.abort, p.status)) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(&R.full[sl], 2u * kBoxBytes + (uint32_t)nx * kBoxK * 8 * 2);
                            unsigned char* dst = ring + sl * kMoeStageBytes;
                            tma_load_3d_hint(dst, &A.tw[r], 0, st * (kBoxK / 64), rowa, &R.full[sl], pol);
                            tma_load_3d_hint(dst + kBoxBytes, &A.tw[r], 0, st * (kBoxK / 64), rowb, &R.full[sl], pol);
                            for (int g = 0; g < nx; ++g)
                                tma_load_3d_keep(dst + 2 * kBoxBytes + g * kBoxK * 8 * 2, &A.tx[r], 0,
                                                 st * (kBoxK / 64), off + ps + 8 * g, &R.full[sl]);
                        }
                    }
                }
            }
            pdl_trigger();
            if (!ok || *R.abort) producer_drain(R, it, kMoeStages);
        }
        return;
    }

    // ---- consumers
    pdl_wait();
    for (int i = tid; i <= p.E; i += kConsumers) s_off[i] = p.offsets[i];
    consumer_sync(kConsumers);
    const int wm = warp & 3, wk = warp >> 2;
    const int g = lane >> 2, tq = lane & 3;
    const int box = wm >> 1, brow = 16 * (wm & 1) + g;
    uint32_t it = 0, ntile = 0;
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
        const int tg = u % ngrp, le = (u / ngrp) % p.El, r = u / (ngrp * p.El);
        const int e = p.ep ? r * p.El + le : le;
        const int ntg = min(TG, tiles - tg * TG);
        const int off = s_off[e], cnt = s_off[e + 1] - off;
        for (int ps = 0; ps < cnt; ps += kMoeTokPass) {
            const int ng = min(kMoeGroups, (cnt - ps + 7) / 8);
            uint4 xr[2][2][kMoeGroups];                 // activation fragments (kept across a unit's tiles)
            for (int i = 0; i < ntg; ++i) {
                const int tb = tg * TG + i;
                float c[kMoeGroups][4];
#pragma unroll
                for (int q = 0; q < kMoeGroups; ++q) c[q][0] = c[q][1] = c[q][2] = c[q][3] = 0.f;
                for (int st = 0; st < spu; ++st, ++it) {
                    const int sl = it % kMoeStages;
                    mbar_wait(&R.full[sl], (it / kMoeStages) & 1, R.abort, p.status);
                    __syncwarp();
                    const int steps_here = min(kBoxK / kKStep, (K - st * kBoxK) / kKStep);
                    // 128-byte-swizzled boxes: 16-byte unit u of the 128-byte row (row, chunk c)
                    // sits at unit u ^ ((4 * row + c) & 7); every row a lane reads has parity g & 1
                    const unsigned char* stage = ring + sl * kMoeStageBytes;
                    const unsigned char* wA = stage + box * kBoxBytes + brow * (kBoxK * 2);
                    const unsigned char* wB = wA + 8 * (kBoxK * 2);
                    if (TG == 1 || i == 0) {
#pragma unroll
                        for (int s2 = 0; s2 < 2; ++s2)
#pragma unroll
                            for (int h = 0; h < 2; ++h)
#pragma unroll
                                for (int q = 0; q < kMoeGroups; ++q)
                                    if (wk + 2 * s2 < steps_here && q < ng) {
                                        const int step = wk + 2 * s2;
                                        xr[s2][h][q] = *reinterpret_cast<const uint4*>(
                                            stage + 2 * kBoxBytes + q * kBoxK * 16 + g * (kBoxK * 2) + step * 128 +
                                            ((h ^ (g & 1)) << 6) + ((tq ^ step) << 4));
                                    }
                    }
#pragma unroll
                    for (int s2 = 0; s2 < 2; ++s2) {
                        const int step = wk + 2 * s2;
                        if (step < steps_here) {
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int off_w = step * 128 + ((h ^ (g & 1)) << 6) + ((tq ^ step) << 4);
                                const uint4 a = *reinterpret_cast<const uint4*>(wA + off_w);
                                const uint4 b = *reinterpret_cast<const uint4*>(wB + off_w);
#pragma unroll
                                for (int q = 0; q < kMoeGroups; ++q) {
                                    if (q < ng) {
                                        const uint4 xv = xr[s2][h][q];
                                        mma_bf16_16816(c[q], a.x, b.x, a.y, b.y, xv.x, xv.y);
                                        mma_bf16_16816(c[q], a.z, b.z, a.w, b.w, xv.z, xv.w);
                                    }
                                }
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&R.empty[sl]);
                }
                if constexpr (DOWN) {
                    // the second K half parks its sums in one of two tile buffers; after one barrier the
                    // first half adds them (half 0 + half 1) and stores the expert's output rows from
                    // registers: lanes g = 0..7 write 8 consecutive rows of one slot. The next tile
                    // writes the other buffer, so no barrier is needed after the reads.
                    float* tb2 = tile + (ntile & 1) * (kTileRows * kMoeTS);
                    ++ntile;
                    if (wk == 1) {
#pragma unroll
                        for (int q = 0; q < kMoeGroups; ++q) {
                            const int c0 = 8 * q + 2 * tq;
                            const int i0 = (16 * wm + g) * kMoeTS + c0, i1 = (16 * wm + g + 8) * kMoeTS + c0;
                            tb2[i0] = c[q][0];
                            tb2[i0 + 1] = c[q][1];
                            tb2[i1] = c[q][2];
                            tb2[i1 + 1] = c[q][3];
                        }
                    }
                    consumer_sync(kConsumers);
                    if (wk == 0) {
                        const int nt = min(kMoeTokPass, cnt - ps);
                        const int row0 = tb * kTileRows + 16 * wm + g;
#pragma unroll
                        for (int q = 0; q < kMoeGroups; ++q) {
                            const int c0 = 8 * q + 2 * tq;
                            const int i0 = (16 * wm + g) * kMoeTS + c0, i1 = (16 * wm + g + 8) * kMoeTS + c0;
#pragma unroll
                            for (int e2 = 0; e2 < 2; ++e2) {
                                if (c0 + e2 < nt) {
                                    float* o = p.o + ((size_t)r * nslot + off + ps + c0 + e2) * p.H + row0;
                                    o[0] = c[q][e2] + tb2[i0 + e2];
                                    o[8] = c[q][2 + e2] + tb2[i1 + e2];
                                }
                            }
                        }
                    }
                } else {
                    // gate/up: tile[row][slot] = half 0 + half 1
#pragma unroll
                    for (int q = 0; q < kMoeGroups; ++q) {
                        const int c0 = 8 * q + 2 * tq;
                        const int i0 = (16 * wm + g) * kMoeTS + c0, i1 = (16 * wm + g + 8) * kMoeTS + c0;
                        if (wk == 0) {
                            tile[i0] = c[q][0];
                            tile[i0 + 1] = c[q][1];
                            tile[i1] = c[q][2];
                            tile[i1 + 1] = c[q][3];
                        }
                    }
                    consumer_sync(kConsumers);
#pragma unroll
                    for (int q = 0; q < kMoeGroups; ++q) {
                        const int c0 = 8 * q + 2 * tq;
                        const int i0 = (16 * wm + g) * kMoeTS + c0, i1 = (16 * wm + g + 8) * kMoeTS + c0;
                        if (wk == 1) {
                            tile[i0] += c[q][0];
                            tile[i0 + 1] += c[q][1];
                            tile[i1] += c[q][2];
                            tile[i1 + 1] += c[q][3];
                        }
                    }
                    consumer_sync(kConsumers);
                    {
                        const int nt = min(kMoeTokPass, cnt - ps);
                        bf16* act = reinterpret_cast<bf16*>(p.act);
                        for (int i2 = tid; i2 < 32 * nt; i2 += kConsumers) {   // 32 consecutive outputs per slot
                            const int q = i2 >> 5, j = i2 & 31;
                            const int slot = off + ps + q;
                            const float rv = p.rinv[slot];
                            const float gt = tile[j * kMoeTS + q] * rv;
                            const float up = tile[(j + 32) * kMoeTS + q] * rv;
                            act[((size_t)r * nslot + slot) * p.Fs + tb * 32 + j] =
                                __float2bfloat16_rn(gt / (1.0f + expf(-gt)) * up);
                        }
                    }
                    consumer_sync(kConsumers);
                }
            }
        }
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

static size_t moe_gemm_smem(int E) {
    return 1024 + (size_t)kMoeStages * kMoeStageBytes + (size_t)2 * kTileRows * kMoeTS * 4 +
           (size_t)(E + 1) * 4 + 16;
}

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
                e = step_stage_map(p.ed[r], p.Fs, p.El * p.H, 32, &A.tw[r]);
                if (e == cudaSuccess)
                    e = step_stage_map(static_cast<const bf16*>(p.act) + (size_t)r * nslot * p.Fs, p.Fs, (int)nslot, 8,
                                       &A.tx[r]);
            } else {
                e = step_stage_map(p.egu[r], p.H, p.El * 2 * p.Fs, 32, &A.tw[r]);
                if (e == cudaSuccess)
                    e = step_stage_map(static_cast<const bf16*>(p.xs) + (size_t)(q.xs_copies > 1 ? r : 0) * nslot * p.H,
                                       p.H, (int)nslot, 8, &A.tx[r]);
            }
            if (e != cudaSuccess) return e;
        }
        const int tiles = down ? p.H / kTileRows : 2 * p.Fs / kTileRows;
        const int TG = (down && (p.Fs + kBoxK - 1) / kBoxK == 1) ? kMoeTG : 1;
        const int U = p.N * p.El * ((tiles + TG - 1) / TG);
        void* args[] = {&A};
        const void* fn = down ? reinterpret_cast<const void*>(moe_gemm_kernel<true>)
                              : reinterpret_cast<const void*>(moe_gemm_kernel<false>);
        e = launch_pdl(fn, args, U < kSMs ? U : kSMs, smem, s, kStreamThreads);
        if (e != cudaSuccess) return e;
        mark(2 + down);
    }
    e = launch_small(reinterpret_cast<const void*>(moe_combine_kernel), &q,
                     p.T * ((p.H + kCombineCols - 1) / kCombineCols), kCombineCols / 4, s);
    mark(4);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace tpk
