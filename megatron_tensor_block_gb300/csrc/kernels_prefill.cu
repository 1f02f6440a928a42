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

#include <algorithm>

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
    CUtensorMap tb;       // B [N, K] boxes 64 x 256, or (B_KN) B [K, N] boxes 64 x 64; 128-byte swizzle
    float* C;             // [M, N]
    int M, N, K;
    int* status;
};

template <bool B_KN>
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
                if (B_KN) {
                    // four [64 K x 64 N] boxes: the tile's N range in 64-element atoms
#pragma unroll
                    for (int nb = 0; nb < kTcBN / 64; ++nb)
                        tma_load_2d_keep(st + kTcABytes + nb * 8192, &g.tb, n0 + nb * 64, kb * kTcBK, &full[s]);
                } else {
                    tma_load_2d_keep(st + kTcABytes, &g.tb, kb * kTcBK, n0, &full[s]);
                }
            }
            // no copy may still be landing when the CTA exits
            volatile int no_abort = 0;
            for (int k = kb > kTcStages ? kb - kTcStages : 0; k < kb; ++k)
                mbar_wait(&full[k % kTcStages], (k / kTcStages) & 1, &no_abort, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = B_KN ? idesc_bf16_bmn(kTcBM, kTcBN) : idesc_bf16(kTcBM, kTcBN);
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
                for (int k = 0; k < kTcBK / 16; ++k) {
                    // MN-major B: 16 K rows of 128 bytes per step; 64-element N atoms 8 KB apart
                    const uint64_t bd = B_KN ? smem_desc_mn_sw128(b0 + k * 2048, 8192, 1024) : smem_desc_sw128(b0 + k * 32);
                    tc_mma(tmem, smem_desc_sw128(a0 + k * 32), bd, idesc, (kb | k) != 0);
                }
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
                                 cudaStream_t s, bool b_kn) {
    TcGemmArgs g;
    memset(&g, 0, sizeof g);
    cudaError_t e = tensor_map_2d(A, K, M, kTcBK, kTcBM, 1, &g.ta);
    if (e == cudaSuccess) e = b_kn ? tensor_map_2d(B, N, K, 64, kTcBK, 1, &g.tb) : tensor_map_2d(B, K, N, kTcBK, kTcBN, 1, &g.tb);
    if (e != cudaSuccess) return e;
    g.C = C;
    g.M = M;
    g.N = N;
    g.K = K;
    g.status = status;
    static bool set[2] = {false, false};
    if (!set[b_kn]) {
        e = cudaFuncSetAttribute(b_kn ? tc_gemm_plain_kernel<true> : tc_gemm_plain_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
        if (e != cudaSuccess) return e;
        set[b_kn] = true;
    }
    dim3 grid(M / kTcBM, N / kTcBN);
    if (b_kn) tc_gemm_plain_kernel<true><<<grid, kTcThreads, kTcSmem, s>>>(g);
    else tc_gemm_plain_kernel<false><<<grid, kTcThreads, kTcSmem, s>>>(g);
    return cudaGetLastError();
}

}  // namespace tpk

namespace tpk {

// ---------------------------------------------------------------------------
// shared pieces of the fused projections
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tc_setup(unsigned char* smem, int nfull, int nempty, uint32_t tmem_cols,
                                         int* status, uint64_t*& full, uint64_t*& empty, uint64_t*& extra,
                                         uint32_t*& tmem_slot, volatile int*& abort_flag, int n_extra,
                                         const uint32_t* extra_counts) {
    full = reinterpret_cast<uint64_t*>(smem);
    empty = full + nfull;
    extra = empty + nempty;
    tmem_slot = reinterpret_cast<uint32_t*>(extra + n_extra);
    abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    if (threadIdx.x == 0) {
        for (int i = 0; i < nfull; ++i) mbar_init(&full[i], 1);
        for (int i = 0; i < nempty; ++i) mbar_init(&empty[i], 1);
        for (int i = 0; i < n_extra; ++i) mbar_init(&extra[i], extra_counts[i]);
        *abort_flag = (smem_u32(smem + 1024) & 1023u) ? 1 : 0;
        if (*abort_flag) set_status(status, TP_ERR_ALIGN);
        fence_mbar_init();
    }
    if ((threadIdx.x >> 5) == 1) tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

__device__ __forceinline__ void tc_teardown(uint64_t* done_bar, uint32_t done_parity, uint32_t tmem,
                                            uint32_t cols) {
    tc_fence_before();
    __syncthreads();
    if ((threadIdx.x >> 5) == 1) {
        volatile int no_abort = 0;
        if (done_bar) mbar_wait(done_bar, done_parity, &no_abort, nullptr);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, cols);
        tmem_relinquish();
    }
}

__device__ __forceinline__ float fbits(uint32_t u) { return __uint_as_float(u); }

// ---------------------------------------------------------------------------
// column-parallel projection with fused epilogue (QKV + RoPE + KV append, or
// gate/up + SwiGLU). Persistent: one CTA per SM walks the 128-token x
// 256-column tiles of every shard; two accumulators in tensor memory
// (2 x 256 columns) let the epilogue of one tile run while the MMAs of the
// next are issued, and the TMA producer runs ahead across tile boundaries.
// ---------------------------------------------------------------------------

enum TcMode : int { TC_QKV = 0, TC_GATEUP = 1 };

struct TcColArgs {
    CUtensorMap ta;                       // normalised activations [copies * T, K], boxes 64 x 128
    CUtensorMap tb[TP_MAX_SHARDS];        // QKV: [qkv_rows, K] boxes 64 x 256; gate/up: [2F', K] boxes 64 x 128
    int T, K, S;                          // tokens, reduction length, tokens per sequence
    int a_row_stride;                     // first A row of shard r = r * a_row_stride (0: shared copy)
    int n_mt, n_nt, N;                    // tiles: token tiles, column tiles per shard, shards
    int gm;                               // token tiles per group (tile order, below)
    int hq_s, hkv_s, d, max_kv, ffn_s;
    const float* bias[TP_MAX_SHARDS];
    const int* pos;                       // [B] first new position of each sequence
    const float2* rope;                   // [max_kv][d/2] (cos, sin)
    bf16* q_out;                          // [N][T][hq_s * d]
    void* kcache[TP_MAX_SHARDS];
    void* vcache[TP_MAX_SHARDS];
    bf16* act;                            // [N][T][F']
    int* status;
};

// tile -> (token tile, column tile, shard). The token tiles are taken in
// groups of gm whose activations fit in L2 with room to spare; within a group
// token tiles vary fastest, so that the CTAs resident at one time share the
// weight tiles they stream, and the group's activations stay in L2 while every
// column tile of every shard passes over them. The weights are read once per
// group, the activations about once.
__device__ __forceinline__ void col_tile(const TcColArgs& g, int tile, int& mt, int& nt, int& r) {
    const int per_g = g.gm * g.n_nt * g.N, grp = tile / per_g, local = tile - grp * per_g;
    const int m0 = grp * g.gm, gm = min(g.gm, g.n_mt - m0);
    mt = m0 + local % gm;
    const int rest = local / gm;
    nt = rest % g.n_nt;
    r = rest / g.n_nt;
}

template <int MODE>
__device__ __forceinline__ void col_epilogue(const TcColArgs& g, uint32_t acc, int mt, int nt, int r, int q, int lane,
                                             bool ok) {
    const int t = mt * kTcBM + 32 * q + lane;
    const bool live = ok && t < g.T;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    if (MODE == TC_GATEUP) {
        for (int c = 0; c < 4; ++c) {
            if (nt * 128 + 32 * c >= g.ffn_s) break;      // ragged last tile (warp-uniform)
            uint32_t gv[32], uv[32];
            tmem_ld32(acc + lane_off + 32 * c, gv);
            tmem_ld32(acc + lane_off + 128 + 32 * c, uv);
            tmem_wait_ld();
            if (live) {
                bf16* dst = g.act + ((size_t)r * g.T + t) * g.ffn_s + nt * 128 + 32 * c;
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    uint4 pk;
                    uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
                    for (int j = 0; j < 8; j += 2) {
                        const float g0 = fbits(gv[i + j]), g1 = fbits(gv[i + j + 1]);
                        const float a0 = g0 / (1.0f + expf(-g0)) * fbits(uv[i + j]);
                        const float a1 = g1 / (1.0f + expf(-g1)) * fbits(uv[i + j + 1]);
                        w[j / 2] = pack_bf16x2(a0, a1);
                    }
                    *reinterpret_cast<uint4*>(dst + i) = pk;
                }
            }
        }
        return;
    }
    const int d = g.d, half = d >> 1;
    const int b = t / g.S, sidx = t - b * g.S;
    const int p = live ? g.pos[b] + sidx : 0;
    const bool in_cache = p >= 0 && p < g.max_kv;
    if (live && !in_cache) set_status(g.status, TP_ERR_CAPACITY);
    const int pr = in_cache ? p : 0;                     // rotary table row (in range on every path)
    const int n_heads = g.hq_s + 2 * g.hkv_s;
    for (int hh = 0; hh < kTcBN / d; ++hh) {
        const int head = (nt * kTcBN) / d + hh;
        if (head >= n_heads) break;                       // ragged last tile (warp-uniform)
        const bool is_q = head < g.hq_s;
        const bool is_k = !is_q && head < g.hq_s + g.hkv_s;
        const bool rot = is_q || is_k;
        bf16* qdst = g.q_out + ((size_t)r * g.T + t) * g.hq_s * d + head * d;
        bf16* cdst = nullptr;
        if (!is_q && in_cache && live) {
            const int kvh = is_k ? head - g.hq_s : head - g.hq_s - g.hkv_s;
            bf16* cache = reinterpret_cast<bf16*>(is_k ? g.kcache[r] : g.vcache[r]);
            cdst = cache + (((size_t)b * g.hkv_s + kvh) * g.max_kv + p) * d;
        }
        const float* bias = g.bias[r];
        for (int c = 0; c < half / 32; ++c) {
            uint32_t lo[32], hi[32];
            tmem_ld32(acc + lane_off + hh * d + 32 * c, lo);
            tmem_ld32(acc + lane_off + hh * d + half + 32 * c, hi);
            tmem_wait_ld();
            if (!live) continue;
            uint32_t plo[16], phi[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                float va0 = fbits(lo[i]), va1 = fbits(lo[i + 1]);
                float vb0 = fbits(hi[i]), vb1 = fbits(hi[i + 1]);
                if (bias) {
                    const int col = head * d + 32 * c + i;
                    va0 += bias[col];
                    va1 += bias[col + 1];
                    vb0 += bias[col + half];
                    vb1 += bias[col + half + 1];
                }
                if (rot) {
                    const float2 cs0 = g.rope[(size_t)pr * half + 32 * c + i];
                    const float2 cs1 = g.rope[(size_t)pr * half + 32 * c + i + 1];
                    const float ra0 = va0 * cs0.x - vb0 * cs0.y, rb0 = va0 * cs0.y + vb0 * cs0.x;
                    const float ra1 = va1 * cs1.x - vb1 * cs1.y, rb1 = va1 * cs1.y + vb1 * cs1.x;
                    va0 = ra0;
                    vb0 = rb0;
                    va1 = ra1;
                    vb1 = rb1;
                }
                plo[i / 2] = pack_bf16x2(va0, va1);
                phi[i / 2] = pack_bf16x2(vb0, vb1);
            }
            bf16* dst = is_q ? qdst : cdst;
            if (dst) {
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    *reinterpret_cast<uint4*>(dst + 32 * c + 2 * i) = make_uint4(plo[i], plo[i + 1], plo[i + 2], plo[i + 3]);
                    *reinterpret_cast<uint4*>(dst + half + 32 * c + 2 * i) =
                        make_uint4(phi[i], phi[i + 1], phi[i + 2], phi[i + 3]);
                }
            }
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(kTcThreads, 1) tc_col_kernel(const __grid_constant__ TcColArgs g) {
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t *full, *empty, *extra;
    uint32_t* tmem_slot;
    volatile int* abort_flag;
    const uint32_t counts[5] = {1, 1, 4, 4, 1};   // acc full x2, acc empty x2 (epilogue warps), done
    tc_setup(smem, kTcStages, kTcStages, 512, g.status, full, empty, extra, tmem_slot, abort_flag, 5, counts);
    uint64_t* acc_full = extra;
    uint64_t* acc_empty = extra + 2;
    uint64_t* done = extra + 4;
    const uint32_t tmem = *tmem_slot;
    unsigned char* stages = smem + 1024;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = g.K / kTcBK;
    const int ntiles = g.n_mt * g.n_nt * g.N;

    if (warp == 0) {
        if (lane == 0 && !*abort_flag) {
            uint32_t it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                int mt, nt, r;
                col_tile(g, tile, mt, nt, r);
                const int arow = r * g.a_row_stride + mt * kTcBM;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % kTcStages;
                    if (!mbar_wait(&empty[s], ((it / kTcStages) & 1) ^ 1, abort_flag, g.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], kTcStageBytes);
                    unsigned char* st = stages + s * kTcStageBytes;
                    tma_load_2d_keep(st, &g.ta, kb * kTcBK, arow, &full[s]);
                    if (MODE == TC_QKV) {
                        tma_load_2d_keep(st + kTcABytes, &g.tb[r], kb * kTcBK, nt * kTcBN, &full[s]);
                    } else {   // 128 gate rows, then the matching 128 up rows
                        tma_load_2d_keep(st + kTcABytes, &g.tb[r], kb * kTcBK, nt * 128, &full[s]);
                        tma_load_2d_keep(st + kTcABytes + kTcBBytes / 2, &g.tb[r], kb * kTcBK, g.ffn_s + nt * 128,
                                         &full[s]);
                    }
                }
            }
            volatile int no_abort = 0;         // no copy may still be landing when the CTA exits
            for (uint32_t k = it > (uint32_t)kTcStages ? it - kTcStages : 0; k < it; ++k)
                mbar_wait(&full[k % kTcStages], (k / kTcStages) & 1, &no_abort, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kTcBM, kTcBN);
            uint32_t it = 0;
            bool ok = !*abort_flag;
            int li = 0;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++li) {
                const int buf = li & 1;
                if (!mbar_wait(&acc_empty[buf], ((li >> 1) & 1) ^ 1, abort_flag, g.status)) break;
                tc_fence_after();
                const uint32_t acc = tmem + 256 * buf;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % kTcStages;
                    if (!mbar_wait(&full[s], (it / kTcStages) & 1, abort_flag, g.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(stages + s * kTcStageBytes), b0 = a0 + kTcABytes;
#pragma unroll
                    for (int k = 0; k < kTcBK / 16; ++k)
                        tc_mma(acc, smem_desc_sw128(a0 + k * 32), smem_desc_sw128(b0 + k * 32), idesc, (kb | k) != 0);
                    tc_commit(smem_u32(&empty[s]));
                }
                if (ok) tc_commit(smem_u32(&acc_full[buf]));
            }
            tc_commit(smem_u32(done));                // fires when every issued MMA has completed
        }
    } else {
        const int q = warp & 3;                        // warps 2..5 -> tensor-memory lane quarters 2,3,0,1
        int li = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++li) {
            const int buf = li & 1;
            bool ok = mbar_wait(&acc_full[buf], (li >> 1) & 1, abort_flag, g.status);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            if (ok) {
                int mt, nt, r;
                col_tile(g, tile, mt, nt, r);
                col_epilogue<MODE>(g, tmem + 256 * buf, mt, nt, r, q, lane, true);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
            if (!ok) break;
        }
    }
    tc_teardown(done, 0, tmem, 512);
}

// ---------------------------------------------------------------------------
// row-parallel projection with the rank-ordered reduction: for one
// 128-token x 256-column output tile, shard r's partial product is
// accumulated in its own tensor-memory buffer (two buffers alternate, so the
// MMAs of shard r+1 run while shard r's partial is read), and the epilogue
// warps add the partials into a running sum held in registers in rank
// order, sum = ((p0 + p1) + p2) + ...; the residual is added last.
// Persistent over the output tiles; 8 epilogue warps, two per lane quarter,
// each holding 128 of the tile's 256 columns for its 32 rows.
// ---------------------------------------------------------------------------

constexpr int kRowBN = 256;
// L2 budgets of the tile orders (MB): a token-tile group's activations in the
// column-parallel kernels, an output-column group's weights in the row-parallel ones
#ifndef TP_COL_GROUP_MB
#define TP_COL_GROUP_MB 32
#endif
#ifndef TP_ROW_GROUP_MB
#define TP_ROW_GROUP_MB 64
#endif
constexpr int kColGroupMB = TP_COL_GROUP_MB, kRowGroupMB = TP_ROW_GROUP_MB;
constexpr int kRowStages = 4;
constexpr int kRowStageBytes = kTcABytes + kRowBN * kTcBK * 2;   // 48 KB
constexpr int kRowSmem = 1024 + kRowStages * kRowStageBytes;
constexpr int kRowThreads = 320;

struct TcRowArgs {
    CUtensorMap ta;                       // per-shard activations stacked [N * T, Kr], boxes 64 x 128
    CUtensorMap tb[TP_MAX_SHARDS];        // shard weights [H, Kr], boxes 64 x 256
    int T, Kr, N, H;
    int n_mt, n_nt;
    int gn;                               // output-column tiles per group (tile order, below)
    const float* resid;                   // [T][H]
    float* out;                           // [T][H]
    int* status;
};

// Tile order of the row-parallel projections (o_proj, down_proj): the output-
// column tiles are taken in groups of gn whose weights (every shard's) fit in
// L2 with room to spare. Within a group output-column tiles vary fastest, so
// the CTAs resident at one time cover a few token tiles across the group's
// columns: a wave reads each of its token tiles' activations (every shard's)
// once, and the group's weights, read by every wave, are loaded evict-last
// while the activations stream evict-first. The activations are read once per
// group. (Token tiles fastest re-read every shard's activations once per wave:
// 2.07 GB of DRAM reads per down_proj launch; one group of all columns, 1.39 GB.)
__device__ __forceinline__ void row_tile(const TcRowArgs& g, int tile, int& m0, int& n0) {
    const int per_g = g.gn * g.n_mt, grp = tile / per_g, local = tile - grp * per_g;
    const int c0 = grp * g.gn, gn = min(g.gn, g.n_nt - c0);
    m0 = (local / gn) * kTcBM;
    n0 = (c0 + local % gn) * kRowBN;
}

__global__ void __launch_bounds__(kRowThreads, 1) tc_row_kernel(const __grid_constant__ TcRowArgs g) {
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t *full, *empty, *extra;
    uint32_t* tmem_slot;
    volatile int* abort_flag;
    const uint32_t counts[5] = {1, 1, 8, 8, 1};   // partial full x2, partial empty x2 (epilogue warps), done
    tc_setup(smem, kRowStages, kRowStages, 512, g.status, full, empty, extra, tmem_slot, abort_flag, 5, counts);
    uint64_t* pfull = extra;
    uint64_t* pempty = extra + 2;
    uint64_t* done = extra + 4;
    const uint32_t tmem = *tmem_slot;
    unsigned char* stages = smem + 1024;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = g.Kr / kTcBK;
    const int ntiles = g.n_mt * g.n_nt;

    if (warp == 0) {
        if (lane == 0 && !*abort_flag) {
            uint32_t it = 0;
            bool ok = true;
            const uint64_t pol_a = l2_evict_first_policy(), pol_b = l2_evict_last_policy();
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                int m0, n0;
                row_tile(g, tile, m0, n0);
                for (int r = 0; r < g.N && ok; ++r)
                    for (int kb = 0; kb < nk; ++kb, ++it) {
                        const int s = it % kRowStages;
                        if (!mbar_wait(&empty[s], ((it / kRowStages) & 1) ^ 1, abort_flag, g.status)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[s], kRowStageBytes);
                        unsigned char* st = stages + s * kRowStageBytes;
                        tma_load_2d(st, &g.ta, kb * kTcBK, r * g.T + m0, &full[s], pol_a);
                        tma_load_2d(st + kTcABytes, &g.tb[r], kb * kTcBK, n0, &full[s], pol_b);
                    }
            }
            volatile int no_abort = 0;
            for (uint32_t k = it > (uint32_t)kRowStages ? it - kRowStages : 0; k < it; ++k)
                mbar_wait(&full[k % kRowStages], (k / kRowStages) & 1, &no_abort, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kTcBM, kRowBN);
            uint32_t it = 0, pi = 0;
            bool ok = !*abort_flag;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x)
                for (int r = 0; r < g.N && ok; ++r, ++pi) {
                    const int buf = pi & 1;
                    if (!mbar_wait(&pempty[buf], ((pi >> 1) & 1) ^ 1, abort_flag, g.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dt = tmem + 256 * buf;
                    for (int kb = 0; kb < nk; ++kb, ++it) {
                        const int s = it % kRowStages;
                        if (!mbar_wait(&full[s], (it / kRowStages) & 1, abort_flag, g.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a0 = smem_u32(stages + s * kRowStageBytes), b0 = a0 + kTcABytes;
#pragma unroll
                        for (int k = 0; k < kTcBK / 16; ++k)
                            tc_mma(dt, smem_desc_sw128(a0 + k * 32), smem_desc_sw128(b0 + k * 32), idesc,
                                   (kb | k) != 0);
                        tc_commit(smem_u32(&empty[s]));
                    }
                    if (ok) tc_commit(smem_u32(&pfull[buf]));
                }
            tc_commit(smem_u32(done));
        }
    } else {
        const int q = warp & 3;                      // warps 2..9 -> lane quarters 2,3,0,1,2,3,0,1
        const int hf = (warp - 2) >> 2;              // which 128 of the 256 columns
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        uint32_t pi = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            int m0, n0;
            row_tile(g, tile, m0, n0);
            float sum[128];
            for (int r = 0; r < g.N; ++r, ++pi) {
                const int buf = pi & 1;
                ok = mbar_wait(&pfull[buf], (pi >> 1) & 1, abort_flag, g.status);
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
                if (ok) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t v[32];
                        tmem_ld32(tmem + lane_off + 256 * buf + 128 * hf + 32 * c, v);
                        tmem_wait_ld();
                        if (r == 0) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) sum[32 * c + i] = fbits(v[i]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) sum[32 * c + i] += fbits(v[i]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&pempty[buf]);
                if (!ok) break;
            }
            const int t = m0 + 32 * q + lane;
            const int n = n0 + 128 * hf;
            if (ok && t < g.T && n < g.H) {
                const size_t o = (size_t)t * g.H + n;
#pragma unroll
                for (int i = 0; i < 128; i += 4) {
                    const float4 rv = *reinterpret_cast<const float4*>(g.resid + o + i);
                    *reinterpret_cast<float4*>(g.out + o + i) =
                        make_float4(rv.x + sum[i], rv.y + sum[i + 1], rv.z + sum[i + 2], rv.w + sum[i + 3]);
                }
            }
        }
    }
    tc_teardown(done, 0, tmem, 512);
}

// ---------------------------------------------------------------------------
// RMSNorm (bf16 output, fully normalised) and the rotary table
// ---------------------------------------------------------------------------

struct NormCopies {
    const float* gamma[TP_MAX_SHARDS];
    int n;
};

// One token per CTA: 1/rms once, then one bf16 copy per distinct gamma,
// copy c at out + c * T * H.
__global__ void __launch_bounds__(256) prefill_norm_kernel(const float* __restrict__ x, const NormCopies gc,
                                                           bf16* __restrict__ out, int T, int H, float eps) {
    __shared__ float wsum[8];
    __shared__ float s_rinv;
    const int t = blockIdx.x, tid = threadIdx.x;
    const float* xr = x + (size_t)t * H;
    float a = 0.f;
    for (int k = tid * 4; k < H; k += 1024) {
        const float4 v = *reinterpret_cast<const float4*>(xr + k);
        a = fmaf(v.x, v.x, a);
        a = fmaf(v.y, v.y, a);
        a = fmaf(v.z, v.z, a);
        a = fmaf(v.w, v.w, a);
    }
    a = warp_sum(a);
    if ((tid & 31) == 0) wsum[tid >> 5] = a;
    __syncthreads();
    if (tid == 0) {
        float ss = 0.f;
        for (int w = 0; w < 8; ++w) ss += wsum[w];
        s_rinv = 1.0f / sqrtf(ss / (float)H + eps);
    }
    __syncthreads();
    const float ri = s_rinv;
    for (int k = tid * 4; k < H; k += 1024) {
        const float4 v = *reinterpret_cast<const float4*>(xr + k);
        for (int c = 0; c < gc.n; ++c) {
            const float4 g4 = *reinterpret_cast<const float4*>(gc.gamma[c] + k);
            uint2 pk;
            pk.x = pack_bf16x2(v.x * ri * g4.x, v.y * ri * g4.y);
            pk.y = pack_bf16x2(v.z * ri * g4.z, v.w * ri * g4.w);
            *reinterpret_cast<uint2*>(out + ((size_t)c * T + t) * H + k) = pk;
        }
    }
}

__global__ void rope_table_kernel(float2* tab, int max_pos, int half, int d, float log2_theta) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= max_pos * half) return;
    const int p = i / half, j = i - p * half;
    float sn, cs;
    sincosf((float)p * exp2f(-(2.0f * j / d) * log2_theta), &sn, &cs);
    tab[i] = make_float2(cs, sn);
}

constexpr int kFtQ = 128, kFtK = 128;          // queries per tile, keys per block

struct FtArgs {
    CUtensorMap tq;                       // q [N*T, hq_s*D], boxes 64 x 128
    CUtensorMap tk[TP_MAX_SHARDS];        // caches [Bmax*Hkv'][max_kv][D], boxes 64 x 128 x 1
    CUtensorMap tv[TP_MAX_SHARDS];
    bf16* out;                            // [N][T][hq_s * D]
    const int* pos;
    int N, B, S, T, hq_s, hkv_s, max_kv;
    float scale_log2;                     // log2(e) / sqrt(D)
    int* status;
};

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* tm, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------------------
// causal prefill attention, two query heads per CTA: the CTA takes one
// 128-query tile for a pair of query heads that share a KV head, so both
// tiles need the same keys. K/V stream once for the pair and the two tiles
// take turns on the tensor cores while the other tile's softmax runs.
//   warp 0    TMA: both Q tiles once, then K and V blocks of 128 keys into a
//             2-stage ring (128-byte swizzle, [group][key][d] tensor map: a
//             block starting before key 0 reads zeros);
//   warp 1    tensor memory (512 columns: S_0, S_1, O_0, O_1) and the MMA
//             thread: S_t = Q_t K_j^T, then O_t += P_t V_j with P_t read from
//             tensor memory (written over S_t as bf16) and V the MN-major
//             operand; S_t of the next block is issued right after O_t's
//             product, so one tile's MMAs run under the other's softmax;
//   warps 2-5 and 6-9: the softmax of tile 0 and 1, one query row per thread:
//             S from tensor memory in one load, masked row max, P =
//             exp2(S * scale - m) written back as bf16, running sum. The
//             running max used for P moves only when a row's max grows by
//             more than 8 (a factor 256, safe in bf16 and fp32); O is then
//             rescaled in tensor memory. The commit that signals S_t of
//             block j follows O_t of block j - 1, so O is complete whenever
//             S is ready.
// Keys of a block that are not the block's own (the last block is loaded
// shifted to end at the last needed key) or lie after the query get
// probability 0. The result is O / l per row.
// ---------------------------------------------------------------------------

constexpr int kFaThreads = 320;
constexpr float kFaRescale = 8.0f;             // log2 of the growth that triggers a rescale
constexpr int kFaKSt = 3, kFaVSt = 2;          // K and V rings: a K slot frees once S is computed

template <int D>
struct FaShape {
    static constexpr int NKB = D / 64;
    static constexpr int QB = kFtQ * D * 2;             // one Q tile
    static constexpr int KB = kFtK * D * 2;             // one K (or V) block
    static constexpr int SMEM = 1024 + 2 * QB + (kFaKSt + kFaVSt) * KB;
};

// A shared-memory descriptor advanced by `bytes` (start address in 16-byte
// units in the low bits; no carry for addresses below 256 KB).
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

template <int D>
__global__ void __launch_bounds__(kFaThreads, 1) attn_fa_prefill_kernel(const __grid_constant__ FtArgs f) {
    using Sh = FaShape<D>;
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;           // [kFaKSt]
    uint64_t* k_empty = k_full + kFaKSt;   // [kFaKSt]
    uint64_t* v_full = k_empty + kFaKSt;   // [kFaVSt]
    uint64_t* v_empty = v_full + kFaVSt;   // [kFaVSt]
    uint64_t* s_full = v_empty + kFaVSt;   // [2] per tile
    uint64_t* p_full = s_full + 2;         // [2] per tile
    uint64_t* o_full = p_full + 2;         // [2] per tile: the last block's product
    uint64_t* done = o_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    unsigned char* sq = smem + 1024;
    unsigned char* sk = sq + 2 * Sh::QB;
    unsigned char* sv = sk + kFaKSt * Sh::KB;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // heaviest query blocks first (causal work grows with the block index)
    const int G = f.hq_s / f.hkv_s, HP = (G + 1) / 2;
    const int nqb = (f.S + kFtQ - 1) / kFtQ;
    int idx = blockIdx.x;
    const int qb = nqb - 1 - idx % nqb;
    idx /= nqb;
    const int hp = idx % HP;
    idx /= HP;
    const int kvh = idx % f.hkv_s;
    idx /= f.hkv_s;
    const int b = idx % f.B;
    const int r = idx / f.B;
    const int h0 = kvh * G + 2 * hp;
    const int ntile = (2 * hp + 1 < G) ? 2 : 1;
    const int p0 = f.pos[b];
    const int rows = min(kFtQ, f.S - qb * kFtQ);
    const int q_first = p0 + qb * kFtQ;
    const int nkeys = max(0, min(q_first + rows, f.max_kv));
    const int nblk = (nkeys + kFtK - 1) / kFtK;
    const int t0 = b * f.S + qb * kFtQ;
    const int grp = b * f.hkv_s + kvh;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < kFaKSt; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < kFaVSt; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);
            mbar_init(&o_full[i], 1);
        }
        mbar_init(done, 1);
        *abort_flag = (smem_u32(sq) & 1023u) ? 1 : 0;
        if (*abort_flag) set_status(f.status, TP_ERR_ALIGN);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0 && !*abort_flag) {
            mbar_arrive_expect_tx(q_full, (uint32_t)(ntile * Sh::QB));
            for (int t = 0; t < ntile; ++t)
#pragma unroll
                for (int kb = 0; kb < Sh::NKB; ++kb)
                    tma_load_2d_keep(sq + t * Sh::QB + kb * (kFtQ * 128), &f.tq, (h0 + t) * D + kb * 64, r * f.T + t0,
                                     q_full);
            // K runs ahead of V: block j's K is needed one product earlier than its V
            int jk = 0, jv = 0;
            bool ok = true;
            while (ok && (jk < nblk || jv < nblk)) {
                const bool do_k = jk < nblk && (jv >= nblk || jk <= jv + kFaKSt - 1);
                const int j = do_k ? jk : jv;
                const int key0 = min(j * kFtK, nkeys - kFtK);   // may be negative: zero fill
                if (do_k) {
                    const int s = j % kFaKSt;
                    if (!(ok = mbar_wait(&k_empty[s], ((j / kFaKSt) & 1) ^ 1, abort_flag, f.status))) break;
                    mbar_arrive_expect_tx(&k_full[s], Sh::KB);
#pragma unroll
                    for (int kb = 0; kb < Sh::NKB; ++kb)
                        tma_load_3d(sk + s * Sh::KB + kb * (kFtK * 128), &f.tk[r], kb * 64, key0, grp, &k_full[s]);
                    ++jk;
                } else {
                    const int s = j % kFaVSt;
                    if (!(ok = mbar_wait(&v_empty[s], ((j / kFaVSt) & 1) ^ 1, abort_flag, f.status))) break;
                    mbar_arrive_expect_tx(&v_full[s], Sh::KB);
#pragma unroll
                    for (int kb = 0; kb < Sh::NKB; ++kb)
                        tma_load_3d(sv + s * Sh::KB + kb * (kFtK * 128), &f.tv[r], kb * 64, key0, grp, &v_full[s]);
                    ++jv;
                }
            }
            volatile int no_abort = 0;
            mbar_wait(q_full, 0, &no_abort, nullptr);
            for (int k = jk > kFaKSt ? jk - kFaKSt : 0; k < jk; ++k)
                mbar_wait(&k_full[k % kFaKSt], (k / kFaKSt) & 1, &no_abort, nullptr);
            for (int k = jv > kFaVSt ? jv - kFaVSt : 0; k < jv; ++k)
                mbar_wait(&v_full[k % kFaVSt], (k / kFaVSt) & 1, &no_abort, nullptr);
        }
    } else if (warp == 1) {
        // the whole warp runs the loop (warp-uniform operands); one elected lane issues
        {
            const uint32_t id_s = idesc_bf16(kFtQ, kFtK);
            const uint32_t id_o = idesc_bf16_bmn(kFtQ, D);
            const uint64_t dq0 = smem_desc_sw128(smem_u32(sq)), dk0 = smem_desc_sw128(smem_u32(sk));
            const uint64_t dv0 = smem_desc_mn_sw128(smem_u32(sv), kFtK * 128, 1024);
            auto issue_s = [&](int t, int j) {          // S_t = Q_t K_j^T
                const uint64_t dq = desc_add(dq0, t * Sh::QB), dk = desc_add(dk0, (j % kFaKSt) * Sh::KB);
#pragma unroll
                for (int kb = 0; kb < Sh::NKB; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        tc_mma_w(tmem + kFtK * t, desc_add(dq, kb * (kFtQ * 128) + k * 32),
                               desc_add(dk, kb * (kFtK * 128) + k * 32), id_s, (kb | k) != 0);
                tc_commit_w(smem_u32(&s_full[t]));
            };
            // every lane waits; the outcome is made warp-uniform so the lanes stay together
            auto wait_all = [&](uint64_t* bar, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, f.status));
            };
            auto wait_k = [&](int j) {
                const bool w = wait_all(&k_full[j % kFaKSt], (j / kFaKSt) & 1);
                tc_fence_after();
                return w;
            };
            bool ok = __all_sync(0xffffffffu, !*abort_flag) && wait_all(q_full, 0);
            if (ok && nblk > 0 && (ok = wait_k(0))) {
                for (int t = 0; t < ntile; ++t) issue_s(t, 0);
                tc_commit_w(smem_u32(&k_empty[0]));
            }
            for (int j = 0; j < nblk && ok; ++j) {
                const uint64_t dv = desc_add(dv0, (j % kFaVSt) * Sh::KB);
                if (!(ok = wait_all(&v_full[j % kFaVSt], (j / kFaVSt) & 1))) break;
                for (int t = 0; t < ntile && ok; ++t) {
                    // O_t += P_t V_j, P_t in the first 64 columns of S_t
                    if (!(ok = wait_all(&p_full[t], j & 1))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kFtK / 16; ++kk)
                        tc_mma_ts_w(tmem + 2 * kFtK + D * t, tmem + kFtK * t + 8 * kk, desc_add(dv, kk * 16 * 128),
                                  id_o, (j | kk) != 0);
                    if (j + 1 == nblk) tc_commit_w(smem_u32(&o_full[t]));
                    if (j + 1 < nblk) {                     // S_t of the next block, after O_t in issue order
                        if (t == 0 && !(ok = wait_k(j + 1))) break;
                        issue_s(t, j + 1);
                    }
                }
                if (j + 1 < nblk) tc_commit_w(smem_u32(&k_empty[(j + 1) % kFaKSt]));
                tc_commit_w(smem_u32(&v_empty[j % kFaVSt]));   // every MMA reading V_j has been issued
            }
            tc_commit_w(smem_u32(done));
        }
    } else {
        const int t = (warp - 2) >> 2;                      // tile
        const int qd = warp & 3;                            // tensor-memory lane quarter
        const int m = 32 * qd + lane;                       // query row of the tile
        const uint32_t lane_off = (uint32_t)(32 * qd) << 16;
        const uint32_t s_col = tmem + lane_off + kFtK * t, o_col = tmem + lane_off + 2 * kFtK + D * t;
        const int q_pos = q_first + m;
        const int warp_first = q_first + 32 * qd;           // the warp's smallest query position
        float m_use = -INFINITY, l_run = 0.f;
        bool ok = t < ntile;
        for (int j = 0; j < nblk && ok; ++j) {
            ok = mbar_wait(&s_full[t], j & 1, abort_flag, f.status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            uint32_t v[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(s_col + 32 * c, v[c]);
            tmem_wait_ld();
            const int key0 = min(j * kFtK, nkeys - kFtK);
            const int lo = j * kFtK, hi = min(lo + kFtK, nkeys);
            // a block whose keys all precede every row of the warp needs no mask
            const bool whole = key0 == lo && hi == lo + kFtK && lo + kFtK - 1 <= warp_first;
            const int kmax = min(hi - 1, q_pos);
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // independent chains
            if (whole) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) mq[i & 3] = fmaxf(mq[i & 3], __uint_as_float(v[c][i]));
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int key = key0 + 32 * c + i;
                        if (key >= lo && key <= kmax) mq[i & 3] = fmaxf(mq[i & 3], __uint_as_float(v[c][i]));
                    }
            }
            const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
            const float m_blk = mx == -INFINITY ? -INFINITY : mx * f.scale_log2;
            // the max used for P moves only on a large growth (or the first keys)
            const bool grow = m_blk > m_use + kFaRescale;
            const float alpha = grow ? ex2_approx(m_use - m_blk) : 1.f;   // 0 when m_use is -inf
            if (grow) m_use = m_blk;
            // P = 2^(S * scale - m) in independent passes (arguments, exponentials,
            // sums, packing) so the exponentials of a row overlap; a masked key's
            // argument is -inf, whose exponential is 0
            float* e = reinterpret_cast<float*>(&v[0][0]);
            if (whole) {
#pragma unroll
                for (int i = 0; i < 128; ++i) e[i] = fmaf(e[i], f.scale_log2, -m_use);
            } else {
#pragma unroll
                for (int i = 0; i < 128; ++i) {
                    const int key = key0 + i;
                    e[i] = (key >= lo && key <= kmax) ? fmaf(e[i], f.scale_log2, -m_use) : -INFINITY;
                }
            }
#pragma unroll
            for (int i = 0; i < 128; ++i) e[i] = ex2_approx(e[i]);
            float sq[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < 128; ++i) sq[i & 7] += e[i];
            const float sum = ((sq[0] + sq[1]) + (sq[2] + sq[3])) + ((sq[4] + sq[5]) + (sq[6] + sq[7]));
            uint32_t pk[2][32];
#pragma unroll
            for (int i = 0; i < 64; ++i) pk[i >> 5][i & 31] = pack_bf16x2(e[2 * i], e[2 * i + 1]);
            l_run = l_run * alpha + sum;
            tmem_st32(s_col, pk[0]);
            tmem_st32(s_col + 32, pk[1]);
            // O holds blocks 0 .. j-1 (complete: their products precede S of this
            // block in the MMA order); rescale it where this row's max moved
            if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(o_col + 32 * c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(o_col + 32 * c, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[t]);
        }
        // the output row: O / l
        if (ok && nblk > 0) {
            ok = mbar_wait(&o_full[t], 0, abort_flag, f.status);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok && t < ntile) {
            tc_fence_after();
            const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
            bf16* dst = f.out + ((size_t)r * f.T + t0 + m) * f.hq_s * D + (h0 + t) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(o_col + 32 * c, o);
                tmem_wait_ld();
                if (m < rows) {
#pragma unroll
                    for (int i = 0; i < 32; i += 8)
                        *reinterpret_cast<uint4*>(dst + 32 * c + i) = make_uint4(
                            pack_bf16x2(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv),
                            pack_bf16x2(__uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv),
                            pack_bf16x2(__uint_as_float(o[i + 4]) * inv, __uint_as_float(o[i + 5]) * inv),
                            pack_bf16x2(__uint_as_float(o[i + 6]) * inv, __uint_as_float(o[i + 7]) * inv));
                }
            }
        }
    }
    tc_teardown(done, 0, tmem, 512);
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

cudaError_t launch_prefill_norm(const float* x, const float* const* gammas, int n_copies, void* out, int T, int H,
                                float eps, cudaStream_t s) {
    if (n_copies < 1 || n_copies > TP_MAX_SHARDS) return cudaErrorInvalidValue;
    NormCopies gc;
    memset(&gc, 0, sizeof gc);
    for (int c = 0; c < n_copies; ++c) gc.gamma[c] = gammas[c];
    gc.n = n_copies;
    if (T > 0) prefill_norm_kernel<<<T, 256, 0, s>>>(x, gc, static_cast<bf16*>(out), T, H, eps);
    return cudaGetLastError();
}

cudaError_t launch_rope_table(float2* tab, int max_pos, int d, double log2_theta, cudaStream_t s) {
    const int n = max_pos * (d / 2);
    rope_table_kernel<<<(n + 255) / 256, 256, 0, s>>>(tab, max_pos, d / 2, d, (float)log2_theta);
    return cudaGetLastError();
}

cudaError_t launch_tc_col(int mode, const PrefillColParams& p, cudaStream_t s) {
    if (p.T <= 0) return cudaSuccess;
    TcColArgs g;
    memset(&g, 0, sizeof g);
    const int copies = p.a_copies > 1 ? p.N : 1;
    cudaError_t e = tensor_map_2d(p.A, p.K, (long)copies * p.T, kTcBK, kTcBM, 1, &g.ta);
    for (int r = 0; r < p.N && e == cudaSuccess; ++r)
        e = tensor_map_2d(p.W[r], p.K, p.rows, kTcBK, mode == TC_QKV ? kTcBN : 128, 1, &g.tb[r]);
    if (e != cudaSuccess) return e;
    g.a_row_stride = copies > 1 ? p.T : 0;
    g.T = p.T;
    g.K = p.K;
    g.S = p.S;
    g.hq_s = p.hq_s;
    g.hkv_s = p.hkv_s;
    g.d = p.d;
    g.max_kv = p.max_kv;
    g.ffn_s = p.ffn_s;
    for (int r = 0; r < p.N; ++r) {
        g.bias[r] = p.bias[r];
        g.kcache[r] = p.kcache[r];
        g.vcache[r] = p.vcache[r];
    }
    g.pos = p.pos;
    g.rope = p.rope;
    g.q_out = static_cast<bf16*>(p.q_out);
    g.act = static_cast<bf16*>(p.act);
    g.status = p.status;
    static bool set[2] = {false, false};
    const void* fn = mode == TC_QKV ? reinterpret_cast<const void*>(tc_col_kernel<TC_QKV>)
                                    : reinterpret_cast<const void*>(tc_col_kernel<TC_GATEUP>);
    if (!set[mode]) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
        if (e != cudaSuccess) return e;
        set[mode] = true;
    }
    g.n_mt = (p.T + kTcBM - 1) / kTcBM;
    g.n_nt = mode == TC_QKV ? (p.rows + kTcBN - 1) / kTcBN : (p.ffn_s + 127) / 128;
    g.N = p.N;
    // token tiles per group: about kColGroupMB of activations per group, every copy counted
    const long tile_bytes = (long)kTcBM * p.K * 2 * copies;
    g.gm = (int)std::max(1L, std::min((long)g.n_mt, ((long)kColGroupMB << 20) / tile_bytes));
    const long tiles = (long)g.n_mt * g.n_nt * g.N;
    if (tiles > INT32_MAX) return cudaErrorInvalidConfiguration;
    const int grid = tiles < kSMs ? (int)tiles : kSMs;
    void* args[] = {&g};
    e = cudaLaunchKernel(fn, dim3(grid), dim3(kTcThreads), args, kTcSmem, s);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_tc_row(const PrefillRowParams& p, cudaStream_t s) {
    if (p.T <= 0) return cudaSuccess;
    TcRowArgs g;
    memset(&g, 0, sizeof g);
    cudaError_t e = tensor_map_2d(p.A, p.Kr, (long)p.N * p.T, kTcBK, kTcBM, 1, &g.ta);
    for (int r = 0; r < p.N && e == cudaSuccess; ++r) e = tensor_map_2d(p.W[r], p.Kr, p.H, kTcBK, kRowBN, 1, &g.tb[r]);
    if (e != cudaSuccess) return e;
    g.T = p.T;
    g.Kr = p.Kr;
    g.N = p.N;
    g.H = p.H;
    g.resid = p.resid;
    g.out = p.out;
    g.status = p.status;
    static bool set = false;
    if (!set) {
        e = cudaFuncSetAttribute(tc_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRowSmem);
        if (e != cudaSuccess) return e;
        set = true;
    }
    g.n_mt = (p.T + kTcBM - 1) / kTcBM;
    g.n_nt = (p.H + kRowBN - 1) / kRowBN;
    // output-column tiles per group: about kRowGroupMB of weights per group
    const long col_bytes = (long)kRowBN * p.Kr * p.N * 2;
    g.gn = (int)std::max(1L, std::min((long)g.n_nt, ((long)kRowGroupMB << 20) / col_bytes));
    const long tiles = (long)g.n_mt * g.n_nt;
    if (tiles > INT32_MAX) return cudaErrorInvalidConfiguration;
    const int grid = tiles < kSMs ? (int)tiles : kSMs;
    tc_row_kernel<<<grid, kRowThreads, kRowSmem, s>>>(g);
    return cudaGetLastError();
}

cudaError_t launch_flash_prefill(const FlashParams& p, cudaStream_t s) {
    const int G = p.hq_s / p.hkv_s;
    const long grid = (long)p.N * p.B * p.hkv_s * ((G + 1) / 2) * ((p.S + kFtQ - 1) / kFtQ);
    if (grid == 0) return cudaSuccess;
    if (grid > INT32_MAX) return cudaErrorInvalidConfiguration;
    FtArgs f;
    memset(&f, 0, sizeof f);
    cudaError_t e = tensor_map_2d(p.q, (long)p.hq_s * p.d, (long)p.N * p.T, 64, kFtQ, 1, &f.tq);
    const long groups = (long)p.max_batch * p.hkv_s;
    for (int r = 0; r < p.N && e == cudaSuccess; ++r) {
        e = tensor_map_3d(p.kcache[r], p.d, p.max_kv, groups, 64, kFtK, 1, &f.tk[r]);
        if (e == cudaSuccess) e = tensor_map_3d(p.vcache[r], p.d, p.max_kv, groups, 64, kFtK, 1, &f.tv[r]);
    }
    if (e != cudaSuccess) return e;
    f.out = static_cast<bf16*>(p.out);
    f.pos = p.pos;
    f.N = p.N;
    f.B = p.B;
    f.S = p.S;
    f.T = p.T;
    f.hq_s = p.hq_s;
    f.hkv_s = p.hkv_s;
    f.max_kv = p.max_kv;
    f.scale_log2 = p.scale * 1.4426950408889634f;
    f.status = p.status;
    static bool set[2] = {false, false};
    const int which = p.d == 128 ? 1 : 0;
    const void* fn = which ? reinterpret_cast<const void*>(attn_fa_prefill_kernel<128>)
                           : reinterpret_cast<const void*>(attn_fa_prefill_kernel<64>);
    const int smem = which ? FaShape<128>::SMEM : FaShape<64>::SMEM;
    if (!set[which]) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        set[which] = true;
    }
    void* args[] = {&f};
    e = cudaLaunchKernel(fn, dim3((unsigned)grid), dim3(kFaThreads), args, smem, s);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace tpk
