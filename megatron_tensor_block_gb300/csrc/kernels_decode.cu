// Decode-regime kernels of the tensor-parallel block: every projection of
// every logical shard in one launch, and split-KV grouped-query attention.
//
// "Multi-GPU & Multi-Node", How tensor parallelism works:
//   step 1 -- column-parallel QKV and gate/up: each shard produces its slice
//             of the outputs (EPI_QKV_ROPE, EPI_SWIGLU);
//   step 2 -- attention over the shard's own heads and KV cache
//             (attn_decode_kernel), activation per shard (EPI_SWIGLU);
//   step 3 -- row-parallel o_proj and down_proj: partial sums added in rank
//             order (EPI_ROWPAR), the single-device form of the all-reduce
//             ("feat: multi-GPU tensor-parallel runtime ...", Problem and
//             Collective backend abstraction).
//
// Skinny GEMM design (decode, T <= 8 tokens): a work unit is 64 output rows
// x one reduction chunk of one shard. Eight warps per CTA: four row groups of
// 16 rows x two interleaved halves of the chunk's 64-element steps. Each
// lane streams its weight fragment straight from HBM with 16-byte loads and
// feeds it to a bf16 m16n8k16 tensor-core MMA whose B operand (the tokens)
// sits in shared memory. Because the order of the reduction index inside an
// MMA is free, a lane's 16 contiguous bytes of a weight row are used as its
// A fragment and the matching 16 bytes of each token row as its B fragment
// -- no shuffles or shared-memory staging of weights.
// Units of a group (chunks, and shards for row-parallel) write fp32 partials;
// the last unit to finish sums them in a fixed order (chunks, then ranks), so
// results do not depend on scheduling.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "stream.cuh"
#include "tp_internal.h"

namespace tpk {

// Global row (within one shard's weight) of row j (0..63) of tile tb. QKV and
// gate/up tiles pair each row with its partner so the epilogue has both:
// rotary pairs (i, i + d/2) of a head, and (gate_i, up_i).
__device__ __forceinline__ int tile_row(int epi, int tb, int j, int head_dim, int ffn_s) {
    if (epi == EPI_QKV_ROPE) {
        const int half = head_dim >> 1;
        const int per_head = half >> 5;
        const int h = tb / per_head, sub = tb - h * per_head;
        const int base = h * head_dim + sub * 32;
        return j < 32 ? base + j : base + half + (j - 32);
    }
    if (epi == EPI_SWIGLU) return j < 32 ? tb * 32 + j : ffn_s + tb * 32 + (j - 32);
    return tb * kTileRows + j;
}

template <typename TW> struct XPad;          // shared-memory row padding: 64 bytes
template <> struct XPad<bf16> { static constexpr int v = 32; };
template <> struct XPad<float> { static constexpr int v = 16; };

// ---------------------------------------------------------------------------
// main loops: one warp, 16 rows x its share of the chunk's 64-wide steps
// ---------------------------------------------------------------------------

template <int U>
__device__ __forceinline__ void mainloop_bf16(const char* pA, const char* pB, const char* px,
                                              int nsteps, int wk, float (&c)[4]) {
    for (int s0 = wk; s0 < nsteps; s0 += 2 * U) {
        uint4 wa[U][2], wb[U][2];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = s0 + 2 * u;
            if (s < nsteps) {
                wa[u][0] = ld_stream16(pA + s * 128);
                wa[u][1] = ld_stream16(pA + s * 128 + 64);
                wb[u][0] = ld_stream16(pB + s * 128);
                wb[u][1] = ld_stream16(pB + s * 128 + 64);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = s0 + 2 * u;
            if (s < nsteps) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 xv = *reinterpret_cast<const uint4*>(px + s * 128 + h * 64);
                    mma_bf16_16816(c, wa[u][h].x, wb[u][h].x, wa[u][h].y, wb[u][h].y, xv.x, xv.y);
                    mma_bf16_16816(c, wa[u][h].z, wb[u][h].z, wa[u][h].w, wb[u][h].w, xv.z, xv.w);
                }
            }
        }
    }
}

// fp32 weights: plain FMA, four rows at a time, lanes along the reduction.
__device__ __forceinline__ void mainloop_f32(const float* W, const int* rows, int K, int k0,
                                             const float* xs, int xstride, int nsteps, int wk,
                                             int lane, float* red_rows /* [16][8] */) {
    for (int rr = 0; rr < 16; rr += 4) {
        float acc[4][kTMax];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int t = 0; t < kTMax; ++t) acc[i][t] = 0.f;
        for (int s = wk; s < nsteps; s += 2) {
            const int kk = s * kKStep + 2 * lane;
            float2 w2[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                w2[i] = __ldg(reinterpret_cast<const float2*>(W + (size_t)rows[rr + i] * K + k0 + kk));
#pragma unroll
            for (int t = 0; t < kTMax; ++t) {
                const float2 x2 = *reinterpret_cast<const float2*>(xs + t * xstride + kk);
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i][t] = fmaf(w2[i].x, x2.x, fmaf(w2[i].y, x2.y, acc[i][t]));
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int t = 0; t < kTMax; ++t) {
                const float v = warp_sum(acc[i][t]);
                if (lane == 0) red_rows[(rr + i) * kTMax + t] = v;
            }
    }
}

// ---------------------------------------------------------------------------
// the skinny-GEMM kernel
// ---------------------------------------------------------------------------

// Cross-unit reduction (chunks in order, then ranks in order) and the
// epilogue of one 64-row tile. `tile` holds this unit's [64][8] partial,
// `ss` its per-token sums of squares. NAMED selects the consumer-only barrier
// (warp-specialised kernels) instead of __syncthreads.
template <typename TW, int EPI, bool NAMED>
__device__ __forceinline__ void unit_finish(const GemvParams& p, int u, int gi, int r, int tb, float* tile,
                                            float* ss, unsigned* s_flag, int tid, int nthreads) {
#define SYNC() do { if (NAMED) consumer_sync(nthreads); else __syncthreads(); } while (0)
    const int upg = p.shape.units_per_group();
    const int T = p.T;
    if (upg > 1) {
        float* mine = p.part + (size_t)u * kPartStride;
        for (int i = tid; i < kTileRows * kTMax; i += nthreads) mine[i] = tile[i];
        if (EPI != EPI_ROWPAR && tid < kTMax) mine[kTileRows * kTMax + tid] = ss[tid];
        bool last;
        if constexpr (NAMED) last = arrive_last_consumers(&p.cnt[gi], (unsigned)upg, nthreads, s_flag);
        else last = arrive_last(&p.cnt[gi], (unsigned)upg);
        if (!last) return;
        const float* base = p.part + (size_t)gi * upg * kPartStride;
        const int C = p.shape.chunks;
        const int nrank = (EPI == EPI_ROWPAR) ? p.shape.shards_per_group : 1;
        // every partial of the group is loaded before any is added (the loads
        // are independent), then summed: chunks in order, then ranks in order
        constexpr int kMaxParts = kMaxGroupUnits;
        const int nvec = (EPI == EPI_ROWPAR ? kTileRows * kTMax : kPartStride) / 4;
        for (int i4 = tid; i4 < nvec; i4 += nthreads) {
            float4 v[kMaxParts];
#pragma unroll
            for (int q = 0; q < kMaxParts; ++q)
                if (q < upg) v[q] = __ldcg(reinterpret_cast<const float4*>(base + (size_t)q * kPartStride) + i4);
            float4 total = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < kMaxParts; ++q) {
                if (q >= upg) break;
                const int rr = q / C, cc = q - rr * C;
                float4& pr = v[rr * C];
                if (cc > 0) {
                    pr.x += v[q].x; pr.y += v[q].y; pr.z += v[q].z; pr.w += v[q].w;
                }
                if (cc == C - 1) {
                    if (rr == 0) total = pr;
                    else { total.x += pr.x; total.y += pr.y; total.z += pr.z; total.w += pr.w; }
                }
            }
            const int i = i4 * 4;
            if (i < kTileRows * kTMax) *reinterpret_cast<float4*>(tile + i) = total;
            else *reinterpret_cast<float4*>(ss + (i - kTileRows * kTMax)) = total;
        }
        SYNC();
    }

    // ---- epilogues
    if (EPI == EPI_ROWPAR) {
        bf16* nout = reinterpret_cast<bf16*>(p.norm_out);
        for (int i = tid; i < kTileRows * T; i += nthreads) {
            const int t = i / kTileRows, j = i - t * kTileRows;
            const int row = tb * kTileRows + j;
            const size_t o = (size_t)t * p.rows + row;
            const float yv = p.resid[o] + tile[j * kTMax + t];
            p.y[o] = yv;
            if (nout) {
                // the next RMSNorm's operands: h * gamma_r for every shard, and
                // this tile's share of sum(h^2)
                for (int r2 = 0; r2 < p.n_shards; ++r2)
                    nout[((size_t)r2 * kTMax + t) * p.rows + row] = __float2bfloat16_rn(yv * p.gamma2[r2][row]);
                tile[j * kTMax + t] = yv;
            }
        }
        if (nout) {
            SYNC();
            if (tid < T) {
                float a = 0.f;
                for (int j = 0; j < kTileRows; ++j) a = fmaf(tile[j * kTMax + tid], tile[j * kTMax + tid], a);
                p.ss_tiles_out[tb * kTMax + tid] = a;
            }
        }
        return;
    }
    const float inv_k = 1.0f / (float)p.K;
    if (EPI == EPI_SWIGLU) {
        TW* out = reinterpret_cast<TW*>(p.act_out);
        for (int i = tid; i < 32 * T; i += nthreads) {
            const int t = i >> 5, j = i & 31;
            const float rinv = 1.0f / sqrtf(ss[t] * inv_k + p.eps);
            const float gt = tile[j * kTMax + t] * rinv;
            const float up = tile[(j + 32) * kTMax + t] * rinv;
            const float a = gt / (1.0f + expf(-gt)) * up;
            Stor<TW>::store(out + ((size_t)r * kTMax + t) * p.ffn_s + tb * 32 + j, a);
        }
        return;
    }
    // EPI_QKV_ROPE (decode: token t is sequence b = t at position pos[t])
    const int d = p.head_dim, half = d >> 1;
    for (int i = tid; i < 32 * T; i += nthreads) {
        const int t = i >> 5, j = i & 31;
        const float rinv = 1.0f / sqrtf(ss[t] * inv_k + p.eps);
        const int rowA = tile_row(EPI_QKV_ROPE, tb, j, d, 0);
        const int head = rowA / d, ii = rowA - head * d;
        float va = tile[j * kTMax + t] * rinv;
        float vb = tile[(j + 32) * kTMax + t] * rinv;
        if (p.bias[r]) {
            va += p.bias[r][rowA];
            vb += p.bias[r][rowA + half];
        }
        const int pos = p.pos[t];
        if (head < p.hq_s + p.hkv_s) {
            float c, sn;
            if constexpr (sizeof(TW) == 4) {
                const double inv_freq = exp2(-(2.0 * ii / d) * p.log2_theta);
                double sd, cd;
                sincos((double)pos * inv_freq, &sd, &cd);
                c = (float)cd;
                sn = (float)sd;
            } else {
                const float inv_freq = exp2f(-(2.0f * ii / d) * (float)p.log2_theta);
                sincosf((float)pos * inv_freq, &sn, &c);
            }
            const float ra = va * c - vb * sn, rb = va * sn + vb * c;
            va = ra;
            vb = rb;
        }
        if (head < p.hq_s) {
            float* q = p.q_out + ((size_t)r * kTMax + t) * p.hq_s * d + head * d + ii;
            q[0] = va;
            q[half] = vb;
        } else {
            const bool is_k = head < p.hq_s + p.hkv_s;
            const int kvh = is_k ? head - p.hq_s : head - p.hq_s - p.hkv_s;
            if (pos < 0 || pos >= p.max_kv) {
                set_status(p.status, TP_ERR_CAPACITY);
                continue;
            }
            TW* cache = reinterpret_cast<TW*>(is_k ? p.kcache[r] : p.vcache[r]);
            TW* dst = cache + (((size_t)t * p.hkv_s + kvh) * p.max_kv + pos) * d + ii;
            Stor<TW>::store(dst, va);
            Stor<TW>::store(dst + half, vb);
        }
    }
#undef SYNC
}

template <typename TW, int EPI>
__global__ void __launch_bounds__(256) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    constexpr int PAD = XPad<TW>::v;
    const int kc = p.shape.kc;
    const int xstride = kc + PAD;                       // elements
    TW* xs = reinterpret_cast<TW*>(smem);
    float* red = reinterpret_cast<float*>(smem + (size_t)kTMax * xstride * sizeof(TW));  // [2][64][8]
    float* tile = red + 2 * kTileRows * kTMax;          // [64][8]
    float* ss = tile + kTileRows * kTMax;               // [8] sum of squares per token

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int u = blockIdx.x;
    const int upg = p.shape.units_per_group();
    const int gi = u / upg, rem = u - gi * upg;
    int r, tb, chunk;
    if (EPI == EPI_ROWPAR) {
        tb = gi;
        r = rem / p.shape.chunks;
        chunk = rem - r * p.shape.chunks;
    } else {
        const int rb = p.shape.groups / p.n_shards;     // row tiles per shard
        r = gi / rb;
        tb = gi - r * rb;
        chunk = rem;
    }
    const int k0 = chunk * kc;
    const int T = p.T;

    // ---- stage the activation chunk in shared memory (tokens >= T are zero)
    if (EPI == EPI_ROWPAR) {
        const TW* a = reinterpret_cast<const TW*>(p.act[r]);
        const int vec_per_row = kc * (int)sizeof(TW) / 16;
        for (int i = tid; i < kTMax * vec_per_row; i += blockDim.x) {
            const int t = i / vec_per_row, v = i - t * vec_per_row;
            uint4 val = make_uint4(0, 0, 0, 0);
            if (t < T) val = *reinterpret_cast<const uint4*>(
                reinterpret_cast<const char*>(a + (size_t)t * p.K + k0) + v * 16);
            *reinterpret_cast<uint4*>(reinterpret_cast<char*>(xs + t * xstride) + v * 16) = val;
        }
    } else {
        // warp w stages token w: x * gamma (the norm's 1/rms is applied in
        // the epilogue) and the chunk's sum of squares.
        const int t = warp;
        const float* g = p.gamma[r];
        float acc = 0.f;
        for (int k = lane * 4; k < kc; k += 128) {
            float4 xv = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < T) xv = *reinterpret_cast<const float4*>(p.x + (size_t)t * p.K + k0 + k);
            const float4 gv = *reinterpret_cast<const float4*>(g + k0 + k);
            acc = fmaf(xv.x, xv.x, acc);
            acc = fmaf(xv.y, xv.y, acc);
            acc = fmaf(xv.z, xv.z, acc);
            acc = fmaf(xv.w, xv.w, acc);
            if constexpr (sizeof(TW) == 2) {
                uint2 pk;
                pk.x = pack_bf16x2(xv.x * gv.x, xv.y * gv.y);
                pk.y = pack_bf16x2(xv.z * gv.z, xv.w * gv.w);
                *reinterpret_cast<uint2*>(xs + t * xstride + k) = pk;
            } else {
                *reinterpret_cast<float4*>(reinterpret_cast<float*>(xs) + t * xstride + k) =
                    make_float4(xv.x * gv.x, xv.y * gv.y, xv.z * gv.z, xv.w * gv.w);
            }
        }
        acc = warp_sum(acc);
        if (lane == 0) ss[t] = acc;
    }
    __syncthreads();

    // ---- main loop
    const int wm = warp & 3, wk = warp >> 2;
    const int nsteps = kc / kKStep;
    if constexpr (sizeof(TW) == 2) {
        const int g = lane >> 2, tq = lane & 3;
        const int rowA = tile_row(EPI, tb, 16 * wm + g, p.head_dim, p.ffn_s);
        const int rowB = tile_row(EPI, tb, 16 * wm + g + 8, p.head_dim, p.ffn_s);
        const TW* W = reinterpret_cast<const TW*>(p.W[r]);
        const char* pA = reinterpret_cast<const char*>(W + (size_t)rowA * p.K + k0) + tq * 16;
        const char* pB = reinterpret_cast<const char*>(W + (size_t)rowB * p.K + k0) + tq * 16;
        const char* px = reinterpret_cast<const char*>(xs + g * xstride) + tq * 16;
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        mainloop_bf16<4>(pA, pB, px, nsteps, wk, c);
        float* rw = red + wk * kTileRows * kTMax;
        rw[(16 * wm + g) * kTMax + 2 * tq] = c[0];
        rw[(16 * wm + g) * kTMax + 2 * tq + 1] = c[1];
        rw[(16 * wm + g + 8) * kTMax + 2 * tq] = c[2];
        rw[(16 * wm + g + 8) * kTMax + 2 * tq + 1] = c[3];
    } else {
        int rows[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) rows[i] = tile_row(EPI, tb, 16 * wm + i, p.head_dim, p.ffn_s);
        mainloop_f32(reinterpret_cast<const float*>(p.W[r]), rows, p.K, k0,
                     reinterpret_cast<const float*>(xs), xstride, nsteps, wk, lane,
                     red + wk * kTileRows * kTMax + 16 * wm * kTMax);
    }
    __syncthreads();
    for (int i = tid; i < kTileRows * kTMax; i += blockDim.x) tile[i] = red[i] + red[kTileRows * kTMax + i];
    __syncthreads();

    unit_finish<TW, EPI, false>(p, u, gi, r, tb, tile, ss, nullptr, tid, blockDim.x);
}

// ---------------------------------------------------------------------------
// split-KV grouped-query attention, one new token per sequence
// ---------------------------------------------------------------------------

template <typename TW>
__device__ __forceinline__ void load8(const TW* p, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<bf16>(const bf16* p, float (&v)[8]) {
    const uint4 u = ld_stream16(p);
    float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z), e = unpack_bf16x2(u.w);
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y; v[4] = c.x; v[5] = c.y; v[6] = e.x; v[7] = e.y;
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&v)[8]) {
    const uint4 u0 = ld_stream16(p), u1 = ld_stream16(p + 4);
    v[0] = __uint_as_float(u0.x); v[1] = __uint_as_float(u0.y); v[2] = __uint_as_float(u0.z); v[3] = __uint_as_float(u0.w);
    v[4] = __uint_as_float(u1.x); v[5] = __uint_as_float(u1.y); v[6] = __uint_as_float(u1.z); v[7] = __uint_as_float(u1.w);
}

constexpr int kMaxGroup = 8;   // query heads per KV head handled by one CTA

template <typename TW, int D>
__global__ void __launch_bounds__(128) attn_decode_kernel(const AttnDecodeParams p) {
    constexpr int LPK = D / 8;           // lanes per key (8 elements each)
    constexpr int KPP = 128 / LPK;       // keys per pass of the CTA
    extern __shared__ __align__(1024) unsigned char smem[];
    const int G = p.hq_s / p.hkv_s;
    float* qs = reinterpret_cast<float*>(smem);          // [G][D]
    float* sc = qs + kMaxGroup * D;                      // [G][chunk]
    float* red = sc + kMaxGroup * kAttnChunk;            // [KPP][G][D]
    __shared__ float s_m[kMaxGroup], s_l[kMaxGroup];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int u = blockIdx.x;
    const int c = u % p.n_chunks;
    const int gi = u / p.n_chunks;                       // ((r*B + b)*hkv_s + kh)
    const int kh = gi % p.hkv_s;
    const int rb = gi / p.hkv_s;
    const int b = rb % p.B, r = rb / p.B;
    const int T = p.B;
    const int pos = p.pos[b];
    const int Lk = min(pos + 1, p.max_kv);
    const int j0 = c * kAttnChunk;
    const int n = max(0, min(Lk - j0, kAttnChunk));

    const size_t qoff = ((size_t)r * kTMax + b) * p.hq_s * D + (size_t)kh * G * D;
    for (int i = tid; i < G * D; i += 128) qs[i] = p.q[qoff + i] * p.scale;
    __syncthreads();

    const TW* Kb = reinterpret_cast<const TW*>(p.kcache[r]) + ((size_t)b * p.hkv_s + kh) * p.max_kv * D;
    const TW* Vb = reinterpret_cast<const TW*>(p.vcache[r]) + ((size_t)b * p.hkv_s + kh) * p.max_kv * D;
    const int ks = tid / LPK, li = tid % LPK;

    // scores s[g][j] = (q_g / sqrt(d)) . k_j
    // (trip counts are uniform across the warp: the shuffles need all lanes)
    for (int base = 0; base < n; base += 4 * KPP) {
        float kv[4][8];
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
            const int jj = base + ks + uu * KPP;
#pragma unroll
            for (int e = 0; e < 8; ++e) kv[uu][e] = 0.f;
            if (jj < n) load8<TW>(Kb + (size_t)(j0 + jj) * D + li * 8, kv[uu]);
        }
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
            const int jj = base + ks + uu * KPP;
            for (int g = 0; g < G; ++g) {
                float dot = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) dot = fmaf(qs[g * D + li * 8 + e], kv[uu][e], dot);
#pragma unroll
                for (int o = LPK / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
                if (li == 0 && jj < n) sc[g * kAttnChunk + jj] = dot;
            }
        }
    }
    __syncthreads();

    // chunk-local softmax statistics (max, sum of exp) per head
    for (int g = warp; g < G; g += 4) {
        float m = -INFINITY;
        for (int j = lane; j < n; j += 32) m = fmaxf(m, sc[g * kAttnChunk + j]);
        m = warp_max(m);
        float l = 0.f;
        for (int j = lane; j < n; j += 32) {
            const float e = expf(sc[g * kAttnChunk + j] - m);
            sc[g * kAttnChunk + j] = e;
            l += e;
        }
        l = warp_sum(l);
        if (lane == 0) {
            s_m[g] = m;
            s_l[g] = l;
        }
    }
    __syncthreads();

    // unnormalised output o[g] = sum_j e[g][j] v_j
    float acc[kMaxGroup][8];
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
    for (int base = 0; base < n; base += 4 * KPP) {
        float vv[4][8];
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
            const int jj = base + ks + uu * KPP;
            if (jj < n) load8<TW>(Vb + (size_t)(j0 + jj) * D + li * 8, vv[uu]);
        }
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
            const int jj = base + ks + uu * KPP;
            if (jj < n) {
#pragma unroll
                for (int g = 0; g < kMaxGroup; ++g) {
                    if (g < G) {
                        const float e = sc[g * kAttnChunk + jj];
#pragma unroll
                        for (int q = 0; q < 8; ++q) acc[g][q] = fmaf(e, vv[uu][q], acc[g][q]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g)
        if (g < G)
#pragma unroll
            for (int q = 0; q < 8; ++q) red[(ks * G + g) * D + li * 8 + q] = acc[g][q];
    __syncthreads();

    const int pstride = G * (D + 2);
    float* mine = p.part + (size_t)u * pstride;
    for (int i = tid; i < G * D; i += 128) {
        float o = red[i];
        for (int k2 = 1; k2 < KPP; ++k2) o += red[k2 * G * D + i];
        mine[i] = o;
    }
    if (tid < G) {
        mine[G * D + tid] = s_m[tid];
        mine[G * D + G + tid] = s_l[tid];
    }
    if (!arrive_last(&p.cnt[gi], (unsigned)p.n_chunks)) return;

    // combine the chunks in chunk order with log-sum-exp weights
    const float* base = p.part + (size_t)gi * p.n_chunks * pstride;
    TW* out = reinterpret_cast<TW*>(p.out) + qoff;
    for (int i = tid; i < G * D; i += 128) {
        const int g = i / D;
        float M = -INFINITY;
        for (int cc = 0; cc < p.n_chunks; ++cc) {
            const float l = __ldcg(base + (size_t)cc * pstride + G * D + G + g);
            if (l > 0.f) M = fmaxf(M, __ldcg(base + (size_t)cc * pstride + G * D + g));
        }
        float den = 0.f, num = 0.f;
        for (int cc = 0; cc < p.n_chunks; ++cc) {
            const float* pc = base + (size_t)cc * pstride;
            const float l = __ldcg(pc + G * D + G + g);
            if (l > 0.f) {
                const float w = expf(__ldcg(pc + G * D + g) - M);
                den = fmaf(l, w, den);
                num = fmaf(__ldcg(pc + i), w, num);
            }
        }
        Stor<TW>::store(out + i, num / den);
    }
}

// ---------------------------------------------------------------------------
// persistent warp-specialised kernels (bf16): one producer thread streams the
// weights (or KV tiles) with bulk asynchronous copies into a ring of shared
// memory stages; eight consumer warps compute from shared memory. Launched
// with programmatic dependent launch: the producer starts streaming data that
// the preceding kernel does not write while that kernel is still running.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void decode_unit(const GemvParams& p, int epi, int u, int& gi, int& r, int& tb,
                                            int& chunk) {
    const int upg = p.shape.units_per_group();
    gi = u / upg;
    const int rem = u - gi * upg;
    if (epi == EPI_ROWPAR) {
        tb = gi;
        r = rem / p.shape.chunks;
        chunk = rem - r * p.shape.chunks;
    } else {
        const int rb = p.shape.groups / p.n_shards;
        r = gi / rb;
        tb = gi - r * rb;
        chunk = rem;
    }
}

// Tensor-map arguments of one projection launch: a map per shard weight,
// boxes of kBoxK x 32 rows (row-major [rows, K] bf16, no swizzle).
struct TmaGemvArgs {
    CUtensorMap tm[TP_MAX_SHARDS];   // weights, boxes of kBoxK x 32 rows
    CUtensorMap tmx;                 // activation operand rows, boxes of kBoxK x 8 rows
    GemvParams p;
};

// Each stage carries, for 64 rows x 256 reduction elements: the two weight
// boxes (rows 0-31 and 32-63 of the tile) and the matching activation box
// (the shard's 8 token rows). Consumers touch only shared memory.
template <int EPI>
__global__ void __launch_bounds__(kStreamThreads, 2) gemv_stream_kernel(const __grid_constant__ TmaGemvArgs A) {
    const GemvParams& p = A.p;
    extern __shared__ __align__(1024) unsigned char smem[];
    const Ring R = ring_setup(smem, kGemvStages);
    unsigned char* ring = smem + kCtrlBytes;
    float* tile = reinterpret_cast<float*>(ring + kGemvStages * kGemvStageBytes);   // [64][8]
    float* ss = tile + kTileRows * kTMax;                                            // [8] (+pad)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int U = p.shape.units();
    const int kc = p.shape.kc;
    const int spu = (kc + kBoxK - 1) / kBoxK;

    if (warp == kConsumers / 32) {                     // ---- producer
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            uint32_t it = 0;
            bool ok = (smem_u32(ring) & 127u) == 0;    // tensor copies need 128-byte aligned destinations
            if (!ok) {
                *R.abort = 1;
                set_status(p.status, TP_ERR_ALIGN);
            }
            // Weights do not depend on the preceding kernel: the first ring's worth
            // of weight boxes is issued before waiting for it; the activation
            // boxes of those stages follow once it has completed.
            const int my_units = ((int)blockIdx.x < U) ? (U - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
            const uint32_t total = (uint32_t)(my_units * spu);
            bool waited = false;
            int npend = 0;
            int pend_x[kGemvStages], pend_y[kGemvStages];
            for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
                int gi, r, tb, chunk;
                decode_unit(p, EPI, u, gi, r, tb, chunk);
                const int rowa = tile_row(EPI, tb, 0, p.head_dim, p.ffn_s);
                const int rowb = tile_row(EPI, tb, 32, p.head_dim, p.ffn_s);
                const int k0 = chunk * kc;
                for (int st = 0; st < spu; ++st, ++it) {
                    const int sl = it % kGemvStages;
                    if (!mbar_wait(&R.empty[sl], ((it / kGemvStages) & 1) ^ 1, R.abort, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&R.full[sl], 2u * kBoxBytes + kXBoxBytes);
                    unsigned char* dst = ring + sl * kGemvStageBytes;
                    tma_load_2d(dst, &A.tm[r], k0 + st * kBoxK, rowa, &R.full[sl], pol);
                    tma_load_2d(dst + kBoxBytes, &A.tm[r], k0 + st * kBoxK, rowb, &R.full[sl], pol);
                    if (waited) {
                        tma_load_2d_keep(dst + 2 * kBoxBytes, &A.tmx, k0 + st * kBoxK, r * kTMax, &R.full[sl]);
                    } else {
                        pend_x[npend] = k0 + st * kBoxK;
                        pend_y[npend] = r * kTMax;
                        ++npend;
                        if (npend == kGemvStages || it + 1 == total) {
                            pdl_wait();                // activations are written by the preceding kernel
                            waited = true;
                            for (int q = 0; q < npend; ++q) {
                                const uint32_t iq = it + 1 - npend + q;
                                const int sq = iq % kGemvStages;
                                tma_load_2d_keep(ring + sq * kGemvStageBytes + 2 * kBoxBytes, &A.tmx, pend_x[q],
                                                 pend_y[q], &R.full[sq]);
                            }
                            npend = 0;
                        }
                    }
                }
            }
            if (!waited && npend > 0) {                // aborted before the flush: complete the stages' bytes
                pdl_wait();
                for (int q = 0; q < npend; ++q) {
                    const uint32_t iq = it - npend + q;
                    const int sq = iq % kGemvStages;
                    tma_load_2d_keep(ring + sq * kGemvStageBytes + 2 * kBoxBytes, &A.tmx, pend_x[q], pend_y[q],
                                     &R.full[sq]);
                }
            }
            pdl_trigger();
            if (!ok || *R.abort) producer_drain(R, it, kGemvStages);
        }
        return;
    }

    // ---- consumers
    pdl_wait();
    const int wm = warp & 3, wk = warp >> 2;
    const int g = lane >> 2, tq = lane & 3;
    const int box = wm >> 1, brow = 16 * (wm & 1) + g;
    const int T = p.T;
    int* s_pos = reinterpret_cast<int*>(ss + kTMax);                  // [8]
    float* s_bias = ss + 2 * kTMax;                                   // [64]
    // values every unit of this CTA needs, loaded once: the sums of squares
    // of the normalised input and the token positions
    if (EPI == EPI_QKV_ROPE && tid < kTMax) s_pos[tid] = tid < T ? p.pos[tid] : 0;
    if (EPI != EPI_ROWPAR) {
        float a = 0.f;                                                // warp t: token t
        if (warp < T)
            for (int q = lane; q < p.n_ss_tiles; q += 32) a += p.ss_tiles[q * kTMax + warp];
        a = warp_sum(a);
        if (lane == 0) ss[warp] = a;
    }
    consumer_sync(kConsumers);
    uint32_t it = 0;
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
        int gi, r, tb, chunk;
        decode_unit(p, EPI, u, gi, r, tb, chunk);
        float bias_v = 0.f;                                           // in flight during the stages
        if (EPI == EPI_QKV_ROPE && tid < kTileRows && p.bias[r])
            bias_v = p.bias[r][tile_row(EPI_QKV_ROPE, tb, tid, p.head_dim, 0)];
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        for (int st = 0; st < spu; ++st, ++it) {
            const int sl = it % kGemvStages;
            mbar_wait(&R.full[sl], (it / kGemvStages) & 1, R.abort, p.status);
            __syncwarp();   // lanes leave the wait loop independently
            const int steps_here = min(kBoxK / kKStep, (kc - st * kBoxK) / kKStep);
            const unsigned char* stage = ring + sl * kGemvStageBytes;
            const unsigned char* wA = stage + box * kBoxBytes + brow * (kBoxK * 2) + tq * 16;
            const unsigned char* wB = wA + 8 * (kBoxK * 2);
            const unsigned char* px = stage + 2 * kBoxBytes + g * (kBoxK * 2) + tq * 16;
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
                const int step = wk + 2 * s2;
                if (step < steps_here) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 a = *reinterpret_cast<const uint4*>(wA + step * 128 + h * 64);
                        const uint4 b = *reinterpret_cast<const uint4*>(wB + step * 128 + h * 64);
                        const uint4 xv = *reinterpret_cast<const uint4*>(px + step * 128 + h * 64);
                        mma_bf16_16816(c, a.x, b.x, a.y, b.y, xv.x, xv.y);
                        mma_bf16_16816(c, a.z, b.z, a.w, b.w, xv.z, xv.w);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&R.empty[sl]);
        }
        // combine the two reduction halves in a fixed order: (half 0) + (half 1)
        const int i0 = (16 * wm + g) * kTMax + 2 * tq, i1 = (16 * wm + g + 8) * kTMax + 2 * tq;
        if (wk == 0) {
            tile[i0] = c[0];
            tile[i0 + 1] = c[1];
            tile[i1] = c[2];
            tile[i1 + 1] = c[3];
        }
        if (EPI == EPI_QKV_ROPE && tid < kTileRows) s_bias[tid] = bias_v;
        consumer_sync(kConsumers);
        if (wk == 1) {
            tile[i0] += c[0];
            tile[i0 + 1] += c[1];
            tile[i1] += c[2];
            tile[i1 + 1] += c[3];
        }
        consumer_sync(kConsumers);
        if (EPI == EPI_ROWPAR) {
            // this unit's partial sum; the rank-ordered reduction runs in a later kernel
            float* mine = p.part + (size_t)u * kPartStride;
            for (int i = tid * 4; i < kTileRows * kTMax; i += kConsumers * 4)
                *reinterpret_cast<float4*>(mine + i) = *reinterpret_cast<const float4*>(tile + i);
        } else if (EPI == EPI_SWIGLU) {
            bf16* out = reinterpret_cast<bf16*>(p.act_out);
            const float inv_k = 1.0f / (float)p.K;
            for (int i = tid; i < 32 * T; i += kConsumers) {
                const int t = i >> 5, j = i & 31;
                const float rinv = 1.0f / sqrtf(ss[t] * inv_k + p.eps);
                const float gt = tile[j * kTMax + t] * rinv;
                const float up = tile[(j + 32) * kTMax + t] * rinv;
                out[((size_t)r * kTMax + t) * p.ffn_s + tb * 32 + j] = __float2bfloat16_rn(gt / (1.0f + expf(-gt)) * up);
            }
        } else {
            const int d = p.head_dim, half = d >> 1;
            const float inv_k = 1.0f / (float)p.K;
            for (int i = tid; i < 32 * T; i += kConsumers) {
                const int t = i >> 5, j = i & 31;
                const float rinv = 1.0f / sqrtf(ss[t] * inv_k + p.eps);
                const int rowA = tile_row(EPI_QKV_ROPE, tb, j, d, 0);
                const int head = rowA / d, ii = rowA - head * d;
                float va = tile[j * kTMax + t] * rinv + s_bias[j];
                float vb = tile[(j + 32) * kTMax + t] * rinv + s_bias[j + 32];
                const int pos = s_pos[t];
                if (head < p.hq_s + p.hkv_s) {
                    float cs, sn;
                    sincosf((float)pos * exp2f(-(2.0f * ii / d) * (float)p.log2_theta), &sn, &cs);
                    const float ra = va * cs - vb * sn, rb = va * sn + vb * cs;
                    va = ra;
                    vb = rb;
                }
                if (head < p.hq_s) {
                    float* q = p.q_out + ((size_t)r * kTMax + t) * p.hq_s * d + head * d + ii;
                    q[0] = va;
                    q[half] = vb;
                } else {
                    const bool is_k = head < p.hq_s + p.hkv_s;
                    const int kvh = is_k ? head - p.hq_s : head - p.hq_s - p.hkv_s;
                    if (pos < 0 || pos >= p.max_kv) {
                        set_status(p.status, TP_ERR_CAPACITY);
                        continue;
                    }
                    bf16* cache = reinterpret_cast<bf16*>(is_k ? p.kcache[r] : p.vcache[r]);
                    bf16* dst = cache + (((size_t)t * p.hkv_s + kvh) * p.max_kv + pos) * d + ii;
                    dst[0] = __float2bfloat16_rn(va);
                    dst[half] = __float2bfloat16_rn(vb);
                }
            }
        }
        consumer_sync(kConsumers);
    }
}

// Rank-ordered reduction of a row-parallel projection's unit partials (the
// single-device all-reduce), one CTA per 64-row tile, thread = (row, token):
//   y = resid + sum_r (sum_c part[tile][r][c])   -- chunks, then ranks, in order
// With norm_out set it also writes the next RMSNorm's operands (y * gamma_r
// for every shard, bf16) and the tile's per-token sums of squares of y.
__global__ void __launch_bounds__(512) rowpar_reduce_kernel(const GemvParams p) {
    pdl_trigger();
    pdl_wait();
    __shared__ float sq[kTileRows][kTMax];
    const int tb = blockIdx.x, tid = threadIdx.x;
    const int j = tid / kTMax, t = tid - j * kTMax;
    const int upg = p.shape.units_per_group(), C = p.shape.chunks;
    const float* base = p.part + (size_t)tb * upg * kPartStride + j * kTMax + t;
    float v[kMaxGroupUnits];
#pragma unroll
    for (int q = 0; q < kMaxGroupUnits; ++q)
        if (q < upg) v[q] = base[(size_t)q * kPartStride];
    // chunks in order within each rank, then ranks in order
    float total = 0.f, pr = 0.f;
#pragma unroll
    for (int q = 0; q < kMaxGroupUnits; ++q) {
        if (q < upg) {
            const int cc = q % C;
            pr = (cc == 0) ? v[q] : pr + v[q];
            if (cc == C - 1) total = (q < C) ? pr : total + pr;
        }
    }
    const int row = tb * kTileRows + j;
    float yv = 0.f;
    if (t < p.T) {
        const size_t o = (size_t)t * p.rows + row;
        yv = p.resid[o] + total;
        p.y[o] = yv;
        if (p.norm_out) {
            bf16* nout = reinterpret_cast<bf16*>(p.norm_out);
            for (int r2 = 0; r2 < p.n_shards; ++r2)
                nout[((size_t)r2 * kTMax + t) * p.rows + row] = __float2bfloat16_rn(yv * p.gamma2[r2][row]);
        }
    }
    if (p.norm_out) {
        sq[j][t] = yv * yv;
        __syncthreads();
        if (tid < kTMax) {
            float a = 0.f;
            for (int jj = 0; jj < kTileRows; ++jj) a += sq[jj][tid];
            p.ss_tiles_out[tb * kTMax + tid] = a;
        }
    }
}

// RMSNorm operand preparation: CTA (t, kb) writes x[t, kb*256 .. +256) * gamma_r
// as bf16 for every shard and that block's sum of squares ss[kb][t] (rows t >= T
// are zero). 64 threads x 4 elements.
__global__ void __launch_bounds__(64) norm_prep_kernel(const NormPrepParams p) {
    pdl_trigger();                                     // the next kernel may start streaming weights
    pdl_wait();
    __shared__ float wsum[2];
    const int t = blockIdx.x, kb = blockIdx.y, tid = threadIdx.x;
    const int k = kb * 256 + tid * 4;
    const bool in = k < p.H;                           // the last block may be ragged (H % 256 != 0)
    const float4 v = (t < p.T && in) ? *reinterpret_cast<const float4*>(p.x + (size_t)t * p.H + k)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r = 0; r < p.N && in; ++r) {
        const float4 gm = __ldg(reinterpret_cast<const float4*>(p.gamma[r] + k));
        uint2 pk;
        pk.x = pack_bf16x2(v.x * gm.x, v.y * gm.y);
        pk.y = pack_bf16x2(v.z * gm.z, v.w * gm.w);
        *reinterpret_cast<uint2*>(reinterpret_cast<bf16*>(p.xg) + ((size_t)r * kTMax + t) * p.H + k) = pk;
    }
    float a = v.x * v.x;
    a = fmaf(v.y, v.y, a);
    a = fmaf(v.z, v.z, a);
    a = fmaf(v.w, v.w, a);
    a = warp_sum(a);
    if ((tid & 31) == 0) wsum[tid >> 5] = a;
    __syncthreads();
    if (tid == 0) p.ss[kb * kTMax + t] = wsum[0] + wsum[1];
}

template <int D, int G>
__global__ void __launch_bounds__(kStreamThreads, 2) attn_stream_kernel(const AttnDecodeParams p) {
    constexpr int SK = kAttnStageBytes / (D * 2);      // keys per stage
    constexpr int LPK = D / 8;                          // lanes per key
    constexpr int KPP = kConsumers / LPK;               // keys per pass
    extern __shared__ __align__(1024) unsigned char smem[];
    const Ring R = ring_setup(smem);
    unsigned char* ring = smem + kCtrlBytes;
    float* qs = reinterpret_cast<float*>(ring + kStages * kAttnStageBytes);   // [8][D]
    float* sc = qs + kMaxGroup * D;                                           // [8][chunk]
    float* red = sc + kMaxGroup * kAttnChunk;                                 // [8 warps][8][D]
    float* s_m = red + 8 * kMaxGroup * D;                                     // [8]
    float* s_l = s_m + kMaxGroup;                                             // [8]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int U = p.N * p.B * p.hkv_s * p.n_chunks;

    if (warp == kConsumers / 32) {                     // ---- producer
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            uint32_t it = 0;
            bool ok = true, waited = false;
            int posv[kTMax];
            for (int b = 0; b < kTMax; ++b) posv[b] = b < p.B ? p.pos[b] : 0;
            for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
                const int c = u % p.n_chunks, gi = u / p.n_chunks;
                const int kh = gi % p.hkv_s, rb = gi / p.hkv_s, b = rb % p.B, r = rb / p.B;
                int pos = posv[0];
#pragma unroll
                for (int bb = 1; bb < kTMax; ++bb)
                    if (bb == b) pos = posv[bb];
                const int Lk = min(pos + 1, p.max_kv);
                const int j0 = c * kAttnChunk;
                const int n = max(0, min(Lk - j0, kAttnChunk));
                const size_t off = (((size_t)b * p.hkv_s + kh) * p.max_kv + j0) * D;
                for (int half = 0; half < 2 && ok; ++half) {
                    const bf16* src = reinterpret_cast<const bf16*>(half ? p.vcache[r] : p.kcache[r]) + off;
                    for (int k0 = 0; k0 < n; k0 += SK, ++it) {
                        const int keys = min(SK, n - k0);
                        // the tile holding the new position is written by the preceding kernel
                        if (!waited && j0 + k0 + keys > pos) {
                            pdl_wait();
                            waited = true;
                        }
                        const int sl = it % kStages;
                        if (!mbar_wait(&R.empty[sl], ((it / kStages) & 1) ^ 1, R.abort, p.status)) {
                            ok = false;
                            break;
                        }
                        const uint32_t bytes = (uint32_t)keys * D * 2u;
                        mbar_arrive_expect_tx(&R.full[sl], bytes);
                        bulk_g2s(ring + sl * kAttnStageBytes, src + (size_t)k0 * D, bytes, &R.full[sl], pol);
                    }
                }
            }
            pdl_trigger();
            if (!ok || *R.abort) producer_drain(R, it);
        }
        return;
    }

    // ---- consumers
    pdl_wait();
    const int ks = tid / LPK, li = tid % LPK;
    int* s_pos = reinterpret_cast<int*>(s_l + kMaxGroup);
    if (tid < kTMax) s_pos[tid] = tid < p.B ? p.pos[tid] : 0;
    // the first unit's queries; later units' are loaded during the previous unit
    float4 qn = make_float4(0.f, 0.f, 0.f, 0.f);
    auto q_load = [&](int u) {
        const int gi = u / p.n_chunks, kh = gi % p.hkv_s, rb = gi / p.hkv_s, b = rb % p.B, r = rb / p.B;
        const size_t qoff = ((size_t)r * kTMax + b) * p.hq_s * D + (size_t)kh * G * D;
        if (tid * 4 < G * D) qn = *reinterpret_cast<const float4*>(p.q + qoff + tid * 4);
    };
    if ((int)blockIdx.x < U) q_load(blockIdx.x);
    consumer_sync(kConsumers);
    uint32_t it = 0;
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
        const int c = u % p.n_chunks;
        const int b = (u / p.n_chunks / p.hkv_s) % p.B;
        const int pos = s_pos[b];
        const int Lk = min(pos + 1, p.max_kv);
        const int j0 = c * kAttnChunk;
        const int n = max(0, min(Lk - j0, kAttnChunk));
        if (tid * 4 < G * D) {
            float4 v = qn;
            v.x *= p.scale; v.y *= p.scale; v.z *= p.scale; v.w *= p.scale;
            *reinterpret_cast<float4*>(qs + tid * 4) = v;
        }
        consumer_sync(kConsumers);
        if (u + (int)gridDim.x < U) q_load(u + gridDim.x);
        float qr[G][8];                                  // this thread's slice of every query of the group
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) qr[g][e] = qs[g * D + li * 8 + e];

        // scores s[g][j] = (q_g / sqrt(d)) . k_j, one K stage at a time
        for (int k0 = 0; k0 < n; k0 += SK, ++it) {
            const int keys = min(SK, n - k0);
            const int sl = it % kStages;
            mbar_wait(&R.full[sl], (it / kStages) & 1, R.abort, p.status);
            __syncwarp();
            const bf16* Kt = reinterpret_cast<const bf16*>(ring + sl * kAttnStageBytes);
#pragma unroll
            for (int kk = 0; kk < SK; kk += KPP) {       // uniform trip count (shuffles below)
                const int key = kk + ks;
                float kv[8];
                if (key < keys) {
                    const uint4 w = *reinterpret_cast<const uint4*>(Kt + key * D + li * 8);
                    const float2 a0 = unpack_bf16x2(w.x), a1 = unpack_bf16x2(w.y), a2 = unpack_bf16x2(w.z),
                                 a3 = unpack_bf16x2(w.w);
                    kv[0] = a0.x; kv[1] = a0.y; kv[2] = a1.x; kv[3] = a1.y;
                    kv[4] = a2.x; kv[5] = a2.y; kv[6] = a3.x; kv[7] = a3.y;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) kv[e] = 0.f;
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    // four independent partial products, then a short tree
                    float d0 = qr[g][0] * kv[0], d1 = qr[g][1] * kv[1], d2 = qr[g][2] * kv[2], d3 = qr[g][3] * kv[3];
                    d0 = fmaf(qr[g][4], kv[4], d0);
                    d1 = fmaf(qr[g][5], kv[5], d1);
                    d2 = fmaf(qr[g][6], kv[6], d2);
                    d3 = fmaf(qr[g][7], kv[7], d3);
                    float dot = (d0 + d1) + (d2 + d3);
#pragma unroll
                    for (int o = LPK / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
                    if (li == 0 && key < keys) sc[g * kAttnChunk + k0 + key] = dot;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&R.empty[sl]);
        }
        consumer_sync(kConsumers);

        // chunk-local softmax statistics per head
        for (int g = warp; g < G; g += kConsumers / 32) {
            float m = -INFINITY;
            for (int j = lane; j < n; j += 32) m = fmaxf(m, sc[g * kAttnChunk + j]);
            m = warp_max(m);
            float l = 0.f;
            for (int j = lane; j < n; j += 32) {
                const float e = expf(sc[g * kAttnChunk + j] - m);
                sc[g * kAttnChunk + j] = e;
                l += e;
            }
            l = warp_sum(l);
            if (lane == 0) {
                s_m[g] = m;
                s_l[g] = l;
            }
        }
        consumer_sync(kConsumers);

        // unnormalised output o[g] = sum_j e[g][j] v_j, one V stage at a time
        float acc[G][8];
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
        for (int k0 = 0; k0 < n; k0 += SK, ++it) {
            const int keys = min(SK, n - k0);
            const int sl = it % kStages;
            mbar_wait(&R.full[sl], (it / kStages) & 1, R.abort, p.status);
            __syncwarp();
            const bf16* Vt = reinterpret_cast<const bf16*>(ring + sl * kAttnStageBytes);
            for (int key = ks; key < keys; key += KPP) {
                const uint4 w = *reinterpret_cast<const uint4*>(Vt + key * D + li * 8);
                float v[8];
                const float2 a0 = unpack_bf16x2(w.x), a1 = unpack_bf16x2(w.y), a2 = unpack_bf16x2(w.z),
                             a3 = unpack_bf16x2(w.w);
                v[0] = a0.x; v[1] = a0.y; v[2] = a1.x; v[3] = a1.y;
                v[4] = a2.x; v[5] = a2.y; v[6] = a3.x; v[7] = a3.y;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float e = sc[g * kAttnChunk + k0 + key];
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[g][q] = fmaf(e, v[q], acc[g][q]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&R.empty[sl]);
        }
        // reduce over the key slots: first within the warp, then across warps
#pragma unroll
        for (int o = LPK; o < 32; o <<= 1)
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[g][q] += __shfl_xor_sync(0xffffffffu, acc[g][q], o);
        if (lane < LPK) {
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int q = 0; q < 8; ++q) red[(warp * kMaxGroup + g) * D + li * 8 + q] = acc[g][q];
        }
        consumer_sync(kConsumers);
        // this chunk's partial (unnormalised output, max, sum); combined later
        const int pstride = G * (D + 2);
        float* mine = p.part + (size_t)u * pstride;
        for (int i = tid; i < G * D; i += kConsumers) {
            const int g = i / D, dd = i - g * D;
            float o = red[g * D + dd];
            for (int w = 1; w < kConsumers / 32; ++w) o += red[(w * kMaxGroup + g) * D + dd];
            mine[i] = o;
        }
        if (tid < G) {
            mine[G * D + tid] = s_m[tid];
            mine[G * D + G + tid] = s_l[tid];
        }
        consumer_sync(kConsumers);
    }
}

// ---------------------------------------------------------------------------
// tensor-core split-KV decode attention (bf16 caches). The keys are the MMA
// rows: S^T = K Q^T with K from shared memory (M = 16 keys per warp) and the
// group's queries as the 8 columns, so no query padding is needed; then
// O^T = V^T P^T with P^T moved into operand form by movmatrix. K and V of 64
// keys arrive per stage as 2-D tensor-map boxes 72 elements wide (head_dim
// 128), which pads every shared row to 144 bytes: ldmatrix reads are free of
// bank conflicts without a swizzle. Rows past the chunk's valid keys (stale
// cache, other groups, or zero fill) are masked in registers (scores to -inf,
// value operands to zero), so the consumers never write the stages.
// Warps 0-3 take the even 64-key blocks of a chunk, warps 4-7 the odd ones;
// each warp keeps a running max, sum and output for its 16 keys per block;
// the eight are merged at the end of the chunk in a fixed tree order.
// ---------------------------------------------------------------------------

constexpr int kAtKeys = 64;                   // keys per stage
constexpr int kAtRing = 5;
constexpr int kAtMaxStage = 4 * kAtKeys * 72 * 2;   // K and V, two column halves each (head_dim 128)
constexpr int kAtSlot = 1024;                 // floats per merge slot (G * head_dim <= 1024)

template <int D>
struct AtShape {
    static constexpr int NB = D / 64;                     // 64-element column halves per row
    static constexpr int PT = D == 128 ? 72 : 64;         // elements per shared row (box width)
    static constexpr int BOX = kAtKeys * PT * 2;          // bytes per box
    static constexpr int STAGE = 2 * NB * BOX;            // K boxes, then V boxes
};

struct TmaAttnArgs {
    CUtensorMap tk[TP_MAX_SHARDS];
    CUtensorMap tv[TP_MAX_SHARDS];
    AttnDecodeParams p;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// transpose of an 8x8 bf16 matrix held as one 32-bit fragment register per lane
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// shared address of the 8-element chunk `chunk` of key row `key` in a part
// (K or V) of a stage made of 64-element-wide boxes
template <int D>
__device__ __forceinline__ uint32_t at_addr(uint32_t part, int key, int chunk) {
    using S = AtShape<D>;
    return part + (chunk >> 3) * S::BOX + key * (S::PT * 2) + (chunk & 7) * 16;
}

size_t attn_tc_smem() {
    return 1024 + (size_t)kAtRing * kAtMaxStage + (size_t)(4 * kAtSlot + 8 * kMaxGroup * 2 + kTMax) * 4;
}

template <int D>
__global__ void __launch_bounds__(kStreamThreads, 1) attn_tc_kernel(const __grid_constant__ TmaAttnArgs A) {
    using S = AtShape<D>;
    constexpr int KS = D / 16;
    const AttnDecodeParams& p = A.p;
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kAtRing;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 16 * kAtRing);
    unsigned char* ring = smem + 1024;
    float* red = reinterpret_cast<float*>(ring + kAtRing * kAtMaxStage);       // [4][kAtSlot]
    float* s_ml = red + 4 * kAtSlot;                                           // [8 warps][8 queries][m, l]
    int* s_pos = reinterpret_cast<int*>(s_ml + 8 * kMaxGroup * 2);             // [8]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.hq_s / p.hkv_s;
    const int U = p.N * p.B * p.hkv_s * p.n_chunks;
    if (tid == 0) {
        for (int i = 0; i < kAtRing; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 4);           // the four warps of one group release a stage
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumers / 32) {             // ---- producer
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            uint32_t it = 0;
            bool ok = (smem_u32(ring) & 127u) == 0, waited = false;
            if (!ok) {
                *abort_flag = 1;
                set_status(p.status, TP_ERR_ALIGN);
            }
            int posv[kTMax];
            for (int b = 0; b < kTMax; ++b) posv[b] = b < p.B ? p.pos[b] : 0;
            for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
                const int c = u % p.n_chunks, gi = u / p.n_chunks;
                const int kh = gi % p.hkv_s, rb = gi / p.hkv_s, b = rb % p.B, r = rb / p.B;
                int pos = posv[0];
#pragma unroll
                for (int bb = 1; bb < kTMax; ++bb)
                    if (bb == b) pos = posv[bb];
                const int Lk = min(pos + 1, p.max_kv);
                const int j0 = c * kAttnChunk;
                const int n = max(0, min(Lk - j0, kAttnChunk));
                const int row0 = (b * p.hkv_s + kh) * p.max_kv + j0;
                for (int k0 = 0; k0 < n; k0 += kAtKeys, ++it) {
                    if (!waited && j0 + k0 + kAtKeys > pos) {   // holds the position just written
                        pdl_wait();
                        waited = true;
                    }
                    const int sl = it % kAtRing;
                    if (!mbar_wait(&empty[sl], ((it / kAtRing) & 1) ^ 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[sl], (uint32_t)S::STAGE);
                    unsigned char* st = ring + sl * kAtMaxStage;
#pragma unroll
                    for (int h = 0; h < S::NB; ++h) {
                        tma_load_2d(st + h * S::BOX, &A.tk[r], h * 64, row0 + k0, &full[sl], pol);
                        tma_load_2d(st + (S::NB + h) * S::BOX, &A.tv[r], h * 64, row0 + k0, &full[sl], pol);
                    }
                }
            }
            pdl_trigger();
            if (!ok || *abort_flag) {
                volatile int no_abort = 0;
                const uint32_t first = it > (uint32_t)kAtRing ? it - kAtRing : 0u;
                for (uint32_t k = first; k < it; ++k)
                    mbar_wait(&full[k % kAtRing], (k / kAtRing) & 1, &no_abort, nullptr);
            }
        }
        return;
    }

    // ---- consumers
    pdl_wait();
    const int grp = warp >> 2, wq = warp & 3;
    const int g = lane >> 2, t = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;
    if (tid < kTMax) s_pos[tid] = tid < p.B ? p.pos[tid] : 0;
    consumer_sync(kConsumers);
    const uint32_t ring_u32 = smem_u32(ring);
    const int q0 = 2 * t, q1 = 2 * t + 1;                 // the two queries of this lane's fragments
    uint32_t it_unit = 0;
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
        const int c = u % p.n_chunks, gi = u / p.n_chunks;
        const int kh = gi % p.hkv_s, rb = gi / p.hkv_s, b = rb % p.B, r = rb / p.B;
        const int pos = s_pos[b];
        const int Lk = min(pos + 1, p.max_kv);
        const int j0 = c * kAttnChunk;
        const int n = max(0, min(Lk - j0, kAttnChunk));
        const int nblk = (n + kAtKeys - 1) / kAtKeys;

        // B operand of S^T = K Q^T: query g, head-dim pairs (16ks + 2t, +1) and (16ks + 8 + 2t, +1)
        uint32_t qb[KS][2];
        {
            const float* qp = p.q + ((size_t)r * kTMax + b) * p.hq_s * D + (size_t)(kh * G + (g < G ? g : 0)) * D;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                if (g < G) {
                    const float2 a = *reinterpret_cast<const float2*>(qp + 16 * ks + 2 * t);
                    const float2 c2 = *reinterpret_cast<const float2*>(qp + 16 * ks + 8 + 2 * t);
                    qb[ks][0] = pack_bf16x2(a.x * p.scale, a.y * p.scale);
                    qb[ks][1] = pack_bf16x2(c2.x * p.scale, c2.y * p.scale);
                } else {
                    qb[ks][0] = qb[ks][1] = 0u;
                }
            }
        }
        float o[KS][4];
#pragma unroll
        for (int dt = 0; dt < KS; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

        for (int blk = grp; blk < nblk; blk += 2) {
            const uint32_t it = it_unit + blk;
            const int sl = it % kAtRing;
            mbar_wait(&full[sl], (it / kAtRing) & 1, abort_flag, p.status);
            __syncwarp();                        // lanes leave the wait loop independently
            const uint32_t kpart = ring_u32 + sl * kAtMaxStage, vpart = kpart + S::NB * S::BOX;
            const int kb = blk * kAtKeys + 16 * wq;          // this warp's first key, relative to the chunk
            // ---- S^T for 16 keys x 8 queries
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(at_addr<D>(kpart, 16 * wq + rr + 8 * (mi & 1), 2 * ks + (mi >> 1)), a0, a1, a2, a3);
                mma_bf16_16816(sc, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
            }
            // ---- online softmax per query over this warp's keys (rows g and g + 8)
            const bool v0 = kb + g < n, v1 = kb + g + 8 < n;
            const float x00 = v0 ? sc[0] : -INFINITY, x01 = v0 ? sc[1] : -INFINITY;
            const float x10 = v1 ? sc[2] : -INFINITY, x11 = v1 ? sc[3] : -INFINITY;
            float mq0 = fmaxf(x00, x10), mq1 = fmaxf(x01, x11);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mq0 = fmaxf(mq0, __shfl_xor_sync(0xffffffffu, mq0, off));
                mq1 = fmaxf(mq1, __shfl_xor_sync(0xffffffffu, mq1, off));
            }
            const float n0 = fmaxf(m0, mq0), n1 = fmaxf(m1, mq1);
            const float al0 = (n0 == -INFINITY) ? 1.f : expf(m0 - n0);
            const float al1 = (n1 == -INFINITY) ? 1.f : expf(m1 - n1);
            const float p00 = (x00 == -INFINITY) ? 0.f : expf(x00 - n0);
            const float p10 = (x10 == -INFINITY) ? 0.f : expf(x10 - n0);
            const float p01 = (x01 == -INFINITY) ? 0.f : expf(x01 - n1);
            const float p11 = (x11 == -INFINITY) ? 0.f : expf(x11 - n1);
            float ps0 = p00 + p10, ps1 = p01 + p11;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                ps0 += __shfl_xor_sync(0xffffffffu, ps0, off);
                ps1 += __shfl_xor_sync(0xffffffffu, ps1, off);
            }
            l0 = l0 * al0 + ps0;
            l1 = l1 * al1 + ps1;
            m0 = n0;
            m1 = n1;
#pragma unroll
            for (int dt = 0; dt < KS; ++dt) {
                o[dt][0] *= al0;
                o[dt][1] *= al1;
                o[dt][2] *= al0;
                o[dt][3] *= al1;
            }
            // ---- O^T += V^T P^T; P^T fragments: (keys 2t, 2t+1 | 8+2t, 9+2t ; query g)
            const uint32_t pb0 = movmatrix_t(pack_bf16x2(p00, p01));
            const uint32_t pb1 = movmatrix_t(pack_bf16x2(p10, p11));
            const uint32_t mlo = (kb + 2 * t < n ? 0x0000FFFFu : 0u) | (kb + 2 * t + 1 < n ? 0xFFFF0000u : 0u);
            const uint32_t mhi = (kb + 8 + 2 * t < n ? 0x0000FFFFu : 0u) | (kb + 9 + 2 * t < n ? 0xFFFF0000u : 0u);
#pragma unroll
            for (int dt = 0; dt < KS; ++dt) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(at_addr<D>(vpart, 16 * wq + rr + 8 * (mi >> 1), 2 * dt + (mi & 1)), a0, a1, a2, a3);
                mma_bf16_16816(o[dt], a0 & mlo, a1 & mlo, a2 & mhi, a3 & mhi, pb0, pb1);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[sl]);
        }
        it_unit += nblk;

        // ---- merge the eight warps: common max, then a fixed tree of sums
        if (g == 0) {
            s_ml[(warp * kMaxGroup + q0) * 2] = m0;
            s_ml[(warp * kMaxGroup + q0) * 2 + 1] = l0;
            s_ml[(warp * kMaxGroup + q1) * 2] = m1;
            s_ml[(warp * kMaxGroup + q1) * 2 + 1] = l1;
        }
        consumer_sync(kConsumers);
        float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            M0 = fmaxf(M0, s_ml[(w * kMaxGroup + q0) * 2]);
            M1 = fmaxf(M1, s_ml[(w * kMaxGroup + q1) * 2]);
        }
        const float c0 = (m0 == -INFINITY) ? 0.f : expf(m0 - M0);
        const float c1 = (m1 == -INFINITY) ? 0.f : expf(m1 - M1);
#pragma unroll
        for (int dt = 0; dt < KS; ++dt) {
            o[dt][0] *= c0;
            o[dt][1] *= c1;
            o[dt][2] *= c0;
            o[dt][3] *= c1;
        }
        // round 1: warps 4-7 -> 0-3; round 2: 2,3 -> 0,1; round 3: 1 -> 0
        for (int half = 4; half >= 1; half >>= 1) {
            if (warp >= half && warp < 2 * half) {
                float* dst = red + (warp - half) * kAtSlot;
#pragma unroll
                for (int dt = 0; dt < KS; ++dt) {
                    if (q0 < G) {
                        dst[q0 * D + 16 * dt + g] = o[dt][0];
                        dst[q0 * D + 16 * dt + g + 8] = o[dt][2];
                    }
                    if (q1 < G) {
                        dst[q1 * D + 16 * dt + g] = o[dt][1];
                        dst[q1 * D + 16 * dt + g + 8] = o[dt][3];
                    }
                }
            }
            consumer_sync(kConsumers);
            if (warp < half) {
                const float* src = red + warp * kAtSlot;
#pragma unroll
                for (int dt = 0; dt < KS; ++dt) {
                    if (q0 < G) {
                        o[dt][0] += src[q0 * D + 16 * dt + g];
                        o[dt][2] += src[q0 * D + 16 * dt + g + 8];
                    }
                    if (q1 < G) {
                        o[dt][1] += src[q1 * D + 16 * dt + g];
                        o[dt][3] += src[q1 * D + 16 * dt + g + 8];
                    }
                }
            }
            consumer_sync(kConsumers);
        }
        if (warp == 0 && (unsigned)u < p.part_units) {
            float* mine = p.part + (size_t)u * G * (D + 2);
#pragma unroll
            for (int dt = 0; dt < KS; ++dt) {
                if (q0 < G) {
                    mine[q0 * D + 16 * dt + g] = o[dt][0];
                    mine[q0 * D + 16 * dt + g + 8] = o[dt][2];
                }
                if (q1 < G) {
                    mine[q1 * D + 16 * dt + g] = o[dt][1];
                    mine[q1 * D + 16 * dt + g + 8] = o[dt][3];
                }
            }
            if (g == 0) {
                float L0 = 0.f, L1 = 0.f;
                for (int w = 0; w < 8; ++w) {
                    const float mw0 = s_ml[(w * kMaxGroup + q0) * 2], mw1 = s_ml[(w * kMaxGroup + q1) * 2];
                    if (mw0 != -INFINITY) L0 += s_ml[(w * kMaxGroup + q0) * 2 + 1] * expf(mw0 - M0);
                    if (mw1 != -INFINITY) L1 += s_ml[(w * kMaxGroup + q1) * 2 + 1] * expf(mw1 - M1);
                }
                if (q0 < G) {
                    mine[G * D + q0] = M0;
                    mine[G * D + G + q0] = L0;
                }
                if (q1 < G) {
                    mine[G * D + q1] = M1;
                    mine[G * D + G + q1] = L1;
                }
            }
        }
        consumer_sync(kConsumers);               // s_ml and red are reused by the next unit
    }
}

// Combines the split-KV chunk partials of one (shard, sequence, KV head)
// group in chunk order with log-sum-exp weights; one CTA per group.
template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnDecodeParams p) {
    pdl_trigger();
    pdl_wait();
    constexpr int kMaxC = 128;                          // chunk statistics held in shared memory
    __shared__ float s_m[kMaxC][kMaxGroup], s_l[kMaxC][kMaxGroup];
    __shared__ float s_den[kMaxGroup], s_M[kMaxGroup];
    const int gi = blockIdx.x, tid = threadIdx.x;
    const int G = p.hq_s / p.hkv_s, pstride = G * (D + 2);
    const int kh = gi % p.hkv_s, rb = gi / p.hkv_s, b = rb % p.B, r = rb / p.B;
    const float* base = p.part + (size_t)gi * p.n_chunks * pstride;
    const int nc = min(p.n_chunks, kMaxC);
    if (p.n_chunks > kMaxC) set_status(p.status, TP_ERR_UNSUPPORTED);
    // all chunks' (max, sum) in one parallel pass
    for (int i = tid; i < nc * 2 * G; i += 256) {
        const int cc = i / (2 * G), q = i - cc * 2 * G;
        const float v = base[(size_t)cc * pstride + G * D + q];
        if (q < G) s_m[cc][q] = v; else s_l[cc][q - G] = v;
    }
    __syncthreads();
    if (tid < G) {
        float M = -INFINITY;
        for (int cc = 0; cc < nc; ++cc)
            if (s_l[cc][tid] > 0.f) M = fmaxf(M, s_m[cc][tid]);
        float den = 0.f;
        for (int cc = 0; cc < nc; ++cc) {
            const float w = s_l[cc][tid] > 0.f ? expf(s_m[cc][tid] - M) : 0.f;
            s_m[cc][tid] = w;                           // reuse as the chunk weight
            den = fmaf(s_l[cc][tid], w, den);
        }
        s_den[tid] = den;
        s_M[tid] = M;
    }
    __syncthreads();
    const size_t qoff = ((size_t)r * kTMax + b) * p.hq_s * D + (size_t)kh * G * D;
    bf16* out = reinterpret_cast<bf16*>(p.out) + qoff;
    for (int i = tid; i < G * D; i += 256) {
        const int g = i / D;
        float num = 0.f;
        int cc = 0;
        for (; cc + 8 <= nc; cc += 8) {                  // eight independent loads in flight
            float v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = base[(size_t)(cc + q) * pstride + i];
#pragma unroll
            for (int q = 0; q < 8; ++q) num = fmaf(v[q], s_m[cc + q][g], num);
        }
        for (; cc < nc; ++cc) num = fmaf(base[(size_t)cc * pstride + i], s_m[cc][g], num);
        out[i] = __float2bfloat16_rn(num / s_den[g]);
    }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

template <typename TW>
static size_t gemv_smem(const GemvParams& p) {
    return (size_t)kTMax * (p.shape.kc + XPad<TW>::v) * sizeof(TW) +
           (size_t)(3 * kTileRows * kTMax + kTMax) * sizeof(float);
}

template <typename TW, int EPI>
static cudaError_t launch_gemv_t(const GemvParams& p, cudaStream_t s) {
    const size_t smem = gemv_smem<TW>(p);
    static int set_bytes = -1;                  // raise the limit once per size (host-side only)
    if ((int)smem > set_bytes) {
        cudaError_t e = cudaFuncSetAttribute(gemv_kernel<TW, EPI>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        set_bytes = (int)smem;
    }
    gemv_kernel<TW, EPI><<<p.shape.units(), 256, smem, s>>>(p);
    return cudaGetLastError();
}

static bool g_pdl = true;
void set_pdl(bool on) { g_pdl = on; }

cudaError_t launch_pdl(const void* fn, void** args, int grid, size_t smem, cudaStream_t s, int threads) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_pdl ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

size_t gemv_stream_smem(int kc) {
    (void)kc;
    // ring | tile [64][8] | ss [8], positions [8], bias [64] (+pad)
    return kCtrlBytes + (size_t)kGemvStages * kGemvStageBytes + (size_t)(kTileRows * kTMax + 96) * 4;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); each distinct map is encoded once and cached.
cudaError_t tensor_map_2d(const void* base, long inner, long rows, int box_inner, int box_rows, int swizzle128,
                          CUtensorMap* out) {
    static std::mutex mu;
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    struct Entry { const void* w; long inner, rows; int bi, br, sw; CUtensorMap tm; };
    static std::vector<Entry> cache;
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : cache)
        if (e.w == base && e.inner == inner && e.rows == rows && e.bi == box_inner && e.br == box_rows &&
            e.sw == swizzle128) {
            *out = e.tm;
            return cudaSuccess;
        }
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void**>(&encode),
                                                         12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || !encode) return e != cudaSuccess ? e : cudaErrorNotSupported;
    }
    cuuint64_t gdim[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)inner * 2};
    cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
    cuuint32_t estride[2] = {1u, 1u};
    Entry ent{base, inner, rows, box_inner, box_rows, swizzle128, {}};
    CUresult r = encode(&ent.tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box,
                        estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (cache.size() > 4096) cache.clear();
    cache.push_back(ent);
    *out = ent.tm;
    return cudaSuccess;
}

static cudaError_t weight_tensor_map(const void* W, int K, int rows, CUtensorMap* out, int box_rows = 32) {
    return tensor_map_2d(W, K, rows, kBoxK, box_rows, 0, out);
}

template <int EPI>
static cudaError_t launch_gemv_stream(const GemvParams& p, cudaStream_t s) {
    const size_t smem = gemv_stream_smem(p.shape.kc);
    static int set_bytes = -1;
    if ((int)smem > set_bytes) {
        cudaError_t e = cudaFuncSetAttribute(gemv_stream_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        // full shared-memory carveout, so a CTA of the next kernel fits beside this one
        e = cudaFuncSetAttribute(gemv_stream_kernel<EPI>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        set_bytes = (int)smem;
    }
    TmaGemvArgs A;
    memset(&A, 0, sizeof A);
    A.p = p;
    for (int r = 0; r < p.n_shards; ++r) {
        cudaError_t e = weight_tensor_map(p.W[r], p.K, p.rows, &A.tm[r]);
        if (e != cudaSuccess) return e;
    }
    cudaError_t ex = weight_tensor_map(p.xact, p.K, p.n_shards * kTMax, &A.tmx, kTMax);
    if (ex != cudaSuccess) return ex;
    const int grid = p.shape.units() < 2 * kSMs ? p.shape.units() : 2 * kSMs;   // two CTAs per SM
    void* args[] = {&A};
    cudaError_t e = launch_pdl(reinterpret_cast<const void*>(gemv_stream_kernel<EPI>), args, grid, smem, s, kStreamThreads);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_norm_prep(const NormPrepParams& p, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kTMax, (p.H + 255) / 256);
    cfg.blockDim = dim3(64);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_pdl ? 1 : 0;
    void* args[] = {const_cast<NormPrepParams*>(&p)};
    cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(norm_prep_kernel), args);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_gemv(const GemvParams& p, int epi, int dtype, cudaStream_t s) {
    if (dtype == TP_BF16) {
        if (epi == EPI_QKV_ROPE) return launch_gemv_stream<EPI_QKV_ROPE>(p, s);
        if (epi == EPI_SWIGLU) return launch_gemv_stream<EPI_SWIGLU>(p, s);
        return launch_gemv_stream<EPI_ROWPAR>(p, s);
    }
    if (epi == EPI_QKV_ROPE) return launch_gemv_t<float, EPI_QKV_ROPE>(p, s);
    if (epi == EPI_SWIGLU) return launch_gemv_t<float, EPI_SWIGLU>(p, s);
    return launch_gemv_t<float, EPI_ROWPAR>(p, s);
}

template <typename TW, int D>
static cudaError_t launch_attn_t(const AttnDecodeParams& p, cudaStream_t s) {
    constexpr int KPP = 128 / (D / 8);
    const size_t smem = (size_t)(kMaxGroup * D + kMaxGroup * kAttnChunk + KPP * kMaxGroup * D) * sizeof(float);
    static bool set = false;
    if (!set) {
        cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<TW, D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        set = true;
    }
    const int grid = p.N * p.B * p.hkv_s * p.n_chunks;
    attn_decode_kernel<TW, D><<<grid, 128, smem, s>>>(p);
    return cudaGetLastError();
}

size_t attn_stream_smem(int d) {
    return kCtrlBytes + (size_t)kStages * kAttnStageBytes +
           (size_t)(kMaxGroup * d + kMaxGroup * kAttnChunk + 8 * kMaxGroup * d + 2 * kMaxGroup + kTMax) * 4;
}

template <int D, int G>
static cudaError_t launch_attn_stream(const AttnDecodeParams& p, cudaStream_t s) {
    const size_t smem = attn_stream_smem(D);
    static bool set = false;
    if (!set) {
        cudaError_t e = cudaFuncSetAttribute(attn_stream_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(attn_stream_kernel<D, G>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        set = true;
    }
    const int U = p.N * p.B * p.hkv_s * p.n_chunks;
    const int grid = U < 2 * kSMs ? U : 2 * kSMs;       // two CTAs per SM: more warps to hide latency
    void* args[] = {const_cast<AttnDecodeParams*>(&p)};
    cudaError_t e = launch_pdl(reinterpret_cast<const void*>(attn_stream_kernel<D, G>), args, grid, smem, s,
                               kStreamThreads);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int D>
static cudaError_t launch_attn_stream_g(const AttnDecodeParams& p, cudaStream_t s) {
    switch (p.hq_s / p.hkv_s) {
        case 1: return launch_attn_stream<D, 1>(p, s);
        case 2: return launch_attn_stream<D, 2>(p, s);
        case 3: return launch_attn_stream<D, 3>(p, s);
        case 4: return launch_attn_stream<D, 4>(p, s);
        case 5: return launch_attn_stream<D, 5>(p, s);
        case 6: return launch_attn_stream<D, 6>(p, s);
        case 7: return launch_attn_stream<D, 7>(p, s);
        default: return launch_attn_stream<D, 8>(p, s);
    }
}

static cudaError_t launch_small_pdl(const void* fn, void** args, int grid, int threads, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_rowpar_reduce(const GemvParams& p, cudaStream_t s) {
    void* args[] = {const_cast<GemvParams*>(&p)};
    return launch_small_pdl(reinterpret_cast<const void*>(rowpar_reduce_kernel), args, p.shape.groups,
                            kTileRows * kTMax, s);
}

cudaError_t launch_attn_combine(const AttnDecodeParams& p, cudaStream_t s) {
    void* args[] = {const_cast<AttnDecodeParams*>(&p)};
    const void* fn = p.d == 64 ? reinterpret_cast<const void*>(attn_combine_kernel<64>)
                               : reinterpret_cast<const void*>(attn_combine_kernel<128>);
    return launch_small_pdl(fn, args, p.N * p.B * p.hkv_s, 256, s);
}

template <int D>
static cudaError_t launch_attn_tc(const AttnDecodeParams& p, cudaStream_t s) {
    using S = AtShape<D>;
    const size_t smem = attn_tc_smem();
    static bool set = false;
    if (!set) {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        set = true;
    }
    if ((p.hq_s / p.hkv_s) * D > kAtSlot) return cudaErrorInvalidValue;
    TmaAttnArgs A;
    memset(&A, 0, sizeof A);
    A.p = p;
    const long rows = (long)p.max_batch * p.hkv_s * p.max_kv;
    for (int r = 0; r < p.N; ++r) {
        cudaError_t e = tensor_map_2d(p.kcache[r], D, rows, S::PT, kAtKeys, 0, &A.tk[r]);
        if (e == cudaSuccess) e = tensor_map_2d(p.vcache[r], D, rows, S::PT, kAtKeys, 0, &A.tv[r]);
        if (e != cudaSuccess) return e;
    }
    const int U = p.N * p.B * p.hkv_s * p.n_chunks;
    const int grid = U < kSMs ? U : kSMs;
    void* args[] = {&A};
    cudaError_t e = launch_pdl(reinterpret_cast<const void*>(attn_tc_kernel<D>), args, grid, smem, s, kStreamThreads);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_attn_decode(const AttnDecodeParams& p, int dtype, cudaStream_t s) {
    if (dtype == TP_BF16) return p.d == 64 ? launch_attn_tc<64>(p, s) : launch_attn_tc<128>(p, s);
    return p.d == 64 ? launch_attn_t<float, 64>(p, s) : launch_attn_t<float, 128>(p, s);
}


// ===========================================================================
// The whole decode step in one persistent launch (bf16).
//
// One CTA per SM runs every stage of the block as a phase:
//   NORM -> QKV (+RoPE, KV append) -> ATTN (split-KV partials) -> COMBINE
//   -> O_PROJ (partials) -> REDUCE (h, next norm operands) -> GATE_UP
//   (+SwiGLU) -> DOWN (partials) -> REDUCE (y)
// separated by grid barriers (a sense-reversing counter in the workspace,
// every wait bounded). The producer thread streams the data of later
// phases that does not depend on earlier ones -- every weight box, and every
// K/V block except the one holding the new position -- through the same
// 5-stage ring while the consumers are still in an earlier phase or waiting
// at a barrier; only the activation boxes (and the new K/V rows) wait for
// the barrier that publishes them. So HBM keeps streaming across phase
// boundaries and no kernel boundary, launch gap or ramp remains inside the
// step. The phases compute exactly what the separate kernels compute.
// ===========================================================================

namespace {
constexpr int kSkRing = 5;
constexpr int kSkStage = kGemvStageBytes;               // 36 KB: 2 weight boxes + activation box, or K+V of 64 keys
constexpr int kSkPhases = 8;                            // barriers inside a step
constexpr int kSkMaxPend = kSkRing;
static_assert(kGemvStageBytes == kAtMaxStage, "the two stage formats share one slot size");
}  // namespace

struct StepArgs {
    CUtensorMap wm[4][TP_MAX_SHARDS];       // weights of qkv, o, gate_up, down (boxes kBoxK x 32)
    CUtensorMap xm[4];                      // their activation operands (boxes kBoxK x 8)
    CUtensorMap tk[TP_MAX_SHARDS];          // K / V caches (boxes 72 or 64 x 64 keys)
    CUtensorMap tv[TP_MAX_SHARDS];
    GemvParams g[4];                        // qkv, o, gate_up, down
    AttnDecodeParams a;
    NormPrepParams np;
    unsigned long long* bar;                // grid-barrier arrival counter (only grows)
    unsigned long long* stamps;             // optional [grid][kStepStamps]: start, 8 barrier arrivals, end (ns)
};

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Grid barrier k of a step has passed once the arrival counter reaches
// base + k * gridDim.x. The counter only grows (by kSkPhases * gridDim.x per
// step, every CTA arriving at every barrier even after an error), so `base`
// is the multiple of that amount at or below the value read at the start.
__device__ __forceinline__ bool sk_passed(const unsigned long long* bar, unsigned long long base, unsigned k) {
    return ld_acquire_u64(bar) >= base + (unsigned long long)k * gridDim.x;
}

__device__ __forceinline__ bool sk_wait_gen(const unsigned long long* bar, unsigned long long base, unsigned k,
                                            volatile int* abort, int* status) {
    if (sk_passed(bar, base, k)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (sk_passed(bar, base, k)) return true;
        if (*abort) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            set_status(status, TP_ERR_TIMEOUT);
            return false;
        }
    }
}

// Consumer side of grid barrier k: every consumer thread of the CTA has
// finished the phase; thread 0 arrives with a release reduction (no reply
// to wait for) and polls the counter with acquire loads.
__device__ __forceinline__ void sk_barrier(unsigned long long* bar, unsigned long long base, unsigned k,
                                           volatile int* abort, int* status, unsigned long long* stamp) {
    consumer_sync(kConsumers);
    if (threadIdx.x == 0) {
        if (stamp) *stamp = global_ns();
        asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(bar) : "memory");
        sk_wait_gen(bar, base, k, abort, status);
    }
    consumer_sync(kConsumers);
}

// ---- producer helpers -------------------------------------------------------

// Stages whose activation box waits for a barrier, oldest first.
struct SkPend {
    int n;
    uint32_t stage[kSkMaxPend];
    int slot[kSkMaxPend], x[kSkMaxPend], y[kSkMaxPend], map[kSkMaxPend];
    unsigned need[kSkMaxPend];
};

// Issues every pending activation box whose barrier has passed, waiting for
// the barriers in order (oldest first).
__device__ __forceinline__ bool sk_flush(SkPend& pd, const StepArgs& A, unsigned char* ring, uint64_t* full,
                                         unsigned long long gen0, volatile int* abort, int* status) {
    bool ok = true;
    for (int i = 0; i < pd.n; ++i) {
        if (ok) ok = sk_wait_gen(A.bar, gen0, pd.need[i], abort, status);
        // the activations were written by other CTAs' ordinary stores
        asm volatile("fence.proxy.async.global;" ::: "memory");
        // issued even after a failed wait: the stage's byte count must complete
        tma_load_2d_keep(ring + pd.slot[i] * kSkStage + 2 * kBoxBytes, &A.xm[pd.map[i]], pd.x[i], pd.y[i],
                         &full[pd.slot[i]]);
    }
    pd.n = 0;
    return ok;
}

// Before the producer reuses the slot of stage `it` (last held by stage
// it - kSkRing): if that stage is still pending, its consumers cannot release
// the slot until its activation box is issued.
__device__ __forceinline__ void sk_before_reuse(SkPend& pd, uint32_t it, const StepArgs& A, unsigned char* ring,
                                                uint64_t* full, unsigned long long gen0, volatile int* abort,
                                                int* status) {
    if (pd.n > 0 && pd.stage[0] + kSkRing <= it) sk_flush(pd, A, ring, full, gen0, abort, status);
}

// Producer of one projection phase: weight boxes at once, the activation box
// once barrier `need` has passed.
__device__ __forceinline__ bool sk_produce_gemv(int epi, int wi, unsigned need, const StepArgs& A, unsigned char* ring,
                                                uint64_t* full, uint64_t* empty, uint32_t& it, SkPend& pd,
                                                unsigned long long gen0, volatile int* abort, uint64_t pol) {
    const GemvParams& p = A.g[wi];
    const int U = p.shape.units();
    const int kc = p.shape.kc;
    const int spu = (kc + kBoxK - 1) / kBoxK;
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
        int gi, r, tb, chunk;
        decode_unit(p, epi, u, gi, r, tb, chunk);
        const int rowa = tile_row(epi, tb, 0, p.head_dim, p.ffn_s);
        const int rowb = tile_row(epi, tb, 32, p.head_dim, p.ffn_s);
        const int k0 = chunk * kc;
        for (int st = 0; st < spu; ++st, ++it) {
            const int sl = it % kSkRing;
            sk_before_reuse(pd, it, A, ring, full, gen0, abort, p.status);
            if (!mbar_wait(&empty[sl], ((it / kSkRing) & 1) ^ 1, abort, p.status)) return false;
            mbar_arrive_expect_tx(&full[sl], 2u * kBoxBytes + kXBoxBytes);
            unsigned char* dst = ring + sl * kSkStage;
            tma_load_2d(dst, &A.wm[wi][r], k0 + st * kBoxK, rowa, &full[sl], pol);
            tma_load_2d(dst + kBoxBytes, &A.wm[wi][r], k0 + st * kBoxK, rowb, &full[sl], pol);
            if (pd.n == 0 && sk_passed(A.bar, gen0, need)) {
                asm volatile("fence.proxy.async.global;" ::: "memory");
                tma_load_2d_keep(dst + 2 * kBoxBytes, &A.xm[wi], k0 + st * kBoxK, r * kTMax, &full[sl]);
            } else {
                pd.stage[pd.n] = it;
                pd.slot[pd.n] = sl;
                pd.x[pd.n] = k0 + st * kBoxK;
                pd.y[pd.n] = r * kTMax;
                pd.map[pd.n] = wi;
                pd.need[pd.n] = need;
                ++pd.n;
            }
        }
    }
    return true;
}

template <int D>
__device__ __forceinline__ bool sk_produce_attn(unsigned need, const StepArgs& A, unsigned char* ring, uint64_t* full,
                                                uint64_t* empty, uint32_t& it, SkPend& pd, unsigned long long gen0,
                                                volatile int* abort, uint64_t pol, const int* posv) {
    using S = AtShape<D>;
    const AttnDecodeParams& p = A.a;
    const int U = p.N * p.B * p.hkv_s * p.n_chunks;
    bool passed = false;
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
        const int c = u % p.n_chunks, gi = u / p.n_chunks;
        const int kh = gi % p.hkv_s, rb = gi / p.hkv_s, b = rb % p.B, r = rb / p.B;
        const int pos = posv[b];
        const int Lk = min(pos + 1, p.max_kv);
        const int j0 = c * kAttnChunk;
        const int n = max(0, min(Lk - j0, kAttnChunk));
        const int row0 = (b * p.hkv_s + kh) * p.max_kv + j0;
        for (int k0 = 0; k0 < n; k0 += kAtKeys, ++it) {
            // the block holding the new position is written by the QKV phase
            if (!passed && j0 + k0 + kAtKeys > pos) {
                sk_flush(pd, A, ring, full, gen0, abort, p.status);
                sk_wait_gen(A.bar, gen0, need, abort, p.status);
                asm volatile("fence.proxy.async.global;" ::: "memory");
                passed = true;
            }
            const int sl = it % kSkRing;
            sk_before_reuse(pd, it, A, ring, full, gen0, abort, p.status);
            if (!mbar_wait(&empty[sl], ((it / kSkRing) & 1) ^ 1, abort, p.status)) return false;
            mbar_arrive_expect_tx(&full[sl], (uint32_t)S::STAGE);
            unsigned char* st = ring + sl * kSkStage;
#pragma unroll
            for (int h = 0; h < S::NB; ++h) {
                tma_load_2d(st + h * S::BOX, &A.tk[r], h * 64, row0 + k0, &full[sl], pol);
                tma_load_2d(st + (S::NB + h) * S::BOX, &A.tv[r], h * 64, row0 + k0, &full[sl], pol);
            }
        }
    }
    return true;
}

// ---- consumer phases ---------------------------------------------------------

// RMSNorm operands: x * gamma_r (bf16) for every shard and per-256-block
// sums of squares; one (token, 256-block) item per warp, all SMs.
__device__ __forceinline__ void sk_norm(const NormPrepParams& p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nkb = (p.H + 255) / 256;
    const int items = kTMax * nkb;
    for (int item = blockIdx.x * 8 + warp; item < items; item += gridDim.x * 8) {
        const int t = item / nkb, kb = item - t * nkb;
        float a = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int k = kb * 256 + h * 128 + lane * 4;
            const bool in = k < p.H;
            const float4 v = (t < p.T && in) ? *reinterpret_cast<const float4*>(p.x + (size_t)t * p.H + k)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
            for (int r = 0; r < p.N && in; ++r) {
                const float4 gm = __ldg(reinterpret_cast<const float4*>(p.gamma[r] + k));
                uint2 pk;
                pk.x = pack_bf16x2(v.x * gm.x, v.y * gm.y);
                pk.y = pack_bf16x2(v.z * gm.z, v.w * gm.w);
                *reinterpret_cast<uint2*>(reinterpret_cast<bf16*>(p.xg) + ((size_t)r * kTMax + t) * p.H + k) = pk;
            }
            a = fmaf(v.x, v.x, a);
            a = fmaf(v.y, v.y, a);
            a = fmaf(v.z, v.z, a);
            a = fmaf(v.w, v.w, a);
        }
        a = warp_sum(a);
        if (lane == 0) p.ss[kb * kTMax + t] = a;
    }
}

// One projection phase on the consumer side (the units of this CTA).
template <int EPI>
__device__ __forceinline__ void sk_gemv(const GemvParams& p, unsigned char* ring, uint64_t* full, uint64_t* empty,
                                        volatile int* abort, uint32_t& it, float* tile, float* ss, int* s_pos,
                                        float* s_bias) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int U = p.shape.units();
    const int kc = p.shape.kc;
    const int spu = (kc + kBoxK - 1) / kBoxK;
    const int wm = warp & 3, wk = warp >> 2;
    const int g = lane >> 2, tq = lane & 3;
    const int box = wm >> 1, brow = 16 * (wm & 1) + g;
    const int T = p.T;
    if ((int)blockIdx.x >= U) return;
    if (EPI == EPI_QKV_ROPE && tid < kTMax) s_pos[tid] = tid < T ? p.pos[tid] : 0;
    if (EPI != EPI_ROWPAR) {
        float a = 0.f;                                 // warp t: token t
        if (warp < T)
            for (int q = lane; q < p.n_ss_tiles; q += 32) a += p.ss_tiles[q * kTMax + warp];
        a = warp_sum(a);
        if (lane == 0) ss[warp] = a;
    }
    consumer_sync(kConsumers);
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
        int gi, r, tb, chunk;
        decode_unit(p, EPI, u, gi, r, tb, chunk);
        float bias_v = 0.f;
        if (EPI == EPI_QKV_ROPE && tid < kTileRows && p.bias[r])
            bias_v = p.bias[r][tile_row(EPI_QKV_ROPE, tb, tid, p.head_dim, 0)];
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        for (int st = 0; st < spu; ++st, ++it) {
            const int sl = it % kSkRing;
            mbar_wait(&full[sl], (it / kSkRing) & 1, abort, p.status);
            __syncwarp();
            const int steps_here = min(kBoxK / kKStep, (kc - st * kBoxK) / kKStep);
            const unsigned char* stage = ring + sl * kSkStage;
            const unsigned char* wA = stage + box * kBoxBytes + brow * (kBoxK * 2) + tq * 16;
            const unsigned char* wB = wA + 8 * (kBoxK * 2);
            const unsigned char* px = stage + 2 * kBoxBytes + g * (kBoxK * 2) + tq * 16;
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
                const int step = wk + 2 * s2;
                if (step < steps_here) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 a = *reinterpret_cast<const uint4*>(wA + step * 128 + h * 64);
                        const uint4 b = *reinterpret_cast<const uint4*>(wB + step * 128 + h * 64);
                        const uint4 xv = *reinterpret_cast<const uint4*>(px + step * 128 + h * 64);
                        mma_bf16_16816(c, a.x, b.x, a.y, b.y, xv.x, xv.y);
                        mma_bf16_16816(c, a.z, b.z, a.w, b.w, xv.z, xv.w);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[sl]);
        }
        const int i0 = (16 * wm + g) * kTMax + 2 * tq, i1 = (16 * wm + g + 8) * kTMax + 2 * tq;
        if (wk == 0) {
            tile[i0] = c[0];
            tile[i0 + 1] = c[1];
            tile[i1] = c[2];
            tile[i1 + 1] = c[3];
        }
        if (EPI == EPI_QKV_ROPE && tid < kTileRows) s_bias[tid] = bias_v;
        consumer_sync(kConsumers);
        if (wk == 1) {
            tile[i0] += c[0];
            tile[i0 + 1] += c[1];
            tile[i1] += c[2];
            tile[i1 + 1] += c[3];
        }
        consumer_sync(kConsumers);
        if (EPI == EPI_ROWPAR) {
            float* mine = p.part + (size_t)u * kPartStride;
            for (int i = tid * 4; i < kTileRows * kTMax; i += kConsumers * 4)
                *reinterpret_cast<float4*>(mine + i) = *reinterpret_cast<const float4*>(tile + i);
        } else if (EPI == EPI_SWIGLU) {
            bf16* out = reinterpret_cast<bf16*>(p.act_out);
            const float inv_k = 1.0f / (float)p.K;
            for (int i = tid; i < 32 * T; i += kConsumers) {
                const int t = i >> 5, j = i & 31;
                const float rinv = 1.0f / sqrtf(ss[t] * inv_k + p.eps);
                const float gt = tile[j * kTMax + t] * rinv;
                const float up = tile[(j + 32) * kTMax + t] * rinv;
                out[((size_t)r * kTMax + t) * p.ffn_s + tb * 32 + j] = __float2bfloat16_rn(gt / (1.0f + expf(-gt)) * up);
            }
        } else {
            const int d = p.head_dim, half = d >> 1;
            const float inv_k = 1.0f / (float)p.K;
            for (int i = tid; i < 32 * T; i += kConsumers) {
                const int t = i >> 5, j = i & 31;
                const float rinv = 1.0f / sqrtf(ss[t] * inv_k + p.eps);
                const int rowA = tile_row(EPI_QKV_ROPE, tb, j, d, 0);
                const int head = rowA / d, ii = rowA - head * d;
                float va = tile[j * kTMax + t] * rinv + s_bias[j];
                float vb = tile[(j + 32) * kTMax + t] * rinv + s_bias[j + 32];
                const int pos = s_pos[t];
                if (head < p.hq_s + p.hkv_s) {
                    float cs, sn;
                    sincosf((float)pos * exp2f(-(2.0f * ii / d) * (float)p.log2_theta), &sn, &cs);
                    const float ra = va * cs - vb * sn, rb = va * sn + vb * cs;
                    va = ra;
                    vb = rb;
                }
                if (head < p.hq_s) {
                    float* q = p.q_out + ((size_t)r * kTMax + t) * p.hq_s * d + head * d + ii;
                    q[0] = va;
                    q[half] = vb;
                } else {
                    const bool is_k = head < p.hq_s + p.hkv_s;
                    const int kvh = is_k ? head - p.hq_s : head - p.hq_s - p.hkv_s;
                    if (pos < 0 || pos >= p.max_kv) {
                        set_status(p.status, TP_ERR_CAPACITY);
                        continue;
                    }
                    bf16* cache = reinterpret_cast<bf16*>(is_k ? p.kcache[r] : p.vcache[r]);
                    bf16* dst = cache + (((size_t)t * p.hkv_s + kvh) * p.max_kv + pos) * d + ii;
                    dst[0] = __float2bfloat16_rn(va);
                    dst[half] = __float2bfloat16_rn(vb);
                }
            }
        }
        consumer_sync(kConsumers);
    }
}

// Attention phase on the consumer side: the units of attn_tc_kernel, with
// every warp waiting for and releasing every stage (the ring is shared with
// the projection phases, whose stages all eight warps release).
template <int D>
__device__ __forceinline__ void sk_attn(const AttnDecodeParams& p, unsigned char* ring, uint64_t* full,
                                        uint64_t* empty, volatile int* abort, uint32_t& it_unit, float* red,
                                        float* s_ml, const int* s_pos) {
    using S = AtShape<D>;
    constexpr int KS = D / 16;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.hq_s / p.hkv_s;
    const int U = p.N * p.B * p.hkv_s * p.n_chunks;
    const int grp = warp >> 2, wq = warp & 3;
    const int g = lane >> 2, t = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;
    const uint32_t ring_u32 = smem_u32(ring);
    const int q0 = 2 * t, q1 = 2 * t + 1;
    (void)tid;
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
        const int c = u % p.n_chunks, gi = u / p.n_chunks;
        const int kh = gi % p.hkv_s, rb = gi / p.hkv_s, b = rb % p.B, r = rb / p.B;
        const int pos = s_pos[b];
        const int Lk = min(pos + 1, p.max_kv);
        const int j0 = c * kAttnChunk;
        const int n = max(0, min(Lk - j0, kAttnChunk));
        const int nblk = (n + kAtKeys - 1) / kAtKeys;
        uint32_t qb[KS][2];
        {
            const float* qp = p.q + ((size_t)r * kTMax + b) * p.hq_s * D + (size_t)(kh * G + (g < G ? g : 0)) * D;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                if (g < G) {
                    const float2 a = *reinterpret_cast<const float2*>(qp + 16 * ks + 2 * t);
                    const float2 c2 = *reinterpret_cast<const float2*>(qp + 16 * ks + 8 + 2 * t);
                    qb[ks][0] = pack_bf16x2(a.x * p.scale, a.y * p.scale);
                    qb[ks][1] = pack_bf16x2(c2.x * p.scale, c2.y * p.scale);
                } else {
                    qb[ks][0] = qb[ks][1] = 0u;
                }
            }
        }
        float o[KS][4];
#pragma unroll
        for (int dt = 0; dt < KS; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        for (int blk = 0; blk < nblk; ++blk) {
            const uint32_t it = it_unit + blk;
            const int sl = it % kSkRing;
            mbar_wait(&full[sl], (it / kSkRing) & 1, abort, p.status);
            __syncwarp();
            if ((blk & 1) == grp) {
                const uint32_t kpart = ring_u32 + sl * kSkStage, vpart = kpart + S::NB * S::BOX;
                const int kb = blk * kAtKeys + 16 * wq;
                float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(at_addr<D>(kpart, 16 * wq + rr + 8 * (mi & 1), 2 * ks + (mi >> 1)), a0, a1, a2, a3);
                    mma_bf16_16816(sc, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
                }
                const bool v0 = kb + g < n, v1 = kb + g + 8 < n;
                const float x00 = v0 ? sc[0] : -INFINITY, x01 = v0 ? sc[1] : -INFINITY;
                const float x10 = v1 ? sc[2] : -INFINITY, x11 = v1 ? sc[3] : -INFINITY;
                float mq0 = fmaxf(x00, x10), mq1 = fmaxf(x01, x11);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mq0 = fmaxf(mq0, __shfl_xor_sync(0xffffffffu, mq0, off));
                    mq1 = fmaxf(mq1, __shfl_xor_sync(0xffffffffu, mq1, off));
                }
                const float n0 = fmaxf(m0, mq0), n1 = fmaxf(m1, mq1);
                const float al0 = (n0 == -INFINITY) ? 1.f : expf(m0 - n0);
                const float al1 = (n1 == -INFINITY) ? 1.f : expf(m1 - n1);
                const float p00 = (x00 == -INFINITY) ? 0.f : expf(x00 - n0);
                const float p10 = (x10 == -INFINITY) ? 0.f : expf(x10 - n0);
                const float p01 = (x01 == -INFINITY) ? 0.f : expf(x01 - n1);
                const float p11 = (x11 == -INFINITY) ? 0.f : expf(x11 - n1);
                float ps0 = p00 + p10, ps1 = p01 + p11;
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    ps0 += __shfl_xor_sync(0xffffffffu, ps0, off);
                    ps1 += __shfl_xor_sync(0xffffffffu, ps1, off);
                }
                l0 = l0 * al0 + ps0;
                l1 = l1 * al1 + ps1;
                m0 = n0;
                m1 = n1;
#pragma unroll
                for (int dt = 0; dt < KS; ++dt) {
                    o[dt][0] *= al0;
                    o[dt][1] *= al1;
                    o[dt][2] *= al0;
                    o[dt][3] *= al1;
                }
                const uint32_t pb0 = movmatrix_t(pack_bf16x2(p00, p01));
                const uint32_t pb1 = movmatrix_t(pack_bf16x2(p10, p11));
                const uint32_t mlo = (kb + 2 * t < n ? 0x0000FFFFu : 0u) | (kb + 2 * t + 1 < n ? 0xFFFF0000u : 0u);
                const uint32_t mhi = (kb + 8 + 2 * t < n ? 0x0000FFFFu : 0u) | (kb + 9 + 2 * t < n ? 0xFFFF0000u : 0u);
#pragma unroll
                for (int dt = 0; dt < KS; ++dt) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(at_addr<D>(vpart, 16 * wq + rr + 8 * (mi >> 1), 2 * dt + (mi & 1)), a0, a1, a2, a3);
                    mma_bf16_16816(o[dt], a0 & mlo, a1 & mlo, a2 & mhi, a3 & mhi, pb0, pb1);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[sl]);
        }
        it_unit += nblk;
        if (g == 0) {
            s_ml[(warp * kMaxGroup + q0) * 2] = m0;
            s_ml[(warp * kMaxGroup + q0) * 2 + 1] = l0;
            s_ml[(warp * kMaxGroup + q1) * 2] = m1;
            s_ml[(warp * kMaxGroup + q1) * 2 + 1] = l1;
        }
        consumer_sync(kConsumers);
        float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            M0 = fmaxf(M0, s_ml[(w * kMaxGroup + q0) * 2]);
            M1 = fmaxf(M1, s_ml[(w * kMaxGroup + q1) * 2]);
        }
        const float c0 = (m0 == -INFINITY) ? 0.f : expf(m0 - M0);
        const float c1 = (m1 == -INFINITY) ? 0.f : expf(m1 - M1);
#pragma unroll
        for (int dt = 0; dt < KS; ++dt) {
            o[dt][0] *= c0;
            o[dt][1] *= c1;
            o[dt][2] *= c0;
            o[dt][3] *= c1;
        }
        for (int half = 4; half >= 1; half >>= 1) {
            if (warp >= half && warp < 2 * half) {
                float* dst = red + (warp - half) * kAtSlot;
#pragma unroll
                for (int dt = 0; dt < KS; ++dt) {
                    if (q0 < G) {
                        dst[q0 * D + 16 * dt + g] = o[dt][0];
                        dst[q0 * D + 16 * dt + g + 8] = o[dt][2];
                    }
                    if (q1 < G) {
                        dst[q1 * D + 16 * dt + g] = o[dt][1];
                        dst[q1 * D + 16 * dt + g + 8] = o[dt][3];
                    }
                }
            }
            consumer_sync(kConsumers);
            if (warp < half) {
                const float* src = red + warp * kAtSlot;
#pragma unroll
                for (int dt = 0; dt < KS; ++dt) {
                    if (q0 < G) {
                        o[dt][0] += src[q0 * D + 16 * dt + g];
                        o[dt][2] += src[q0 * D + 16 * dt + g + 8];
                    }
                    if (q1 < G) {
                        o[dt][1] += src[q1 * D + 16 * dt + g];
                        o[dt][3] += src[q1 * D + 16 * dt + g + 8];
                    }
                }
            }
            consumer_sync(kConsumers);
        }
        if (warp == 0 && (unsigned)u < p.part_units) {
            float* mine = p.part + (size_t)u * G * (D + 2);
#pragma unroll
            for (int dt = 0; dt < KS; ++dt) {
                if (q0 < G) {
                    mine[q0 * D + 16 * dt + g] = o[dt][0];
                    mine[q0 * D + 16 * dt + g + 8] = o[dt][2];
                }
                if (q1 < G) {
                    mine[q1 * D + 16 * dt + g] = o[dt][1];
                    mine[q1 * D + 16 * dt + g + 8] = o[dt][3];
                }
            }
            if (g == 0) {
                float L0 = 0.f, L1 = 0.f;
                for (int w = 0; w < 8; ++w) {
                    const float mw0 = s_ml[(w * kMaxGroup + q0) * 2], mw1 = s_ml[(w * kMaxGroup + q1) * 2];
                    if (mw0 != -INFINITY) L0 += s_ml[(w * kMaxGroup + q0) * 2 + 1] * expf(mw0 - M0);
                    if (mw1 != -INFINITY) L1 += s_ml[(w * kMaxGroup + q1) * 2 + 1] * expf(mw1 - M1);
                }
                if (q0 < G) {
                    mine[G * D + q0] = M0;
                    mine[G * D + G + q0] = L0;
                }
                if (q1 < G) {
                    mine[G * D + q1] = M1;
                    mine[G * D + G + q1] = L1;
                }
            }
        }
        consumer_sync(kConsumers);
    }
}

// Split-KV combine: one (group, query head) item per warp, all SMs. Lanes
// hold the chunk statistics (chunk = lane, lane + 32, ...), the warp forms
// the common maximum and denominator, then each lane combines four output
// elements at a time in chunk order.
template <int D>
__device__ __forceinline__ void sk_combine(const AttnDecodeParams& p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.hq_s / p.hkv_s, pstride = G * (D + 2);
    const int n_groups = p.N * p.B * p.hkv_s;
    const int nc = p.n_chunks;
    for (int item = blockIdx.x * 8 + warp; item < n_groups * G; item += gridDim.x * 8) {
        const int gi = item / G, gq = item - gi * G;
        const int kh = gi % p.hkv_s, rb = gi / p.hkv_s, b = rb % p.B, r = rb / p.B;
        const float* base = p.part + (size_t)gi * nc * pstride;
        float M = -INFINITY;
        for (int cc = lane; cc < nc; cc += 32) {
            const float l = base[(size_t)cc * pstride + G * D + G + gq];
            if (l > 0.f) M = fmaxf(M, base[(size_t)cc * pstride + G * D + gq]);
        }
        M = warp_max(M);
        float den = 0.f;
        for (int cc = lane; cc < nc; cc += 32) {
            const float l = base[(size_t)cc * pstride + G * D + G + gq];
            if (l > 0.f) den = fmaf(l, expf(base[(size_t)cc * pstride + G * D + gq] - M), den);
        }
        den = warp_sum(den);
        const float inv = den > 0.f ? 1.0f / den : 0.f;
        bf16* out = reinterpret_cast<bf16*>(p.out) + ((size_t)r * kTMax + b) * p.hq_s * D + (size_t)(kh * G + gq) * D;
        for (int d0 = lane * 4; d0 < D; d0 += 128) {
            float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int cc = 0; cc < nc; ++cc) {
                const float* pc = base + (size_t)cc * pstride;
                const float l = pc[G * D + G + gq];
                const float w = l > 0.f ? expf(pc[G * D + gq] - M) : 0.f;
                // the partial stride G*(D+2) floats need not be a multiple of 4: scalar loads
                const float* pv = pc + gq * D + d0;
                num.x = fmaf(pv[0], w, num.x);
                num.y = fmaf(pv[1], w, num.y);
                num.z = fmaf(pv[2], w, num.z);
                num.w = fmaf(pv[3], w, num.w);
            }
            uint2 pk;
            pk.x = pack_bf16x2(num.x * inv, num.y * inv);
            pk.y = pack_bf16x2(num.z * inv, num.w * inv);
            *reinterpret_cast<uint2*>(out + d0) = pk;
        }
    }
}

// Rank-ordered reduction of a row-parallel phase's partials: one 8-row slice
// of a 64-row tile per warp, all SMs; lane = (row, token pair). Chunks are
// summed in order within each rank, then ranks in order, then the residual.
// With norm_out it writes the next norm's operands (y * gamma_r, bf16, every
// shard) and per-(8-row slice, token) sums of squares.
__device__ __forceinline__ void sk_reduce(const GemvParams& p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int upg = p.shape.units_per_group(), C = p.shape.chunks;
    const int j8 = lane >> 2, tp = lane & 3;
    for (int item = blockIdx.x * 8 + warp; item < p.shape.groups * 8; item += gridDim.x * 8) {
        const int tb = item >> 3, sl = item & 7;
        const int j = sl * 8 + j8;                     // row within the tile
        const float* base = p.part + (size_t)tb * upg * kPartStride + j * kTMax + 2 * tp;
        float2 v[kMaxGroupUnits];
#pragma unroll
        for (int q = 0; q < kMaxGroupUnits; ++q)
            if (q < upg) v[q] = *reinterpret_cast<const float2*>(base + (size_t)q * kPartStride);
        float2 total = make_float2(0.f, 0.f), pr = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < kMaxGroupUnits; ++q) {
            if (q < upg) {
                const int cc = q % C;
                pr = (cc == 0) ? v[q] : make_float2(pr.x + v[q].x, pr.y + v[q].y);
                if (cc == C - 1) total = (q < C) ? pr : make_float2(total.x + pr.x, total.y + pr.y);
            }
        }
        const int row = tb * kTileRows + j;
        float sq[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int t = 2 * tp + e;
            float yv = 0.f;
            if (t < p.T) {
                const size_t o = (size_t)t * p.rows + row;
                yv = p.resid[o] + (e ? total.y : total.x);
                p.y[o] = yv;
                if (p.norm_out) {
                    bf16* nout = reinterpret_cast<bf16*>(p.norm_out);
                    for (int r2 = 0; r2 < p.n_shards; ++r2)
                        nout[((size_t)r2 * kTMax + t) * p.rows + row] = __float2bfloat16_rn(yv * p.gamma2[r2][row]);
                }
            }
            sq[e] = yv * yv;
        }
        if (p.norm_out) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], off);
                sq[1] += __shfl_xor_sync(0xffffffffu, sq[1], off);
            }
            if (j8 == 0) {
                p.ss_tiles_out[(size_t)item * kTMax + 2 * tp] = sq[0];
                p.ss_tiles_out[(size_t)item * kTMax + 2 * tp + 1] = sq[1];
            }
        }
    }
}

size_t decode_step_smem() {
    // ring | red [4][kAtSlot] | s_ml [8][8][2] | tile [64][8] | ss, pos, bias, wsum
    return 1024 + (size_t)kSkRing * kSkStage +
           (size_t)(4 * kAtSlot + 8 * kMaxGroup * 2 + kTileRows * kTMax + kTMax + kTMax + 96 + 8) * 4;
}

template <int D>
__global__ void __launch_bounds__(kStreamThreads, 1) decode_step_kernel(const __grid_constant__ StepArgs A) {
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kSkRing;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 16 * kSkRing);
    unsigned long long* s_gen0 = reinterpret_cast<unsigned long long*>(smem + 16 * kSkRing + 8);
    unsigned char* ring = smem + 1024;
    float* red = reinterpret_cast<float*>(ring + kSkRing * kSkStage);
    float* s_ml = red + 4 * kAtSlot;
    float* tile = s_ml + 8 * kMaxGroup * 2;
    float* ss = tile + kTileRows * kTMax;
    int* s_pos = reinterpret_cast<int*>(ss + kTMax);
    float* s_bias = reinterpret_cast<float*>(s_pos + kTMax);
    float* wsum = s_bias + 96;
    int* status = A.a.status;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < kSkRing; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumers / 32);
        }
        *abort_flag = (smem_u32(ring) & 127u) ? 1 : 0;
        if (*abort_flag) set_status(status, TP_ERR_ALIGN);
        // read before this CTA arrives anywhere: fewer than gridDim.x arrivals of
        // this step can precede it
        const unsigned long long per_step = (unsigned long long)kSkPhases * gridDim.x;
        const unsigned long long c = ld_acquire_u64(A.bar);
        *s_gen0 = c - c % per_step;
        fence_mbar_init();
    }
    __syncthreads();
    const unsigned long long gen0 = *s_gen0;

    if (warp == kConsumers / 32) {                     // ---- producer
        if (lane == 0 && !*abort_flag) {
            const uint64_t pol = l2_evict_first_policy();
            uint32_t it = 0;
            SkPend pd;
            pd.n = 0;
            int posv[kTMax];
            for (int b = 0; b < kTMax; ++b) posv[b] = b < A.a.B ? A.a.pos[b] : 0;
            bool ok = sk_produce_gemv(EPI_QKV_ROPE, 0, 1, A, ring, full, empty, it, pd, gen0, abort_flag, pol);
            if (ok) ok = sk_produce_attn<D>(2, A, ring, full, empty, it, pd, gen0, abort_flag, pol, posv);
            if (ok) ok = sk_produce_gemv(EPI_ROWPAR, 1, 4, A, ring, full, empty, it, pd, gen0, abort_flag, pol);
            if (ok) ok = sk_produce_gemv(EPI_SWIGLU, 2, 6, A, ring, full, empty, it, pd, gen0, abort_flag, pol);
            if (ok) ok = sk_produce_gemv(EPI_ROWPAR, 3, 7, A, ring, full, empty, it, pd, gen0, abort_flag, pol);
            sk_flush(pd, A, ring, full, gen0, abort_flag, status);
            // no copy may still be landing when the CTA exits
            volatile int no_abort = 0;
            const uint32_t first = it > (uint32_t)kSkRing ? it - kSkRing : 0u;
            for (uint32_t k = first; k < it; ++k) mbar_wait(&full[k % kSkRing], (k / kSkRing) & 1, &no_abort, nullptr);
        }
        return;
    }

    // ---- consumers
    unsigned long long* st = A.stamps && blockIdx.x < kMaxStepCtas ? A.stamps + (size_t)blockIdx.x * kStepStamps : nullptr;
    if (st && tid == 0) st[0] = global_ns();
    if (tid < kTMax) s_pos[tid] = tid < A.a.B ? A.a.pos[tid] : 0;
    uint32_t it = 0;
    sk_norm(A.np);
    sk_barrier(A.bar, gen0, 1, abort_flag, status, st ? st + 1 : nullptr);
    sk_gemv<EPI_QKV_ROPE>(A.g[0], ring, full, empty, abort_flag, it, tile, ss, s_pos, s_bias);
    sk_barrier(A.bar, gen0, 2, abort_flag, status, st ? st + 2 : nullptr);
    if (tid < kTMax) s_pos[tid] = tid < A.a.B ? A.a.pos[tid] : 0;
    consumer_sync(kConsumers);
    sk_attn<D>(A.a, ring, full, empty, abort_flag, it, red, s_ml, s_pos);
    sk_barrier(A.bar, gen0, 3, abort_flag, status, st ? st + 3 : nullptr);
    sk_combine<D>(A.a);
    sk_barrier(A.bar, gen0, 4, abort_flag, status, st ? st + 4 : nullptr);
    sk_gemv<EPI_ROWPAR>(A.g[1], ring, full, empty, abort_flag, it, tile, ss, s_pos, s_bias);
    sk_barrier(A.bar, gen0, 5, abort_flag, status, st ? st + 5 : nullptr);
    sk_reduce(A.g[1]);
    sk_barrier(A.bar, gen0, 6, abort_flag, status, st ? st + 6 : nullptr);
    sk_gemv<EPI_SWIGLU>(A.g[2], ring, full, empty, abort_flag, it, tile, ss, s_pos, s_bias);
    sk_barrier(A.bar, gen0, 7, abort_flag, status, st ? st + 7 : nullptr);
    sk_gemv<EPI_ROWPAR>(A.g[3], ring, full, empty, abort_flag, it, tile, ss, s_pos, s_bias);
    sk_barrier(A.bar, gen0, 8, abort_flag, status, st ? st + 8 : nullptr);
    sk_reduce(A.g[3]);
    if (st && tid == 0) st[kStepStamps - 1] = global_ns();
}

cudaError_t launch_decode_step(const DecodeStepParams& P, cudaStream_t s) {
    const size_t smem = decode_step_smem();
    const int D = P.a.d;
    const void* fn = D == 64 ? reinterpret_cast<const void*>(decode_step_kernel<64>)
                             : reinterpret_cast<const void*>(decode_step_kernel<128>);
    static int grid_sz[2] = {0, 0};
    const int which = D == 64 ? 0 : 1;
    if (!grid_sz[which]) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        int dev = 0, sms = 0, per_sm = 0;
        e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kStreamThreads, smem);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        grid_sz[which] = sms;                          // one CTA per SM
    }
    StepArgs A;
    memset(&A, 0, sizeof A);
    const int epis[4] = {EPI_QKV_ROPE, EPI_ROWPAR, EPI_SWIGLU, EPI_ROWPAR};
    (void)epis;
    for (int i = 0; i < 4; ++i) {
        const GemvParams& p = P.g[i];
        A.g[i] = p;
        for (int r = 0; r < p.n_shards; ++r) {
            cudaError_t e = weight_tensor_map(p.W[r], p.K, p.rows, &A.wm[i][r]);
            if (e != cudaSuccess) return e;
        }
        cudaError_t e = weight_tensor_map(p.xact, p.K, p.n_shards * kTMax, &A.xm[i], kTMax);
        if (e != cudaSuccess) return e;
    }
    A.a = P.a;
    A.np = P.np;
    const long rows = (long)P.a.max_batch * P.a.hkv_s * P.a.max_kv;
    for (int r = 0; r < P.a.N; ++r) {
        const int pt = D == 128 ? AtShape<128>::PT : AtShape<64>::PT;
        cudaError_t e = tensor_map_2d(P.a.kcache[r], D, rows, pt, kAtKeys, 0, &A.tk[r]);
        if (e == cudaSuccess) e = tensor_map_2d(P.a.vcache[r], D, rows, pt, kAtKeys, 0, &A.tv[r]);
        if (e != cudaSuccess) return e;
    }
    A.bar = P.bar;
    A.stamps = P.stamps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_sz[which]);
    cfg.blockDim = dim3(kStreamThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {&A};
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace tpk
