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

cudaError_t launch_attn_decode(const AttnDecodeParams& p, int dtype, cudaStream_t s) {
    if (dtype == TP_BF16) return p.d == 64 ? launch_attn_stream_g<64>(p, s) : launch_attn_stream_g<128>(p, s);
    return p.d == 64 ? launch_attn_t<float, 64>(p, s) : launch_attn_t<float, 128>(p, s);
}

}  // namespace tpk
