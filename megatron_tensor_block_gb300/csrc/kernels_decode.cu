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

// Unit u of a projection -> (group, shard, 64-row tile, reduction chunk).
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
static_assert(32 * kTMax <= kConsumers, "one QKV epilogue output per consumer thread");
constexpr int kQStage = 3584;                 // bf16 elements of q staged for the attention phase (7 KB)
constexpr int kQSegs = 7;                     // segments whose q is staged
constexpr int kSegTab = 8;                    // attention segments per CTA listed ahead of the phase

template <int D>
struct AtShape {
    static constexpr int NB = D / 64;                     // 64-element column halves per row
    static constexpr int PT = D == 128 ? 72 : 64;         // elements per shared row (box width)
    static constexpr int BOX = kAtKeys * PT * 2;          // bytes per box
    static constexpr int STAGE = 2 * NB * BOX;            // K boxes, then V boxes
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

// 3-D bf16 tensor [d2][d1][d0] (d0 contiguous), boxes box0 x box1 x 1; not cached.
cudaError_t tensor_map_3d(const void* base, long d0, long d1, long d2, int box0, int box1, int swizzle128,
                          CUtensorMap* out) {
    static std::mutex mu;
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void**>(&encode),
                                                         12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || !encode) return e != cudaSuccess ? e : cudaErrorNotSupported;
    }
    cuuint64_t gdim[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
    cuuint64_t gstride[2] = {(cuuint64_t)d0 * 2, (cuuint64_t)d0 * d1 * 2};
    cuuint32_t box[3] = {(cuuint32_t)box0, (cuuint32_t)box1, 1u};
    cuuint32_t estride[3] = {1u, 1u, 1u};
    CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstride, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

static cudaError_t weight_tensor_map(const void* W, int K, int rows, CUtensorMap* out, int box_rows = 32) {
    return tensor_map_2d(W, K, rows, kBoxK, box_rows, 0, out);
}

// Stage boxes of the streaming GEMVs (decode step, MoE experts): a [rows][K]
// bf16 matrix viewed as [rows][K / 64][64] so one box ({64, 4, box_rows}:
// box_rows rows x 256 columns) lands 128-byte swizzled in shared memory.
// K % 64 == 0.
cudaError_t step_stage_map(const void* W, int K, int rows, int box_rows, CUtensorMap* out) {
    static std::mutex mu;
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    struct Entry { const void* w; int K, rows, br; CUtensorMap tm; };
    static std::vector<Entry> cache;
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : cache)
        if (e.w == W && e.K == K && e.rows == rows && e.br == box_rows) {
            *out = e.tm;
            return cudaSuccess;
        }
    if (K % 64) return cudaErrorInvalidValue;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void**>(&encode),
                                                         12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || !encode) return e != cudaSuccess ? e : cudaErrorNotSupported;
    }
    cuuint64_t gdim[3] = {64u, (cuuint64_t)(K / 64), (cuuint64_t)rows};
    cuuint64_t gstride[2] = {128u, (cuuint64_t)K * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)(kBoxK / 64), (cuuint32_t)box_rows};
    cuuint32_t estride[3] = {1u, 1u, 1u};
    CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(W), gdim, gstride, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    cache.push_back({W, K, rows, box_rows, *out});
    return cudaSuccess;
}

// fp32 projections (bf16 decode runs as one launch: launch_decode_step)
cudaError_t launch_gemv(const GemvParams& p, int epi, int dtype, cudaStream_t s) {
    if (dtype != TP_F32) return cudaErrorInvalidValue;
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

cudaError_t launch_attn_decode(const AttnDecodeParams& p, int dtype, cudaStream_t s) {
    if (dtype != TP_F32) return cudaErrorInvalidValue;
    return p.d == 64 ? launch_attn_t<float, 64>(p, s) : launch_attn_t<float, 128>(p, s);
}


// ===========================================================================
// The whole decode step in one persistent launch (bf16).
//
// One CTA per SM runs every stage of the block as a phase:
//   NORM | QKV (+RoPE, KV append) | ATTN (+split-KV combine) |
//   O_PROJ (+rank-ordered reduce, next norm operands) | GATE_UP (+SwiGLU) |
//   DOWN (+rank-ordered reduce)
// separated by five grid barriers (a monotonic arrival counter in the
// workspace; every wait bounded). Each phase's work -- 256-element reduction
// stages of the projections, or keys of the attention -- is laid out in one
// flattened order and split into one contiguous range per CTA: whole tiles
// for the column-parallel phases and o_proj, an even split of the down
// stages, and for attention two key shares -- CTAs without a QKV tile take
// the larger one and prefetch it into L2 while QKV runs. A 64-row tile (or
// KV group) whose range straddles two CTAs gets one fp32 partial per CTA; one
// CTA combines them in CTA order and runs the epilogue: for down tiles the
// one holding the tile's last stage, polling (value, epoch) pieces; for a
// KV group the one holding its last keys, after a per-group counter. Results
// are deterministic and no extra phase is needed.
// The producer thread streams the data of later phases that does not depend
// on earlier ones -- every weight box, and every K/V block except the one
// holding the new position -- through the same 5-stage ring while the
// consumers are still busy or at a barrier; only the activation boxes (and
// the new K/V rows) wait for the barrier that publishes them.
// ===========================================================================

namespace {
constexpr int kSkRing = 5;
constexpr int kSkStage = kGemvStageBytes;               // 36 KB: 2 weight boxes + activation box, or K+V of 64 keys
constexpr int kSkBarriers = 5;                          // grid barriers inside a step
constexpr int kSkMaxPend = kSkRing;
static_assert(kGemvStageBytes == kAtMaxStage, "the two stage formats share one slot size");
static_assert(kStepStamps == 2 * (kSkBarriers + 1) + 1, "stamps: start, per phase streaming done + arrival");
}  // namespace

struct StepArgs {
    CUtensorMap wm[4][TP_MAX_SHARDS];       // weights of qkv, o, gate_up, down (boxes kBoxK x 32)
    CUtensorMap xm[4];                      // their activation operands (boxes kBoxK x 8)
    CUtensorMap tk[TP_MAX_SHARDS];          // K / V caches (boxes 72 or 64 x 64 keys)
    CUtensorMap tv[TP_MAX_SHARDS];
    GemvParams g[4];                        // qkv, o, gate_up, down; shape.chunks = partial slots per tile
    AttnDecodeParams a;                     // n_chunks = partial slots per KV group
    NormPrepParams np;
    unsigned long long* bar;                // grid-barrier arrival counter (only grows)
    // Arrivals after the QKV phase, one per CTA and launch (only grows). The
    // consumers do not wait at barrier 2 (the attention phase polls q's
    // epochs), so a CTA may reach barrier 3 before another reaches barrier 2,
    // and the shared counter can pass barrier 2's target early; the key block
    // holding a new position waits on this count instead.
    unsigned long long* kv_ready;
    unsigned long long* stamps;             // optional [grid][kStepStamps]: start, barrier arrivals, end (ns)
    unsigned bar_extra;                     // test hook: extra arrivals every grid barrier waits for (0)
};

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Grid barrier k of a step has passed once the arrival counter reaches
// base + k * gridDim.x. The counter only grows (by kSkBarriers * gridDim.x per
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

// Every CTA of this launch has counted its QKV phase done: kv_ready reaches
// (launch index + 1) * grid (+ the test hook's extra, like every barrier).
__device__ __forceinline__ bool sk_wait_kv(const StepArgs& A, unsigned long long gen0, volatile int* abort,
                                           int* status) {
    const unsigned long long per_step = (unsigned long long)kSkBarriers * gridDim.x;
    const unsigned long long want = (gen0 / per_step + 1ull) * gridDim.x + gen0 % per_step;
    if (ld_acquire_u64(A.kv_ready) >= want) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (ld_acquire_u64(A.kv_ready) >= want) return true;
        if (*abort) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            set_status(status, TP_ERR_TIMEOUT);
            return false;
        }
    }
}

// ---- flattened work split ------------------------------------------------------

// Per-CTA share of W work items (at least `min_r`, so partial slots per tile
// stay bounded for any grid size up to kMaxStepCtas).
__device__ __forceinline__ int sk_share(int W, int min_r) {
    const int r = (W + (int)gridDim.x - 1) / (int)gridDim.x;
    return r > min_r ? r : min_r;
}

// Attention keys of the one-launch step: CTAs 0..na-1 (those holding a QKV
// tile) take ra keys each, the others -- idle during the QKV phase, when they
// prefetch their keys into L2 -- take rb = ra * kIdleKeyNum / kIdleKeyDen
// (rounded up). ra is at least min_r, so a
// KV group of max_kv keys spans at most ceil(max_kv / min_r) + 1 CTAs.
constexpr int kIdleKeyNum = 4, kIdleKeyDen = 3;     // an idle CTA's key share relative to a busy one's (measured best)
struct KeySplit {
    int ra, rb, na;
};
__device__ __forceinline__ KeySplit sk_key_split(int total, int min_r, int busy) {
    KeySplit s;
    s.na = busy > 0 && busy < (int)gridDim.x ? busy : (int)gridDim.x;
    const long long units = (long long)s.na * kIdleKeyDen + (long long)((int)gridDim.x - s.na) * kIdleKeyNum;
    s.ra = max((int)(((long long)total * kIdleKeyDen + units - 1) / units), min_r);
    s.rb = s.na < (int)gridDim.x ? (s.ra * kIdleKeyNum + kIdleKeyDen - 1) / kIdleKeyDen : s.ra;
    return s;
}
// First key of CTA c (c = gridDim.x gives the end), clipped to the key space.
__device__ __forceinline__ int sk_key_start(const KeySplit& s, int c, int total) {
    const long long k = c <= s.na ? (long long)c * s.ra : (long long)s.na * s.ra + (long long)(c - s.na) * s.rb;
    return (int)min(k, (long long)total);
}
// CTA holding key k (k inside the key space).
__device__ __forceinline__ int sk_key_cta(const KeySplit& s, int k) {
    const long long ka = (long long)s.na * s.ra;
    return k < ka ? k / s.ra : s.na + (int)((k - ka) / s.rb);
}

// Projection tiles ("segments"): column-parallel -- one 64-row tile of one
// shard per group (decode_unit with one unit per group); row-parallel -- the
// shards of 64-row output tile tb are segments tb*N .. tb*N + N-1. Each has
// S = ceil(K / 256) stages; stage f of the phase is stage f % S of segment f / S.
__device__ __forceinline__ void sk_segment(const GemvParams& p, int epi, int seg, int& r, int& tb) {
    if (epi == EPI_ROWPAR) {
        tb = seg / p.n_shards;
        r = seg - tb * p.n_shards;
    } else {
        const int rb = p.shape.groups / p.n_shards;
        r = seg / rb;
        tb = seg - r * rb;
    }
}

__device__ __forceinline__ int sk_nseg(const GemvParams& p, int epi) {
    return epi == EPI_ROWPAR ? p.shape.groups * p.n_shards : p.shape.groups;
}

// Stages per CTA of a projection phase. Column-parallel phases take whole
// tiles (a tile split over CTAs would need a cross-CTA finish before its
// epilogue, which costs more than the imbalance). A row-parallel phase either
// gives each CTA whole output tiles -- every shard's piece, reduced in rank
// order inside the CTA (whole_tiles) -- or is split evenly, its pieces then
// reduced by the CTA holding the tile's last stage, which polls them as
// (value, epoch) pairs (without a pair buffer: by the CTA that arrives last).
__device__ __forceinline__ int sk_phase_share(const GemvParams& p, int epi, int S) {
    const int nseg = sk_nseg(p, epi);
    if (epi != EPI_ROWPAR) return S * ((nseg + (int)gridDim.x - 1) / (int)gridDim.x);
    if (p.whole_tiles)                                  // every shard of an output tile in one CTA
        return S * p.n_shards * ((p.shape.groups + (int)gridDim.x - 1) / (int)gridDim.x);
    const int W = nseg * S;
    return sk_share(W, (W + kMaxStepCtas - 1) / kMaxStepCtas);
}

// CTAs that own stages of segment `seg`: first .. last.
__device__ __forceinline__ void sk_owners(int seg, int S, int R, int& first, int& last) {
    first = (seg * S) / R;
    last = (seg * S + S - 1) / R;
}

// ---- attention key space -------------------------------------------------------

// Groups (shard r, sequence b, KV head kh) in order ((r * B + b) * Hkv' + kh),
// each holding len_b = min(pos_b + 1, max_kv) keys, laid end to end.
struct KeySpace {
    int len[kTMax];
    int pre[kTMax + 1];      // keys of sequences before b, times Hkv'
    int per_r;               // keys of one shard
    int total;
};

__device__ __forceinline__ KeySpace sk_keyspace(const AttnDecodeParams& p, const int* posv) {
    KeySpace ks;
    ks.pre[0] = 0;
#pragma unroll
    for (int b = 0; b < kTMax; ++b) {
        const int l = b < p.B ? min(max(posv[b] + 1, 0), p.max_kv) : 0;
        ks.len[b] = l;
        ks.pre[b + 1] = ks.pre[b] + l * p.hkv_s;
    }
    ks.per_r = ks.pre[kTMax];
    ks.total = ks.per_r * p.N;
    return ks;
}

// Group holding flattened key k, the key's offset in it, and the group's
// first flattened key.
__device__ __forceinline__ void sk_locate(const KeySpace& ks, const AttnDecodeParams& p, int k, int& gi, int& b,
                                          int& off, int& gstart) {
    const int r = k / ks.per_r;
    const int rem = k - r * ks.per_r;
    b = 0;
#pragma unroll
    for (int bb = 1; bb < kTMax; ++bb)
        if (bb < p.B && ks.pre[bb] <= rem) b = bb;
    const int rem2 = rem - ks.pre[b];
    const int kh = rem2 / ks.len[b];
    off = rem2 - kh * ks.len[b];
    gi = (r * p.B + b) * p.hkv_s + kh;
    gstart = r * ks.per_r + ks.pre[b] + kh * ks.len[b];
}

// ---- finisher warp ----------------------------------------------------------------
//
// When a piece of a projection tile that other CTAs share is stored, or a
// phase is done, consumer thread 0 posts a job to a small shared-memory queue
// and the consumers go on streaming. A tenth warp takes the jobs in order: it
// publishes the CTA's stores, counts the arrival for the tile, and if this
// CTA arrived last the consumers sum the pieces in CTA order and run the
// epilogue at the phase end. A KV group split over CTAs is finished instead
// by the CTA holding its last keys (it streams them last): the others
// release-increment the group's counter after storing their pieces.

constexpr int kJobs = 8;
enum SkJobType : int { JOB_COL = 0, JOB_ROW = 1, JOB_GRP = 2, JOB_PHASE = 3, JOB_END = 4 };
struct SkJob {
    int type, pi, idx;
    unsigned expected;
};
constexpr int kMaxFin = 16;             // finishes one CTA can owe in a phase
struct SkQueue {
    SkJob job[kJobs];
    uint64_t full[kJobs];
    uint64_t empty[kJobs];
    uint64_t drained;                   // the finisher has taken every job up to a phase end
    SkJob fin[kMaxFin];                 // tiles / groups this CTA arrived last on, this phase
    int n_fin;
};

// Consumer thread 0 only: the stores the job covers were made before a
// consumer_sync; the mbarrier arrival orders them before the finisher's wait.
// Every consumer thread counts the posts (jn stays uniform across them).
__device__ __forceinline__ void sk_post(SkQueue* qu, uint32_t jn, int type, int pi, int idx, unsigned expected,
                                        volatile int* abort, int* status) {
    const int sl = jn % kJobs;
    mbar_wait(&qu->empty[sl], ((jn / kJobs) & 1) ^ 1, abort, status);
    qu->job[sl].type = type;
    qu->job[sl].pi = pi;
    qu->job[sl].idx = idx;
    qu->job[sl].expected = expected;
    mbar_arrive(&qu->full[sl]);
}

// ---- producer helpers -------------------------------------------------------

// Stages whose activation box waits for a barrier, oldest first.
struct SkPend {
    int n;
    uint32_t stage[kSkMaxPend];
    int slot[kSkMaxPend], x[kSkMaxPend], y[kSkMaxPend], map[kSkMaxPend];
    unsigned need[kSkMaxPend];
};

// Issues every pending activation box, waiting for the barriers in order.
// Returns the last barrier waited for (0 if none was pending).
__device__ __forceinline__ unsigned sk_flush(SkPend& pd, const StepArgs& A, unsigned char* ring, uint64_t* full,
                                             unsigned long long gen0, volatile int* abort, int* status) {
    bool ok = true;
    unsigned last = 0;
    for (int i = 0; i < pd.n; ++i) {
        last = pd.need[i];
        if (ok) ok = sk_wait_gen(A.bar, gen0, pd.need[i], abort, status);
        // the activations were written by other CTAs' ordinary stores
        asm volatile("fence.proxy.async.global;" ::: "memory");
        // issued even after a failed wait: the stage's byte count must complete
        tma_load_3d_keep(ring + pd.slot[i] * kSkStage + 2 * kBoxBytes, &A.xm[pd.map[i]], 0, pd.x[i] >> 6, pd.y[i],
                         &full[pd.slot[i]]);
    }
    pd.n = 0;
    return last;
}

// Stage range [f0, f1) of this CTA in a projection phase; S stages per segment.
__device__ __forceinline__ void sk_gemv_range(const GemvParams& p, int epi, int& f0, int& f1, int& S) {
    S = (p.K + kBoxK - 1) / kBoxK;
    const int W = sk_nseg(p, epi) * S;
    const int R = sk_phase_share(p, epi, S);
    f0 = min((int)blockIdx.x * R, W);
    f1 = min(f0 + R, W);
}

// Positions and the attention key space, read by the producer thread once the
// dependency on the preceding launch is resolved.
struct SkKeys {
    KeySpace ks;
    int posv[kTMax];
    int k0, k1;            // this CTA's attention keys
    bool ready;
};

__device__ __forceinline__ void sk_keys_ready(SkKeys& K, const StepArgs& A) {
    if (K.ready) return;
    pdl_wait();                                         // cache rows and positions of the preceding step
    for (int b = 0; b < kTMax; ++b) K.posv[b] = b < A.a.B ? A.a.pos[b] : 0;
    K.ks = sk_keyspace(A.a, K.posv);
    const KeySplit sp = sk_key_split(K.ks.total, step_min_keys(A.a.max_kv), A.a.key_busy);
    K.k0 = sk_key_start(sp, (int)blockIdx.x, K.ks.total);
    K.k1 = sk_key_start(sp, (int)blockIdx.x + 1, K.ks.total);
    K.ready = true;
}

// One attention segment: the CTA's keys of one group, walked from the end of
// the CTA's range backwards (the block holding a new position comes last).
struct SkSeg {
    int k, len, row0, r, j_new;     // j_new: first block offset holding the new position
};

__device__ __forceinline__ SkSeg sk_attn_segment(const SkKeys& K, const AttnDecodeParams& p, int ke) {
    int gi, b, off, gstart;
    sk_locate(K.ks, p, ke - 1, gi, b, off, gstart);
    SkSeg g;
    g.k = max(K.k0, gstart);
    sk_locate(K.ks, p, g.k, gi, b, off, gstart);
    g.len = ke - g.k;
    const int kh = gi % p.hkv_s;
    g.r = gi / (p.hkv_s * p.B);
    g.row0 = (b * p.hkv_s + kh) * p.max_kv + off;
    g.j_new = K.posv[b] - off - kAtKeys + 1;
    return g;
}

// Producer of one projection phase: weight boxes at once, the activation box
// once barrier `need` has passed. The per-stage path is kept short (one
// thread issues every copy of the CTA): segment geometry is computed once per
// segment, the ring slot and parity advance incrementally.
__device__ __forceinline__ bool sk_produce_gemv(int epi, int wi, unsigned need, const StepArgs& A, unsigned char* ring,
                                                uint64_t* full, uint64_t* empty, uint32_t& it, SkPend& pd,
                                                unsigned long long gen0, volatile int* abort, uint64_t pol) {
    const GemvParams& p = A.g[wi];
    int f0, f1, S;
    sk_gemv_range(p, epi, f0, f1, S);
    if (f0 >= f1) return true;
    // the barrier is polled once per phase (an acquire load is an L2 round trip
    // the producer would otherwise pay per stage); once pending boxes have been
    // flushed, the barrier is known to have passed
    bool passed = sk_passed(A.bar, gen0, need);
    if (passed) {
        // every earlier barrier has passed too: issue what is still pending
        sk_flush(pd, A, ring, full, gen0, abort, p.status);
        asm volatile("fence.proxy.async.global;" ::: "memory");   // activations written by ordinary stores
    }
    // first stage that reuses the slot of the oldest pending stage
    uint32_t flush_at = pd.n > 0 ? pd.stage[0] + kSkRing : 0xffffffffu;
    uint32_t sl = it % kSkRing, par = ((it / kSkRing) & 1) ^ 1;
    const CUtensorMap* xm = &A.xm[wi];
    int seg = f0 / S, st = f0 - seg * S;
    for (int f = f0; f < f1; ++seg, st = 0) {
        int r, tb;
        sk_segment(p, epi, seg, r, tb);
        const CUtensorMap* wmap = &A.wm[wi][r];
        const int rowa = tile_row(epi, tb, 0, p.head_dim, p.ffn_s);
        const int rowb = tile_row(epi, tb, 32, p.head_dim, p.ffn_s);
        const int y = r * kTMax;
        const int n = min(S - st, f1 - f);
        f += n;
        for (int x = st * kBoxK, xe = (st + n) * kBoxK; x < xe; x += kBoxK, ++it) {
            if (it >= flush_at) {
                // the flushed boxes may all belong to an earlier phase
                passed = sk_flush(pd, A, ring, full, gen0, abort, p.status) >= need ||
                         sk_passed(A.bar, gen0, need);
                if (passed) asm volatile("fence.proxy.async.global;" ::: "memory");
                flush_at = 0xffffffffu;
            }
            if (!mbar_wait(&empty[sl], par, abort, p.status)) return false;
            mbar_arrive_expect_tx(&full[sl], 2u * kBoxBytes + kXBoxBytes);
            unsigned char* dst = ring + sl * kSkStage;
            tma_load_3d_hint(dst, wmap, 0, x >> 6, rowa, &full[sl], pol);
            tma_load_3d_hint(dst + kBoxBytes, wmap, 0, x >> 6, rowb, &full[sl], pol);
            if (passed) {
                tma_load_3d_keep(dst + 2 * kBoxBytes, xm, 0, x >> 6, y, &full[sl]);
            } else {
                if (pd.n == 0) flush_at = it + kSkRing;
                pd.stage[pd.n] = it;
                pd.slot[pd.n] = sl;
                pd.x[pd.n] = x;
                pd.y[pd.n] = y;
                pd.map[pd.n] = wi;
                pd.need[pd.n] = need;
                ++pd.n;
            }
            if (++sl == kSkRing) {
                sl = 0;
                par ^= 1;
            }
        }
    }
    return true;
}

template <int D>
__device__ __forceinline__ bool sk_produce_attn(unsigned need, const StepArgs& A, unsigned char* ring, uint64_t* full,
                                                uint64_t* empty, uint32_t& it, SkPend& pd, SkKeys& keys,
                                                unsigned long long gen0, volatile int* abort, uint64_t pol) {
    using S = AtShape<D>;
    const AttnDecodeParams& p = A.a;
    sk_keys_ready(keys, A);
    if ((int)blockIdx.x >= p.key_busy && p.key_busy < (int)gridDim.x) {
        // no QKV tile here: pull this CTA's K and V rows into L2 while the
        // other CTAs run the QKV phase (its share of keys is the larger one)
        for (int ke = keys.k1; ke > keys.k0;) {
            const SkSeg g = sk_attn_segment(keys, p, ke);
            const size_t rb = (size_t)D * sizeof(bf16);
            const char* kb = static_cast<const char*>(p.kcache[g.r]) + (size_t)g.row0 * rb;
            const char* vb = static_cast<const char*>(p.vcache[g.r]) + (size_t)g.row0 * rb;
            const size_t n = (size_t)g.len * rb;
            for (size_t o = 0; o < n; o += 32768) {
                const uint32_t sz = (uint32_t)min((size_t)32768, n - o);
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(kb + o), "r"(sz) : "memory");
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(vb + o), "r"(sz) : "memory");
            }
            ke = g.k;
        }
    }
    bool passed = false;
    uint32_t flush_at = pd.n > 0 ? pd.stage[0] + kSkRing : 0xffffffffu;
    uint32_t sl = it % kSkRing, par = ((it / kSkRing) & 1) ^ 1;
    // segments in reverse order: a block holding a new position (a group's last
    // keys) comes last in the CTA's range, so everything before it can stream
    // while the QKV phase is still running
    for (int ke = keys.k1; ke > keys.k0;) {
        const SkSeg g = sk_attn_segment(keys, p, ke);
        const CUtensorMap* tk = &A.tk[g.r];
        const CUtensorMap* tv = &A.tv[g.r];
        for (int j = 0; j < g.len; j += kAtKeys, ++it) {
            if (!passed && j >= g.j_new) {              // written by the QKV phase
                sk_flush(pd, A, ring, full, gen0, abort, p.status);
                flush_at = 0xffffffffu;
                sk_wait_kv(A, gen0, abort, p.status);
                asm volatile("fence.proxy.async.global;" ::: "memory");
                passed = true;
            }
            if (it >= flush_at) {
                sk_flush(pd, A, ring, full, gen0, abort, p.status);
                flush_at = 0xffffffffu;
            }
            if (!mbar_wait(&empty[sl], par, abort, p.status)) return false;
            mbar_arrive_expect_tx(&full[sl], (uint32_t)S::STAGE);
            unsigned char* st = ring + sl * kSkStage;
#pragma unroll
            for (int h = 0; h < S::NB; ++h) {
                tma_load_2d(st + h * S::BOX, tk, h * 64, g.row0 + j, &full[sl], pol);
                tma_load_2d(st + (S::NB + h) * S::BOX, tv, h * 64, g.row0 + j, &full[sl], pol);
            }
            if (++sl == kSkRing) {
                sl = 0;
                par ^= 1;
            }
        }
        ke = g.k;
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

// QKV output i of tile tb (token i / 32, tile rows i % 32 and i % 32 + 32,
// a rotary pair): the factors that do not depend on the projection -- the
// token's 1/rms, the biases and the rotation -- and their application.
// A (value, epoch) pair is one aligned 64-bit store: a reader that sees the
// epoch sees the value written with it.
__device__ __forceinline__ void sk_pair_st(unsigned long long* p, float v, unsigned ep) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p),
                 "l"(((unsigned long long)ep << 32) | __float_as_uint(v))
                 : "memory");
}

__device__ __forceinline__ unsigned long long sk_pair_ld(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Two consecutive pairs (16-byte aligned), polled until both carry epoch ep
// (bounded: gives up after kWaitLimitNs or when the CTA has given up).
__device__ __forceinline__ float2 sk_pair_wait2(const unsigned long long* p, unsigned ep, volatile int* abort,
                                                int* status) {
    unsigned long long a, b;
    uint64_t t0 = 0;
    while (true) {
        asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
        if (((unsigned)(a >> 32) == ep && (unsigned)(b >> 32) == ep) || *abort) break;
        if (!t0) t0 = global_ns();
        else if (global_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            set_status(status, TP_ERR_TIMEOUT);
            break;
        }
    }
    return make_float2(__uint_as_float((unsigned)a), __uint_as_float((unsigned)b));
}

struct QkvPrep {
    float rinv, ba, bb, cs, sn;
};

__device__ __forceinline__ QkvPrep sk_qkv_prep(const GemvParams& p, int r, int tb, int i, const float* ss,
                                               const int* s_pos, const float* s_bias) {
    const int d = p.head_dim, half = d >> 1;
    const int t = i >> 5, j = i & 31;
    QkvPrep q;
    q.rinv = 1.0f / sqrtf(ss[t] * (1.0f / (float)p.K) + p.eps);
    const int rowA = tile_row(EPI_QKV_ROPE, tb, j, d, 0);
    const int head = rowA / d, ii = rowA - head * d;
    q.ba = q.bb = 0.f;
    if (s_bias) {
        q.ba = s_bias[j];
        q.bb = s_bias[j + 32];
    } else if (p.bias[r]) {
        q.ba = p.bias[r][rowA];
        q.bb = p.bias[r][rowA + half];
    }
    q.cs = 1.f;
    q.sn = 0.f;
    if (head < p.hq_s + p.hkv_s)                        // q and k rotate, v does not
        sincosf((float)s_pos[t] * exp2f(-(2.0f * ii / d) * (float)p.log2_theta), &q.sn, &q.cs);
    return q;
}

__device__ __forceinline__ void sk_qkv_apply(const GemvParams& p, int r, int tb, int i, const float* tile,
                                             const int* s_pos, const QkvPrep& q, unsigned ep) {
    const int d = p.head_dim, half = d >> 1;
    const int t = i >> 5, j = i & 31;
    const int rowA = tile_row(EPI_QKV_ROPE, tb, j, d, 0);
    const int head = rowA / d, ii = rowA - head * d;
    const float va = tile[j * kTMax + t] * q.rinv + q.ba;
    const float vb = tile[(j + 32) * kTMax + t] * q.rinv + q.bb;
    const float ra = va * q.cs - vb * q.sn, rb = va * q.sn + vb * q.cs;
    if (head < p.hq_s) {
        const size_t o = ((size_t)r * kTMax + t) * p.hq_s * d + head * d + ii;
        p.q_out[o] = ra;
        p.q_out[o + half] = rb;
        if (p.q_pairs) {                                // read by the attention phase without a grid barrier
            sk_pair_st(p.q_pairs + o, ra, ep);
            sk_pair_st(p.q_pairs + o + half, rb, ep);
        }
    } else {
        const bool is_k = head < p.hq_s + p.hkv_s;
        const int kvh = is_k ? head - p.hq_s : head - p.hq_s - p.hkv_s;
        const int pos = s_pos[t];
        if (pos < 0 || pos >= p.max_kv) {
            set_status(p.status, TP_ERR_CAPACITY);
            return;
        }
        bf16* cache = reinterpret_cast<bf16*>(is_k ? p.kcache[r] : p.vcache[r]);
        bf16* dst = cache + (((size_t)t * p.hkv_s + kvh) * p.max_kv + pos) * d + ii;
        dst[0] = __float2bfloat16_rn(ra);
        dst[half] = __float2bfloat16_rn(rb);
    }
}

// Epilogue of a column-parallel tile whose full sum is in `tile` ([64][8]).
// Threads tid0, tid0 + nthr, ... of the caller share the outputs. The bias of
// the tile's rows comes from s_bias (shared) or, when null, from global memory.
template <int EPI>
__device__ __forceinline__ void sk_col_epilogue(const GemvParams& p, int r, int tb, const float* tile, const float* ss,
                                                const int* s_pos, const float* s_bias, unsigned ep, int tid0 = -1,
                                                int nthr = kConsumers) {
    const int tid = tid0 < 0 ? (int)threadIdx.x : tid0, T = p.T;
    if (EPI == EPI_SWIGLU) {
        bf16* out = reinterpret_cast<bf16*>(p.act_out);
        const float inv_k = 1.0f / (float)p.K;
        for (int i = tid; i < 32 * T; i += nthr) {
            const int t = i >> 5, j = i & 31;
            const float rinv = 1.0f / sqrtf(ss[t] * inv_k + p.eps);
            const float gt = tile[j * kTMax + t] * rinv;
            const float up = tile[(j + 32) * kTMax + t] * rinv;
            out[((size_t)r * kTMax + t) * p.ffn_s + tb * 32 + j] = __float2bfloat16_rn(gt / (1.0f + expf(-gt)) * up);
        }
    } else {
        for (int i = tid; i < 32 * T; i += nthr)
            sk_qkv_apply(p, r, tb, i, tile, s_pos, sk_qkv_prep(p, r, tb, i, ss, s_pos, s_bias), ep);
    }
}

// ---- finishing tiles and groups shared by several CTAs -----------------------

// Finisher warp: publishes the CTA's stores covered by the job and counts its
// arrival for the tile or group; true in the CTA that arrived last (which
// resets the counter and will read every piece).
__device__ __forceinline__ bool fin_arrive(unsigned* cnt, unsigned expected) {
    unsigned last = 0;
    if ((threadIdx.x & 31) == 0) {
        __threadfence();
        const unsigned old = atomicAdd(cnt, 1u);
        last = old + 1 == expected;
        if (last) {
            *cnt = 0u;
            __threadfence();
        }
    }
    return __shfl_sync(0xffffffffu, last, 0) != 0;
}

// Consumers: column-parallel tile `seg` -- the pieces summed in CTA order into
// `tile`, then the epilogue (the tile's bias read from global memory).
template <int EPI>
__device__ __forceinline__ void sk_col_finish(const GemvParams& p, int seg, int np, float* tile, const float* ss,
                                              const int* s_pos, unsigned ep) {
    const int tid = threadIdx.x;
    constexpr int kMaxSplit = 8;
    const int nsplit = p.shape.chunks;
    for (int i = tid * 2; i < kTileRows * kTMax; i += kConsumers * 2) {
        float2 v[kMaxSplit];
#pragma unroll
        for (int q = 0; q < kMaxSplit; ++q)
            if (q < np) v[q] = __ldcg(reinterpret_cast<const float2*>(p.part + ((size_t)seg * nsplit + q) * kPartStride + i));
        float2 acc = v[0];
#pragma unroll
        for (int q = 1; q < kMaxSplit; ++q)
            if (q < np) acc = make_float2(acc.x + v[q].x, acc.y + v[q].y);
        for (int q = kMaxSplit; q < np; ++q) {
            const float2 x = __ldcg(reinterpret_cast<const float2*>(p.part + ((size_t)seg * nsplit + q) * kPartStride + i));
            acc = make_float2(acc.x + x.x, acc.y + x.y);
        }
        *reinterpret_cast<float2*>(tile + i) = acc;
    }
    consumer_sync(kConsumers);
    int r, tb;
    sk_segment(p, EPI, seg, r, tb);
    sk_col_epilogue<EPI>(p, r, tb, tile, ss, s_pos, nullptr, ep);
    consumer_sync(kConsumers);
}

// Output rows of a row-parallel tile, per thread: row j of tile tb, tokens
// 2*tp and 2*tp + 1. y = residual + sum; the next norm's operands
// bf16(y * gamma_r) for every shard, and per-8-row sums of squares.
__device__ __forceinline__ void sk_row_out(const GemvParams& p, int tb, float2 total, float2 res, const float* g2) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j8 = lane >> 2, tp = lane & 3;
    const int row = tb * kTileRows + warp * 8 + j8;
    float sq[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int t = 2 * tp + e;
        float yv = 0.f;
        if (t < p.T) {
            const size_t o = (size_t)t * p.rows + row;
            yv = (e ? res.y : res.x) + (e ? total.y : total.x);
            p.y[o] = yv;
            if (p.norm_out) {
                bf16* nout = reinterpret_cast<bf16*>(p.norm_out);
                for (int r2 = 0; r2 < p.n_shards; ++r2)
                    nout[((size_t)r2 * kTMax + t) * p.rows + row] = __float2bfloat16_rn(yv * g2[r2]);
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
            const size_t item = (size_t)tb * 8 + warp;
            p.ss_tiles_out[item * kTMax + 2 * tp] = sq[0];
            p.ss_tiles_out[item * kTMax + 2 * tp + 1] = sq[1];
        }
    }
}

// The inputs of a tile's output rows that do not depend on the phase (the
// residual and the next norm's gamma), copied asynchronously into this
// thread's slots of `slot` ([2 + TP_MAX_SHARDS] floats per thread) when the
// tile starts, so its epilogue does not wait on a round trip to L2.
constexpr int kRowSlot = 2 + TP_MAX_SHARDS;

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void sk_row_prefetch(const GemvParams& p, int tb, float* slot) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j8 = lane >> 2, tp = lane & 3;
    const int row = tb * kTileRows + warp * 8 + j8;
    float* my = slot + threadIdx.x * kRowSlot;
#pragma unroll
    for (int e = 0; e < 2; ++e)
        if (2 * tp + e < p.T) cp_async4(my + e, p.resid + (size_t)(2 * tp + e) * p.rows + row);
    if (p.norm_out)
        for (int r2 = 0; r2 < p.n_shards; ++r2) cp_async4(my + 2 + r2, p.gamma2[r2] + row);
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Consumers: row-parallel output tile tb -- pieces (CTA order) within each
// rank, then ranks in order, then the residual; with norm_out also the next
// norm's operands and per-(8-row slice, token) sums of squares. One 8-row
// slice per warp; lane = (row, token pair).
__device__ __forceinline__ void sk_row_finish(const GemvParams& p, int tb, int S, int R) {
    constexpr int kPer = 2;                            // pieces per shard held in registers
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j8 = lane >> 2, tp = lane & 3;
    const int j = warp * 8 + j8;
    const int nsplit = p.shape.chunks;
    auto piece = [&](int r, int c) {
        return reinterpret_cast<const float2*>(p.part + ((size_t)(tb * p.n_shards + r) * nsplit + c) * kPartStride +
                                               j * kTMax + 2 * tp);
    };
    // the residual and gamma are read with the pieces: one round trip
    const int row = tb * kTileRows + j;
    float2 res = make_float2(0.f, 0.f);
    if (2 * tp < p.T) res.x = __ldcg(p.resid + (size_t)(2 * tp) * p.rows + row);
    if (2 * tp + 1 < p.T) res.y = __ldcg(p.resid + (size_t)(2 * tp + 1) * p.rows + row);
    float g2[TP_MAX_SHARDS];
#pragma unroll
    for (int r2 = 0; r2 < TP_MAX_SHARDS; ++r2) g2[r2] = p.norm_out && r2 < p.n_shards ? p.gamma2[r2][row] : 0.f;
    int cnt_r[TP_MAX_SHARDS];
    float2 v[TP_MAX_SHARDS][kPer];
#pragma unroll
    for (int r = 0; r < TP_MAX_SHARDS; ++r) {
        cnt_r[r] = 0;
        if (r < p.n_shards) {
            int first, last;
            sk_owners(tb * p.n_shards + r, S, R, first, last);
            cnt_r[r] = last - first + 1;
#pragma unroll
            for (int c = 0; c < kPer; ++c)
                if (c < cnt_r[r]) v[r][c] = __ldcg(piece(r, c));
        }
    }
    float2 total = make_float2(0.f, 0.f);
#pragma unroll
    for (int r = 0; r < TP_MAX_SHARDS; ++r) {
        if (r < p.n_shards) {
            float2 pr = v[r][0];
#pragma unroll
            for (int c = 1; c < kPer; ++c)
                if (c < cnt_r[r]) pr = make_float2(pr.x + v[r][c].x, pr.y + v[r][c].y);
            for (int c = kPer; c < cnt_r[r]; ++c) {
                const float2 x = __ldcg(piece(r, c));
                pr = make_float2(pr.x + x.x, pr.y + x.y);
            }
            total = r == 0 ? pr : make_float2(total.x + pr.x, total.y + pr.y);
        }
    }
    sk_row_out(p, tb, total, res, g2);
}

// (value, epoch) pairs: a 64-bit word per value, the epoch of the launch
// that wrote it in the high half. A single-copy-atomic 64-bit access needs no
// fence or counter: a reader that sees the current epoch sees the value.
__device__ __forceinline__ unsigned long long sk_pack(float v, unsigned ep) {
    return ((unsigned long long)ep << 32) | __float_as_uint(v);
}
__device__ __forceinline__ void sk_pair_store2(unsigned long long* p, float a, float b, unsigned ep) {
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(sk_pack(a, ep)), "l"(sk_pack(b, ep))
                 : "memory");
}
__device__ __forceinline__ void sk_pair_load2(const unsigned long long* p, unsigned long long& a,
                                              unsigned long long& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

// Consumers: row-parallel output tile tb split over CTAs, combined by the CTA
// holding its last stage. Every thread polls its (row, token pair) of every
// piece at once until all carry this launch's epoch (bounded), then sums
// the pieces in CTA order within each rank, the ranks in order, and adds the
// residual -- the order of the counted finish, without its fence, counter
// and second round trip.
__device__ __forceinline__ void sk_row_combine(const GemvParams& p, int tb, int S, int R, unsigned ep,
                                               volatile int* abort) {
    constexpr int kPer = 2;                            // pieces per shard polled from registers
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j8 = lane >> 2, tp = lane & 3;
    const int j = warp * 8 + j8;
    const int nsplit = p.shape.chunks;
    auto piece = [&](int r, int c) {
        return p.pairs + ((size_t)(tb * p.n_shards + r) * nsplit + c) * (kTileRows * kTMax) + j * kTMax + 2 * tp;
    };
    const int row = tb * kTileRows + j;
    float2 res = make_float2(0.f, 0.f);
    if (2 * tp < p.T) res.x = __ldcg(p.resid + (size_t)(2 * tp) * p.rows + row);
    if (2 * tp + 1 < p.T) res.y = __ldcg(p.resid + (size_t)(2 * tp + 1) * p.rows + row);
    float g2[TP_MAX_SHARDS];
#pragma unroll
    for (int r2 = 0; r2 < TP_MAX_SHARDS; ++r2) g2[r2] = p.norm_out && r2 < p.n_shards ? p.gamma2[r2][row] : 0.f;
    int cnt_r[TP_MAX_SHARDS];
    unsigned long long va[TP_MAX_SHARDS][kPer], vb[TP_MAX_SHARDS][kPer];
#pragma unroll
    for (int r = 0; r < TP_MAX_SHARDS; ++r) {
        cnt_r[r] = 0;
        if (r < p.n_shards) {
            int first, last;
            sk_owners(tb * p.n_shards + r, S, R, first, last);
            cnt_r[r] = last - first + 1;
        }
#pragma unroll
        for (int c = 0; c < kPer; ++c) va[r][c] = vb[r][c] = 0ull;
    }
    auto cur = [&](unsigned long long a, unsigned long long b) {
        return (unsigned)(a >> 32) == ep && (unsigned)(b >> 32) == ep;
    };
    uint64_t t0 = 0;
    for (int round = 0;; ++round) {
#pragma unroll
        for (int r = 0; r < TP_MAX_SHARDS; ++r)
#pragma unroll
            for (int c = 0; c < kPer; ++c)
                if (c < cnt_r[r] && !cur(va[r][c], vb[r][c])) sk_pair_load2(piece(r, c), va[r][c], vb[r][c]);
        bool all = true;
#pragma unroll
        for (int r = 0; r < TP_MAX_SHARDS; ++r)
#pragma unroll
            for (int c = 0; c < kPer; ++c)
                if (c < cnt_r[r]) all = all && cur(va[r][c], vb[r][c]);
        if (all) break;
        if (round == 0) t0 = global_ns();
        if (*abort) break;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            set_status(p.status, TP_ERR_TIMEOUT);
            break;
        }
    }
    float2 total = make_float2(0.f, 0.f);
#pragma unroll
    for (int r = 0; r < TP_MAX_SHARDS; ++r) {
        if (r < p.n_shards) {
            float2 pr = make_float2(__uint_as_float((unsigned)va[r][0]), __uint_as_float((unsigned)vb[r][0]));
#pragma unroll
            for (int c = 1; c < kPer; ++c)
                if (c < cnt_r[r])
                    pr = make_float2(pr.x + __uint_as_float((unsigned)va[r][c]),
                                     pr.y + __uint_as_float((unsigned)vb[r][c]));
            for (int c = kPer; c < cnt_r[r]; ++c) {        // more pieces than registers: one at a time
                unsigned long long a = 0ull, b = 0ull;
                const uint64_t t1 = global_ns();
                while (true) {
                    sk_pair_load2(piece(r, c), a, b);
                    if (cur(a, b) || *abort) break;
                    if (global_ns() - t1 > kWaitLimitNs) {
                        *abort = 1;
                        set_status(p.status, TP_ERR_TIMEOUT);
                        break;
                    }
                }
                pr = make_float2(pr.x + __uint_as_float((unsigned)a), pr.y + __uint_as_float((unsigned)b));
            }
            total = r == 0 ? pr : make_float2(total.x + pr.x, total.y + pr.y);
        }
    }
    __syncwarp();
    sk_row_out(p, tb, total, res, g2);
}

// Consumers: output tile tb of a row-parallel phase whose rank-ordered sum
// over the shards is in `acc` ([64][8]); the tile's inputs were prefetched
// into `slot` by sk_row_prefetch.
__device__ __forceinline__ void sk_row_epilogue(const GemvParams& p, int tb, const float* acc, const float* slot) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = warp * 8 + (lane >> 2), tp = lane & 3;
    asm volatile("cp.async.wait_all;" ::: "memory");    // this thread's own copies
    const float* my = slot + threadIdx.x * kRowSlot;
    const float2 res = make_float2(my[0], my[1]);
    const float2 total = make_float2(acc[j * kTMax + 2 * tp], acc[j * kTMax + 2 * tp + 1]);
    sk_row_out(p, tb, total, res, my + 2);
}

// One projection phase on the consumer side: this CTA's stage range, one
// segment (tile of one shard) at a time.
template <int EPI>
__device__ __forceinline__ void sk_gemv(const GemvParams& p, int pi, unsigned char* ring, uint64_t* full,
                                        uint64_t* empty, volatile int* abort, uint32_t& it, float* tile, float* acc,
                                        float* ss, int* s_pos, float* s_bias, float* slot, SkQueue* qu,
                                        uint32_t& jn, uint32_t& jf, unsigned ep) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = (p.K + kBoxK - 1) / kBoxK;
    const int W = sk_nseg(p, EPI) * S;
    const int R = sk_phase_share(p, EPI, S);
    const int f0 = min((int)blockIdx.x * R, W), f1 = min(f0 + R, W);
    const int wm = warp & 3, wk = warp >> 2;
    const int g = lane >> 2, tq = lane & 3;
    const int box = wm >> 1, brow = 16 * (wm & 1) + g;
    if (f0 >= f1) return;
    if (EPI == EPI_QKV_ROPE && tid < kTMax) s_pos[tid] = tid < p.T ? p.pos[tid] : 0;
    if (EPI != EPI_ROWPAR) {
        float a = 0.f;                                 // warp t: token t
        if (warp < p.T)
            for (int q = lane; q < p.n_ss_tiles; q += 32) a += p.ss_tiles[q * kTMax + warp];
        a = warp_sum(a);
        if (lane == 0) ss[warp] = a;
    }
    consumer_sync(kConsumers);
    for (int f = f0; f < f1;) {
        const int seg = f / S, st0 = f - seg * S;
        const int st1 = min(S, st0 + (f1 - f));       // this CTA's stages of the segment: [st0, st1)
        int r, tb;
        sk_segment(p, EPI, seg, r, tb);
        if (EPI == EPI_ROWPAR && p.whole_tiles && r == 0) sk_row_prefetch(p, tb, slot);
        int first, last;
        sk_owners(seg, S, R, first, last);
        if (EPI == EPI_QKV_ROPE && first == last && tid < 32 * p.T) {
            // this CTA runs the tile's epilogue: its projection-independent
            // factors are computed while the weights stream (thread-private slots)
            const QkvPrep q = sk_qkv_prep(p, r, tb, tid, ss, s_pos, nullptr);
            float* my = slot + tid * 8;
            my[0] = q.rinv;
            my[1] = q.ba;
            my[2] = q.bb;
            my[3] = q.cs;
            my[4] = q.sn;
        }
        // four independent accumulators (per 64-element step half and 16-byte
        // half) so the tensor-core ops of a stage do not form one dependent chain
        float ca[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) ca[q][0] = ca[q][1] = ca[q][2] = ca[q][3] = 0.f;
        for (int st = st0; st < st1; ++st, ++it) {
            const int sl = it % kSkRing;
            mbar_wait(&full[sl], (it / kSkRing) & 1, abort, p.status);
            __syncwarp();
            const int steps_here = min(kBoxK / kKStep, (p.K - st * kBoxK) / kKStep);
            // Boxes are 128-byte swizzled: 16-byte unit u of the 128-byte row
            // (row, chunk c) sits at unit u ^ ((4 * row + c) & 7). A lane reads
            // unit 4h + tq of chunk `step` in rows of its own parity (g & 1), so
            // the eight rows a quarter warp touches fall on distinct banks.
            const unsigned char* stage = ring + sl * kSkStage;
            const unsigned char* wA = stage + box * kBoxBytes + brow * (kBoxK * 2);
            const unsigned char* wB = wA + 8 * (kBoxK * 2);
            const unsigned char* px = stage + 2 * kBoxBytes + g * (kBoxK * 2);
            uint4 fa[2][2], fb[2][2], fx[2][2];
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int step = wk + 2 * s2;
                    if (step < steps_here) {
                        const int off = step * 128 + ((h ^ (g & 1)) << 6) + ((tq ^ step) << 4);
                        fa[s2][h] = *reinterpret_cast<const uint4*>(wA + off);
                        fb[s2][h] = *reinterpret_cast<const uint4*>(wB + off);
                        fx[s2][h] = *reinterpret_cast<const uint4*>(px + off);
                    }
                }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[sl]);       // the fragments are in registers
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (wk + 2 * s2 < steps_here) {
                        float* cq = ca[2 * s2 + h];
                        float(&cc)[4] = *reinterpret_cast<float(*)[4]>(cq);
                        mma_bf16_16816(cc, fa[s2][h].x, fb[s2][h].x, fa[s2][h].y, fb[s2][h].y, fx[s2][h].x,
                                       fx[s2][h].y);
                        mma_bf16_16816(cc, fa[s2][h].z, fb[s2][h].z, fa[s2][h].w, fb[s2][h].w, fx[s2][h].z,
                                       fx[s2][h].w);
                    }
                }
        }
        float c[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) c[e] = (ca[0][e] + ca[1][e]) + (ca[2][e] + ca[3][e]);
        f += st1 - st0;
        // this CTA's sum over its stages of the segment: (half 0) + (half 1)
        const int i0 = (16 * wm + g) * kTMax + 2 * tq, i1 = (16 * wm + g + 8) * kTMax + 2 * tq;
        if (wk == 0) {
            tile[i0] = c[0];
            tile[i0 + 1] = c[1];
            tile[i1] = c[2];
            tile[i1 + 1] = c[3];
        }
        consumer_sync(kConsumers);
        if (wk == 1) {
            tile[i0] += c[0];
            tile[i0 + 1] += c[1];
            tile[i1] += c[2];
            tile[i1 + 1] += c[3];
        }
        consumer_sync(kConsumers);
        const int nsplit = p.shape.chunks;
        if (EPI == EPI_ROWPAR && p.whole_tiles) {       // this CTA holds every shard of output tile tb
            for (int i = tid; i < kTileRows * kTMax; i += kConsumers)
                acc[i] = r == 0 ? tile[i] : acc[i] + tile[i];   // ((p0 + p1) + p2) + ...
            consumer_sync(kConsumers);
            if (r == p.n_shards - 1) {
                sk_row_epilogue(p, tb, acc, slot);
                consumer_sync(kConsumers);
            }
            continue;
        }
        if (EPI != EPI_ROWPAR && first == last) {      // the whole tile was this CTA's
            if (EPI == EPI_QKV_ROPE) {
                if (tid < 32 * p.T) {
                    const float* my = slot + tid * 8;
                    sk_qkv_apply(p, r, tb, tid, tile, s_pos, QkvPrep{my[0], my[1], my[2], my[3], my[4]}, ep);
                }
            } else {
                sk_col_epilogue<EPI>(p, r, tb, tile, ss, s_pos, s_bias, ep);
            }
            consumer_sync(kConsumers);
            continue;
        }
        if (EPI == EPI_ROWPAR && p.pairs) {              // the piece as (value, epoch) pairs, polled by the combiner
            unsigned long long* pm = p.pairs + ((size_t)seg * nsplit + ((int)blockIdx.x - first)) * (kTileRows * kTMax);
            for (int i = tid * 2; i < kTileRows * kTMax; i += kConsumers * 2) sk_pair_store2(pm + i, tile[i], tile[i + 1], ep);
            consumer_sync(kConsumers);                  // `tile` may be reused
            continue;
        }
        float* mine = p.part + ((size_t)seg * nsplit + ((int)blockIdx.x - first)) * kPartStride;
        for (int i = tid * 4; i < kTileRows * kTMax; i += kConsumers * 4)
            *reinterpret_cast<float4*>(mine + i) = *reinterpret_cast<const float4*>(tile + i);
        consumer_sync(kConsumers);                      // the piece is stored; `tile` may be reused
        if (tid == 0) {
            if (EPI == EPI_ROWPAR) {
                // the last piece of output tile tb posts the job that counts the tile's arrivals
                unsigned expected = 0;
                for (int r2 = 0; r2 < p.n_shards; ++r2) {
                    int a1, a2;
                    sk_owners(tb * p.n_shards + r2, S, R, a1, a2);
                    expected += (unsigned)(a2 - a1 + 1);
                }
                sk_post(qu, jn, JOB_ROW, pi, tb, expected, abort, p.status);
            } else {
                sk_post(qu, jn, JOB_COL, pi, seg, (unsigned)(last - first + 1), abort, p.status);
            }
        }
        ++jn;
        ++jf;
    }
    if (EPI == EPI_ROWPAR && p.pairs) {
        // output tiles whose last stage is this CTA's: it combines their pieces
        const int per_tile = p.n_shards * S;
        for (int tb = (f0 + 1 + per_tile - 1) / per_tile - 1; (tb + 1) * per_tile <= f1; ++tb) {
            if (tb < 0) continue;
            sk_row_combine(p, tb, S, R, ep, abort);
        }
    }
}

// The CTA's attention segments, listed once at the start of the step (they
// depend only on the positions) so the attention phase starts without walking
// the key space. More than kSegTab segments: the phase walks it instead.
struct SkSegInfo {
    int gi, b, kh, r, gstart, len, n, qoff;
};

template <int D>
__device__ __forceinline__ void sk_seg_table(const AttnDecodeParams& p, SkSegInfo* tab, int* s_nseg) {
    pdl_wait();                                         // positions of the preceding step
    int posv[kTMax];
    for (int b = 0; b < kTMax; ++b) posv[b] = b < p.B ? p.pos[b] : 0;
    const KeySpace ks = sk_keyspace(p, posv);
    const int G = p.hq_s / p.hkv_s;
    const KeySplit sp = sk_key_split(ks.total, step_min_keys(p.max_kv), p.key_busy);
    const int k0 = sk_key_start(sp, (int)blockIdx.x, ks.total), k1 = sk_key_start(sp, (int)blockIdx.x + 1, ks.total);
    int n = 0;
    for (int ke = k1; ke > k0 && n <= kSegTab; ++n) {
        int gi, b, off, gstart;
        sk_locate(ks, p, ke - 1, gi, b, off, gstart);
        const int k = max(k0, gstart);
        if (n < kSegTab) {
            SkSegInfo& e = tab[n];
            e.gi = gi;
            e.b = b;
            e.kh = gi % p.hkv_s;
            e.r = gi / (p.hkv_s * p.B);
            e.gstart = gstart;
            e.len = ks.len[b];
            e.n = ke - k;
            e.qoff = ((e.r * kTMax + b) * p.hq_s + e.kh * G) * D;
        }
        ke = k;
    }
    *s_nseg = n;                                        // kSegTab + 1: too many to list
}

// Attention phase on the consumer side: this CTA's key range, one group
// segment at a time (every warp waits for and releases every stage; the
// 64-key blocks of a segment alternate between warps 0-3 and 4-7). A segment
// holding a whole group writes the normalised output directly; otherwise
// the CTA stores (max, sum, unnormalised output) and the last of the group's
// CTAs combines them in CTA order.
template <int D>
__device__ __forceinline__ void sk_attn(const AttnDecodeParams& p, unsigned char* ring, uint64_t* full,
                                        uint64_t* empty, volatile int* abort, uint32_t& it, float* red,
                                        float* s_ml2, float* s_cmb, const int* s_pos, bf16* qs,
                                        const SkSegInfo* tab, const int* s_nseg, uint64_t* tab_ready,
                                        SkQueue* qu, uint32_t& jn, unsigned ep) {
    using S = AtShape<D>;
    constexpr int KS = D / 16;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.hq_s / p.hkv_s;
    const int grp = warp >> 2, wq = warp & 3;
    const int g = lane >> 2, t = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;
    const uint32_t ring_u32 = smem_u32(ring);
    const int q0 = 2 * t, q1 = 2 * t + 1;
    const int pstride = G * (D + 2);
    const KeySpace ks = sk_keyspace(p, s_pos);
    const KeySplit sp = sk_key_split(ks.total, step_min_keys(p.max_kv), p.key_busy);
    const int k0 = sk_key_start(sp, (int)blockIdx.x, ks.total), k1 = sk_key_start(sp, (int)blockIdx.x + 1, ks.total);
    // q of the CTA's first segments, scaled and rounded to bf16 once and staged
    // in shared memory: one round trip of loads for all of them instead of one
    // per segment (q was written by other CTAs in the QKV phase)
    mbar_wait(tab_ready, 0, abort, p.status);
    const int nseg = *s_nseg;
    const bool listed = nseg <= kSegTab;
    const int qper = G * D;
    const int nq = listed ? min(min(nseg, kQSegs), kQStage / qper) : 0;
    {
        constexpr int kPer = kQStage / kConsumers;
        static_assert(kPer <= 32, "one bit per staged value");
        const int n = nq * qper;
        float v[kPer];
        if (p.q_pairs) {
            // poll the (value, epoch) pairs: every load of a round in flight, the
            // missing ones reloaded until each carries this launch's epoch
            unsigned long long u[kPer];
            unsigned need = 0;
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const int idx = tid + i * kConsumers;
                if (idx < n) {
                    const int sg = idx / qper;
                    u[i] = sk_pair_ld(p.q_pairs + tab[sg].qoff + (idx - sg * qper));
                    if ((unsigned)(u[i] >> 32) != ep) need |= 1u << i;
                }
            }
            uint64_t t0 = 0;
            while (need) {
                if (*abort) break;
                if (!t0) t0 = global_ns();
                else if (global_ns() - t0 > kWaitLimitNs) {
                    *abort = 1;
                    set_status(p.status, TP_ERR_TIMEOUT);
                    break;
                }
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    if (need & (1u << i)) {
                        const int idx = tid + i * kConsumers, sg = idx / qper;
                        u[i] = sk_pair_ld(p.q_pairs + tab[sg].qoff + (idx - sg * qper));
                        if ((unsigned)(u[i] >> 32) == ep) need &= ~(1u << i);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < kPer; ++i) v[i] = __uint_as_float((unsigned)u[i]);
        } else {
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const int idx = tid + i * kConsumers;
                if (idx < n) {
                    const int sg = idx / qper;
                    v[i] = __ldcg(p.q + tab[sg].qoff + (idx - sg * qper));
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int idx = tid + i * kConsumers;
            if (idx < n) qs[idx] = __float2bfloat16_rn(v[i] * p.scale);
        }
    }
    consumer_sync(kConsumers);
    int ui = 0;
    for (int ke = k1; ke > k0; ++ui) {                  // segments in reverse order (as the producer)
        int gi, b, gstart, len, n, kh, r;
        if (listed) {
            const SkSegInfo& e = tab[ui];
            gi = e.gi;
            b = e.b;
            gstart = e.gstart;
            len = e.len;
            n = e.n;                                    // keys of this segment
            kh = e.kh;
            r = e.r;
        } else {
            int off;
            sk_locate(ks, p, ke - 1, gi, b, off, gstart);
            len = ks.len[b];
            n = ke - max(k0, gstart);
            kh = gi % p.hkv_s;
            r = gi / (p.hkv_s * p.B);
        }
        ke -= n;
        const int nblk = (n + kAtKeys - 1) / kAtKeys;
        uint32_t qb[KS][2];
        if (ui < nq) {
            const bf16* qp = qs + ui * qper + (g < G ? g : 0) * D;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                qb[kk][0] = g < G ? *reinterpret_cast<const uint32_t*>(qp + 16 * kk + 2 * t) : 0u;
                qb[kk][1] = g < G ? *reinterpret_cast<const uint32_t*>(qp + 16 * kk + 8 + 2 * t) : 0u;
            }
        } else {
            const size_t qo = ((size_t)r * kTMax + b) * p.hq_s * D + (size_t)(kh * G + (g < G ? g : 0)) * D;
            const float* qp = p.q + qo;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                if (g < G) {
                    const float2 a = p.q_pairs ? sk_pair_wait2(p.q_pairs + qo + 16 * kk + 2 * t, ep, abort, p.status)
                                               : __ldcg(reinterpret_cast<const float2*>(qp + 16 * kk + 2 * t));
                    const float2 c2 = p.q_pairs
                                          ? sk_pair_wait2(p.q_pairs + qo + 16 * kk + 8 + 2 * t, ep, abort, p.status)
                                          : __ldcg(reinterpret_cast<const float2*>(qp + 16 * kk + 8 + 2 * t));
                    qb[kk][0] = pack_bf16x2(a.x * p.scale, a.y * p.scale);
                    qb[kk][1] = pack_bf16x2(c2.x * p.scale, c2.y * p.scale);
                } else {
                    qb[kk][0] = qb[kk][1] = 0u;
                }
            }
        }
        float o[KS][4];
#pragma unroll
        for (int dt = 0; dt < KS; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        for (int blk = 0; blk < nblk; ++blk, ++it) {
            const int sl = it % kSkRing;
            mbar_wait(&full[sl], (it / kSkRing) & 1, abort, p.status);
            __syncwarp();
            if ((blk & 1) == grp) {
                const uint32_t kpart = ring_u32 + sl * kSkStage, vpart = kpart + S::NB * S::BOX;
                const int kb = blk * kAtKeys + 16 * wq;          // relative to the segment
                float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(at_addr<D>(kpart, 16 * wq + rr + 8 * (mi & 1), 2 * kk + (mi >> 1)), a0, a1, a2, a3);
                    mma_bf16_16816(sc, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
                }
                const bool v0 = kb + g < n, v1 = kb + g + 8 < n;
                const float x00 = v0 ? sc[0] : -INFINITY, x01 = v0 ? sc[1] : -INFINITY;
                const float x10 = v1 ? sc[2] : -INFINITY, x11 = v1 ? sc[3] : -INFINITY;
                float mq0 = fmaxf(x00, x10), mq1 = fmaxf(x01, x11);
#pragma unroll
                for (int sh = 4; sh < 32; sh <<= 1) {
                    mq0 = fmaxf(mq0, __shfl_xor_sync(0xffffffffu, mq0, sh));
                    mq1 = fmaxf(mq1, __shfl_xor_sync(0xffffffffu, mq1, sh));
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
                for (int sh = 4; sh < 32; sh <<= 1) {
                    ps0 += __shfl_xor_sync(0xffffffffu, ps0, sh);
                    ps1 += __shfl_xor_sync(0xffffffffu, ps1, sh);
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

        // ---- merge the eight warps: common max per query, every warp's rescaled
        // output into its slot, then all threads sum the slots in warp order
        const int first = sk_key_cta(sp, gstart), last = sk_key_cta(sp, gstart + len - 1);
        const int nc = last - first + 1;
        // A KV group split over CTAs is combined by the CTA holding its last keys
        // (its block with the new position streams last, so it normally finishes
        // last): it waits for the other nc - 1 pieces here, and their loads go out
        // during the merge below.
        const bool owner = nc > 1 && (int)blockIdx.x == last;
        if (owner && tid == 0) {
            const unsigned want = (unsigned)(nc - 1);
            if (ld_acquire_u32(p.cnt + gi) != want) {
                const uint64_t t0 = global_ns();
                while (ld_acquire_u32(p.cnt + gi) != want) {
                    if (*abort) break;
                    if (global_ns() - t0 > kWaitLimitNs) {
                        *abort = 1;
                        set_status(p.status, TP_ERR_TIMEOUT);
                        break;
                    }
                }
            }
            p.cnt[gi] = 0u;                             // counters are zero at every launch
        }
        float* s_ml = s_ml2 + (ui & 1) * (8 * kMaxGroup * 2);   // double-buffered across segments
        if (g == 0) {
            s_ml[(warp * kMaxGroup + q0) * 2] = m0;
            s_ml[(warp * kMaxGroup + q0) * 2 + 1] = l0;
            s_ml[(warp * kMaxGroup + q1) * 2] = m1;
            s_ml[(warp * kMaxGroup + q1) * 2 + 1] = l1;
        }
        consumer_sync(kConsumers);                      // also orders the pieces' loads after the wait
        const float* base = p.part + (size_t)gi * p.n_chunks * pstride;
        constexpr int kEarly = 2;                       // pieces loaded before the merge's second half
        const bool early = owner && G * D <= 2 * kConsumers;
        float em[kEarly][2], el[kEarly][2], evv[kEarly][2];
        if (early) {
#pragma unroll
            for (int cc = 0; cc < kEarly; ++cc)
#pragma unroll
                for (int o = 0; o < 2; ++o) {
                    const int i = tid + o * kConsumers;
                    if (cc < nc - 1 && i < G * D) {
                        const float* pc = base + (size_t)cc * pstride;
                        em[cc][o] = __ldcg(pc + G * D + i / D);
                        el[cc][o] = __ldcg(pc + G * D + G + i / D);
                        evv[cc][o] = __ldcg(pc + i);
                    }
                }
        }
        float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            M0 = fmaxf(M0, s_ml[(w * kMaxGroup + q0) * 2]);
            M1 = fmaxf(M1, s_ml[(w * kMaxGroup + q1) * 2]);
        }
        const float c0 = (m0 == -INFINITY) ? 0.f : expf(m0 - M0);
        const float c1 = (m1 == -INFINITY) ? 0.f : expf(m1 - M1);
        float* dst = red + warp * kAtSlot;
#pragma unroll
        for (int dt = 0; dt < KS; ++dt) {
            if (q0 < G) {
                dst[q0 * D + 16 * dt + g] = o[dt][0] * c0;
                dst[q0 * D + 16 * dt + g + 8] = o[dt][2] * c0;
            }
            if (q1 < G) {
                dst[q1 * D + 16 * dt + g] = o[dt][1] * c1;
                dst[q1 * D + 16 * dt + g + 8] = o[dt][3] * c1;
            }
        }
        if (warp == 0) {                                // this segment's (max, sum) per query: lane 4w + t
            const int w = lane >> 2;                    // holds warp w's share of queries 2t, 2t + 1
            const float mw0 = s_ml[(w * kMaxGroup + q0) * 2], mw1 = s_ml[(w * kMaxGroup + q1) * 2];
            float L0 = mw0 == -INFINITY ? 0.f : s_ml[(w * kMaxGroup + q0) * 2 + 1] * expf(mw0 - M0);
            float L1 = mw1 == -INFINITY ? 0.f : s_ml[(w * kMaxGroup + q1) * 2 + 1] * expf(mw1 - M1);
#pragma unroll
            for (int sh = 4; sh < 32; sh <<= 1) {
                L0 += __shfl_xor_sync(0xffffffffu, L0, sh);
                L1 += __shfl_xor_sync(0xffffffffu, L1, sh);
            }
            if (lane < 4) {
                if (q0 < G) {
                    s_cmb[q0] = M0;
                    s_cmb[kMaxGroup + q0] = L0;
                }
                if (q1 < G) {
                    s_cmb[q1] = M1;
                    s_cmb[kMaxGroup + q1] = L1;
                }
            }
        }
        consumer_sync(kConsumers);
        bf16* out = reinterpret_cast<bf16*>(p.out) + ((size_t)r * kTMax + b) * p.hq_s * D + (size_t)kh * G * D;
        if (nc == 1) {                                  // the whole group: normalise and store
            for (int i = tid; i < G * D; i += kConsumers) {
                float acc = red[i];
#pragma unroll
                for (int w = 1; w < 8; ++w) acc += red[w * kAtSlot + i];
                const float L = s_cmb[kMaxGroup + i / D];
                out[i] = __float2bfloat16_rn(L > 0.f ? acc / L : 0.f);
            }
            continue;                                   // slots are rewritten after the next segment's first barrier
        }
        if (!owner) {                                   // a piece of a group another CTA finishes
            float* mine = p.part + ((size_t)gi * p.n_chunks + ((int)blockIdx.x - first)) * pstride;
            for (int i = tid; i < G * D; i += kConsumers) {
                float acc = red[i];
#pragma unroll
                for (int w = 1; w < 8; ++w) acc += red[w * kAtSlot + i];
                mine[i] = acc;
            }
            if (tid < G) {
                mine[G * D + tid] = s_cmb[tid];
                mine[G * D + G + tid] = s_cmb[kMaxGroup + tid];
            }
            consumer_sync(kConsumers);                  // the piece is stored; the slots may be reused
            // the finisher warp publishes the piece (its release would hold up this thread)
            if (tid == 0) sk_post(qu, jn, JOB_GRP, 0, gi, 0u, abort, p.status);
            ++jn;
            continue;
        }
        // owner: the pieces in CTA order -- max, weights exp(m_c - M), sum of
        // l_c w_c, sum of O_c w_c -- with its own piece (in shared memory) last
        constexpr int kMaxSplit = 8;                    // pieces loaded in one batch (more: one at a time)
        int o_idx = 0;
        for (int i = tid; i < G * D; i += kConsumers, ++o_idx) {
            const int gq = i / D;
            float pm[kMaxSplit], pl[kMaxSplit], pv[kMaxSplit];
#pragma unroll
            for (int cc = 0; cc < kMaxSplit; ++cc) {
                if (cc < nc - 1) {
                    if (early && cc < kEarly) {
                        pm[cc] = o_idx ? em[cc][1] : em[cc][0];
                        pl[cc] = o_idx ? el[cc][1] : el[cc][0];
                        pv[cc] = o_idx ? evv[cc][1] : evv[cc][0];
                    } else {
                        const float* pc = base + (size_t)cc * pstride;
                        pm[cc] = __ldcg(pc + G * D + gq);
                        pl[cc] = __ldcg(pc + G * D + G + gq);
                        pv[cc] = __ldcg(pc + i);
                    }
                }
            }
            float own = red[i];
#pragma unroll
            for (int w = 1; w < 8; ++w) own += red[w * kAtSlot + i];
            const float mo = s_cmb[gq], lo = s_cmb[kMaxGroup + gq];
            float M = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < kMaxSplit; ++cc)
                if (cc < nc - 1 && pl[cc] > 0.f) M = fmaxf(M, pm[cc]);
            for (int cc = kMaxSplit; cc < nc - 1; ++cc)
                if (__ldcg(base + (size_t)cc * pstride + G * D + G + gq) > 0.f)
                    M = fmaxf(M, __ldcg(base + (size_t)cc * pstride + G * D + gq));
            if (lo > 0.f) M = fmaxf(M, mo);
            float den = 0.f, num = 0.f;
#pragma unroll
            for (int cc = 0; cc < kMaxSplit; ++cc) {
                if (cc < nc - 1) {
                    const float w = pl[cc] > 0.f ? expf(pm[cc] - M) : 0.f;
                    den = fmaf(pl[cc], w, den);
                    num = fmaf(pv[cc], w, num);
                }
            }
            for (int cc = kMaxSplit; cc < nc - 1; ++cc) {
                const float* pc = base + (size_t)cc * pstride;
                const float l = __ldcg(pc + G * D + G + gq);
                const float w = l > 0.f ? expf(__ldcg(pc + G * D + gq) - M) : 0.f;
                den = fmaf(l, w, den);
                num = fmaf(__ldcg(pc + i), w, num);
            }
            const float wo = lo > 0.f ? expf(mo - M) : 0.f;
            den = fmaf(lo, wo, den);
            num = fmaf(own, wo, num);
            out[i] = __float2bfloat16_rn(num * (den > 0.f ? 1.0f / den : 0.f));
        }
    }
}

constexpr int kStepThreads = kStreamThreads + 32;       // + the finisher warp

size_t decode_step_smem() {
    // ring | red [8][kAtSlot] | s_ml [2][8][8][2] | tile [64][8] | ss, pos, bias | s_cmb | ftile [64][8] |
    // queue | table-ready barrier | segment table [kSegTab] | segment count (8 bytes) | staged q [kQStage] bf16
    return 1024 + (size_t)kSkRing * kSkStage +
           (size_t)(8 * kAtSlot + 2 * 8 * kMaxGroup * 2 + kTileRows * kTMax + kTMax + kTMax + 96 + 2 * kMaxGroup +
                    kTileRows * kTMax) * 4 +
           sizeof(SkQueue) + 8 + kSegTab * sizeof(SkSegInfo) + 8 + (size_t)kQStage * 2;
}

// The finisher warp: the jobs of the consumers, in order. Piece jobs are
// counted for their tile or group; a tile or group this CTA arrived last on
// goes to the CTA's finish list. A phase-end job releases the consumers, who
// run the finish list with all their threads.
__device__ __forceinline__ void sk_finisher(const StepArgs& A, SkQueue* qu, volatile int* abort) {
    const int lane = threadIdx.x & 31;
    int* status = A.a.status;
    for (uint32_t fj = 0;; ++fj) {
        const int sl = fj % kJobs;
        const bool ok = mbar_wait(&qu->full[sl], (fj / kJobs) & 1, abort, status);
        __syncwarp();
        if (!__all_sync(0xffffffffu, ok)) return;       // the consumers stopped posting (error already set)
        const SkJob j = qu->job[sl];
        if (j.type == JOB_GRP) {                        // an attention piece stored: count it for the group
            if (lane == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(A.a.cnt + j.idx) : "memory");
        } else if (j.type == JOB_COL || j.type == JOB_ROW) {
            unsigned* cnt = A.g[j.pi].cnt;
            if (fin_arrive(cnt + j.idx, j.expected) && lane == 0) {
                if (qu->n_fin < kMaxFin) qu->fin[qu->n_fin++] = j;
                else set_status(status, TP_ERR_UNSUPPORTED);
            }
        } else if (lane == 0) {
            mbar_arrive(&qu->drained);                   // every earlier job is done
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&qu->empty[sl]);
        if (j.type == JOB_END) return;
    }
}

// Consumers at the end of phase k (k = 1..kSkBarriers; k = kSkBarriers + 1 is
// the last phase, which has no barrier): hand the phase end to the finisher,
// run the finishes this CTA owes, then arrive at grid barrier k and wait. A
// phase in which this CTA posted no piece job owes no finish: it skips the
// hand-over (except the last, whose end job lets the finisher exit). `jf`
// counts the posts that can make this CTA owe a finish, `jf_mark` its value at
// the previous phase end, `nd` the hand-overs so far.
template <int D>
__device__ __forceinline__ void sk_phase_end(const StepArgs& A, unsigned long long base, unsigned k,
                                             volatile int* abort, SkQueue* qu, uint32_t& jn, uint32_t jf, uint32_t& jf_mark,
                                             uint32_t& nd, float* tile, const float* ss, const int* s_pos,
                                             float* red, float* s_inv, unsigned long long* st, bool wait = true) {
    int* status = A.a.status;
    const bool hand_over = jf != jf_mark || k > kSkBarriers;
    consumer_sync(kConsumers);
    if (threadIdx.x == 0) {
        if (st) st[2 * k - 1] = global_ns();
        if (hand_over) sk_post(qu, jn, k > kSkBarriers ? JOB_END : JOB_PHASE, 0, (int)k, 0u, abort, status);
    }
    int nf = 0;
    if (hand_over) {
        ++jn;
        mbar_wait(&qu->drained, nd & 1, abort, status);
        ++nd;
        nf = *reinterpret_cast<volatile int*>(&qu->n_fin);
    }
    jf_mark = jf;
    for (int f = 0; f < nf; ++f) {
        const SkJob j = qu->fin[f];
        if (j.type == JOB_COL) {
            const unsigned ep = (unsigned)(base / ((unsigned long long)kSkBarriers * gridDim.x)) + 1u;
            if (j.pi == 0) sk_col_finish<EPI_QKV_ROPE>(A.g[0], j.idx, (int)j.expected, tile, ss, s_pos, ep);
            else sk_col_finish<EPI_SWIGLU>(A.g[2], j.idx, (int)j.expected, tile, ss, s_pos, ep);
        } else if (j.type == JOB_ROW) {
            const GemvParams& p = A.g[j.pi];
            const int S = (p.K + kBoxK - 1) / kBoxK;
            sk_row_finish(p, j.idx, S, sk_phase_share(p, EPI_ROWPAR, S));
        }
    }
    consumer_sync(kConsumers);
    if (threadIdx.x == 0) {
        if (nf) qu->n_fin = 0;
        if (st) st[2 * k] = global_ns();
        if (k <= kSkBarriers) {
            if (k == 2) asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(A.kv_ready) : "memory");
            asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(A.bar) : "memory");
            if (wait) {                                 // (else the next phase polls its inputs' epochs)
                sk_wait_gen(A.bar, base, k, abort, status);
                __threadfence();
            }
        }
    }
    consumer_sync(kConsumers);
}

template <int D>
__global__ void __maxnreg__(168) decode_step_kernel(const __grid_constant__ StepArgs A) {
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kSkRing;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 16 * kSkRing);
    unsigned long long* s_gen0 = reinterpret_cast<unsigned long long*>(smem + 16 * kSkRing + 8);
    unsigned char* ring = smem + 1024;
    float* red = reinterpret_cast<float*>(ring + kSkRing * kSkStage);
    float* s_ml = red + 8 * kAtSlot;
    float* tile = s_ml + 2 * 8 * kMaxGroup * 2;
    float* ss = tile + kTileRows * kTMax;
    int* s_pos = reinterpret_cast<int*>(ss + kTMax);
    float* s_bias = reinterpret_cast<float*>(s_pos + kTMax);
    float* s_cmb = s_bias + 96;
    float* ftile = s_cmb + 2 * kMaxGroup;
    SkQueue* qu = reinterpret_cast<SkQueue*>(ftile + kTileRows * kTMax);
    uint64_t* tab_ready = reinterpret_cast<uint64_t*>(qu + 1);
    SkSegInfo* seg_tab = reinterpret_cast<SkSegInfo*>(tab_ready + 1);
    int* s_nseg = reinterpret_cast<int*>(seg_tab + kSegTab);
    bf16* qs = reinterpret_cast<bf16*>(s_nseg + 2);
    int* status = A.a.status;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < kSkRing; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumers / 32);
        }
        for (int i = 0; i < kJobs; ++i) {
            mbar_init(&qu->full[i], 1);
            mbar_init(&qu->empty[i], 1);
        }
        mbar_init(&qu->drained, 1);
        mbar_init(tab_ready, 1);
        qu->n_fin = 0;
        *abort_flag = (smem_u32(ring) & 1023u) ? 1 : 0;       // 128-byte-swizzled boxes need 1024-byte alignment
        if (*abort_flag) set_status(status, TP_ERR_ALIGN);
        // read before this CTA arrives anywhere: fewer than gridDim.x arrivals of
        // this step can precede it
        const unsigned long long per_step = (unsigned long long)kSkBarriers * gridDim.x;
        const unsigned long long c = ld_acquire_u64(A.bar);
        // bar_extra (a test hook, 0 otherwise) raises every barrier's target
        // above what the grid's arrivals reach, so the waits run out; the
        // arrivals themselves, and so the next launch's base, are unchanged
        *s_gen0 = c - c % per_step + A.bar_extra;
        fence_mbar_init();
    }
    __syncthreads();
    const unsigned long long gen0 = *s_gen0;
    // this launch's epoch: the barrier counter grows by kSkBarriers * gridDim.x a launch (never 0)
    const unsigned ep = (unsigned)(gen0 / ((unsigned long long)kSkBarriers * gridDim.x)) + 1u;
    unsigned long long* st =
        A.stamps && blockIdx.x < kMaxStepCtas ? A.stamps + (size_t)blockIdx.x * kStepStamps : nullptr;

    if (warp == kConsumers / 32) {                     // ---- producer
        if (lane == 0 && !*abort_flag) {
            const uint64_t pol = l2_evict_first_policy();
            uint32_t it = 0;
            SkPend pd;
            pd.n = 0;
            SkKeys keys;
            keys.ready = false;
            // weights do not depend on the preceding step: QKV streams at once; the
            // activation boxes wait for barrier 1, which follows the consumers' wait
            bool ok = sk_produce_gemv(EPI_QKV_ROPE, 0, 1, A, ring, full, empty, it, pd, gen0, abort_flag, pol);
            if (ok) ok = sk_produce_attn<D>(2, A, ring, full, empty, it, pd, keys, gen0, abort_flag, pol);
            if (ok) ok = sk_produce_gemv(EPI_ROWPAR, 1, 3, A, ring, full, empty, it, pd, gen0, abort_flag, pol);
            if (ok) ok = sk_produce_gemv(EPI_SWIGLU, 2, 4, A, ring, full, empty, it, pd, gen0, abort_flag, pol);
            if (ok) ok = sk_produce_gemv(EPI_ROWPAR, 3, 5, A, ring, full, empty, it, pd, gen0, abort_flag, pol);
            sk_flush(pd, A, ring, full, gen0, abort_flag, status);
            // no copy may still be landing when the CTA exits
            volatile int no_abort = 0;
            const uint32_t first = it > (uint32_t)kSkRing ? it - kSkRing : 0u;
            for (uint32_t k = first; k < it; ++k) mbar_wait(&full[k % kSkRing], (k / kSkRing) & 1, &no_abort, nullptr);
        }
        return;
    }
    if (warp == kConsumers / 32 + 1) {                 // ---- finisher
        if (lane == 0) {
            sk_seg_table<D>(A.a, seg_tab, s_nseg);
            mbar_arrive(tab_ready);
        }
        __syncwarp();
        sk_finisher(A, qu, abort_flag);
        return;
    }

    // ---- consumers
    if (st && tid == 0) st[0] = global_ns();
    pdl_wait();                                         // x, positions and caches of the preceding step
    if (tid < kTMax) s_pos[tid] = tid < A.a.B ? A.a.pos[tid] : 0;
    consumer_sync(kConsumers);
    uint32_t it = 0, jn = 0, jf = 0, jf_mark = 0, nd = 0;
    sk_norm(A.np);
    sk_phase_end<D>(A, gen0, 1, abort_flag, qu, jn, jf, jf_mark, nd, tile, ss, s_pos, red, s_cmb, st);
    sk_gemv<EPI_QKV_ROPE>(A.g[0], 0, ring, full, empty, abort_flag, it, tile, ftile, ss, s_pos, s_bias, red, qu, jn, jf, ep);
    // with q published as (value, epoch) pairs the consumers only arrive at barrier 2 (the producer still
    // waits for it before loading the key block holding a new position)
    sk_phase_end<D>(A, gen0, 2, abort_flag, qu, jn, jf, jf_mark, nd, tile, ss, s_pos, red, s_cmb, st,
                    A.a.q_pairs == nullptr);
    sk_attn<D>(A.a, ring, full, empty, abort_flag, it, red, s_ml, s_cmb, s_pos, qs, seg_tab, s_nseg, tab_ready, qu,
               jn, ep);
    sk_phase_end<D>(A, gen0, 3, abort_flag, qu, jn, jf, jf_mark, nd, tile, ss, s_pos, red, s_cmb, st);
    sk_gemv<EPI_ROWPAR>(A.g[1], 1, ring, full, empty, abort_flag, it, tile, ftile, ss, s_pos, s_bias, red, qu, jn, jf, ep);
    sk_phase_end<D>(A, gen0, 4, abort_flag, qu, jn, jf, jf_mark, nd, tile, ss, s_pos, red, s_cmb, st);
    sk_gemv<EPI_SWIGLU>(A.g[2], 2, ring, full, empty, abort_flag, it, tile, ftile, ss, s_pos, s_bias, red, qu, jn, jf, ep);
    sk_phase_end<D>(A, gen0, 5, abort_flag, qu, jn, jf, jf_mark, nd, tile, ss, s_pos, red, s_cmb, st);
    pdl_trigger();                                      // the next launch may start streaming its weights
    sk_gemv<EPI_ROWPAR>(A.g[3], 3, ring, full, empty, abort_flag, it, tile, ftile, ss, s_pos, s_bias, red, qu, jn, jf, ep);
    sk_phase_end<D>(A, gen0, kSkBarriers + 1, abort_flag, qu, jn, jf, jf_mark, nd, tile, ss, s_pos, red, s_cmb, st);
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
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kStepThreads, smem);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        grid_sz[which] = sms < kMaxStepCtas ? sms : kMaxStepCtas;   // one CTA per SM
    }
    StepArgs A;
    memset(&A, 0, sizeof A);
    for (int i = 0; i < 4; ++i) {
        const GemvParams& p = P.g[i];
        A.g[i] = p;
        for (int r = 0; r < p.n_shards; ++r) {
            cudaError_t e = step_stage_map(p.W[r], p.K, p.rows, 32, &A.wm[i][r]);
            if (e != cudaSuccess) return e;
        }
        cudaError_t e = step_stage_map(p.xact, p.K, p.n_shards * kTMax, kTMax, &A.xm[i]);
        if (e != cudaSuccess) return e;
    }
    A.a = P.a;
    {
        // CTAs holding a QKV tile: whole tiles, ceil(tiles / grid) per CTA
        const int tiles = P.g[0].shape.groups, g = grid_sz[which];
        const int per = (tiles + g - 1) / g;
        A.a.key_busy = (tiles + per - 1) / per;
    }
    A.np = P.np;
    const long rows = (long)P.a.max_batch * P.a.hkv_s * P.a.max_kv;
    for (int r = 0; r < P.a.N; ++r) {
        const int pt = D == 128 ? AtShape<128>::PT : AtShape<64>::PT;
        cudaError_t e = tensor_map_2d(P.a.kcache[r], D, rows, pt, kAtKeys, 0, &A.tk[r]);
        if (e == cudaSuccess) e = tensor_map_2d(P.a.vcache[r], D, rows, pt, kAtKeys, 0, &A.tv[r]);
        if (e != cudaSuccess) return e;
    }
    A.bar = P.bar;
    A.kv_ready = P.kv_ready;
    A.stamps = P.stamps;
    A.bar_extra = P.bar_extra;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_sz[which]);
    cfg.blockDim = dim3(kStepThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    // One CTA per SM and every SM taken: once the preceding kernel's CTAs have
    // left, all of this grid is resident (the grid barriers rely on it; their
    // waits are bounded, so a grid that could not become resident would end
    // with TP_ERR_TIMEOUT, not hang). Programmatic serialization lets CTAs start
    // streaming weights on SMs the preceding step has already left.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_pdl ? 1 : 0;
    void* args[] = {&A};
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace tpk
