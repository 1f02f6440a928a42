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
#include "common.cuh"
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

template <typename TW, int EPI>
__global__ void __launch_bounds__(256) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
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

    // ---- cross-unit reduction: chunks in order, then ranks in order
    if (upg > 1) {
        float* mine = p.part + (size_t)u * kPartStride;
        for (int i = tid; i < kTileRows * kTMax; i += blockDim.x) mine[i] = tile[i];
        if (EPI != EPI_ROWPAR && tid < kTMax) mine[kTileRows * kTMax + tid] = ss[tid];
        if (!arrive_last(&p.cnt[gi], (unsigned)upg)) return;
        const float* base = p.part + (size_t)gi * upg * kPartStride;
        const int C = p.shape.chunks;
        const int nrank = (EPI == EPI_ROWPAR) ? p.shape.shards_per_group : 1;
        for (int i = tid; i < kPartStride; i += blockDim.x) {
            if (EPI == EPI_ROWPAR && i >= kTileRows * kTMax) break;
            float total = 0.f;
            for (int rr = 0; rr < nrank; ++rr) {
                float pr = __ldcg(base + (size_t)(rr * C) * kPartStride + i);
                for (int cc = 1; cc < C; ++cc) pr += __ldcg(base + (size_t)(rr * C + cc) * kPartStride + i);
                total = (rr == 0) ? pr : total + pr;
            }
            if (i < kTileRows * kTMax) tile[i] = total; else ss[i - kTileRows * kTMax] = total;
        }
        __syncthreads();
    }

    // ---- epilogues
    if (EPI == EPI_ROWPAR) {
        for (int i = tid; i < kTileRows * T; i += blockDim.x) {
            const int t = i / kTileRows, j = i - t * kTileRows;
            const size_t o = (size_t)t * p.rows + tb * kTileRows + j;
            p.y[o] = p.resid[o] + tile[j * kTMax + t];
        }
        return;
    }
    const float inv_k = 1.0f / (float)p.K;
    if (EPI == EPI_SWIGLU) {
        TW* out = reinterpret_cast<TW*>(p.act_out);
        for (int i = tid; i < 32 * T; i += blockDim.x) {
            const int t = i >> 5, j = i & 31;
            const float rinv = 1.0f / sqrtf(ss[t] * inv_k + p.eps);
            const float gt = tile[j * kTMax + t] * rinv;
            const float up = tile[(j + 32) * kTMax + t] * rinv;
            const float a = gt / (1.0f + expf(-gt)) * up;
            Stor<TW>::store(out + ((size_t)r * T + t) * p.ffn_s + tb * 32 + j, a);
        }
        return;
    }
    // EPI_QKV_ROPE (decode: token t is sequence b = t at position pos[t])
    const int d = p.head_dim, half = d >> 1;
    for (int i = tid; i < 32 * T; i += blockDim.x) {
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
            const double inv_freq = exp2(-(2.0 * ii / d) * p.log2_theta);
            double sn, cs;
            sincos((double)pos * inv_freq, &sn, &cs);
            const float c = (float)cs, s = (float)sn;
            const float ra = va * c - vb * s, rb = va * s + vb * c;
            va = ra;
            vb = rb;
        }
        if (head < p.hq_s) {
            float* q = p.q_out + ((size_t)r * T + t) * p.hq_s * d + head * d + ii;
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
    extern __shared__ __align__(16) unsigned char smem[];
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

    const size_t qoff = ((size_t)r * T + b) * p.hq_s * D + (size_t)kh * G * D;
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

cudaError_t launch_gemv(const GemvParams& p, int epi, int dtype, cudaStream_t s) {
    if (dtype == TP_BF16) {
        if (epi == EPI_QKV_ROPE) return launch_gemv_t<bf16, EPI_QKV_ROPE>(p, s);
        if (epi == EPI_SWIGLU) return launch_gemv_t<bf16, EPI_SWIGLU>(p, s);
        return launch_gemv_t<bf16, EPI_ROWPAR>(p, s);
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

cudaError_t launch_attn_decode(const AttnDecodeParams& p, int dtype, cudaStream_t s) {
    if (dtype == TP_BF16) return p.d == 64 ? launch_attn_t<bf16, 64>(p, s) : launch_attn_t<bf16, 128>(p, s);
    return p.d == 64 ? launch_attn_t<float, 64>(p, s) : launch_attn_t<float, 128>(p, s);
}

}  // namespace tpk
