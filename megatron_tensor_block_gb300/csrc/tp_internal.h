// Internal declarations shared by the C-ABI layer (tp_api.cu) and the kernel
// translation units. Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "tp_block.h"

namespace tpk {

constexpr int kTileRows = 64;     // output rows per skinny-GEMM work unit
constexpr int kTMax = 8;          // tokens per decode step handled in one pass
constexpr int kKStep = 64;        // reduction elements per warp step
constexpr int kSMs = 152;         // GB300 streaming multiprocessors
constexpr int kAttnChunk = 256;   // keys per split-KV work unit (fp32 decode)
constexpr int kStepChunk = 128;   // keys per split-KV work unit of the one-launch bf16 decode step
constexpr int kPartStride = kTileRows * kTMax + kTMax;   // floats per unit partial
constexpr int kMaxKcTma = 512;
constexpr int kMaxGroupUnits = 16;  // partials reduced by one finisher (register-resident)    // reduction chunk bound of the tensor-map projection kernel

// Shape of one skinny-GEMM launch: `groups` output tiles, each reduced from
// `units_per_group` work units (`shards_per_group` shards x `chunks` chunks).
struct GemvShape {
    int groups = 0;
    int shards_per_group = 1;
    int chunks = 1;
    int kc = 0;                 // reduction elements per unit
#ifdef __CUDACC__
    __host__ __device__
#endif
    int units() const { return groups * shards_per_group * chunks; }
#ifdef __CUDACC__
    __host__ __device__
#endif
    int units_per_group() const { return shards_per_group * chunks; }
};

enum Epi : int { EPI_QKV_ROPE = 0, EPI_SWIGLU = 1, EPI_ROWPAR = 2 };

// Parameters of one skinny-GEMM launch (decode projections). One struct for
// all epilogues; fields an epilogue does not use are ignored.
struct GemvParams {
    const void* W[TP_MAX_SHARDS];      // per-shard weight [rows, K]
    int n_shards;
    int rows;                          // rows per shard (column-par) or H (row-par)
    int K;                             // reduction length per shard
    int T;                             // tokens (<= kTMax)
    GemvShape shape;
    // activation: normalised input (column-parallel) ...
    const float* x;                    // [T, K] float32 (residual stream)
    const float* gamma[TP_MAX_SHARDS]; // per-shard replicated norm weight [K]
    float eps;
    // ... or per-shard activation (row-parallel), storage type of W
    const void* act[TP_MAX_SHARDS];    // [T, K]
    // workspace
    float* part;                       // [units][kPartStride]
    unsigned* cnt;                     // [groups]
    int* status;
    // EPI_QKV_ROPE
    const float* bias[TP_MAX_SHARDS];  // [rows] or NULL
    float* q_out;                      // [N][T][Hq' d]
    void* kcache[TP_MAX_SHARDS];
    void* vcache[TP_MAX_SHARDS];
    const int* pos;                    // [B]
    int hq_s, hkv_s, head_dim, max_kv;
    double log2_theta;
    // EPI_SWIGLU
    void* act_out;                     // [N][T][F']
    int ffn_s;
    // EPI_ROWPAR
    const float* resid;                // [T][rows]
    float* y;                          // [T][rows]
    // tensor-map (bf16) kernel: activations arrive through the copy pipeline
    const void* xact;                  // [N * kTMax][K] bf16 operand rows (shard r at row r*kTMax)
    const float* ss_in;                // QKV: [kTMax] sums of squares of x
    const float* ss_tiles;             // gate/up: [n_ss_tiles][kTMax] partial sums of squares of h
    int n_ss_tiles;
    void* norm_out;                    // o_proj: [N][kTMax][H] bf16(h * gamma_ffn_r), or NULL
    float* ss_tiles_out;               // o_proj: [H / 8][kTMax] per-8-row sums of squares
    const float* gamma2[TP_MAX_SHARDS];
    int whole_tiles;                   // one-launch step, row-parallel: each CTA takes every shard of its output tiles
    // one-launch step, row-parallel tiles split over CTAs: pieces as (value, epoch)
    // pairs [segments][chunks][kTileRows * kTMax], polled by the tile's combiner; or NULL
    unsigned long long* pairs;
    // one-launch step, QKV: the rotated queries also as (value, epoch) pairs [N][kTMax][Hq' d],
    // polled by the attention phase instead of a grid barrier; or NULL
    unsigned long long* q_pairs;
};

// RMSNorm operand preparation: xg[r][t][k] = bf16(x[t][k] * gamma_r[k]),
// ss[t] = sum_k x[t][k]^2 (rows t >= T are zero).
struct NormPrepParams {
    const float* x;
    const float* gamma[TP_MAX_SHARDS];
    int N, T, H;
    void* xg;
    float* ss;
};

struct AttnDecodeParams {
    const float* q;                    // [N][T][Hq' d] rotated queries
    const void* kcache[TP_MAX_SHARDS]; // [Bmax][Hkv'][max_kv][d]
    const void* vcache[TP_MAX_SHARDS];
    const int* pos;                    // [B]
    int N, B, hq_s, hkv_s, d, max_kv, max_batch, n_chunks;
    float scale;                       // 1/sqrt(d)
    float* part;                       // [groups][n_chunks][G*(d+2)]
    unsigned* cnt;                     // [groups]
    void* out;                         // [N][kTMax][Hq' d] storage type
    int* status;
    unsigned part_units;               // capacity of `part` in chunk partials
    int key_busy;                      // one-launch step: CTAs 0..key_busy-1 hold a QKV tile (the rest take a
                                       // larger attention key share, prefetched into L2 during QKV)
    const unsigned long long* q_pairs; // one-launch step: q as (value, epoch) pairs [N][kTMax][Hq' d]
};

struct CopyDesc {
    const void* src;    // NULL: fill zeros
    void* dst;
    int64_t rows;
    int64_t row_bytes;
    int64_t src_pitch;  // bytes
    int64_t dst_pitch;  // bytes
};
constexpr int kMaxCopyDescs = 48;
struct CopyBatch {
    CopyDesc d[kMaxCopyDescs];
    int n;
};

// Expert-sliced MoE feed-forward block (bf16), slots = (token, choice) pairs.
struct MoeParams {
    int N, T, H, E, top_k, Fs;             // Fs: expert FFN width per shard
    int El, ep;                            // experts per shard (E, or E/N with expert parallelism); ep: 1 when
                                           // shard r holds the whole experts [r*El, (r+1)*El)
    float eps;
    const float* x;                        // [T][H]
    const float* logits;                   // [T][E]
    const float* gamma[TP_MAX_SHARDS];     // [H] per shard
    const void* egu[TP_MAX_SHARDS];        // [El][2Fs][H]: gate rows then up rows per expert
    const void* ed[TP_MAX_SHARDS];         // [El][H][Fs]
    int* ids;                              // [T*k] chosen experts, descending logit
    float* wts;                            // [T*k] renormalised routing weights
    int* offsets;                          // [E+1] bucket starts (slot order)
    int* perm;                             // [T*k] slot -> flat choice index t*k + j
    int* slot_of;                          // [T*k] flat choice index -> slot
    float* rinv;                           // [T*k] 1/rms of each slot's token
    void* xs;                              // [xs_copies][T*k][H] bf16: x_t * gamma_r in slot order
    int xs_copies;                         // 1 when every shard points at the same gamma, else N
    void* act;                             // [N][T*k][Fs] bf16: SwiGLU outputs per slot
    float* o;                              // [N][T*k][H] expert outputs per slot
    float* y;                              // [T][H]
    int* status;
};
// marks: optional events recorded before routing, after the routing kernels,
// after each expert GEMM and after the combine (n_marks <= 5)
cudaError_t launch_moe(const MoeParams& p, cudaStream_t s, cudaEvent_t const* marks = nullptr, int n_marks = 0);

// 2-D bf16 tensor map [rows, inner] with boxes box_inner x box_rows (cached).
cudaError_t tensor_map_2d(const void* base, long inner, long rows, int box_inner, int box_rows, int swizzle128,
                          CUtensorMap* out);
cudaError_t tensor_map_3d(const void* base, long d0, long d1, long d2, int box0, int box1, int swizzle128,
                          CUtensorMap* out);
// Streaming-GEMV stage boxes: [rows][K] bf16 as [rows][K/64][64], boxes of
// box_rows rows x 256 columns, 128-byte swizzled (cached). K % 64 == 0.
cudaError_t step_stage_map(const void* W, int K, int rows, int box_rows, CUtensorMap* out);

// tcgen05 GEMM, C[M, N] (fp32) = A[M, K] * B[N, K]^T (bf16, K-major),
// M % 128 == 0, N % 256 == 0, K % 64 == 0.
cudaError_t launch_tc_gemm_plain(const void* A, const void* B, float* C, int M, int N, int K, int* status,
                                 cudaStream_t s, bool b_kn = false);

// Prefill (tcgen05) projections and attention.
struct PrefillColParams {
    const void* A;                        // normalised activations [a_copies][T, K] bf16
    int a_copies;                         // 1: every shard reads copy 0; N: shard r reads copy r
    const void* W[TP_MAX_SHARDS];         // QKV: [qkv_rows, K]; gate/up: [2F', K]
    int N, T, K, rows, S;
    int hq_s, hkv_s, d, max_kv, ffn_s;
    const float* bias[TP_MAX_SHARDS];
    const int* pos;
    const float2* rope;
    void* q_out;                          // [N][T][hq_s d] bf16
    void* kcache[TP_MAX_SHARDS];
    void* vcache[TP_MAX_SHARDS];
    void* act;                            // [N][T][F'] bf16
    int* status;
};
struct PrefillRowParams {
    const void* A;                        // [N][T][Kr] bf16 (shard activations stacked)
    const void* W[TP_MAX_SHARDS];         // [H, Kr] bf16
    int N, T, Kr, H;
    const float* resid;
    float* out;
    int* status;
};
struct FlashParams {
    const void* q;
    void* kcache[TP_MAX_SHARDS];
    void* vcache[TP_MAX_SHARDS];
    void* out;
    const int* pos;
    int N, B, S, T, hq_s, hkv_s, max_kv, d;   // d: head_dim, 64 or 128
    int max_batch;                        // cache extent: groups = max_batch * hkv_s
    float scale;
    int* status;
};
// bf16 RMSNorm of x [T, H]: n_copies outputs (one per gamma), copy c at out + c*T*H
cudaError_t launch_prefill_norm(const float* x, const float* const* gammas, int n_copies, void* out, int T, int H,
                                float eps, cudaStream_t s);
cudaError_t launch_rope_table(float2* tab, int max_pos, int d, double log2_theta, cudaStream_t s);
cudaError_t launch_tc_col(int mode, const PrefillColParams& p, cudaStream_t s);   // 0: QKV, 1: gate/up
cudaError_t launch_tc_row(const PrefillRowParams& p, cudaStream_t s);
cudaError_t launch_flash_prefill(const FlashParams& p, cudaStream_t s);

// The whole bf16 decode step in one persistent cooperative launch.
struct DecodeStepParams {
    GemvParams g[4];                      // qkv, o, gate_up, down (as for the separate launches)
    AttnDecodeParams a;
    NormPrepParams np;
    unsigned long long* bar;              // grid-barrier arrival counter in the workspace (zero-initialised)
    unsigned long long* kv_ready;         // arrivals after the QKV phase (new K/V rows written), zero-initialised
    unsigned long long* stamps;           // optional per-CTA phase end times
    unsigned bar_extra;                   // test hook: arrivals every grid barrier waits for beyond the grid (0)
};
cudaError_t launch_decode_step(const DecodeStepParams& p, cudaStream_t s);
constexpr int kMaxStepCtas = 256;        // stamp rows reserved in the workspace
constexpr int kStepMinKeys = 128;        // smallest key range per CTA in the step's attention phase
// Key range per CTA at least kStepMinKeys and large enough that a KV group of
// max_kv keys is split over at most 32 CTAs.
#ifdef __CUDACC__
__host__ __device__
#endif
inline int step_min_keys(int max_kv) {
    const int m = (max_kv + 30) / 31;
    return m > kStepMinKeys ? m : kStepMinKeys;
}
constexpr int kStepStamps = 13;          // per CTA: start, then per phase: streaming done, arrival (or end)

// Several decode blocks in one persistent launch: every CTA streams its own
// weight and KV tiles for all layers through a ring of 16 KB slots, and the
// activations between phases travel as (value, epoch) pairs so a consumer
// polls the data itself instead of a grid barrier.
constexpr int kChainThreads = 384;       // eight consumer warps, then a warpgroup holding the producer warp
constexpr int kChainSlot = 16384;        // bytes per ring slot
constexpr int kChainMaxSlots = 12;
constexpr int kChainMaxItems = 40;       // items of one projection phase per CTA
constexpr int kChainMaxCtas = 160;
constexpr int kChainMaps = 6;            // per layer and shard: wqkv, wo, wgu, wd, K cache, V cache
struct ChainLayer {
    const float* bqkv[TP_MAX_SHARDS];    // QKV bias or null
    const float* g_attn[TP_MAX_SHARDS];
    const float* g_ffn[TP_MAX_SHARDS];
    void* kc[TP_MAX_SHARDS];             // [max_batch][hkv_s][max_kv][d] bf16
    void* vc[TP_MAX_SHARDS];
};
struct ChainArgs {
    int H, N, hq_s, hkv_s, d, G, qkv_rows, F_s, T, max_batch, max_kv, L, grid;
    int ck;                              // keys per attention tile (16 KB of K)
    int n_slots;
    int kc[4];                           // chunks of 64 columns per box: qkv, o, gate/up (each half), down
    int nl[4];                           // loads per 8-row item and shard: qkv, o, gate/up, down
    float eps, log2_theta, qscale;       // qscale = log2(e) / sqrt(d)
    const CUtensorMap* maps;             // [L][kChainMaps][N], 64-byte aligned, device memory
    const ChainLayer* layers;            // [L], device memory
    const int* tab;                      // per projection phase p: starts [grid + 1] at tab_off[p], items after
    int tab_off[4];
    const int* att_rank;                 // [grid]: the CTA's place in the attention round robin
    const float* x;                      // [T][H] input of layer 0
    float* y;                            // [T][H] output of the last layer
    const int* pos;                      // [T]
    const float2* rope;                  // [max_kv][d/2]: (cos, sin) of pos * theta^(-2e/d)
    const unsigned long long* cbase;     // start of the pair buffers (polling offsets are relative to it)
    unsigned long long* fx;              // [max_batch][H] layer inputs (layers 1..)
    unsigned long long* fq;              // [N][max_batch][qkv_rows] projections before rotation
    unsigned long long* fp;              // [N * max_batch * hkv_s][maxch][G (d + 2)] attention partials:
                                         // output [G][d / 2] (unnormalised, two bf16 values a pair), then
                                         // (max, sum) per head
    unsigned long long* fh;              // [max_batch][H] residual stream after attention
    unsigned long long* fa;              // [max_batch][N][F_s / 2] SwiGLU outputs, two bf16 values a pair
    int maxch;
    unsigned* gen;                       // launch counter (epochs) and CTAs finished
    unsigned* done;
    int* gabort;
    int* status;
    unsigned long long* stamps;          // optional [grid][L][5 phases][inputs arrived, outputs stored] (ns)
    int xa_stride;                       // bf16 elements per token row of the operand buffer
    int sm_misc, sm_xin, sm_xa, sm_gam, sm_att, sm_stage, sm_qs, sm_res, sm_part, sm_carry,
        sm_ring;                         // shared-memory offsets
};
// Fills the shared-memory offsets of `a` (N, max_batch, H, xa_stride, d,
// n_slots set) and returns the dynamic shared-memory bytes of a launch.
size_t chain_smem(ChainArgs& a);
cudaError_t launch_chain(const ChainArgs& a, size_t smem, cudaStream_t s);
// 3-D bf16 map over a [rows][K] matrix viewed as [rows][K/64][64], boxes of
// {64, kc, box_rows}, 128-byte swizzled, written to `out` (any memory).
cudaError_t chain_map(const void* W, long K, long rows, int kc, int box_rows, CUtensorMap* out);

// Logits of the final hidden state over the vocab-parallel head (bf16 rows of
// every shard stacked in rank order; rows >= org_vocab are padding, not written).
constexpr int kHeadThreads = 288;        // eight consumer warps + a copy-issuing warp
constexpr int kHeadMaxStages = 16;
struct HeadArgs {
    const void* W[TP_MAX_SHARDS];        // [rows_s][H] bf16 per shard
    int N, rows_s, org_vocab, H, T, grid;
    long rpc;                            // rows per CTA (a multiple of rs)
    int rs, ns, ring_off, cps;           // rows per stage, stages, ring offset in shared memory, CTAs per SM
    const float* x;                      // [T][H]
    const float* gamma;                  // [H]
    float eps;
    float* logits;                       // [T][org_vocab]
    int* status;                         // nullable
};
// Picks the stage geometry of `a` (H set) for smem_max bytes; returns the launch's shared-memory bytes.
size_t head_smem(HeadArgs& a, int smem_max);
cudaError_t launch_lm_head(const HeadArgs& a, size_t smem, cudaStream_t s);

// launchers (return the launch's cudaError_t)
cudaError_t launch_gemv(const GemvParams& p, int epi, int dtype, cudaStream_t s);
void set_pdl(bool on);   // programmatic dependent launch between the kernels of a call (default on)
// Launch with the programmatic-stream-serialisation attribute (unless switched off).
cudaError_t launch_pdl(const void* fn, void** args, int grid, size_t smem, cudaStream_t s, int threads);
cudaError_t launch_attn_decode(const AttnDecodeParams& p, int dtype, cudaStream_t s);
cudaError_t launch_copy_batch(const CopyBatch& b, cudaStream_t s);
cudaError_t launch_reduce_partials(const float* partials, const float* resid, const float* bias,
                                   float* out, int N, int64_t M, int64_t H, cudaStream_t s);

}  // namespace tpk
