/*
 * tp_block.h -- C ABI of the Megatron column/row tensor-parallel block with
 * N logical shards on one GPU (sm_103a).
 *
 * Sources, by page title and section:
 *  [RT]  "feat: multi-GPU tensor-parallel runtime with per-rank device
 *        placement and cross-GPU collectives": Problem (ranks run on one
 *        device and their partial outputs are summed locally), Design /
 *        Forward execution (replicated residual stream; reductions after
 *        o_proj and after down_proj), Collective backend abstraction
 *        (copy-and-reduce), Acceptance criteria (clear errors, no silent
 *        wrong results).
 *  [GA]  "Gather tensor-parallel sharded parameters on read in a trace":
 *        Change (shard-dim rule, replicated tensors, vocab padding dropped to
 *        org_vocab_size, fused rows grouped by rank, gathered tensor is a
 *        copy).
 *  [MG]  "Multi-GPU & Multi-Node": How tensor parallelism works (steps 1-3,
 *        replicated norms), Supported architectures (expert slicing, or
 *        expert parallelism, with a replicated router), Requirements &
 *        constraints (divisibility).
 *
 * Conventions for every call:
 *  - All tensor arguments are plain pointers to DEVICE memory on the current
 *    CUDA device unless stated otherwise; the caller owns them. No call keeps
 *    a pointer after it returns, and no call frees caller memory.
 *  - Matrices are row-major [out, in] (y = x @ W^T). Storage type of weight
 *    matrices and KV caches is the plan's dtype; 1-D parameters (norm gamma,
 *    biases), hidden states, router logits and partial sums are float32.
 *  - `stream` is a cudaStream_t passed as void* (NULL: legacy default
 *    stream). Calls that launch work are asynchronous on that stream.
 *  - Every call validates its arguments on the host before any launch and
 *    returns TP_OK (0) or a negative tp_status; nothing aborts, prints or
 *    falls back to the CPU. tp_last_error() gives a message for the last
 *    failing call on the calling thread.
 *  - Launching calls require the current device to be compute capability
 *    10.3 (sm_103a); otherwise they return TP_ERR_UNSUPPORTED.
 */
#ifndef TP_BLOCK_H
#define TP_BLOCK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TP_MAX_SHARDS 8
#define TP_ABI_VERSION 1

typedef enum tp_status {
    TP_OK = 0,
    TP_ERR_INVALID_ARG = -1,   /* bad size, mode or enum value */
    TP_ERR_INDIVISIBLE = -2,   /* heads / kv heads / FFN not divisible by tp */
    TP_ERR_UNSUPPORTED = -3,   /* device is not sm_103, or shape outside the kernels' range */
    TP_ERR_NULL = -4,          /* a required pointer is NULL */
    TP_ERR_ALIGN = -5,         /* a pointer is not 16-byte aligned */
    TP_ERR_SHAPE = -6,         /* sizes inconsistent with the plan */
    TP_ERR_CAPACITY = -7,      /* position + new tokens exceeds max_kv, or workspace too small */
    TP_ERR_CUDA = -8,          /* a CUDA runtime call or launch failed */
    TP_ERR_TIMEOUT = -9        /* a bounded device-side wait gave up */
} tp_status;

typedef enum tp_dtype { TP_F32 = 0, TP_BF16 = 1 } tp_dtype;

typedef enum tp_mode {
    TP_MODE_DECODE = 0,   /* one new token per sequence at pos[b] */
    TP_MODE_PREFILL = 1,  /* T_per_seq new tokens per sequence at pos[b].. (causal) */
    TP_MODE_MOE_FFN = 2   /* feed-forward half only, MoE (sliced or expert-parallel, per the plan) */
} tp_mode;

/* Kinds of sharded parameter ([GA] Change): which dim is split and how the
 * gather reassembles it. */
typedef enum tp_param_kind {
    TP_PARAM_REPLICATED = 0,      /* no shard stamp: every shard holds the whole tensor */
    TP_PARAM_COLWISE = 1,         /* column-parallel: output dim (dim 0) split */
    TP_PARAM_ROWWISE = 2,         /* row-parallel: input dim (dim 1) split */
    TP_PARAM_FUSED_QKV = 3,       /* [q_r; k_r; v_r] per shard; gathers rank-grouped */
    TP_PARAM_FUSED_GATE_UP = 4,   /* [gate_r; up_r] per shard; gathers rank-grouped */
    TP_PARAM_PACKED_COLWISE = 5,  /* any stacked segments, per-shard slices stacked */
    TP_PARAM_VOCAB_PARALLEL = 6   /* rows padded to a multiple of 64*tp, split; gather cuts to org_vocab */
} tp_param_kind;

/* Shape of one block. Attention fields may be 0 for an MoE-only block
 * (TP_MODE_MOE_FFN); expert fields are 0 for a dense block. */
typedef struct tp_model_desc {
    int64_t hidden;        /* H */
    int64_t n_heads;       /* Hq */
    int64_t n_kv_heads;    /* Hkv */
    int64_t head_dim;      /* d */
    int64_t ffn;           /* F (dense SwiGLU intermediate) */
    int64_t n_experts;     /* E (0: dense) */
    int64_t top_k;         /* experts per token */
    int64_t expert_ffn;    /* Fe */
    int64_t org_vocab;     /* lm_head rows before padding (0: no head) */
    double eps;            /* RMSNorm epsilon */
    double rope_theta;     /* rotary base */
    int32_t dtype;         /* tp_dtype of weight matrices and KV caches */
    int32_t has_qkv_bias;  /* 1: q/k/v biases present */
    int64_t max_batch;     /* sequences per call */
    int64_t max_tokens;    /* B * T_per_seq per call */
    int64_t max_kv;        /* KV cache capacity (positions) per sequence */
    int32_t expert_parallel; /* MoE sharding: 0 expert slicing (every shard holds 1/tp of every expert's
                              * FFN width), 1 expert parallelism (shard r holds the whole experts
                              * [r*E/tp, (r+1)*E/tp); E must divide by tp) */
    int32_t reserved0;       /* must be 0 */
} tp_model_desc;

typedef struct tp_plan_s* tp_plan_t;

/* Sizes derived by tp_plan. Row counts are per shard; *_bytes are per shard. */
typedef struct tp_plan_info {
    int32_t tp;
    int32_t reduce_points;       /* row-parallel reductions per block: 2 dense, 1 MoE-only */
    int64_t hq_shard;            /* Hq' = Hq/tp */
    int64_t hkv_shard;           /* Hkv' */
    int64_t ffn_shard;           /* F' */
    int64_t expert_ffn_shard;    /* Fe' (Fe/tp when sliced, Fe with expert parallelism) */
    int64_t qkv_rows;            /* (Hq' + 2 Hkv') d */
    int64_t vocab_padded;        /* org_vocab rounded up to a multiple of 64*tp */
    int64_t vocab_rows_shard;    /* vocab_padded / tp */
    int64_t wqkv_bytes, bqkv_bytes, wo_bytes, wgu_bytes, wd_bytes, gamma_bytes;
    int64_t egu_bytes, ed_bytes;
    int64_t kv_cache_bytes;      /* one of K or V: [max_batch][Hkv'][max_kv][d] */
    int64_t lm_head_bytes;       /* [vocab_rows_shard][H] */
    int64_t workspace_bytes;     /* scratch for tp_block_forward, any mode */
    int64_t weight_bytes_shard;  /* all matrices of one shard */
    int64_t weight_bytes_total;  /* all shards */
    /* MoE routing tables inside the workspace (byte offsets, for inspection
     * after a MOE_FFN call): chosen expert ids int32 [T*top_k], bucket starts
     * int32 [E+1], slot -> choice index int32 [T*top_k]. -1 without experts. */
    int64_t moe_ids_offset, moe_bucket_offset, moe_perm_offset;
    int64_t experts_shard;       /* experts held per shard: E sliced, E/tp with expert parallelism */
    int64_t noalloc_scratch_bytes; /* bytes of the static array a DECODE call of
                                  * tp_block_forward_noalloc uses (0 without an
                                  * attention block); must be <= TP_NOALLOC_SCRATCH_BYTES */
} tp_plan_info;

/* Full (unsharded) block weights, caller-owned device memory. */
typedef struct tp_block_weights {
    const void* wq;          /* [Hq d, H] */
    const void* wk;          /* [Hkv d, H] */
    const void* wv;          /* [Hkv d, H] */
    const float* bq;         /* [Hq d] or NULL */
    const float* bk;         /* [Hkv d] or NULL */
    const float* bv;         /* [Hkv d] or NULL */
    const void* wo;          /* [H, Hq d] */
    const void* w_gate;      /* [F, H] */
    const void* w_up;        /* [F, H] */
    const void* w_down;      /* [H, F] */
    const float* gamma_attn; /* [H] */
    const float* gamma_ffn;  /* [H] */
    const void* e_gate;      /* [E, Fe, H] */
    const void* e_up;        /* [E, Fe, H] */
    const void* e_down;      /* [E, H, Fe] */
} tp_block_weights;

/* Per-shard tensors, caller-allocated with the sizes in tp_plan_info. */
typedef struct tp_shard_set {
    void* wqkv[TP_MAX_SHARDS];        /* [qkv_rows, H]: rows q_r, then k_r, then v_r */
    float* bqkv[TP_MAX_SHARDS];       /* [qkv_rows] or NULL */
    void* wo[TP_MAX_SHARDS];          /* [H, Hq' d]: columns r*Hq'd.. of o_proj */
    void* wgu[TP_MAX_SHARDS];         /* [2F', H]: gate_r rows then up_r rows */
    void* wd[TP_MAX_SHARDS];          /* [H, F']: columns r*F'.. of down_proj */
    float* gamma_attn[TP_MAX_SHARDS]; /* [H] replicated copy */
    float* gamma_ffn[TP_MAX_SHARDS];  /* [H] replicated copy */
    void* egu[TP_MAX_SHARDS];         /* [E, 2Fe', H]: per expert gate_r then up_r rows; expert
                                       * parallel: [E/tp, 2Fe, H], experts r*E/tp.. whole */
    void* ed[TP_MAX_SHARDS];          /* [E, H, Fe']: per expert columns r*Fe'.. of down; expert
                                       * parallel: [E/tp, H, Fe] */
} tp_shard_set;

/* Per-shard KV caches: shard r owns KV heads [r Hkv', (r+1) Hkv').
 * Layout [max_batch][Hkv'][max_kv][d] in the plan dtype; keys are stored
 * after the rotary embedding. */
typedef struct tp_kv_set {
    void* k[TP_MAX_SHARDS];
    void* v[TP_MAX_SHARDS];
} tp_kv_set;

/* ---------------------------------------------------------------- plan */

/* Validates `d` for `tp` logical shards and builds a host-only plan
 * ([MG] Requirements & constraints: heads, KV heads and the FFN width must
 * divide by the degree; [RT] Design: the reduction points after o_proj and
 * down_proj). Makes no CUDA call. The plan is owned by the caller and freed
 * with tp_plan_destroy.
 * Errors: TP_ERR_NULL (d or out NULL), TP_ERR_INVALID_ARG (tp outside
 * 1..TP_MAX_SHARDS, non-positive sizes, Hq % Hkv != 0, unknown dtype),
 * TP_ERR_INDIVISIBLE (Hq, Hkv, F or Fe not divisible by tp),
 * TP_ERR_UNSUPPORTED (sizes outside what the kernels handle: head_dim not 64
 * or 128, H or per-shard widths not multiples of 64). */
tp_status tp_plan(const tp_model_desc* d, int32_t tp, tp_plan_t* out);

/* Frees a plan. NULL is accepted. */
void tp_plan_destroy(tp_plan_t plan);

/* Copies the derived sizes into `out` (host memory). */
tp_status tp_plan_get_info(tp_plan_t plan, tp_plan_info* out);

/* Writes a one-line text description (per-shard bytes and shapes, showing
 * that each shard holds about 1/tp of the weights, [RT] Acceptance
 * criteria) into `buf` (host, `n` bytes, NUL-terminated, truncated). */
tp_status tp_plan_describe(tp_plan_t plan, char* buf, size_t n);

/* ----------------------------------------------------- shard and gather */

/* Builds every shard's tensors from the full block weights ([MG] How tensor
 * parallelism works: QKV and gate/up split their output dim, o_proj and
 * down_proj their input dim; norms replicated; [MG] Supported architectures:
 * each shard holds 1/tp of every expert, or with expert_parallel the whole
 * experts r*E/tp .. (r+1)*E/tp - 1). Bit-exact copies, asynchronous on
 * `stream`. Pointers in `full` that the block does not use may be NULL.
 * Errors: TP_ERR_NULL, TP_ERR_ALIGN (matrix pointers must be 16-byte
 * aligned), TP_ERR_UNSUPPORTED, TP_ERR_CUDA. */
tp_status tp_shard_weights(tp_plan_t plan, const tp_block_weights* full,
                           const tp_shard_set* out, void* stream);

/* Shards one tensor of kind `k`. `full` is [rows, cols] of `dtype`
 * (TP_F32 or TP_BF16); `shards_out` is a HOST array of tp device pointers,
 * each sized for one shard. Fused kinds take `segments` (host array of
 * `n_segments` row counts summing to `rows`); for FUSED_QKV and
 * FUSED_GATE_UP a NULL `segments` means the plan's (Hq d, Hkv d, Hkv d) or
 * (F, F). VOCAB_PARALLEL takes rows = org_vocab and writes padding rows of
 * zeros at the tail of the last shard. REPLICATED copies to every shard.
 * Errors: TP_ERR_NULL, TP_ERR_SHAPE (a dim not divisible as required),
 * TP_ERR_INVALID_ARG, TP_ERR_CUDA. */
tp_status tp_shard_param(tp_plan_t plan, int32_t k, const void* full,
                         int64_t rows, int64_t cols, int32_t dtype,
                         const int64_t* segments, int32_t n_segments,
                         void* const* shards_out, void* stream);

/* All-gathers a sharded parameter into `out` ([GA] Change):
 *  REPLICATED: out = shard 0 ([rows, cols]);
 *  COLWISE / FUSED_QKV / FUSED_GATE_UP / PACKED_COLWISE: shards stacked on
 *    dim 0 in rank order ([tp*rows, cols]); fused rows therefore come back
 *    grouped by rank, the layout whose x @ W^T equals the concatenated shard
 *    outputs;
 *  ROWWISE: shards concatenated on dim 1 ([rows, tp*cols]);
 *  VOCAB_PARALLEL: shards stacked, rows >= org_vocab dropped
 *    ([org_vocab, cols]).
 * `shards` is a HOST array of tp device pointers, each [rows, cols] of
 * `dtype`. `out` is caller-allocated at the full size. The result is a copy;
 * the shards are read only. Bit-exact. Uses 16-byte vector copies when rows
 * are 16-byte aligned, element copies otherwise (no error).
 * Errors: TP_ERR_NULL, TP_ERR_SHAPE (e.g. org_vocab > tp*rows),
 * TP_ERR_INVALID_ARG, TP_ERR_CUDA. */
tp_status tp_gather_param(tp_plan_t plan, int32_t k, const void* const* shards,
                          int64_t rows_per_shard, int64_t cols_per_shard,
                          int32_t dtype, void* out, void* stream);

/* Places a full KV cache into the per-shard caches ([MG] How tensor
 * parallelism works, step 2: each shard attends over its own heads' cache;
 * shard r owns KV heads [r Hkv', (r+1) Hkv'), contiguous groups, so every
 * query head's KV head sits on the same shard):
 *   kv->k[r][b][h][p][:] = k_full[b][r Hkv' + h][p][:]   for p < L,
 * and the same for V. k_full and v_full are DEVICE [B][Hkv][L][d] in the
 * plan dtype (keys already rotated); the shard caches are the
 * [max_batch][Hkv'][max_kv][d] buffers of tp_kv_set. Positions >= L and
 * sequences >= B of the shard caches are left as they are. Bit-exact copies,
 * asynchronous on `stream`; the full cache is only read.
 * Errors: TP_ERR_NULL, TP_ERR_INVALID_ARG (no attention block), TP_ERR_SHAPE
 * (B outside 1..max_batch), TP_ERR_CAPACITY (L outside 0..max_kv),
 * TP_ERR_UNSUPPORTED, TP_ERR_CUDA. */
tp_status tp_shard_kv(tp_plan_t plan, const void* k_full, const void* v_full, int64_t B, int64_t L,
                      const tp_kv_set* kv, void* stream);

/* ------------------------------------------------------------- forward */

/* Zeroes the control words (completion counters, status) at the start of a
 * workspace. Call once after allocating a workspace and before its first
 * tp_block_forward; the kernels leave the counters at zero after each
 * call. `bytes` >= tp_plan_info.workspace_bytes. */
tp_status tp_workspace_init(tp_plan_t plan, void* workspace, size_t bytes, void* stream);

/* One tensor-parallel block over all tp logical shards ([MG] How tensor
 * parallelism works, steps 1-3; [RT] Design / Forward execution):
 *   DECODE / PREFILL:  h = x + sum_r Attn_r(RMSNorm(x)) Wo_r^T,
 *                      y = h + sum_r SwiGLU_r(RMSNorm(h)) Wd_r^T,
 *     column-parallel QKV and gate/up per shard, rotate-half RoPE, K/V
 *     appended to each shard's cache at positions pos[b]..pos[b]+T_per_seq-1,
 *     grouped-query attention over the shard's own heads (causal), and the
 *     row-parallel partials summed in rank order (((p0 + p1) + p2) + ...)
 *     in float32 before the residual is added.
 *   MOE_FFN: y = x + sum_r sum_j w_tj SwiGLU_{e_tj, r}(RMSNorm(x)_t), with
 *     softmax top-k routing of `router_logits` ([T, E] float32), ties to the
 *     lower expert id, weights renormalised; j-order then rank-order sums.
 *     With expert_parallel, SwiGLU_{e, r} is the whole expert e on the shard
 *     holding it and 0 on the others.
 * x and y are float32 [B*T_per_seq, H], rows sequence-major, y != x. pos is
 * DEVICE int32 [B]. `workspace` holds `workspace_bytes` >= the plan's
 * workspace_bytes and was set up by tp_workspace_init. Results are
 * deterministic (byte-identical across calls on the same inputs).
 * Positions past max_kv are not written; the kernels record
 * TP_ERR_CAPACITY in the workspace status word (tp_get_device_status).
 * PREFILL runs on bf16 plans only. It normalises once per distinct gamma
 * pointer: shards that point at one replicated gamma tensor share one
 * normalised copy of the activations (same values either way). Its
 * activations between stages are stored as bf16 (normalised inputs, q,
 * attention output, SwiGLU output) and accumulated in float32; the
 * row-parallel partials and the residual stream stay float32.
 * Errors: TP_ERR_NULL, TP_ERR_SHAPE (B or tokens above the plan's maxima,
 * T_per_seq != 1 in DECODE), TP_ERR_CAPACITY (workspace too small,
 * T_per_seq > max_kv), TP_ERR_INVALID_ARG (mode not valid for the plan),
 * TP_ERR_UNSUPPORTED (PREFILL or MOE_FFN on an fp32 plan), TP_ERR_ALIGN,
 * TP_ERR_CUDA. */
tp_status tp_block_forward(tp_plan_t plan, const tp_shard_set* w, const tp_kv_set* kv,
                           const float* x, float* y, const int32_t* pos,
                           int32_t B, int32_t T_per_seq, int32_t mode,
                           const float* router_logits,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Size of the library-owned scratch array used by tp_block_forward_noalloc,
 * per device: 16 MiB. */
#define TP_NOALLOC_SCRATCH_BYTES (16 * 1024 * 1024)

/* DECODE forward (same computation, kernels and results as tp_block_forward
 * with TP_MODE_DECODE, T_per_seq = 1) for callers that cannot allocate
 * device memory: code that runs while a CUDA graph is being captured, where
 * an allocation is not allowed; plug-ins inside a host program that owns all
 * device memory through its own pool; and latency-bound loops that cannot
 * afford the synchronisation an allocation may cause. Instead of a caller
 * workspace it uses one static device array of TP_NOALLOC_SCRATCH_BYTES that
 * each GPU loading this library holds until the process exits. The pages have
 * no counterpart of this entry point; it is an interface convenience.
 *  - The caller still passes every input and output (weights, caches, x, y,
 *    pos, as for tp_block_forward). The call allocates nothing: no cudaMalloc,
 *    no cudaFree, no allocating library routine.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture. Later calls only enqueue work.
 *  - Every call on a device shares the one array, which keeps the last call's
 *    contents. Each call first clears, on `stream`, the control words
 *    (counters, status word, grid-barrier counter) and the buffer of
 *    cross-SM pieces, so nothing an earlier call left is taken as this
 *    call's. Calls whose work overlaps on the GPU (other streams, other host
 *    threads) race on the array and give wrong results: issue them on one
 *    stream, or serialise them.
 *  - The array must hold the plan's whole decode footprint,
 *    tp_plan_info.noalloc_scratch_bytes: control words, decode buffers and
 *    the piece buffer (the Llama-3-8B-shaped block at tp 4, batch 8,
 *    max_kv 2049 needs about 11 MB). Larger plans are rejected with
 *    TP_ERR_CAPACITY before any GPU work. The footprint does not depend on
 *    max_tokens (prefill and MoE buffers are not used here).
 *  - Positions past max_kv are skipped as in tp_block_forward and recorded
 *    as TP_ERR_CAPACITY in the array's status word; a bounded device wait
 *    that gives up records TP_ERR_TIMEOUT there. tp_noalloc_status reads it.
 * Errors: TP_ERR_NULL, TP_ERR_INVALID_ARG (no attention block, y == x),
 * TP_ERR_SHAPE (B outside 1..min(max_batch, 8)), TP_ERR_CAPACITY,
 * TP_ERR_ALIGN, TP_ERR_UNSUPPORTED, TP_ERR_CUDA. */
tp_status tp_block_forward_noalloc(tp_plan_t plan, const tp_shard_set* w, const tp_kv_set* kv,
                                   const float* x, float* y, const int32_t* pos, int32_t B,
                                   void* stream);

/* Reads the status word of the current device's static array (TP_OK, or the
 * first device-detected error of the latest tp_block_forward_noalloc call
 * on this device, which cleared it) into *out (host). Synchronises `stream`;
 * pass the stream of that call. Like the entry point, the first call on a
 * device looks up the array's address. No counterpart on the pages.
 * Errors: TP_ERR_NULL, TP_ERR_UNSUPPORTED, TP_ERR_CUDA. */
tp_status tp_noalloc_status(int32_t* out, void* stream);

/* ------------------------------------------- several decode blocks, one launch */

typedef struct tp_stack_s* tp_stack_t;

/* Prepares DECODE over a stack of n_layers blocks of one plan, layer l with
 * its own shard tensors w[l] and KV caches kv[l] (HOST arrays of n_layers
 * entries of caller-owned device pointers, as for tp_block_forward). Layer
 * l's output is layer l+1's input: the decoder of [MG] How tensor
 * parallelism works, steps 1-3, repeated per layer, with the pages' fused
 * per-rank block graphs ([MG] CUDA graphs; [RT] Design) taken to one launch
 * for all layers. The handle owns a small device buffer (TMA descriptors of
 * every weight and cache, item tables); it reads the pointers, not the
 * data, so weights and caches may change between calls but must not move.
 * Requires a bf16 plan with head_dim 64 or 128, at most 8 query heads per KV
 * head and max_batch <= 8. Allocates (cudaMalloc) and synchronises once.
 * Errors: TP_ERR_NULL, TP_ERR_INVALID_ARG (no attention block, n_layers
 * outside 1..255), TP_ERR_UNSUPPORTED (dtype, shape limits above), TP_ERR_ALIGN,
 * TP_ERR_CUDA. */
tp_status tp_stack_create(tp_plan_t plan, int32_t n_layers, const tp_shard_set* w,
                          const tp_kv_set* kv, tp_stack_t* out);

/* Frees a stack handle and its device buffer. NULL is accepted. */
void tp_stack_destroy(tp_stack_t stack);

/* CTAs of one tp_stack_decode launch (one per SM, at most 160); 0 for NULL. */
int32_t tp_stack_ctas(tp_stack_t stack);

/* Measurement hook: while set, every tp_stack_decode launch writes
 * %globaltimer nanoseconds into `stamps` (DEVICE uint64, rows x n_layers x
 * 5 x 2, caller-owned and zeroed by the caller): for CTA c, layer l and
 * phase p (0 QKV, 1 attention, 2 o_proj, 3 gate/up, 4 down) the time the
 * phase's inputs had arrived and the time its last output was stored.
 * Phases in which a CTA has no work keep their entries. rows >= the
 * stack's CTA count; NULL clears the hook.
 * Errors: TP_ERR_NULL (stack), TP_ERR_SHAPE (rows too small). */
tp_status tp_stack_set_stamps(tp_stack_t stack, uint64_t* stamps, int32_t rows);

/* One decode token per sequence through every layer of the stack: the same
 * values as n_layers calls of tp_block_forward (DECODE, T_per_seq = 1)
 * chained through the layers, up to float32 summation order and the bf16
 * rounding of the projection operands; K/V rows of every layer appended at
 * pos[b]. x and y are float32 [B, H] (16-byte aligned, y != x); pos is DEVICE
 * int32 [B], the same for every layer. `workspace` is a tp_workspace_init'ed
 * workspace of at least the plan's workspace_bytes (its own region of it:
 * the call may share a workspace with the other modes, but calls on one
 * workspace must not overlap on the GPU). One kernel launch, no allocation:
 * the call may be captured in a CUDA graph. A device-side wait that gives up
 * (1 s) records TP_ERR_TIMEOUT in the status word; a position outside
 * 0..max_kv-1 records TP_ERR_CAPACITY and is not written.
 * Errors: TP_ERR_NULL, TP_ERR_INVALID_ARG, TP_ERR_SHAPE (B outside
 * 1..min(max_batch, 8)), TP_ERR_CAPACITY (workspace too small), TP_ERR_ALIGN,
 * TP_ERR_CUDA. */
tp_status tp_stack_decode(tp_stack_t stack, const float* x, float* y, const int32_t* pos, int32_t B,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Logits of the final hidden state over the vocab-parallel head ([GA] Change:
 * the head split by vocabulary rows, padded to a multiple of 64*tp with the
 * padding at the tail of the last shard, padding dropped on gather; [MG] How
 * tensor parallelism works: the norm before it replicated):
 *   logits[t][v] = RMSNorm(x[t]) . W[v],   v < org_vocab,
 * with RMSNorm(x) = x / sqrt(mean(x^2) + eps) * gamma and W the shards
 * stacked in rank order. Each shard's rows give its column-parallel logits;
 * writing only v < org_vocab is the gather (padding never reaches `logits`).
 * head_shards: HOST array of tp device pointers, each [vocab_rows_shard, H]
 * bf16 (as tp_shard_param with TP_PARAM_VOCAB_PARALLEL writes them). gamma
 * float32 [H], x float32 [T, H], logits float32 [T, org_vocab], all device,
 * 16-byte aligned. The norm's operand x * gamma is rounded to bf16 for the
 * products, which accumulate in float32. `device_status` (nullable, device
 * int32) receives TP_ERR_TIMEOUT if a bounded wait gives up. One launch.
 * Errors: TP_ERR_NULL, TP_ERR_INVALID_ARG (no head in the plan),
 * TP_ERR_UNSUPPORTED (not bf16), TP_ERR_SHAPE (T outside 1..8), TP_ERR_ALIGN,
 * TP_ERR_CUDA. */
tp_status tp_lm_head_forward(tp_plan_t plan, const void* const* head_shards, const float* gamma,
                             const float* x, int32_t T, float* logits, int32_t* device_status,
                             void* stream);

/* Standalone rank-order reduction ([RT] Collective backend abstraction,
 * copy-and-reduce; [MG] Local TP: the add after the copies):
 *   out[m, :] = residual[m, :] + (((p_0 + p_1) + p_2) + ... + p_{tp-1})[m, :] + bias
 * partials is float32 [tp][M][H] (contiguous), residual float32 [M, H] or
 * NULL, bias float32 [H] or NULL (a row-parallel bias is replicated and
 * added once, after the sum), out float32 [M, H]. out may alias residual.
 * Errors: TP_ERR_NULL, TP_ERR_SHAPE (M < 0), TP_ERR_CUDA. */
tp_status tp_reduce_partials(tp_plan_t plan, const float* partials, const float* residual,
                             const float* bias, float* out, int64_t M, void* stream);

/* Tensor-core GEMM, the primitive of the prefill-regime projections:
 *   C[M, N] = A[M, K] * B[N, K]^T
 * A and B are bf16, row-major with K contiguous (B in the [out, in] weight
 * layout), C is float32 row-major; accumulation in float32 on the tcgen05
 * tensor cores. Requires M % 128 == 0, N % 256 == 0, K % 64 == 0 and
 * 16-byte aligned pointers. `device_status` is a DEVICE int32 (or NULL) that
 * receives TP_ERR_TIMEOUT / TP_ERR_ALIGN if a bounded device wait gives up.
 * Errors: TP_ERR_NULL, TP_ERR_SHAPE, TP_ERR_ALIGN, TP_ERR_UNSUPPORTED,
 * TP_ERR_CUDA. */
tp_status tp_gemm_bf16(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K,
                       int32_t* device_status, void* stream);

/* As tp_gemm_bf16 with B given as [K, N] row-major bf16 (N contiguous), so
 * C = A @ B: the tensor cores read B through its MN-major operand form (the
 * form the prefill attention uses for P @ V). Same shape rules and errors. */
tp_status tp_gemm_bf16_kn(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K,
                          int32_t* device_status, void* stream);

/* Reads the workspace status word (TP_OK or the first device-detected error
 * since tp_workspace_init) into *out (host). Synchronises `stream`. After
 * TP_ERR_TIMEOUT the workspace's counters may be left mid-way: call
 * tp_workspace_init on it before the next forward. */
tp_status tp_get_device_status(void* workspace, int32_t* out, void* stream);

/* Measurement hook: while set, tp_block_forward records events[i]
 * (cudaEvent_t values passed as void*, created by the caller) on its stream
 * before launching stage i and events[n_events-1] after the last stage, so
 * a caller can time each kernel. DECODE and PREFILL have 5 stages
 * (norm+qkv+rope+KV append, attention, o_proj+reduce, norm+gate_up+swiglu,
 * down+reduce): pass 6 events. MOE_FFN has 4 (routing and bucketing, expert
 * gate/up, expert down, weighted combine): pass 5. While the hook is set,
 * DECODE and MOE_FFN launch without programmatic dependent launch, so each
 * event pair brackets its own kernels only. n_events = 0 or events = NULL
 * clears the hook. The array is copied. */
tp_status tp_profile_stages(tp_plan_t plan, void* const* events, int32_t n_events);

/* bf16 DECODE runs the whole block as one persistent launch whose phases
 * are: RMSNorm operands; QKV (+RoPE, KV append); attention (+split-KV
 * combine); o_proj (+rank-ordered reduce, next norm operands); gate/up
 * (+SwiGLU); down (+rank-ordered reduce). While the hook above is set, that
 * launch also records per-CTA device timestamps at its start and, for each
 * of its 6 phases, when the CTA's own streaming work of the phase is done
 * and when it arrives at the phase's grid barrier (or ends), and events[0] /
 * events[n_events-1] bracket the launch. This call reads the timestamps of
 * the last such step and writes the first `n` (1..12) intervals in
 * microseconds to out_us (host): for phase i, out_us[2i] = streaming (latest
 * previous arrival to latest streaming done) and out_us[2i+1] = finishing
 * (latest streaming done to latest arrival). `median_us` (nullable) receives
 * the same intervals measured to the median CTA instead of the latest (the
 * gap is load imbalance). Synchronises `stream`. Errors: TP_ERR_NULL, TP_ERR_INVALID_ARG
 * (no profiled bf16 decode step yet), TP_ERR_CUDA. */
tp_status tp_profile_phases(tp_plan_t plan, double* out_us, double* median_us, int32_t n, void* stream);

/* The raw timestamps behind tp_profile_phases: `rows` CTAs (one per SM, in
 * launch order) x 13 values (start; then per phase: streaming done, barrier
 * arrival or end), %globaltimer nanoseconds, copied to `out` (host). */
tp_status tp_profile_phase_stamps(tp_plan_t plan, uint64_t* out, int32_t rows, void* stream);

/* Test hook for the bounded-wait path ([RT] Acceptance criteria: no silent
 * wrong results). While on (1), every bf16 DECODE launch of this plan waits
 * at each of its grid barriers for one arrival more than its CTAs make, as
 * if one CTA had been lost: the first barrier's wait gives up after the 1 s
 * limit, the launch records TP_ERR_TIMEOUT in the workspace status word, and
 * every CTA leaves through its abort path (all waits are bounded, so the
 * launch ends within a few seconds). The output and the KV rows at pos are
 * then undefined; call tp_workspace_init on the workspace before its next
 * forward. Off (0) by default; nothing in the library turns it on. No
 * counterpart on the pages.
 * Errors: TP_ERR_NULL, TP_ERR_INVALID_ARG (on not 0 or 1). */
tp_status tp_debug_withhold_arrival(tp_plan_t plan, int32_t on);

/* ----------------------------------------------------------------- misc */

/* Message for the last failing call on this thread ("" if none). Never fails. */
const char* tp_last_error(void);

/* TP_ABI_VERSION. */
int32_t tp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TP_BLOCK_H */
