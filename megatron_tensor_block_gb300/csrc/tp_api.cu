// C ABI of the tensor-parallel block library: plan validation and sizes,
// workspace layout, argument checks, and the launch sequence of each call.
// Every step of the block runs in the kernels of this library; there is no
// host-side or CPU fallback path.
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <new>
#include <vector>

#include "tp_internal.h"

using namespace tpk;

// ---------------------------------------------------------------- errors

static thread_local char g_err[512];

static tp_status fail(tp_status code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

static tp_status ok() {
    g_err[0] = '\0';
    return TP_OK;
}

static tp_status cuda_fail(cudaError_t e, const char* what) {
    return fail(TP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define TP_CUDA(call, what)                              \
    do {                                                 \
        cudaError_t e_ = (call);                         \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

// ---------------------------------------------------------------- plan

struct tp_plan_s {
    tp_model_desc d;
    int N = 1;
    tp_plan_info info{};
    bool dense = false, moe = false;
    size_t esz = 4;                     // bytes per stored weight/KV element
    // decode launch shapes
    GemvShape g_qkv, g_o, g_gu, g_down;
    int attn_chunks = 0, attn_groups = 0, step_chunks = 0;
    int step_split[4] = {0, 0, 0, 0};   // partial slots per tile of each projection phase (one-launch step)
    size_t off_step_part = 0;           // their partials (one region, reused phase after phase)
    // workspace layout (byte offsets)
    size_t off_status = 0, off_cnt_qkv = 0, off_cnt_attn = 0, off_cnt_o = 0, off_cnt_gu = 0,
           off_cnt_down = 0, off_step_bar = 0, off_kv_ready = 0, ctrl_bytes = 0;
    size_t off_stamps = 0;              // per-CTA phase end times of the decode step (profiling)
    size_t off_q = 0, off_attn_part = 0, off_attn_out = 0, off_h = 0, off_act = 0;
    size_t off_part_qkv = 0, off_part_o = 0, off_part_gu = 0, off_part_down = 0;
    size_t off_xg = 0, off_ss = 0, off_hg = 0, off_ss_tiles = 0;   // bf16 normalised operands
    // MoE buffers (share the data region with the decode buffers)
    size_t off_m_ids = 0, off_m_wts = 0, off_m_off = 0, off_m_perm = 0, off_m_slot = 0, off_m_rinv = 0,
           off_m_xs = 0, off_m_act = 0, off_m_o = 0, ws_moe_end = 0;
    // prefill buffers (share the data region with the decode and MoE buffers)
    size_t off_p_xn = 0, off_p_q = 0, off_p_ao = 0, off_p_h = 0, off_p_act = 0, off_p_rope = 0, ws_prefill_end = 0;
    size_t ws_bytes = 0;
    size_t ws_decode_end = 0;           // end of the decode buffers (control words included)
    // multi-layer decode (tp_stack_decode): control words, then its own pair buffers
    // at the end of the workspace (no other mode writes them, so no stale epoch matches)
    size_t off_step_pairs = 0;
    // tp_block_forward_noalloc: the decode buffers, then the down pieces' pair
    // buffer right after them (the workspace path keeps it at off_step_pairs)
    size_t na_pairs_off = 0, na_pairs_bytes = 0, na_end = 0;
    // q of the one-launch step as (value, epoch) pairs, right after the down pieces (both layouts)
    size_t off_q_pairs = 0, q_pairs_bytes = 0;
    size_t off_c_ctrl = 0, off_c_x = 0, off_c_q = 0, off_c_p = 0, off_c_h = 0, off_c_a = 0,
           off_c_begin = 0, off_c_end = 0;
    int c_ck = 0, c_maxch = 0;
    // measurement hook (tp_profile_stages)
    cudaEvent_t stage_ev[16] = {};
    int n_stage_ev = 0;
    char* last_stamps_ws = nullptr;     // workspace of the last profiled decode step
    unsigned dbg_bar_extra = 0;         // test hook (tp_debug_withhold_arrival): 0 in every product path
};

static void stage_mark(tp_plan_t P, int i, cudaStream_t s) {
    if (i < P->n_stage_ev && P->stage_ev[i]) cudaEventRecord(P->stage_ev[i], s);
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Smallest number of reduction chunks per shard such that the launch has at
// least `target` work units, with chunk lengths that are whole 64-element
// steps, at least two steps (both k-halves of a CTA busy) and at most
// `max_steps` steps (shared-memory bound).
static int pick_chunks(int steps, long units_per_chunk, int max_steps, long target, int max_chunks) {
    int best = -1;
    for (int C = 1; C <= steps && C <= max_chunks; ++C) {
        if (steps % C) continue;
        const int len = steps / C;
        if (len > max_steps) continue;
        if (len < 2 && steps >= 2) continue;
        best = C;
        if (units_per_chunk * C >= target) return C;
    }
    return best > 0 ? best : steps;
}

static GemvShape make_shape(int groups, int shards_per_group, int K, size_t esz) {
    GemvShape s;
    if (esz == 2) {
        // bf16: persistent tensor-map kernel. Column-parallel tiles take the whole
        // reduction (no cross-CTA partials); row-parallel tiles split each shard's
        // reduction into whole 256-element stages until there are >= 3 units per SM.
        s.groups = groups;
        s.shards_per_group = shards_per_group;
        s.chunks = 1;
        const int stages = (K + 255) / 256;
        if (shards_per_group > 1) {
            for (int C = 1; C <= stages && shards_per_group * C <= kMaxGroupUnits; ++C) {
                if (stages % C) continue;
                s.chunks = C;
                if ((long)groups * shards_per_group * C >= 6L * kSMs) break;
            }
            if (K % (s.chunks * 64) || (K / s.chunks) % 64) s.chunks = 1;
        }
        s.kc = K / s.chunks;
        return s;
    }
    s.groups = groups;
    s.shards_per_group = shards_per_group;
    const int steps = K / kKStep;
    // bf16 runs on the persistent streaming kernel (one CTA per SM walking its
    // units round-robin): ~6 units per CTA keeps the tail short. fp32 runs
    // one CTA per unit.
    const int max_steps = (esz == 2 ? kMaxKcTma : 1024) / kKStep;
    const long target = esz == 2 ? 3L * kSMs : 4L * kSMs;
    s.chunks = pick_chunks(steps, (long)groups * shards_per_group, max_steps, target,
                           kMaxGroupUnits / shards_per_group);
    s.kc = K / s.chunks;
    return s;
}

extern "C" tp_status tp_plan(const tp_model_desc* d, int32_t tp, tp_plan_t* out) {
    if (!d || !out) return fail(TP_ERR_NULL, "tp_plan: desc and out must not be NULL");
    *out = nullptr;
    if (tp < 1 || tp > TP_MAX_SHARDS)
        return fail(TP_ERR_INVALID_ARG, "tp_plan: tp=%d outside 1..%d", tp, TP_MAX_SHARDS);
    if (d->dtype != TP_F32 && d->dtype != TP_BF16)
        return fail(TP_ERR_INVALID_ARG, "tp_plan: unknown dtype %d", d->dtype);
    if (d->hidden <= 0) return fail(TP_ERR_INVALID_ARG, "tp_plan: hidden must be positive");
    const bool dense = d->n_heads > 0;
    const bool moe = d->n_experts > 0;
    if (!dense && !moe) return fail(TP_ERR_INVALID_ARG, "tp_plan: neither attention heads nor experts given");
    if (d->max_batch <= 0 || d->max_tokens <= 0)
        return fail(TP_ERR_INVALID_ARG, "tp_plan: max_batch and max_tokens must be positive");
    if (d->org_vocab < 0) return fail(TP_ERR_INVALID_ARG, "tp_plan: org_vocab must be >= 0");
    if (!(d->eps >= 0.0)) return fail(TP_ERR_INVALID_ARG, "tp_plan: eps must be >= 0");
    if (dense) {
        if (d->n_kv_heads <= 0 || d->head_dim <= 0 || d->ffn <= 0 || d->max_kv <= 0)
            return fail(TP_ERR_INVALID_ARG, "tp_plan: n_kv_heads, head_dim, ffn and max_kv must be positive");
        if (d->n_heads % d->n_kv_heads)
            return fail(TP_ERR_INVALID_ARG, "tp_plan: n_heads=%lld not a multiple of n_kv_heads=%lld",
                        (long long)d->n_heads, (long long)d->n_kv_heads);
        if (!(d->rope_theta > 0.0)) return fail(TP_ERR_INVALID_ARG, "tp_plan: rope_theta must be positive");
        if (d->n_heads % tp)
            return fail(TP_ERR_INDIVISIBLE, "tp_plan: n_heads=%lld not divisible by tp=%d", (long long)d->n_heads, tp);
        if (d->n_kv_heads % tp)
            return fail(TP_ERR_INDIVISIBLE, "tp_plan: n_kv_heads=%lld not divisible by tp=%d", (long long)d->n_kv_heads, tp);
        if (d->ffn % tp)
            return fail(TP_ERR_INDIVISIBLE, "tp_plan: ffn=%lld not divisible by tp=%d", (long long)d->ffn, tp);
    }
    if (d->reserved0 != 0) return fail(TP_ERR_INVALID_ARG, "tp_plan: reserved0 must be 0");
    if (!moe && d->expert_parallel) return fail(TP_ERR_INVALID_ARG, "tp_plan: expert_parallel without experts");
    if (moe) {
        if (d->top_k < 1 || d->top_k > d->n_experts || d->expert_ffn <= 0)
            return fail(TP_ERR_INVALID_ARG, "tp_plan: need 1 <= top_k <= n_experts and expert_ffn > 0");
        if (d->expert_parallel != 0 && d->expert_parallel != 1)
            return fail(TP_ERR_INVALID_ARG, "tp_plan: expert_parallel must be 0 or 1");
        if (d->expert_parallel && d->n_experts % tp)
            return fail(TP_ERR_INDIVISIBLE, "tp_plan: n_experts=%lld not divisible by tp=%d (expert parallelism)",
                        (long long)d->n_experts, tp);
        if (!d->expert_parallel && d->expert_ffn % tp)
            return fail(TP_ERR_INDIVISIBLE, "tp_plan: expert_ffn=%lld not divisible by tp=%d", (long long)d->expert_ffn, tp);
    }
    // ranges the kernels handle
    if (d->hidden % 64) return fail(TP_ERR_UNSUPPORTED, "tp_plan: hidden must be a multiple of 64");
    if (dense) {
        if (d->head_dim != 64 && d->head_dim != 128)
            return fail(TP_ERR_UNSUPPORTED, "tp_plan: head_dim must be 64 or 128");
        if ((d->ffn / tp) % 64) return fail(TP_ERR_UNSUPPORTED, "tp_plan: ffn/tp must be a multiple of 64");
        if (d->n_heads / d->n_kv_heads > 8)
            return fail(TP_ERR_UNSUPPORTED, "tp_plan: more than 8 query heads per KV head");
    }
    if (moe && (d->expert_ffn / (d->expert_parallel ? 1 : tp)) % 64)
        return fail(TP_ERR_UNSUPPORTED, "tp_plan: the expert FFN width per shard must be a multiple of 64");
    if (moe && (d->n_experts > 64 || d->top_k > 8))
        return fail(TP_ERR_UNSUPPORTED, "tp_plan: MoE supports up to 64 experts and top_k <= 8");

    tp_plan_s* P = new (std::nothrow) tp_plan_s();
    if (!P) return fail(TP_ERR_INVALID_ARG, "tp_plan: out of host memory");
    P->d = *d;
    P->N = tp;
    P->dense = dense;
    P->moe = moe;
    P->esz = d->dtype == TP_BF16 ? 2 : 4;
    const int64_t N = tp, H = d->hidden, esz = (int64_t)P->esz;
    tp_plan_info& I = P->info;
    I.tp = tp;
    I.reduce_points = dense ? 2 : 1;
    if (dense) {
        I.hq_shard = d->n_heads / N;
        I.hkv_shard = d->n_kv_heads / N;
        I.ffn_shard = d->ffn / N;
        I.qkv_rows = (I.hq_shard + 2 * I.hkv_shard) * d->head_dim;
        I.wqkv_bytes = I.qkv_rows * H * esz;
        I.bqkv_bytes = d->has_qkv_bias ? I.qkv_rows * 4 : 0;
        I.wo_bytes = H * I.hq_shard * d->head_dim * esz;
        I.wgu_bytes = 2 * I.ffn_shard * H * esz;
        I.wd_bytes = H * I.ffn_shard * esz;
        I.kv_cache_bytes = d->max_batch * I.hkv_shard * d->max_kv * d->head_dim * esz;
    }
    I.gamma_bytes = H * 4;
    if (moe) {
        I.expert_ffn_shard = d->expert_parallel ? d->expert_ffn : d->expert_ffn / N;
        I.experts_shard = d->expert_parallel ? d->n_experts / N : d->n_experts;
        I.egu_bytes = I.experts_shard * 2 * I.expert_ffn_shard * H * esz;
        I.ed_bytes = I.experts_shard * H * I.expert_ffn_shard * esz;
    }
    if (d->org_vocab > 0) {
        const int64_t m = 64 * N;
        I.vocab_padded = (d->org_vocab + m - 1) / m * m;
        I.vocab_rows_shard = I.vocab_padded / N;
        I.lm_head_bytes = I.vocab_rows_shard * H * esz;
    }
    I.weight_bytes_shard = I.wqkv_bytes + I.wo_bytes + I.wgu_bytes + I.wd_bytes + I.egu_bytes + I.ed_bytes;
    I.weight_bytes_total = I.weight_bytes_shard * N;

    // ---- workspace layout: control words first, then the data buffers
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
    P->off_status = take(sizeof(int));   // offset 0 in every layout (tp_noalloc_status relies on it)
    if (dense) {
        const int hd = (int)d->head_dim;
        P->g_qkv = make_shape((int)(N * I.qkv_rows / kTileRows), 1, (int)H, P->esz);
        P->g_o = make_shape((int)(H / kTileRows), (int)N, (int)(I.hq_shard * hd), P->esz);
        P->g_gu = make_shape((int)(N * I.ffn_shard / 32), 1, (int)H, P->esz);
        P->g_down = make_shape((int)(H / kTileRows), (int)N, (int)I.ffn_shard, P->esz);
        P->attn_chunks = (int)((d->max_kv + kAttnChunk - 1) / kAttnChunk);
        // one-launch step: a KV group is split over at most ceil(max_kv / keys per CTA) + 1 <= 32 CTAs
        {
            const int mk = step_min_keys((int)d->max_kv);
            P->step_chunks = (int)((d->max_kv + mk - 1) / mk) + 1;
        }
        P->attn_groups = (int)(N * (d->max_batch < kTMax ? d->max_batch : kTMax) * I.hkv_shard);
        P->off_cnt_qkv = take(sizeof(unsigned) * P->g_qkv.groups);
        P->off_cnt_attn = take(sizeof(unsigned) * P->attn_groups);
        P->off_cnt_o = take(sizeof(unsigned) * P->g_o.groups);
        P->off_cnt_gu = take(sizeof(unsigned) * P->g_gu.groups);
        P->off_cnt_down = take(sizeof(unsigned) * P->g_down.groups);
        P->off_step_bar = take(sizeof(unsigned long long));
        P->off_kv_ready = take(sizeof(unsigned long long));   // QKV epilogues done (one arrival per CTA and launch)
        P->off_c_ctrl = take(4 * sizeof(unsigned));   // launch counter, CTAs finished, abort flag
    }
    P->ctrl_bytes = off;
    if (dense) {
        const int64_t hd = d->head_dim, G = d->n_heads / d->n_kv_heads;
        P->off_q = take((size_t)kTMax * d->n_heads * hd * 4);
        P->off_attn_part = take((size_t)P->attn_groups * std::max(P->attn_chunks, P->step_chunks) * G * (hd + 2) * 4);
        P->off_attn_out = take((size_t)kTMax * d->n_heads * hd * esz);
        P->off_h = take((size_t)kTMax * H * 4);
        P->off_act = take((size_t)kTMax * d->ffn * esz);
        P->off_part_qkv = take((size_t)P->g_qkv.units() * kPartStride * 4);
        P->off_part_o = take((size_t)P->g_o.units() * kPartStride * 4);
        P->off_part_gu = take((size_t)P->g_gu.units() * kPartStride * 4);
        P->off_part_down = take((size_t)P->g_down.units() * kPartStride * 4);
        P->off_xg = take((size_t)N * kTMax * H * 2);
        P->off_ss = take((size_t)(H / 256 + 1) * kTMax * 4);
        P->off_hg = take((size_t)N * kTMax * H * 2);
        P->off_ss_tiles = take((size_t)(H / 8) * kTMax * 4);
        P->off_stamps = take((size_t)kMaxStepCtas * kStepStamps * 8);
        {
            // projection phases of the one-launch step: segments x stages, split
            // evenly over at most kMaxStepCtas CTAs (each CTA takes >= W / kMaxStepCtas)
            const int64_t segs[4] = {P->g_qkv.groups, P->g_o.groups * N, P->g_gu.groups, P->g_down.groups * N};
            const int64_t Ks[4] = {H, I.hq_shard * hd, H, I.ffn_shard};
            size_t need = 0;
            for (int i = 0; i < 4; ++i) {
                const int64_t S = (Ks[i] + 255) / 256, W = segs[i] * S;
                const int64_t rmin = (W + kMaxStepCtas - 1) / kMaxStepCtas;
                P->step_split[i] = (int)((S + rmin - 1) / rmin + 1);
                need = std::max(need, (size_t)segs[i] * P->step_split[i] * kPartStride * 4);
            }
            P->off_step_part = take(need);
        }
        P->ws_decode_end = off;
    }
    if (dense && d->dtype == TP_BF16) {
        off = P->ctrl_bytes;
        const int64_t Tm = d->max_tokens, hd = d->head_dim;
        P->off_p_xn = take((size_t)N * Tm * H * 2);              // one bf16 copy per distinct gamma
        P->off_p_q = take((size_t)Tm * d->n_heads * hd * 2);     // [N][T][Hq' d]
        P->off_p_ao = take((size_t)Tm * d->n_heads * hd * 2);
        P->off_p_h = take((size_t)Tm * H * 4);
        P->off_p_act = take((size_t)Tm * d->ffn * 2);            // [N][T][F']
        P->off_p_rope = take((size_t)d->max_kv * (hd / 2) * 8);  // (cos, sin) per position and pair
        P->ws_prefill_end = off;
    }
    if (moe) {
        off = P->ctrl_bytes;
        const int64_t ns = d->max_tokens * d->top_k, Fs = I.expert_ffn_shard;
        P->off_m_ids = take((size_t)ns * 4);
        P->off_m_wts = take((size_t)ns * 4);
        P->off_m_off = take((size_t)(d->n_experts + 1) * 4);
        P->off_m_perm = take((size_t)ns * 4);
        P->off_m_slot = take((size_t)ns * 4);
        P->off_m_rinv = take((size_t)ns * 4);
        P->off_m_xs = take((size_t)N * ns * H * 2);
        P->off_m_act = take((size_t)N * ns * Fs * 2);
        P->off_m_o = take((size_t)N * ns * H * 4);
        P->ws_moe_end = off;
        I.moe_ids_offset = (int64_t)P->off_m_ids;
        I.moe_bucket_offset = (int64_t)P->off_m_off;
        I.moe_perm_offset = (int64_t)P->off_m_perm;
    } else {
        I.moe_ids_offset = I.moe_bucket_offset = I.moe_perm_offset = -1;
    }
    P->ws_bytes = std::max(P->ws_decode_end, std::max(P->ws_moe_end, P->ws_prefill_end));
    if (P->ws_bytes < P->ctrl_bytes) P->ws_bytes = P->ctrl_bytes;
    if (dense && d->dtype == TP_BF16 && (d->head_dim == 64 || d->head_dim == 128)) {
        off = P->ws_bytes;
        const int64_t MB = d->max_batch, hd = d->head_dim, G = d->n_heads / d->n_kv_heads;
        P->c_ck = (int)(8192 / hd);                              // keys per 16 KB tile of K
        P->c_maxch = (int)((d->max_kv + P->c_ck - 1) / P->c_ck);
        const int64_t groups = N * MB * I.hkv_shard;
        P->off_c_begin = off;
        // split row-parallel tiles of the one-launch step: (value, epoch) pieces of the down phase
        P->na_pairs_bytes = (size_t)P->g_down.groups * N * P->step_split[3] * kTileRows * kTMax * 8;
        P->off_step_pairs = take(P->na_pairs_bytes);
        P->q_pairs_bytes = (size_t)kTMax * d->n_heads * hd * 8;
        P->off_q_pairs = take(P->q_pairs_bytes);
        P->off_c_x = take((size_t)MB * H * 8);
        P->off_c_q = take((size_t)N * MB * I.qkv_rows * 8);
        P->off_c_p = take((size_t)groups * P->c_maxch * G * (hd + 2) * 8);
        P->off_c_h = take((size_t)MB * H * 8);
        P->off_c_a = take((size_t)N * MB * I.ffn_shard * 8);
        P->off_c_end = off;
        P->ws_bytes = off;
    }
    I.workspace_bytes = (int64_t)P->ws_bytes;
    if (dense) {
        // every byte a decode step writes: control words, decode buffers, pair buffer
        P->na_end = P->ws_decode_end;
        if (P->off_step_pairs) {
            // the same two pair buffers, contiguous, after the decode buffers
            P->na_pairs_off = align256(P->ws_decode_end);
            P->na_end = align256(P->na_pairs_off + (P->off_q_pairs - P->off_step_pairs) + P->q_pairs_bytes);
        }
        I.noalloc_scratch_bytes = (int64_t)P->na_end;
    }
    *out = P;
    return ok();
}

extern "C" void tp_plan_destroy(tp_plan_t plan) { delete plan; }

extern "C" tp_status tp_plan_get_info(tp_plan_t plan, tp_plan_info* out) {
    if (!plan || !out) return fail(TP_ERR_NULL, "tp_plan_get_info: NULL argument");
    *out = plan->info;
    return ok();
}

extern "C" tp_status tp_plan_describe(tp_plan_t plan, char* buf, size_t n) {
    if (!plan || !buf || n == 0) return fail(TP_ERR_NULL, "tp_plan_describe: NULL argument");
    const tp_plan_info& I = plan->info;
    const double total = (double)I.weight_bytes_total, shard = (double)I.weight_bytes_shard;
    snprintf(buf, n,
             "tensor parallelism: %d logical shards on one GPU; per shard: qkv [%lld x %lld], "
             "o [%lld x %lld], gate_up [%lld x %lld], down [%lld x %lld], experts %lld x [%lld x %lld]; "
             "weights %.3f MB per shard = %.4f of %.3f MB total; %d reductions per block; workspace %lld bytes",
             I.tp, (long long)I.qkv_rows, (long long)plan->d.hidden, (long long)plan->d.hidden,
             (long long)(I.hq_shard * plan->d.head_dim), (long long)(2 * I.ffn_shard), (long long)plan->d.hidden,
             (long long)plan->d.hidden, (long long)I.ffn_shard, (long long)plan->d.n_experts,
             (long long)(2 * I.expert_ffn_shard), (long long)plan->d.hidden, shard / 1e6,
             total > 0 ? shard / total : 0.0, total / 1e6, I.reduce_points, (long long)I.workspace_bytes);
    return ok();
}

// ---------------------------------------------------------------- device checks

static tp_status check_device() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(TP_ERR_UNSUPPORTED, "no usable CUDA device: %s", cudaGetErrorString(e));
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
        return fail(TP_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major, minor);
    return TP_OK;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// ---------------------------------------------------------------- shard / gather

namespace {
struct Batcher {
    CopyBatch b{};
    cudaStream_t s;
    cudaError_t err = cudaSuccess;
    explicit Batcher(cudaStream_t st) : s(st) { b.n = 0; }
    void add(const void* src, void* dst, int64_t rows, int64_t row_bytes, int64_t sp, int64_t dp) {
        if (rows <= 0 || row_bytes <= 0) return;
        if (b.n == kMaxCopyDescs) flush();
        b.d[b.n++] = CopyDesc{src, dst, rows, row_bytes, sp, dp};
    }
    void flush() {
        if (b.n && err == cudaSuccess) err = launch_copy_batch(b, s);
        b.n = 0;
    }
};
const char* cptr(const void* p, int64_t off) { return static_cast<const char*>(p) + off; }
char* mptr(void* p, int64_t off) { return static_cast<char*>(p) + off; }
}  // namespace

extern "C" tp_status tp_shard_weights(tp_plan_t plan, const tp_block_weights* full,
                                      const tp_shard_set* out, void* stream) {
    if (!plan || !full || !out) return fail(TP_ERR_NULL, "tp_shard_weights: NULL argument");
    tp_status st = check_device();
    if (st) return st;
    const tp_model_desc& d = plan->d;
    const int N = plan->N;
    const tp_plan_info& I = plan->info;
    const int64_t H = d.hidden, es = (int64_t)plan->esz;
    if (!full->gamma_attn && plan->dense) return fail(TP_ERR_NULL, "tp_shard_weights: gamma_attn is NULL");
    if (!full->gamma_ffn) return fail(TP_ERR_NULL, "tp_shard_weights: gamma_ffn is NULL");
    for (int r = 0; r < N; ++r)
        if (!out->gamma_ffn[r] || (plan->dense && !out->gamma_attn[r]))
            return fail(TP_ERR_NULL, "tp_shard_weights: shard %d gamma buffer is NULL", r);
    Batcher B(static_cast<cudaStream_t>(stream));
    if (plan->dense) {
        const void* need[] = {full->wq, full->wk, full->wv, full->wo, full->w_gate, full->w_up, full->w_down};
        for (const void* p : need) {
            if (!p) return fail(TP_ERR_NULL, "tp_shard_weights: a dense weight pointer is NULL");
            if (!aligned16(p)) return fail(TP_ERR_ALIGN, "tp_shard_weights: weight pointers must be 16-byte aligned");
        }
        if (d.has_qkv_bias && (!full->bq || !full->bk || !full->bv))
            return fail(TP_ERR_NULL, "tp_shard_weights: plan has q/k/v biases but a bias pointer is NULL");
        const int64_t hd = d.head_dim, qr = I.hq_shard * hd, kr = I.hkv_shard * hd, Fs = I.ffn_shard;
        for (int r = 0; r < N; ++r) {
            if (!out->wqkv[r] || !out->wo[r] || !out->wgu[r] || !out->wd[r] || (d.has_qkv_bias && !out->bqkv[r]))
                return fail(TP_ERR_NULL, "tp_shard_weights: shard %d output buffer is NULL", r);
            const int64_t row = H * es;
            // fused [q_r; k_r; v_r]
            B.add(cptr(full->wq, r * qr * row), mptr(out->wqkv[r], 0), qr, row, row, row);
            B.add(cptr(full->wk, r * kr * row), mptr(out->wqkv[r], qr * row), kr, row, row, row);
            B.add(cptr(full->wv, r * kr * row), mptr(out->wqkv[r], (qr + kr) * row), kr, row, row, row);
            if (d.has_qkv_bias) {
                B.add(cptr(full->bq, r * qr * 4), mptr(out->bqkv[r], 0), 1, qr * 4, qr * 4, qr * 4);
                B.add(cptr(full->bk, r * kr * 4), mptr(out->bqkv[r], qr * 4), 1, kr * 4, kr * 4, kr * 4);
                B.add(cptr(full->bv, r * kr * 4), mptr(out->bqkv[r], (qr + kr) * 4), 1, kr * 4, kr * 4, kr * 4);
            }
            // o_proj: columns [r*Hq'd, (r+1)*Hq'd)
            B.add(cptr(full->wo, r * qr * es), out->wo[r], H, qr * es, d.n_heads * hd * es, qr * es);
            // fused [gate_r; up_r]
            B.add(cptr(full->w_gate, r * Fs * row), mptr(out->wgu[r], 0), Fs, row, row, row);
            B.add(cptr(full->w_up, r * Fs * row), mptr(out->wgu[r], Fs * row), Fs, row, row, row);
            // down_proj: columns [r*F', (r+1)*F')
            B.add(cptr(full->w_down, r * Fs * es), out->wd[r], H, Fs * es, d.ffn * es, Fs * es);
            B.add(full->gamma_attn, out->gamma_attn[r], 1, H * 4, H * 4, H * 4);
        }
    }
    if (plan->moe) {
        if (!full->e_gate || !full->e_up || !full->e_down)
            return fail(TP_ERR_NULL, "tp_shard_weights: expert weight pointer is NULL");
        const int64_t E = d.n_experts, Fe = d.expert_ffn, Fs = I.expert_ffn_shard, row = H * es;
        for (int r = 0; r < N && d.expert_parallel; ++r) {
            if (!out->egu[r] || !out->ed[r]) return fail(TP_ERR_NULL, "tp_shard_weights: shard %d expert buffer is NULL", r);
            // whole experts [r*E/N, (r+1)*E/N): gate rows then up rows of each -> [E/N][2Fe][H], down -> [E/N][H][Fe]
            const int64_t per = I.experts_shard, e0 = r * per;
            B.add(cptr(full->e_gate, e0 * Fe * row), mptr(out->egu[r], 0), per, Fe * row, Fe * row, 2 * Fe * row);
            B.add(cptr(full->e_up, e0 * Fe * row), mptr(out->egu[r], Fe * row), per, Fe * row, Fe * row, 2 * Fe * row);
            B.add(cptr(full->e_down, e0 * H * Fe * es), out->ed[r], per * H, Fe * es, Fe * es, Fe * es);
        }
        for (int r = 0; r < N && !d.expert_parallel; ++r) {
            if (!out->egu[r] || !out->ed[r]) return fail(TP_ERR_NULL, "tp_shard_weights: shard %d expert buffer is NULL", r);
            // every expert: gate rows and up rows [r*Fe', (r+1)*Fe') -> [E][2Fe'][H]
            B.add(cptr(full->e_gate, r * Fs * row), mptr(out->egu[r], 0), E, Fs * row, Fe * row, 2 * Fs * row);
            B.add(cptr(full->e_up, r * Fs * row), mptr(out->egu[r], Fs * row), E, Fs * row, Fe * row, 2 * Fs * row);
            // down columns [r*Fe', (r+1)*Fe') of every [H, Fe] -> [E][H][Fe']
            B.add(cptr(full->e_down, r * Fs * es), out->ed[r], E * H, Fs * es, Fe * es, Fs * es);
        }
    }
    for (int r = 0; r < N; ++r) B.add(full->gamma_ffn, out->gamma_ffn[r], 1, H * 4, H * 4, H * 4);
    B.flush();
    if (B.err != cudaSuccess) return cuda_fail(B.err, "tp_shard_weights: copy launch");
    return ok();
}

static tp_status default_segments(tp_plan_t plan, int32_t k, const int64_t* segments, int32_t nseg,
                                  int64_t rows, int64_t* seg, int* ns) {
    if (segments && nseg > 0) {
        if (nseg > 16) return fail(TP_ERR_INVALID_ARG, "at most 16 segments");
        for (int i = 0; i < nseg; ++i) seg[i] = segments[i];
        *ns = nseg;
    } else if (k == TP_PARAM_FUSED_QKV && plan->dense) {
        seg[0] = plan->d.n_heads * plan->d.head_dim;
        seg[1] = seg[2] = plan->d.n_kv_heads * plan->d.head_dim;
        *ns = 3;
    } else if (k == TP_PARAM_FUSED_GATE_UP && plan->dense) {
        seg[0] = seg[1] = plan->d.ffn;
        *ns = 2;
    } else {
        return fail(TP_ERR_INVALID_ARG, "fused/packed kind needs segment row counts");
    }
    int64_t sum = 0;
    for (int i = 0; i < *ns; ++i) {
        if (seg[i] <= 0 || seg[i] % plan->N) return fail(TP_ERR_SHAPE, "segment %d rows %lld not divisible by tp=%d", i, (long long)seg[i], plan->N);
        sum += seg[i];
    }
    if (sum != rows) return fail(TP_ERR_SHAPE, "segments sum to %lld rows, tensor has %lld", (long long)sum, (long long)rows);
    return TP_OK;
}

extern "C" tp_status tp_shard_param(tp_plan_t plan, int32_t k, const void* full, int64_t rows,
                                    int64_t cols, int32_t dtype, const int64_t* segments,
                                    int32_t n_segments, void* const* shards_out, void* stream) {
    if (!plan || !full || !shards_out) return fail(TP_ERR_NULL, "tp_shard_param: NULL argument");
    if (dtype != TP_F32 && dtype != TP_BF16) return fail(TP_ERR_INVALID_ARG, "tp_shard_param: unknown dtype");
    if (rows <= 0 || cols <= 0) return fail(TP_ERR_SHAPE, "tp_shard_param: rows and cols must be positive");
    const int N = plan->N;
    for (int r = 0; r < N; ++r)
        if (!shards_out[r]) return fail(TP_ERR_NULL, "tp_shard_param: shard %d pointer is NULL", r);
    tp_status st = check_device();
    if (st) return st;
    const int64_t es = dtype == TP_BF16 ? 2 : 4, row = cols * es;
    Batcher B(static_cast<cudaStream_t>(stream));
    switch (k) {
        case TP_PARAM_REPLICATED:
            for (int r = 0; r < N; ++r) B.add(full, shards_out[r], rows, row, row, row);
            break;
        case TP_PARAM_COLWISE: {
            if (rows % N) return fail(TP_ERR_SHAPE, "tp_shard_param: rows %lld not divisible by tp", (long long)rows);
            const int64_t R = rows / N;
            for (int r = 0; r < N; ++r) B.add(cptr(full, r * R * row), shards_out[r], R, row, row, row);
            break;
        }
        case TP_PARAM_ROWWISE: {
            if (cols % N) return fail(TP_ERR_SHAPE, "tp_shard_param: cols %lld not divisible by tp", (long long)cols);
            const int64_t C = cols / N;
            for (int r = 0; r < N; ++r) B.add(cptr(full, r * C * es), shards_out[r], rows, C * es, row, C * es);
            break;
        }
        case TP_PARAM_FUSED_QKV:
        case TP_PARAM_FUSED_GATE_UP:
        case TP_PARAM_PACKED_COLWISE: {
            int64_t seg[16];
            int ns = 0;
            st = default_segments(plan, k, segments, n_segments, rows, seg, &ns);
            if (st) return st;
            for (int r = 0; r < N; ++r) {
                int64_t src0 = 0, dst0 = 0;
                for (int i = 0; i < ns; ++i) {
                    const int64_t R = seg[i] / N;
                    B.add(cptr(full, (src0 + r * R) * row), mptr(shards_out[r], dst0 * row), R, row, row, row);
                    src0 += seg[i];
                    dst0 += R;
                }
            }
            break;
        }
        case TP_PARAM_VOCAB_PARALLEL: {
            const int64_t m = 64 * (int64_t)N, padded = (rows + m - 1) / m * m, R = padded / N;
            for (int r = 0; r < N; ++r) {
                int64_t have = rows - r * R;
                have = have < 0 ? 0 : (have > R ? R : have);
                B.add(cptr(full, r * R * row), shards_out[r], have, row, row, row);
                B.add(nullptr, mptr(shards_out[r], have * row), R - have, row, row, row);
            }
            break;
        }
        default:
            return fail(TP_ERR_INVALID_ARG, "tp_shard_param: unknown kind %d", k);
    }
    B.flush();
    if (B.err != cudaSuccess) return cuda_fail(B.err, "tp_shard_param: copy launch");
    return ok();
}

extern "C" tp_status tp_gather_param(tp_plan_t plan, int32_t k, const void* const* shards,
                                     int64_t rows_per_shard, int64_t cols_per_shard, int32_t dtype,
                                     void* out, void* stream) {
    if (!plan || !shards || !out) return fail(TP_ERR_NULL, "tp_gather_param: NULL argument");
    if (dtype != TP_F32 && dtype != TP_BF16) return fail(TP_ERR_INVALID_ARG, "tp_gather_param: unknown dtype");
    if (rows_per_shard <= 0 || cols_per_shard <= 0)
        return fail(TP_ERR_SHAPE, "tp_gather_param: rows and cols must be positive");
    const int N = plan->N;
    for (int r = 0; r < N; ++r)
        if (!shards[r]) return fail(TP_ERR_NULL, "tp_gather_param: shard %d pointer is NULL", r);
    if (k < TP_PARAM_REPLICATED || k > TP_PARAM_VOCAB_PARALLEL)
        return fail(TP_ERR_INVALID_ARG, "tp_gather_param: unknown kind %d", k);
    const int64_t org = plan->d.org_vocab;
    if (k == TP_PARAM_VOCAB_PARALLEL && (org <= 0 || org > N * rows_per_shard))
        return fail(TP_ERR_SHAPE, "tp_gather_param: org_vocab=%lld outside 1..%lld", (long long)org,
                    (long long)(N * rows_per_shard));
    tp_status st = check_device();
    if (st) return st;
    const int64_t es = dtype == TP_BF16 ? 2 : 4, R = rows_per_shard, C = cols_per_shard, row = C * es;
    Batcher B(static_cast<cudaStream_t>(stream));
    if (k == TP_PARAM_REPLICATED) {
        B.add(shards[0], out, R, row, row, row);
    } else if (k == TP_PARAM_ROWWISE) {
        for (int r = 0; r < N; ++r) B.add(shards[r], mptr(out, r * row), R, row, row, N * row);
    } else {
        for (int r = 0; r < N; ++r) {
            int64_t n = R;
            if (k == TP_PARAM_VOCAB_PARALLEL) {
                n = org - r * R;
                n = n < 0 ? 0 : (n > R ? R : n);
            }
            B.add(shards[r], mptr(out, r * R * row), n, row, row, row);
        }
    }
    B.flush();
    if (B.err != cudaSuccess) return cuda_fail(B.err, "tp_gather_param: copy launch");
    return ok();
}

extern "C" tp_status tp_shard_kv(tp_plan_t plan, const void* k_full, const void* v_full, int64_t B, int64_t L,
                                 const tp_kv_set* kv, void* stream) {
    if (!plan || !k_full || !v_full || !kv) return fail(TP_ERR_NULL, "tp_shard_kv: NULL argument");
    if (!plan->dense) return fail(TP_ERR_INVALID_ARG, "tp_shard_kv: the plan has no attention block");
    const tp_model_desc& d = plan->d;
    if (B < 1 || B > d.max_batch)
        return fail(TP_ERR_SHAPE, "tp_shard_kv: B=%lld outside 1..max_batch (%lld)", (long long)B,
                    (long long)d.max_batch);
    if (L < 0 || L > d.max_kv)
        return fail(TP_ERR_CAPACITY, "tp_shard_kv: L=%lld outside 0..max_kv (%lld)", (long long)L, (long long)d.max_kv);
    const int N = plan->N;
    for (int r = 0; r < N; ++r)
        if (!kv->k[r] || !kv->v[r]) return fail(TP_ERR_NULL, "tp_shard_kv: shard %d cache pointer is NULL", r);
    tp_status st = check_device();
    if (st) return st;
    if (L == 0) return ok();
    const int64_t Hs = plan->info.hkv_shard, Hkv = d.n_kv_heads, hd = d.head_dim;
    const int64_t es = (int64_t)plan->esz, run = L * hd * es;   // one head's first L positions
    Batcher Bt(static_cast<cudaStream_t>(stream));
    for (int r = 0; r < N; ++r)
        for (int64_t b = 0; b < B; ++b) {
            // heads r*Hs .. r*Hs+Hs-1 of sequence b: contiguous in the full cache,
            // one max_kv-long row each in the shard's cache
            const int64_t src = ((b * Hkv) + r * Hs) * run, dst = b * Hs * d.max_kv * hd * es;
            Bt.add(cptr(k_full, src), mptr(kv->k[r], dst), Hs, run, run, d.max_kv * hd * es);
            Bt.add(cptr(v_full, src), mptr(kv->v[r], dst), Hs, run, run, d.max_kv * hd * es);
        }
    Bt.flush();
    if (Bt.err != cudaSuccess) return cuda_fail(Bt.err, "tp_shard_kv: copy launch");
    return ok();
}

// ---------------------------------------------------------------- forward

extern "C" tp_status tp_workspace_init(tp_plan_t plan, void* workspace, size_t bytes, void* stream) {
    if (!plan || !workspace) return fail(TP_ERR_NULL, "tp_workspace_init: NULL argument");
    if (bytes < plan->ws_bytes)
        return fail(TP_ERR_CAPACITY, "tp_workspace_init: workspace %zu bytes < required %zu", bytes, plan->ws_bytes);
    if (!aligned16(workspace)) return fail(TP_ERR_ALIGN, "tp_workspace_init: workspace must be 16-byte aligned");
    tp_status st = check_device();
    if (st) return st;
    TP_CUDA(cudaMemsetAsync(workspace, 0, plan->ctrl_bytes, static_cast<cudaStream_t>(stream)),
            "tp_workspace_init: memset");
    if (plan->off_c_end > plan->off_c_begin)   // pair buffers: epoch 0 is never current
        TP_CUDA(cudaMemsetAsync(static_cast<char*>(workspace) + plan->off_c_begin, 0,
                                plan->off_c_end - plan->off_c_begin, static_cast<cudaStream_t>(stream)),
                "tp_workspace_init: memset");
    return ok();
}

// bf16 decode: every stage in one persistent launch (the launch sequence of
// the separate fp32 kernels below, as phases of one kernel).
static tp_status decode_step_bf16(tp_plan_t P, const tp_shard_set* w, const tp_kv_set* kv, const float* x, float* y,
                                  const int32_t* pos, int B, char* ws, size_t pairs_off, cudaStream_t s,
                                  const GemvParams& q, const NormPrepParams& np) {
    const tp_model_desc& d = P->d;
    const tp_plan_info& I = P->info;
    const int N = P->N, T = B, hd = (int)d.head_dim;
    int* status = reinterpret_cast<int*>(ws + P->off_status);
    DecodeStepParams st{};
    st.np = np;
    st.g[0] = q;
    float* part = reinterpret_cast<float*>(ws + P->off_step_part);
    st.g[0].part = part;
    st.g[0].shape.chunks = P->step_split[0];

    AttnDecodeParams& a = st.a;
    a.q = q.q_out;
    for (int r = 0; r < N; ++r) {
        a.kcache[r] = kv->k[r];
        a.vcache[r] = kv->v[r];
    }
    a.pos = pos;
    a.N = N;
    a.B = B;
    a.hq_s = (int)I.hq_shard;
    a.hkv_s = (int)I.hkv_shard;
    a.d = hd;
    a.max_kv = (int)d.max_kv;
    a.max_batch = (int)d.max_batch;
    a.n_chunks = P->step_chunks;
    a.scale = (float)(1.0 / std::sqrt((double)hd));
    a.part = reinterpret_cast<float*>(ws + P->off_attn_part);
    a.cnt = reinterpret_cast<unsigned*>(ws + P->off_cnt_attn);
    a.out = ws + P->off_attn_out;
    a.status = status;
    a.part_units = (unsigned)(P->attn_groups * P->step_chunks);

    float* h = reinterpret_cast<float*>(ws + P->off_h);
    GemvParams& o = st.g[1];
    o.n_shards = N;
    o.rows = (int)d.hidden;
    o.K = (int)(I.hq_shard * hd);
    o.T = T;
    o.shape = P->g_o;
    o.shape.chunks = P->step_split[1];
    o.part = part;
    o.whole_tiles = 1;                                  // 64 output tiles x every shard: reduced inside each CTA
    o.cnt = reinterpret_cast<unsigned*>(ws + P->off_cnt_o);
    o.status = status;
    o.resid = x;
    o.y = h;
    for (int r = 0; r < N; ++r) {
        o.W[r] = w->wo[r];
        o.gamma2[r] = w->gamma_ffn[r];
    }
    o.xact = ws + P->off_attn_out;
    o.norm_out = ws + P->off_hg;
    o.ss_tiles_out = reinterpret_cast<float*>(ws + P->off_ss_tiles);

    GemvParams& g = st.g[2];
    g.n_shards = N;
    g.rows = (int)(2 * I.ffn_shard);
    g.K = (int)d.hidden;
    g.T = T;
    g.shape = P->g_gu;
    g.shape.chunks = P->step_split[2];
    g.part = part;
    g.cnt = reinterpret_cast<unsigned*>(ws + P->off_cnt_gu);
    g.eps = (float)d.eps;
    g.status = status;
    g.act_out = ws + P->off_act;
    g.ffn_s = (int)I.ffn_shard;
    for (int r = 0; r < N; ++r) {
        g.W[r] = w->wgu[r];
        g.gamma[r] = w->gamma_ffn[r];
    }
    g.xact = ws + P->off_hg;
    g.ss_tiles = reinterpret_cast<const float*>(ws + P->off_ss_tiles);
    g.n_ss_tiles = (int)(d.hidden / 8);                 // per 8-row slice (the step's reduce phase)

    GemvParams& dn = st.g[3];
    dn.n_shards = N;
    dn.rows = (int)d.hidden;
    dn.K = (int)I.ffn_shard;
    dn.T = T;
    dn.shape = P->g_down;
    dn.shape.chunks = P->step_split[3];
    dn.part = part;
    dn.cnt = reinterpret_cast<unsigned*>(ws + P->off_cnt_down);
    dn.status = status;
    dn.resid = h;
    dn.y = y;
    for (int r = 0; r < N; ++r) dn.W[r] = w->wd[r];
    dn.xact = ws + P->off_act;
    dn.pairs = pairs_off ? reinterpret_cast<unsigned long long*>(ws + pairs_off) : nullptr;
    // q pairs sit at the same distance after the down pieces in the workspace and no-alloc layouts
    unsigned long long* qp =
        pairs_off ? reinterpret_cast<unsigned long long*>(ws + pairs_off + (P->off_q_pairs - P->off_step_pairs)) : nullptr;
    st.g[0].q_pairs = qp;
    st.a.q_pairs = qp;

    st.bar = reinterpret_cast<unsigned long long*>(ws + P->off_step_bar);
    st.kv_ready = reinterpret_cast<unsigned long long*>(ws + P->off_kv_ready);
    st.bar_extra = P->dbg_bar_extra;
    st.stamps = P->n_stage_ev > 0 ? reinterpret_cast<unsigned long long*>(ws + P->off_stamps) : nullptr;
    P->last_stamps_ws = st.stamps ? ws : nullptr;
    // with per-step events recorded around the launch, launch without programmatic overlap
    set_pdl(P->n_stage_ev == 0);
    stage_mark(P, 0, s);
    cudaError_t e = launch_decode_step(st, s);
    if (e != cudaSuccess) return cuda_fail(e, "tp_block_forward: decode step launch");
    for (int i = 1; i < P->n_stage_ev; ++i) stage_mark(P, i, s);
    return ok();
}

// `pairs_off`: byte offset of the down pieces' (value, epoch) buffer in `ws`
// (0: none, the counted finish instead).
static tp_status forward_decode(tp_plan_t P, const tp_shard_set* w, const tp_kv_set* kv, const float* x,
                                float* y, const int32_t* pos, int B, char* ws, size_t pairs_off, cudaStream_t s) {
    const tp_model_desc& d = P->d;
    const tp_plan_info& I = P->info;
    const int N = P->N, T = B;
    for (int r = 0; r < N; ++r) {
        if (!w->wqkv[r] || !w->wo[r] || !w->wgu[r] || !w->wd[r] || !w->gamma_attn[r] || !w->gamma_ffn[r])
            return fail(TP_ERR_NULL, "tp_block_forward: shard %d weight pointer is NULL", r);
        if (d.has_qkv_bias && !w->bqkv[r]) return fail(TP_ERR_NULL, "tp_block_forward: shard %d bias is NULL", r);
        if (!kv->k[r] || !kv->v[r]) return fail(TP_ERR_NULL, "tp_block_forward: shard %d KV cache is NULL", r);
        const void* al[] = {w->wqkv[r], w->wo[r], w->wgu[r], w->wd[r], w->gamma_attn[r], w->gamma_ffn[r]};
        for (const void* p : al)
            if (!aligned16(p)) return fail(TP_ERR_ALIGN, "tp_block_forward: shard %d pointer not 16-byte aligned", r);
    }
    int* status = reinterpret_cast<int*>(ws + P->off_status);
    const size_t es = P->esz;
    // with per-stage events recorded between the launches, launch without
    // programmatic overlap so each event brackets exactly one stage
    set_pdl(P->n_stage_ev == 0);
    const int hd = (int)d.head_dim;

    GemvParams q{};
    q.n_shards = N;
    q.rows = (int)I.qkv_rows;
    q.K = (int)d.hidden;
    q.T = T;
    q.shape = P->g_qkv;
    q.x = x;
    q.eps = (float)d.eps;
    q.part = reinterpret_cast<float*>(ws + P->off_part_qkv);
    q.cnt = reinterpret_cast<unsigned*>(ws + P->off_cnt_qkv);
    q.status = status;
    q.q_out = reinterpret_cast<float*>(ws + P->off_q);
    q.pos = pos;
    q.hq_s = (int)I.hq_shard;
    q.hkv_s = (int)I.hkv_shard;
    q.head_dim = hd;
    q.max_kv = (int)d.max_kv;
    q.log2_theta = std::log2(d.rope_theta);
    for (int r = 0; r < N; ++r) {
        q.W[r] = w->wqkv[r];
        q.gamma[r] = w->gamma_attn[r];
        q.bias[r] = d.has_qkv_bias ? w->bqkv[r] : nullptr;
        q.kcache[r] = kv->k[r];
        q.vcache[r] = kv->v[r];
    }
    const bool bf = d.dtype == TP_BF16;
    cudaError_t e;
    if (bf) {
        // bf16 projections take their RMSNorm operands pre-scaled:
        // x * gamma_r for every shard, and sum(x^2) per token
        NormPrepParams np{};
        np.x = x;
        for (int r = 0; r < N; ++r) np.gamma[r] = w->gamma_attn[r];
        np.N = N;
        np.T = T;
        np.H = (int)d.hidden;
        np.xg = ws + P->off_xg;
        np.ss = reinterpret_cast<float*>(ws + P->off_ss);
        q.xact = ws + P->off_xg;
        q.ss_tiles = np.ss;
        q.n_ss_tiles = (int)((d.hidden + 255) / 256);
        return decode_step_bf16(P, w, kv, x, y, pos, B, ws, pairs_off, s, q, np);
    }
    // fp32: one launch per stage
    stage_mark(P, 0, s);
    e = launch_gemv(q, EPI_QKV_ROPE, d.dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "tp_block_forward: qkv launch");

    AttnDecodeParams a{};
    a.q = q.q_out;
    for (int r = 0; r < N; ++r) {
        a.kcache[r] = kv->k[r];
        a.vcache[r] = kv->v[r];
    }
    a.pos = pos;
    a.N = N;
    a.B = B;
    a.hq_s = (int)I.hq_shard;
    a.hkv_s = (int)I.hkv_shard;
    a.d = hd;
    a.max_kv = (int)d.max_kv;
    a.max_batch = (int)d.max_batch;
    a.n_chunks = P->attn_chunks;
    a.scale = (float)(1.0 / std::sqrt((double)hd));
    a.part = reinterpret_cast<float*>(ws + P->off_attn_part);
    a.cnt = reinterpret_cast<unsigned*>(ws + P->off_cnt_attn);
    a.out = ws + P->off_attn_out;
    a.status = status;
    a.part_units = (unsigned)(P->attn_groups * P->attn_chunks);
    stage_mark(P, 1, s);
    e = launch_attn_decode(a, d.dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "tp_block_forward: attention launch");

    float* h = reinterpret_cast<float*>(ws + P->off_h);
    GemvParams o{};
    o.n_shards = N;
    o.rows = (int)d.hidden;
    o.K = (int)(I.hq_shard * hd);
    o.T = T;
    o.shape = P->g_o;
    o.part = reinterpret_cast<float*>(ws + P->off_part_o);
    o.cnt = reinterpret_cast<unsigned*>(ws + P->off_cnt_o);
    o.status = status;
    o.resid = x;
    o.y = h;
    for (int r = 0; r < N; ++r) {
        o.W[r] = w->wo[r];
        o.act[r] = ws + P->off_attn_out + (size_t)r * kTMax * o.K * es;
        o.gamma2[r] = w->gamma_ffn[r];
    }
    stage_mark(P, 2, s);
    e = launch_gemv(o, EPI_ROWPAR, d.dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "tp_block_forward: o_proj launch");

    GemvParams g{};
    g.n_shards = N;
    g.rows = (int)(2 * I.ffn_shard);
    g.K = (int)d.hidden;
    g.T = T;
    g.shape = P->g_gu;
    g.x = h;
    g.eps = (float)d.eps;
    g.part = reinterpret_cast<float*>(ws + P->off_part_gu);
    g.cnt = reinterpret_cast<unsigned*>(ws + P->off_cnt_gu);
    g.status = status;
    g.act_out = ws + P->off_act;
    g.ffn_s = (int)I.ffn_shard;
    for (int r = 0; r < N; ++r) {
        g.W[r] = w->wgu[r];
        g.gamma[r] = w->gamma_ffn[r];
    }
    stage_mark(P, 3, s);
    e = launch_gemv(g, EPI_SWIGLU, d.dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "tp_block_forward: gate_up launch");

    GemvParams dn{};
    dn.n_shards = N;
    dn.rows = (int)d.hidden;
    dn.K = (int)I.ffn_shard;
    dn.T = T;
    dn.shape = P->g_down;
    dn.part = reinterpret_cast<float*>(ws + P->off_part_down);
    dn.cnt = reinterpret_cast<unsigned*>(ws + P->off_cnt_down);
    dn.status = status;
    dn.resid = h;
    dn.y = y;
    for (int r = 0; r < N; ++r) {
        dn.W[r] = w->wd[r];
        dn.act[r] = ws + P->off_act + (size_t)r * kTMax * dn.K * es;
    }
    stage_mark(P, 4, s);
    e = launch_gemv(dn, EPI_ROWPAR, d.dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "tp_block_forward: down launch");
    stage_mark(P, 5, s);
    return ok();
}

static tp_status forward_moe(tp_plan_t P, const tp_shard_set* w, const float* x, float* y, const float* logits,
                             int T, char* ws, cudaStream_t s) {
    const tp_model_desc& d = P->d;
    const int N = P->N;
    for (int r = 0; r < N; ++r) {
        if (!w->egu[r] || !w->ed[r] || !w->gamma_ffn[r])
            return fail(TP_ERR_NULL, "tp_block_forward: shard %d expert weights or gamma_ffn NULL", r);
        if (!aligned16(w->egu[r]) || !aligned16(w->ed[r]) || !aligned16(w->gamma_ffn[r]))
            return fail(TP_ERR_ALIGN, "tp_block_forward: shard %d expert pointer not 16-byte aligned", r);
    }
    if (!aligned16(logits)) return fail(TP_ERR_ALIGN, "tp_block_forward: router_logits not 16-byte aligned");
    MoeParams m{};
    m.N = N;
    m.T = T;
    m.H = (int)d.hidden;
    m.E = (int)d.n_experts;
    m.top_k = (int)d.top_k;
    m.Fs = (int)P->info.expert_ffn_shard;
    m.El = (int)P->info.experts_shard;
    m.ep = d.expert_parallel;
    m.eps = (float)d.eps;
    m.x = x;
    m.logits = logits;
    for (int r = 0; r < N; ++r) {
        m.gamma[r] = w->gamma_ffn[r];
        m.egu[r] = w->egu[r];
        m.ed[r] = w->ed[r];
    }
    m.ids = reinterpret_cast<int*>(ws + P->off_m_ids);
    m.wts = reinterpret_cast<float*>(ws + P->off_m_wts);
    m.offsets = reinterpret_cast<int*>(ws + P->off_m_off);
    m.perm = reinterpret_cast<int*>(ws + P->off_m_perm);
    m.slot_of = reinterpret_cast<int*>(ws + P->off_m_slot);
    m.rinv = reinterpret_cast<float*>(ws + P->off_m_rinv);
    m.xs = ws + P->off_m_xs;
    m.act = ws + P->off_m_act;
    m.o = reinterpret_cast<float*>(ws + P->off_m_o);
    m.y = y;
    m.status = reinterpret_cast<int*>(ws + P->off_status);
    set_pdl(P->n_stage_ev == 0);
    cudaError_t e = launch_moe(m, s, P->stage_ev, P->n_stage_ev < 5 ? P->n_stage_ev : 5);
    if (e != cudaSuccess) return cuda_fail(e, "tp_block_forward: MoE launch");
    return ok();
}

// Prefill: B sequences of S new tokens each (T = B*S rows, sequence-major).
// Stages: RMSNorm -> column-parallel QKV + RoPE + KV append (tensor cores)
// -> causal attention per shard -> row-parallel o_proj with the rank-ordered
// reduction and residual -> RMSNorm -> column-parallel gate/up + SwiGLU ->
// row-parallel down + reduction + residual.
static tp_status forward_prefill(tp_plan_t P, const tp_shard_set* w, const tp_kv_set* kv, const float* x, float* y,
                                 const int32_t* pos, int B, int S, char* ws, cudaStream_t s) {
    const tp_model_desc& d = P->d;
    const tp_plan_info& I = P->info;
    const int N = P->N, T = B * S, H = (int)d.hidden, hd = (int)d.head_dim;
    for (int r = 0; r < N; ++r) {
        if (!w->wqkv[r] || !w->wo[r] || !w->wgu[r] || !w->wd[r] || !w->gamma_attn[r] || !w->gamma_ffn[r])
            return fail(TP_ERR_NULL, "tp_block_forward: shard %d weight pointer is NULL", r);
        if (d.has_qkv_bias && !w->bqkv[r]) return fail(TP_ERR_NULL, "tp_block_forward: shard %d bias is NULL", r);
        if (!kv->k[r] || !kv->v[r]) return fail(TP_ERR_NULL, "tp_block_forward: shard %d KV cache is NULL", r);
        const void* al[] = {w->wqkv[r], w->wo[r], w->wgu[r], w->wd[r], w->gamma_attn[r], w->gamma_ffn[r],
                            kv->k[r], kv->v[r]};
        for (const void* p : al)
            if (!aligned16(p)) return fail(TP_ERR_ALIGN, "tp_block_forward: shard %d pointer not 16-byte aligned", r);
    }
    int* status = reinterpret_cast<int*>(ws + P->off_status);
    void* xn = ws + P->off_p_xn;
    void* q = ws + P->off_p_q;
    void* ao = ws + P->off_p_ao;
    float* h = reinterpret_cast<float*>(ws + P->off_p_h);
    void* act = ws + P->off_p_act;
    float2* rope = reinterpret_cast<float2*>(ws + P->off_p_rope);
    // the gamma of a replicated norm is one tensor: shards that point at the
    // same gamma share one normalised copy
    auto distinct = [&](const float* const* g) {
        for (int r = 1; r < N; ++r)
            if (g[r] != g[0]) return N;
        return 1;
    };
    const int na = distinct(w->gamma_attn), nf = distinct(w->gamma_ffn);
    cudaError_t e;
    const double log2_theta = std::log2(d.rope_theta);
    stage_mark(P, 0, s);
    e = launch_rope_table(rope, (int)d.max_kv, hd, log2_theta, s);
    if (e == cudaSuccess) e = launch_prefill_norm(x, w->gamma_attn, na, xn, T, H, (float)d.eps, s);
    if (e != cudaSuccess) return cuda_fail(e, "tp_block_forward: prefill norm launch");

    PrefillColParams c{};
    c.A = xn;
    c.a_copies = na;
    c.N = N;
    c.T = T;
    c.K = H;
    c.rows = (int)I.qkv_rows;
    c.S = S;
    c.hq_s = (int)I.hq_shard;
    c.hkv_s = (int)I.hkv_shard;
    c.d = hd;
    c.max_kv = (int)d.max_kv;
    c.ffn_s = (int)I.ffn_shard;
    for (int r = 0; r < N; ++r) {
        c.W[r] = w->wqkv[r];
        c.bias[r] = d.has_qkv_bias ? w->bqkv[r] : nullptr;
        c.kcache[r] = kv->k[r];
        c.vcache[r] = kv->v[r];
    }
    c.pos = pos;
    c.rope = rope;
    c.q_out = q;
    c.act = act;
    c.status = status;
    e = launch_tc_col(0, c, s);
    if (e != cudaSuccess) return cuda_fail(e, "tp_block_forward: prefill QKV launch");
    stage_mark(P, 1, s);

    FlashParams f{};
    f.q = q;
    for (int r = 0; r < N; ++r) {
        f.kcache[r] = kv->k[r];
        f.vcache[r] = kv->v[r];
    }
    f.out = ao;
    f.pos = pos;
    f.N = N;
    f.B = B;
    f.S = S;
    f.T = T;
    f.hq_s = (int)I.hq_shard;
    f.hkv_s = (int)I.hkv_shard;
    f.max_kv = (int)d.max_kv;
    f.max_batch = (int)d.max_batch;
    f.d = hd;
    f.scale = (float)(1.0 / std::sqrt((double)hd));
    f.status = status;
    e = launch_flash_prefill(f, s);
    if (e != cudaSuccess) return cuda_fail(e, "tp_block_forward: prefill attention launch");
    stage_mark(P, 2, s);

    PrefillRowParams o{};
    o.A = ao;
    o.N = N;
    o.T = T;
    o.Kr = (int)(I.hq_shard * hd);
    o.H = H;
    for (int r = 0; r < N; ++r) o.W[r] = w->wo[r];
    o.resid = x;
    o.out = h;
    o.status = status;
    e = launch_tc_row(o, s);
    if (e != cudaSuccess) return cuda_fail(e, "tp_block_forward: prefill o_proj launch");
    stage_mark(P, 3, s);

    e = launch_prefill_norm(h, w->gamma_ffn, nf, xn, T, H, (float)d.eps, s);
    if (e != cudaSuccess) return cuda_fail(e, "tp_block_forward: prefill norm launch");
    c.a_copies = nf;
    c.rows = (int)(2 * I.ffn_shard);
    for (int r = 0; r < N; ++r) c.W[r] = w->wgu[r];
    e = launch_tc_col(1, c, s);
    if (e != cudaSuccess) return cuda_fail(e, "tp_block_forward: prefill gate/up launch");
    stage_mark(P, 4, s);

    PrefillRowParams dn{};
    dn.A = act;
    dn.N = N;
    dn.T = T;
    dn.Kr = (int)I.ffn_shard;
    dn.H = H;
    for (int r = 0; r < N; ++r) dn.W[r] = w->wd[r];
    dn.resid = h;
    dn.out = y;
    dn.status = status;
    e = launch_tc_row(dn, s);
    if (e != cudaSuccess) return cuda_fail(e, "tp_block_forward: prefill down launch");
    stage_mark(P, 5, s);
    return ok();
}

extern "C" tp_status tp_block_forward(tp_plan_t plan, const tp_shard_set* w, const tp_kv_set* kv,
                                      const float* x, float* y, const int32_t* pos, int32_t B,
                                      int32_t T_per_seq, int32_t mode, const float* router_logits,
                                      void* workspace, size_t workspace_bytes, void* stream) {
    if (!plan || !w || !x || !y || !workspace) return fail(TP_ERR_NULL, "tp_block_forward: NULL argument");
    if (x == y) return fail(TP_ERR_INVALID_ARG, "tp_block_forward: y must not alias x");
    if (B < 1 || T_per_seq < 1) return fail(TP_ERR_SHAPE, "tp_block_forward: B and T_per_seq must be >= 1");
    if (B > plan->d.max_batch || (int64_t)B * T_per_seq > plan->d.max_tokens)
        return fail(TP_ERR_SHAPE, "tp_block_forward: B=%d x T=%d exceeds the plan's max_batch/max_tokens", B, T_per_seq);
    if (workspace_bytes < plan->ws_bytes)
        return fail(TP_ERR_CAPACITY, "tp_block_forward: workspace %zu bytes < required %zu", workspace_bytes,
                    plan->ws_bytes);
    if (!aligned16(workspace) || !aligned16(x) || !aligned16(y))
        return fail(TP_ERR_ALIGN, "tp_block_forward: x, y and workspace must be 16-byte aligned");
    tp_status st = check_device();
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    (void)router_logits;
    if (mode == TP_MODE_DECODE) {
        if (!plan->dense) return fail(TP_ERR_INVALID_ARG, "tp_block_forward: DECODE needs an attention block");
        if (!kv || !pos) return fail(TP_ERR_NULL, "tp_block_forward: DECODE needs kv and pos");
        if (T_per_seq != 1) return fail(TP_ERR_SHAPE, "tp_block_forward: DECODE takes T_per_seq == 1");
        if (B > kTMax) return fail(TP_ERR_SHAPE, "tp_block_forward: DECODE handles at most %d sequences", kTMax);
        return forward_decode(plan, w, kv, x, y, pos, B, ws, plan->off_step_pairs, s);
    }
    if (mode == TP_MODE_MOE_FFN) {
        if (!plan->moe) return fail(TP_ERR_INVALID_ARG, "tp_block_forward: MOE_FFN needs a plan with experts");
        if (!router_logits) return fail(TP_ERR_NULL, "tp_block_forward: MOE_FFN needs router_logits");
        if (plan->d.dtype != TP_BF16) return fail(TP_ERR_UNSUPPORTED, "tp_block_forward: MOE_FFN runs on bf16 weights");
        if (plan->d.hidden % 256 || plan->info.expert_ffn_shard % 256)
            return fail(TP_ERR_UNSUPPORTED, "tp_block_forward: MOE_FFN needs hidden and expert_ffn/tp multiples of 256");
        return forward_moe(plan, w, x, y, router_logits, B * T_per_seq, ws, s);
    }
    if (mode == TP_MODE_PREFILL) {
        if (!plan->dense) return fail(TP_ERR_INVALID_ARG, "tp_block_forward: PREFILL needs an attention block");
        if (!kv || !pos) return fail(TP_ERR_NULL, "tp_block_forward: PREFILL needs kv and pos");
        if (plan->d.dtype != TP_BF16)
            return fail(TP_ERR_UNSUPPORTED, "tp_block_forward: PREFILL runs on bf16 weights (fp32 plans: DECODE)");
        if ((int64_t)T_per_seq > plan->d.max_kv)
            return fail(TP_ERR_CAPACITY, "tp_block_forward: T_per_seq=%d exceeds max_kv=%lld", T_per_seq,
                        (long long)plan->d.max_kv);
        return forward_prefill(plan, w, kv, x, y, pos, B, T_per_seq, ws, s);
    }
    return fail(TP_ERR_INVALID_ARG, "tp_block_forward: unknown mode %d", mode);
}

extern "C" tp_status tp_reduce_partials(tp_plan_t plan, const float* partials, const float* residual,
                                        const float* bias, float* out, int64_t M, void* stream) {
    if (!plan || !partials || !out) return fail(TP_ERR_NULL, "tp_reduce_partials: NULL argument");
    if (M < 0) return fail(TP_ERR_SHAPE, "tp_reduce_partials: M must be >= 0");
    tp_status st = check_device();
    if (st) return st;
    cudaError_t e = launch_reduce_partials(partials, residual, bias, out, plan->N, M, plan->d.hidden,
                                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tp_reduce_partials: launch");
    return ok();
}

extern "C" tp_status tp_gemm_bf16(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K,
                                  int32_t* device_status, void* stream) {
    if (!A || !B || !C) return fail(TP_ERR_NULL, "tp_gemm_bf16: NULL operand");
    if (M <= 0 || N <= 0 || K <= 0 || M % 128 || N % 256 || K % 64 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return fail(TP_ERR_SHAPE, "tp_gemm_bf16: need M %% 128 == 0, N %% 256 == 0, K %% 64 == 0 (got %lld, %lld, %lld)",
                    (long long)M, (long long)N, (long long)K);
    if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return fail(TP_ERR_ALIGN, "tp_gemm_bf16: pointers must be 16-byte aligned");
    tp_status st = check_device();
    if (st) return st;
    cudaError_t e = launch_tc_gemm_plain(A, B, C, (int)M, (int)N, (int)K, device_status, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tp_gemm_bf16: launch");
    return ok();
}

extern "C" tp_status tp_gemm_bf16_kn(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K,
                                     int32_t* device_status, void* stream) {
    if (!A || !B || !C) return fail(TP_ERR_NULL, "tp_gemm_bf16_kn: NULL operand");
    if (M <= 0 || N <= 0 || K <= 0 || M % 128 || N % 256 || K % 64 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return fail(TP_ERR_SHAPE, "tp_gemm_bf16_kn: need M %% 128 == 0, N %% 256 == 0, K %% 64 == 0 (got %lld, %lld, %lld)",
                    (long long)M, (long long)N, (long long)K);
    if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return fail(TP_ERR_ALIGN, "tp_gemm_bf16_kn: pointers must be 16-byte aligned");
    tp_status st = check_device();
    if (st) return st;
    cudaError_t e = launch_tc_gemm_plain(A, B, C, (int)M, (int)N, (int)K, device_status, static_cast<cudaStream_t>(stream),
                                         true);
    if (e != cudaSuccess) return cuda_fail(e, "tp_gemm_bf16_kn: launch");
    return ok();
}

extern "C" tp_status tp_get_device_status(void* workspace, int32_t* out, void* stream) {
    if (!workspace || !out) return fail(TP_ERR_NULL, "tp_get_device_status: NULL argument");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    TP_CUDA(cudaMemcpyAsync(out, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s), "tp_get_device_status: copy");
    TP_CUDA(cudaStreamSynchronize(s), "tp_get_device_status: sync");
    return ok();
}

extern "C" tp_status tp_profile_stages(tp_plan_t plan, void* const* events, int32_t n_events) {
    if (!plan) return fail(TP_ERR_NULL, "tp_profile_stages: plan is NULL");
    if (n_events < 0 || n_events > 16) return fail(TP_ERR_INVALID_ARG, "tp_profile_stages: 0..16 events");
    plan->n_stage_ev = events ? n_events : 0;
    for (int i = 0; i < plan->n_stage_ev; ++i) plan->stage_ev[i] = static_cast<cudaEvent_t>(events[i]);
    return ok();
}

extern "C" tp_status tp_profile_phases(tp_plan_t plan, double* out_us, double* median_us, int32_t n,
                                       void* stream) {
    if (!plan || !out_us) return fail(TP_ERR_NULL, "tp_profile_phases: NULL argument");
    if (n < 1 || n > kStepStamps - 1) return fail(TP_ERR_INVALID_ARG, "tp_profile_phases: n must be 1..%d", kStepStamps - 1);
    if (!plan->last_stamps_ws)
        return fail(TP_ERR_INVALID_ARG, "tp_profile_phases: no bf16 DECODE step ran while tp_profile_stages was set");
    int dev = 0, sms = 0;
    TP_CUDA(cudaGetDevice(&dev), "tp_profile_phases: cudaGetDevice");
    TP_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "tp_profile_phases: SM count");
    const int rows = sms < kMaxStepCtas ? sms : kMaxStepCtas;
    std::vector<unsigned long long> h((size_t)rows * kStepStamps);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    TP_CUDA(cudaMemcpyAsync(h.data(), plan->last_stamps_ws + plan->off_stamps, h.size() * 8, cudaMemcpyDeviceToHost, s),
            "tp_profile_phases: copy");
    TP_CUDA(cudaStreamSynchronize(s), "tp_profile_phases: sync");
    // phase i ends when its barrier completes, i.e. at the latest arrival
    unsigned long long prev = ~0ull;
    for (int c = 0; c < rows; ++c) prev = std::min(prev, h[(size_t)c * kStepStamps]);
    std::vector<unsigned long long> arr(rows);
    for (int i = 0; i < n; ++i) {
        unsigned long long end = 0;
        for (int c = 0; c < rows; ++c) {
            arr[c] = h[(size_t)c * kStepStamps + i + 1];
            end = std::max(end, arr[c]);
        }
        out_us[i] = end >= prev ? (double)(end - prev) * 1e-3 : 0.0;
        if (median_us) {
            std::nth_element(arr.begin(), arr.begin() + rows / 2, arr.end());
            const unsigned long long med = arr[rows / 2];
            median_us[i] = med >= prev ? (double)(med - prev) * 1e-3 : 0.0;
        }
        prev = end;
    }
    return ok();
}

extern "C" tp_status tp_profile_phase_stamps(tp_plan_t plan, uint64_t* out, int32_t rows, void* stream) {
    if (!plan || !out) return fail(TP_ERR_NULL, "tp_profile_phase_stamps: NULL argument");
    if (rows < 1 || rows > kMaxStepCtas) return fail(TP_ERR_INVALID_ARG, "tp_profile_phase_stamps: rows 1..%d", kMaxStepCtas);
    if (!plan->last_stamps_ws)
        return fail(TP_ERR_INVALID_ARG, "tp_profile_phase_stamps: no bf16 DECODE step ran while tp_profile_stages was set");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    TP_CUDA(cudaMemcpyAsync(out, plan->last_stamps_ws + plan->off_stamps, (size_t)rows * kStepStamps * 8,
                            cudaMemcpyDeviceToHost, s), "tp_profile_phase_stamps: copy");
    TP_CUDA(cudaStreamSynchronize(s), "tp_profile_phase_stamps: sync");
    return ok();
}

extern "C" tp_status tp_debug_withhold_arrival(tp_plan_t plan, int32_t on) {
    if (!plan) return fail(TP_ERR_NULL, "tp_debug_withhold_arrival: NULL plan");
    if (on != 0 && on != 1) return fail(TP_ERR_INVALID_ARG, "tp_debug_withhold_arrival: on must be 0 or 1");
    plan->dbg_bar_extra = (unsigned)on;
    return ok();
}

extern "C" const char* tp_last_error(void) { return g_err; }

extern "C" int32_t tp_version(void) { return TP_ABI_VERSION; }

// ---------------------------------------------------------------- decode with library-owned scratch

// Scratch of tp_block_forward_noalloc: one array in device global memory per
// GPU that loads this library, held until the process exits. Host code must
// not use the array's name as an address (on the host it only stands for the
// symbol); its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TP_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};
}  // namespace

// Device address of the array on the current device, looked up once per
// device (with that device current) and remembered.
static tp_status noalloc_scratch(void** out) {
    int dev = 0;
    TP_CUDA(cudaGetDevice(&dev), "tp_block_forward_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(TP_ERR_UNSUPPORTED, "tp_block_forward_noalloc: device index %d above %d", dev, kMaxDevices - 1);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "tp_block_forward_noalloc: cudaGetSymbolAddress");
        if (!p) return fail(TP_ERR_CUDA, "tp_block_forward_noalloc: no device address for the scratch array");
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return TP_OK;
}

extern "C" tp_status tp_block_forward_noalloc(tp_plan_t plan, const tp_shard_set* w, const tp_kv_set* kv,
                                              const float* x, float* y, const int32_t* pos, int32_t B,
                                              void* stream) {
    if (!plan || !w || !kv || !x || !y || !pos) return fail(TP_ERR_NULL, "tp_block_forward_noalloc: NULL argument");
    if (!plan->dense) return fail(TP_ERR_INVALID_ARG, "tp_block_forward_noalloc: the plan has no attention block");
    if (x == y) return fail(TP_ERR_INVALID_ARG, "tp_block_forward_noalloc: y must not alias x");
    if (B < 1 || B > plan->d.max_batch || B > kTMax)
        return fail(TP_ERR_SHAPE, "tp_block_forward_noalloc: B=%d outside 1..min(max_batch, %d)", B, kTMax);
    // na_end covers every byte the decode step touches: control words, the
    // decode buffers and the down pieces' pair buffer placed right after them
    if (plan->na_end > (size_t)TP_NOALLOC_SCRATCH_BYTES)
        return fail(TP_ERR_CAPACITY,
                    "tp_block_forward_noalloc: this plan's decode needs %zu bytes of scratch; the static array "
                    "holds %lld (use tp_block_forward with a caller workspace)",
                    plan->na_end, (long long)TP_NOALLOC_SCRATCH_BYTES);
    if (!aligned16(x) || !aligned16(y)) return fail(TP_ERR_ALIGN, "tp_block_forward_noalloc: x and y must be 16-byte aligned");
    tp_status st = check_device();
    if (st) return st;
    void* scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(scratch);
    // The array keeps whatever the previous call (of any plan) left. Counters,
    // status word and grid-barrier counter start at zero, so this launch's
    // epoch is 1; the pair buffer starts at zero too, so no piece of an
    // earlier call (also epoch 1) can pass for one of this call's.
    TP_CUDA(cudaMemsetAsync(base, 0, plan->ctrl_bytes, s), "tp_block_forward_noalloc: clearing counters");
    if (plan->na_pairs_off)
        TP_CUDA(cudaMemsetAsync(base + plan->na_pairs_off, 0, plan->na_end - plan->na_pairs_off, s),
                "tp_block_forward_noalloc: clearing the pair buffers");
    return forward_decode(plan, w, kv, x, y, pos, B, base, plan->na_pairs_off, s);
}

extern "C" tp_status tp_noalloc_status(int32_t* out, void* stream) {
    if (!out) return fail(TP_ERR_NULL, "tp_noalloc_status: NULL argument");
    tp_status st = check_device();
    if (st) return st;
    void* scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the status word is the first word of every plan's layout
    TP_CUDA(cudaMemcpyAsync(out, scratch, sizeof(int32_t), cudaMemcpyDeviceToHost, s), "tp_noalloc_status: copy");
    TP_CUDA(cudaStreamSynchronize(s), "tp_noalloc_status: sync");
    return ok();
}

// ---------------------------------------------------------------- several decode blocks in one launch

struct tp_stack_s {
    tp_plan_t plan = nullptr;
    int L = 0;
    void* dev = nullptr;         // tensor maps, layer records, item tables (device memory)
    tpk::ChainArgs a{};          // per-call fields filled by tp_stack_decode
    size_t smem = 0;
};

namespace {

// Chunks of 64 columns per box (odd, at most kmax) and loads per item for a
// reduction of nch chunks.
void chain_split(int nch, int kmax, int& kc, int& nl) {
    const int n = (nch + kmax - 1) / kmax;
    kc = (nch + n - 1) / n;
    if (!(kc & 1)) ++kc;
    nl = (nch + kc - 1) / kc;
}

}  // namespace

extern "C" tp_status tp_stack_create(tp_plan_t plan, int32_t n_layers, const tp_shard_set* w, const tp_kv_set* kv,
                                     tp_stack_t* out) {
    using namespace tpk;
    if (!plan || !w || !kv || !out) return fail(TP_ERR_NULL, "tp_stack_create: NULL argument");
    *out = nullptr;
    const tp_model_desc& d = plan->d;
    const tp_plan_info& I = plan->info;
    if (!plan->dense) return fail(TP_ERR_INVALID_ARG, "tp_stack_create: the plan has no attention block");
    if (d.dtype != TP_BF16) return fail(TP_ERR_UNSUPPORTED, "tp_stack_create: bf16 plans only");
    if (plan->off_c_end <= plan->off_c_begin || plan->c_ck <= 0)
        return fail(TP_ERR_UNSUPPORTED, "tp_stack_create: head_dim must be 64 or 128");
    if (n_layers < 1 || n_layers > 255) return fail(TP_ERR_INVALID_ARG, "tp_stack_create: n_layers %d outside 1..255", n_layers);
    const int N = plan->N, H = (int)d.hidden, hd = (int)d.head_dim, G = (int)(d.n_heads / d.n_kv_heads);
    const int MB = (int)d.max_batch, hq_s = (int)I.hq_shard, hkv_s = (int)I.hkv_shard, F_s = (int)I.ffn_shard;
    const int qkv_rows = (int)I.qkv_rows;
    if (G > 8) return fail(TP_ERR_UNSUPPORTED, "tp_stack_create: at most 8 query heads per KV head (got %d)", G);
    if (MB > kTMax) return fail(TP_ERR_UNSUPPORTED, "tp_stack_create: max_batch above %d", kTMax);
    const long groups = (long)N * MB * hkv_s;
    for (int l = 0; l < n_layers; ++l)
        for (int r = 0; r < N; ++r) {
            const tp_shard_set& s = w[l];
            if (!s.wqkv[r] || !s.wo[r] || !s.wgu[r] || !s.wd[r] || !s.gamma_attn[r] || !s.gamma_ffn[r] ||
                !kv[l].k[r] || !kv[l].v[r])
                return fail(TP_ERR_NULL, "tp_stack_create: layer %d shard %d pointer is NULL", l, r);
            if (d.has_qkv_bias && !s.bqkv[r]) return fail(TP_ERR_NULL, "tp_stack_create: layer %d shard %d bias is NULL", l, r);
            const void* al[] = {s.wqkv[r], s.wo[r], s.wgu[r], s.wd[r], s.gamma_attn[r], s.gamma_ffn[r], kv[l].k[r],
                                kv[l].v[r]};
            for (const void* p : al)
                if (!aligned16(p)) return fail(TP_ERR_ALIGN, "tp_stack_create: layer %d shard %d pointer not 16-byte aligned", l, r);
        }
    tp_status st = check_device();
    if (st) return st;
    int dev = 0, sms = 0, smem_max = 0;
    TP_CUDA(cudaGetDevice(&dev), "tp_stack_create: cudaGetDevice");
    TP_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "tp_stack_create: SM count");
    TP_CUDA(cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev), "tp_stack_create: smem");
    const int grid = std::min(sms, kChainMaxCtas);

    ChainArgs A{};
    A.H = H;
    A.N = N;
    A.hq_s = hq_s;
    A.hkv_s = hkv_s;
    A.d = hd;
    A.G = G;
    A.qkv_rows = qkv_rows;
    A.F_s = F_s;
    A.max_batch = MB;
    A.max_kv = (int)d.max_kv;
    A.L = n_layers;
    A.grid = grid;
    A.ck = plan->c_ck;
    A.maxch = plan->c_maxch;
    A.eps = (float)d.eps;
    A.log2_theta = (float)std::log2(d.rope_theta);
    A.qscale = (float)(1.4426950408889634 / std::sqrt((double)hd));
    chain_split(H / 64, 15, A.kc[0], A.nl[0]);
    chain_split(hq_s * hd / 64, 15, A.kc[1], A.nl[1]);
    chain_split(H / 64, 7, A.kc[2], A.nl[2]);
    chain_split(F_s / 64, 15, A.kc[3], A.nl[3]);
    for (int k = 0; k < 4; ++k) {   // loads per item stay small (the kernel's item decoding assumes at most 64)
        const int loads = (k == 1 || k == 3 ? N : 1) * A.nl[k];
        if (loads > 64)
            return fail(TP_ERR_UNSUPPORTED, "tp_stack_create: %d loads per item of phase %d exceed 64", loads, k);
    }
    A.xa_stride = std::max(N * hq_s * hd, N * F_s) + 8;   // bf16 operands of o_proj and down
    size_t smem = 0;
    for (A.n_slots = kChainMaxSlots; A.n_slots >= 4; --A.n_slots) {
        smem = chain_smem(A);
        if (smem <= (size_t)smem_max) break;
    }
    if (A.n_slots < 4)
        return fail(TP_ERR_UNSUPPORTED, "tp_stack_create: operands of this shape leave no room for the weight ring");

    // ---- items of the projection phases: each phase dealt round robin over
    // the CTAs (a phase lasts as long as its busiest CTA), starting each phase
    // after the CTAs the previous phases loaded most, so the bytes spread too
    const int nph[4] = {N * qkv_rows / 8, H / 8, N * F_s / 8, H / 8};
    const long bph[4] = {16L * H, 16L * N * hq_s * hd, 32L * H, 16L * N * F_s};
    // o_proj and down items: one residual double pair per consumer thread (items x tokens x 4 <= 256)
    const int cap[4] = {kChainMaxItems, std::min(kChainMaxItems, 64 / MB), kChainMaxItems,
                        std::min(kChainMaxItems, 64 / MB)};
    std::vector<long> load(grid, 0);
    std::vector<std::vector<int>> own(4 * (size_t)grid);
    const int order_ph[4] = {3, 2, 0, 1};                   // down, gate/up, qkv, o_proj
    for (int k = 0; k < 4; ++k) {
        const int p = order_ph[k];
        if (nph[p] > (long)grid * cap[p])
            return fail(TP_ERR_UNSUPPORTED, "tp_stack_create: %d items of phase %d exceed %d CTAs x %d", nph[p], p, grid,
                        cap[p]);
        std::vector<int> by_load(grid);
        for (int c = 0; c < grid; ++c) by_load[c] = c;
        std::stable_sort(by_load.begin(), by_load.end(), [&](int x, int y) { return load[x] < load[y]; });
        for (int i = 0; i < nph[p]; ++i) {
            const int c = by_load[i % grid];
            own[(size_t)p * grid + c].push_back(i);
            load[c] += bph[p];
        }
    }
    for (auto& v : own) std::sort(v.begin(), v.end());   // shard-major: one normalised operand per shard run
    std::vector<int> tab;
    for (int p = 0; p < 4; ++p) {
        A.tab_off[p] = (int)tab.size();
        int acc = 0;
        for (int c = 0; c < grid; ++c) {
            tab.push_back(acc);
            acc += (int)own[(size_t)p * grid + c].size();
        }
        tab.push_back(acc);
        for (int c = 0; c < grid; ++c)
            for (int id : own[(size_t)p * grid + c]) tab.push_back(id);
    }
    // attention items go round robin over the CTAs, least loaded first
    std::vector<int> order(grid);
    for (int c = 0; c < grid; ++c) order[c] = c;
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return load[x] < load[y]; });
    std::vector<int> rank(grid);
    for (int i = 0; i < grid; ++i) rank[order[i]] = i;

    // ---- device buffer: maps [L][6][N], layer records [L], tables, ranks
    const size_t n_maps = (size_t)n_layers * kChainMaps * N;
    const size_t off_lay = n_maps * sizeof(CUtensorMap);
    const size_t off_tab = off_lay + (size_t)n_layers * sizeof(ChainLayer);
    const size_t off_rank = off_tab + tab.size() * sizeof(int);
    const size_t off_rope = (off_rank + (size_t)grid * sizeof(int) + 15) & ~(size_t)15;
    const size_t bytes = off_rope + (size_t)d.max_kv * (hd / 2) * 2 * sizeof(float);
    std::vector<unsigned char> host(bytes, 0);
    CUtensorMap* maps = reinterpret_cast<CUtensorMap*>(host.data());
    ChainLayer* lays = reinterpret_cast<ChainLayer*>(host.data() + off_lay);
    const long kv_rows = (long)MB * hkv_s * d.max_kv;
    for (int l = 0; l < n_layers; ++l) {
        for (int r = 0; r < N; ++r) {
            CUtensorMap* m = maps + (size_t)l * kChainMaps * N;
            cudaError_t e = chain_map(w[l].wqkv[r], H, qkv_rows, A.kc[0], 8, &m[0 * N + r]);
            if (e == cudaSuccess) e = chain_map(w[l].wo[r], (long)hq_s * hd, H, A.kc[1], 8, &m[1 * N + r]);
            if (e == cudaSuccess) e = chain_map(w[l].wgu[r], H, 2L * F_s, A.kc[2], 8, &m[2 * N + r]);
            if (e == cudaSuccess) e = chain_map(w[l].wd[r], F_s, H, A.kc[3], 8, &m[3 * N + r]);
            if (e == cudaSuccess) e = chain_map(kv[l].k[r], hd, kv_rows, hd / 64, A.ck, &m[4 * N + r]);
            if (e == cudaSuccess) e = chain_map(kv[l].v[r], hd, kv_rows, hd / 64, A.ck, &m[5 * N + r]);
            if (e != cudaSuccess) return cuda_fail(e, "tp_stack_create: tensor map");
            lays[l].bqkv[r] = d.has_qkv_bias ? w[l].bqkv[r] : nullptr;
            lays[l].g_attn[r] = w[l].gamma_attn[r];
            lays[l].g_ffn[r] = w[l].gamma_ffn[r];
            lays[l].kc[r] = kv[l].k[r];
            lays[l].vc[r] = kv[l].v[r];
        }
    }
    memcpy(host.data() + off_tab, tab.data(), tab.size() * sizeof(int));
    memcpy(host.data() + off_rank, rank.data(), (size_t)grid * sizeof(int));
    // rotary table: angle pos * theta^(-2e/d) for pair e, in double, rounded once
    float* rope = reinterpret_cast<float*>(host.data() + off_rope);
    for (long p = 0; p < d.max_kv; ++p)
        for (int e = 0; e < hd / 2; ++e) {
            const double ang = (double)p * std::pow(d.rope_theta, -2.0 * e / hd);
            rope[(p * (hd / 2) + e) * 2] = (float)std::cos(ang);
            rope[(p * (hd / 2) + e) * 2 + 1] = (float)std::sin(ang);
        }
    tp_stack_s* S = new (std::nothrow) tp_stack_s();
    if (!S) return fail(TP_ERR_INVALID_ARG, "tp_stack_create: out of host memory");
    cudaError_t e = cudaMalloc(&S->dev, bytes);
    if (e == cudaSuccess) e = cudaMemcpy(S->dev, host.data(), bytes, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        if (S->dev) cudaFree(S->dev);
        delete S;
        return cuda_fail(e, "tp_stack_create: device tables");
    }
    unsigned char* db = static_cast<unsigned char*>(S->dev);
    A.maps = reinterpret_cast<const CUtensorMap*>(db);
    A.layers = reinterpret_cast<const ChainLayer*>(db + off_lay);
    A.tab = reinterpret_cast<const int*>(db + off_tab);
    A.att_rank = reinterpret_cast<const int*>(db + off_rank);
    A.rope = reinterpret_cast<const float2*>(db + off_rope);
    S->plan = plan;
    S->L = n_layers;
    S->a = A;
    S->smem = smem;
    *out = S;
    return ok();
}

extern "C" tp_status tp_stack_set_stamps(tp_stack_t stack, uint64_t* stamps, int32_t rows) {
    if (!stack) return fail(TP_ERR_NULL, "tp_stack_set_stamps: NULL stack");
    if (stamps && rows < stack->a.grid)
        return fail(TP_ERR_SHAPE, "tp_stack_set_stamps: %d rows < %d CTAs", rows, stack->a.grid);
    stack->a.stamps = reinterpret_cast<unsigned long long*>(stamps);
    return ok();
}

extern "C" int32_t tp_stack_ctas(tp_stack_t stack) { return stack ? stack->a.grid : 0; }

extern "C" void tp_stack_destroy(tp_stack_t stack) {
    if (!stack) return;
    if (stack->dev) cudaFree(stack->dev);
    delete stack;
}

extern "C" tp_status tp_stack_decode(tp_stack_t stack, const float* x, float* y, const int32_t* pos, int32_t B,
                                     void* workspace, size_t workspace_bytes, void* stream) {
    if (!stack || !x || !y || !pos || !workspace) return fail(TP_ERR_NULL, "tp_stack_decode: NULL argument");
    tp_plan_t P = stack->plan;
    if (x == y) return fail(TP_ERR_INVALID_ARG, "tp_stack_decode: y must not alias x");
    if (B < 1 || B > P->d.max_batch || B > tpk::kTMax)
        return fail(TP_ERR_SHAPE, "tp_stack_decode: B=%d outside 1..min(max_batch, %d)", B, tpk::kTMax);
    if (workspace_bytes < P->ws_bytes)
        return fail(TP_ERR_CAPACITY, "tp_stack_decode: workspace %zu bytes < required %zu", workspace_bytes, P->ws_bytes);
    if (!aligned16(workspace) || !aligned16(x) || !aligned16(y))
        return fail(TP_ERR_ALIGN, "tp_stack_decode: x, y and workspace must be 16-byte aligned");
    char* ws = static_cast<char*>(workspace);
    tpk::ChainArgs A = stack->a;
    A.T = B;
    A.x = x;
    A.y = y;
    A.pos = pos;
    A.cbase = reinterpret_cast<const unsigned long long*>(ws + P->off_c_begin);
    A.fx = reinterpret_cast<unsigned long long*>(ws + P->off_c_x);
    A.fq = reinterpret_cast<unsigned long long*>(ws + P->off_c_q);
    A.fp = reinterpret_cast<unsigned long long*>(ws + P->off_c_p);
    A.fh = reinterpret_cast<unsigned long long*>(ws + P->off_c_h);
    A.fa = reinterpret_cast<unsigned long long*>(ws + P->off_c_a);
    unsigned* cw = reinterpret_cast<unsigned*>(ws + P->off_c_ctrl);
    A.gen = cw;
    A.done = cw + 1;
    A.gabort = reinterpret_cast<int*>(cw + 2);
    A.status = reinterpret_cast<int*>(ws + P->off_status);
    TP_CUDA(tpk::launch_chain(A, stack->smem, static_cast<cudaStream_t>(stream)), "tp_stack_decode: launch");
    return ok();
}

// ---------------------------------------------------------------- logits over the vocab-parallel head

extern "C" tp_status tp_lm_head_forward(tp_plan_t plan, const void* const* head_shards, const float* gamma,
                                        const float* x, int32_t T, float* logits, int32_t* device_status,
                                        void* stream) {
    if (!plan || !head_shards || !gamma || !x || !logits) return fail(TP_ERR_NULL, "tp_lm_head_forward: NULL argument");
    const tp_model_desc& d = plan->d;
    const tp_plan_info& I = plan->info;
    if (d.org_vocab <= 0) return fail(TP_ERR_INVALID_ARG, "tp_lm_head_forward: the plan has no head (org_vocab 0)");
    if (d.dtype != TP_BF16) return fail(TP_ERR_UNSUPPORTED, "tp_lm_head_forward: bf16 heads only");
    if (T < 1 || T > tpk::kTMax) return fail(TP_ERR_SHAPE, "tp_lm_head_forward: T=%d outside 1..%d", T, tpk::kTMax);
    const int N = plan->N;
    for (int r = 0; r < N; ++r) {
        if (!head_shards[r]) return fail(TP_ERR_NULL, "tp_lm_head_forward: shard %d is NULL", r);
        if (!aligned16(head_shards[r])) return fail(TP_ERR_ALIGN, "tp_lm_head_forward: shard %d not 16-byte aligned", r);
    }
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(logits))
        return fail(TP_ERR_ALIGN, "tp_lm_head_forward: x, gamma and logits must be 16-byte aligned");
    tp_status st = check_device();
    if (st) return st;
    int dev = 0, sms = 0, smem_max = 0;
    TP_CUDA(cudaGetDevice(&dev), "tp_lm_head_forward: cudaGetDevice");
    TP_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "tp_lm_head_forward: SM count");
    TP_CUDA(cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev), "tp_lm_head_forward: smem");
    tpk::HeadArgs A{};
    for (int r = 0; r < N; ++r) A.W[r] = head_shards[r];
    A.N = N;
    A.rows_s = (int)I.vocab_rows_shard;
    A.org_vocab = (int)d.org_vocab;
    A.H = (int)d.hidden;
    A.T = T;
    A.grid = sms;
    A.x = x;
    A.gamma = gamma;
    A.eps = (float)d.eps;
    A.logits = logits;
    A.status = reinterpret_cast<int*>(device_status);
    const size_t smem = tpk::head_smem(A, smem_max);
    if (A.ns < 2) return fail(TP_ERR_UNSUPPORTED, "tp_lm_head_forward: hidden size too large for the stage ring");
    A.grid = sms * A.cps;
    const long total = (long)N * A.rows_s;
    long rpc = (total + A.grid - 1) / A.grid;
    A.rpc = (rpc + A.rs - 1) / A.rs * A.rs;
    TP_CUDA(tpk::launch_lm_head(A, smem, static_cast<cudaStream_t>(stream)), "tp_lm_head_forward: launch");
    return ok();
}
