// Several decode blocks in one persistent launch, latency first.
//
// The computation of every layer is the decode block of "Tensor Parallelism
// in llama.cpp" (How tensor parallelism works, steps 1-3): column-parallel
// QKV with RoPE and a per-shard KV append, grouped-query attention over the
// shard's own heads, the row-parallel o_proj whose shard partials are summed
// in rank order before the residual, then the same for SwiGLU gate/up and
// down_proj. Layer l's output is layer l+1's input.
//
// GB300 design: one CTA per SM; a producer warp streams each CTA's weight and
// KV tiles for all layers through a ring of 16 KB slots (TMA, 128-byte
// swizzled 3-D boxes), so weights are in shared memory before the activation
// they multiply exists. A step with one or two loads per CTA (QKV, o_proj) is
// computed a row per warp; a step with more (gate/up, down) splits its loads
// into tasks, one load (or a K part of one) per warp, each warp multiplying
// all rows of its load with one operand load per 16-byte unit, and the tasks'
// partial sums meet in shared memory in a fixed order. One copy of the code
// serves all four projection steps, since the launch's speed follows the
// size of the code each layer runs.
//
// Activations move between steps as 8-byte pairs (a value, or two bf16
// values, and a 32-bit epoch) written with one store: a consumer polls the
// data itself, which replaces "store, fence, arrive, poll a counter, load"
// by one round trip to L2 per step. The residual stream and q, k, v cross as
// fp32; the SwiGLU outputs and the attention chunk outputs, which feed bf16
// operands, cross as bf16 pairs, so that every step's input fits one round
// trip. Every CTA that needs a whole vector (the RMSNorm statistics, the
// split-KV combine) computes it itself from the pairs instead of waiting for
// another CTA to do it.
//
// Phases of a layer and the CTA items of each (8 output rows per item; the
// host balances the bytes of all items over the CTAs):
//   QKV  rows 8i..8i+7 of shard r's [q_r; k_r; v_r] (+ bias)     -> fq
//   ATT  keys of one (shard, sequence, KV head) group, one 16 KB tile of K
//        and of V; RoPE of q and of the new key, online softmax  -> fp
//   O    output rows 8i.., every shard (rank order) + residual   -> fh
//   GU   SwiGLU rows 8i.. of shard r                              -> fa
//   D    output rows 8i.., every shard (rank order) + residual   -> fx / y
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "stream.cuh"
#include "tp_internal.h"

namespace tpk {

namespace {

constexpr int kCW = 8;            // consumer warps
constexpr int kCT = kCW * 32;     // consumer threads
constexpr int kProducerRegs = 40, kConsumerRegs = 232;   // registers per thread after the split
enum { PH_QKV = 0, PH_O = 1, PH_GU = 2, PH_D = 3 };   // projection phases (item tables)

// ---- (value, epoch) pairs -------------------------------------------------------
//
// A pair is one naturally aligned 8-byte word, written and read as a unit
// (relaxed, GPU scope: the exchange never leaves the device), so a reader that
// sees the epoch it expects sees the value written with it.

__device__ __forceinline__ unsigned long long ll_pack(float v, unsigned ep) {
    return ((unsigned long long)ep << 32) | __float_as_uint(v);
}
__device__ __forceinline__ void ll_st(unsigned long long* p, float v, unsigned ep) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(ll_pack(v, ep)) : "memory");
}
// two adjacent pairs with one 16-byte store (16-byte aligned; each pair stays one unit)
__device__ __forceinline__ void ll_st2(unsigned long long* p, float v0, float v1, unsigned ep) {
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(ll_pack(v0, ep)), "l"(ll_pack(v1, ep))
                 : "memory");
}
__device__ __forceinline__ void ll_ld2(const unsigned long long* p, unsigned long long& a, unsigned long long& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ bool ll_ok(unsigned long long v, unsigned ep) { return (unsigned)(v >> 32) == ep; }
__device__ __forceinline__ float ll_val(unsigned long long v) { return __uint_as_float((unsigned)v); }

// Bounded polling: gives up after kWaitLimitNs, or at once when this CTA or
// any other has given up (the CTA-local flag, then the workspace flag).
struct Poll {
    uint64_t t0 = 0;
    int rounds = 0;
};
__device__ __forceinline__ bool poll_more(Poll& pl, const ChainArgs& A, volatile int* abort) {
    if (*abort) return false;
    if (pl.rounds++ == 0) pl.t0 = global_ns();
    if ((pl.rounds & 15) == 0) {
        if (*reinterpret_cast<volatile int*>(A.gabort)) {
            *abort = 1;
            return false;
        }
        if (global_ns() - pl.t0 > kWaitLimitNs) {
            *abort = 1;
            *reinterpret_cast<volatile int*>(A.gabort) = 1;
            set_status(A.status, TP_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}



// Barrier of the consumer warps that also ORs a flag over them, so that every
// consumer takes the same branch after it.
__device__ __forceinline__ bool csync_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(kCT)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"r"(kCT) : "memory"); }


// ---- ring -------------------------------------------------------------------------

struct CRing {
    uint64_t* full;
    uint64_t* empty;
    unsigned char* base;   // slot 0, 1024-byte aligned
    int ns;
    volatile int* abort;
};

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// (a copy that has landed is taken without the blocking wait)
__device__ __forceinline__ unsigned char* ring_wait(const CRing& R, uint32_t k, int* status) {
    const uint32_t par = (k / R.ns) & 1;
    if (!mbar_test(&R.full[k % R.ns], par)) mbar_wait(&R.full[k % R.ns], par, R.abort, status);
    return R.base + (size_t)(k % R.ns) * kChainSlot;
}
// Every consumer warp releases every load it waited for.
__device__ __forceinline__ void ring_release(const CRing& R, uint32_t k) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&R.empty[k % R.ns]);
}

// ---- polling ----------------------------------------------------------------------
//
// A wait on pairs keeps every load of a round in flight: NB double pairs
// (16 bytes: two pairs) per thread in registers, at double-pair offsets
// off[u] from base (off < 0: none), the missing ones reloaded each round
// until every pair carries epoch ep.
constexpr int kPoll = 8;
template <int NB>
__device__ __forceinline__ bool ll_wait2(const unsigned long long* base, const int (&off)[NB],
                                         unsigned long long (&v)[NB][2], unsigned ep, const ChainArgs& A,
                                         volatile int* abort) {
    unsigned need = 0;
#pragma unroll
    for (int u = 0; u < NB; ++u)
        if (off[u] >= 0) {
            ll_ld2(base + 2 * (size_t)off[u], v[u][0], v[u][1]);
            need |= 1u << u;
        }
    Poll pl;
    while (true) {
#pragma unroll
        for (int u = 0; u < NB; ++u)
            if ((need >> u & 1) && ll_ok(v[u][0], ep) && ll_ok(v[u][1], ep)) need &= ~(1u << u);
        if (!need) return true;
        if (!poll_more(pl, A, abort)) return false;
#pragma unroll
        for (int u = 0; u < NB; ++u)
            if (need >> u & 1) ll_ld2(base + 2 * (size_t)off[u], v[u][0], v[u][1]);
    }
}

// Polls the double pairs of an index space 0..n-1 (thread: tid, tid + kCT,
// ...; NB per round trip): src(i) is the double-pair offset from the
// workspace region base, put(i, a, b) consumes the two values.
template <int NB = kPoll, class Src, class Put>
__device__ __forceinline__ bool poll_space(const ChainArgs& A, int n, unsigned ep, volatile int* abort, Src src,
                                           Put put) {
    bool ok = true;
#pragma unroll 1
    for (int i0 = threadIdx.x; i0 < n; i0 += NB * kCT) {
        int off[NB];
        unsigned long long v[NB][2];
#pragma unroll
        for (int u = 0; u < NB; ++u) {
            const int i = i0 + u * kCT;
            off[u] = i < n ? src(i) : -1;
        }
        ok = ll_wait2<NB>(A.cbase, off, v, ep, A, abort) && ok;
#pragma unroll
        for (int u = 0; u < NB; ++u)
            if (off[u] >= 0) put(i0 + u * kCT, ll_val(v[u][0]), ll_val(v[u][1]));
    }
    return ok;
}

// double-pair offset of a pair buffer element from the region base
__device__ __forceinline__ int dp_off(const ChainArgs& A, const unsigned long long* p) {
    return (int)((p - A.cbase) >> 1);
}

// ---- projection micro-kernel --------------------------------------------------------
//
// A load holds 8 weight rows as [row][kc chunks][64] bf16 (128-byte lines,
// 16-byte unit u of line L stored at u ^ (L & 7)); gate/up loads hold two
// such boxes half a slot apart. With at most 8 tokens a row's dot products are
// CUDA-core work (the MMA shapes would be at least half empty). A task is one
// warp's share of a load: all its rows over a range of 16-byte K units, lane l
// taking units l, l + 32, ...: the operand unit is loaded once and multiplied
// into every row, fp32 sums per lane, then one transposing butterfly.
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float dot8f(const uint4 w, const float (&x)[8], float s) {
    s = fmaf(bf_lo(w.x), x[0], s);
    s = fmaf(bf_hi(w.x), x[1], s);
    s = fmaf(bf_lo(w.y), x[2], s);
    s = fmaf(bf_hi(w.y), x[3], s);
    s = fmaf(bf_lo(w.z), x[4], s);
    s = fmaf(bf_hi(w.z), x[5], s);
    s = fmaf(bf_lo(w.w), x[6], s);
    s = fmaf(bf_hi(w.w), x[7], s);
    return s;
}

// Sums each of the NR values over the warp's 32 lanes. Round by round every
// lane gives away half of its values and keeps the other half (lanes with the
// round's offset bit set keep the upper half), so NR sums cost NR - 1 + (5 -
// log2 NR) shuffles; lane l returns the total of value l >> (5 - log2 NR).
template <int NR, int SZ>
__device__ __forceinline__ float lane_reduce(float (&a)[SZ]) {
    static_assert(NR <= SZ, "values to reduce");
    const int lane = threadIdx.x & 31;
    int o = 16;
#pragma unroll
    for (int n = NR; n > 1; n >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = up ? a[i] : a[i + n / 2];
            const float keep = up ? a[i + n / 2] : a[i];
            a[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float v = a[0];
#pragma unroll
    for (; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ uint32_t lds32(const void* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// ---- shared memory ---------------------------------------------------------------------

struct ChainSmem {
    int ctrl, misc, xin, xa, gam, att, stage, qs, res, part, carry, ring, total;
};
constexpr int kMiscBytes = 4096;
constexpr int kPsBytes = 16 * (128 + 8) * 2;    // attention query tile [16 rows][d + 8] bf16
constexpr int kStageFloats = 11 * 128;      // q (G <= 8 heads), new k, new v of one group, rotation
__host__ __device__ inline int al16(int x) { return (x + 15) & ~15; }
constexpr int kPartFloats = kTMax * 16;    // one task's partial sums: [token][up to 16 rows]
__host__ __device__ inline ChainSmem chain_layout(int N, int MB, int H, int xs, int d, int ns) {
    ChainSmem L;
    int o = 0;
    L.ctrl = o;  o += 256;                                   // full[12], empty[12], abort
    L.misc = o;  o += kMiscBytes;
    L.xin = o;   o = al16(o + MB * H * 4);
    L.xa = o;    o = al16(o + MB * xs * 2);
    L.gam = o;   o = al16(o + N * H * 4);                     // the shards' gammas of a phase (float32)
    L.att = o;   o += kCW * 8 * d * 4;                       // per-warp attention outputs [warp][head][d]
    L.stage = o; o += kStageFloats * 4;
    L.qs = o;    o = al16(o + kPsBytes + 2 * d * 2);           // probabilities [key][8 heads], new k, v (bf16)
    L.res = o;   o = al16(o + kChainMaxItems * MB * 8 * 4);
    L.part = o;  o += kCW * kPartFloats * 4;                  // the partial sums of a wave of tasks
    L.carry = o; o += 2 * kTMax * 8 * 2 * 4;                  // an item's fold state across waves (two copies)
    o = (o + 1023) & ~1023;
    L.ring = o;  o += ns * kChainSlot;
    L.total = o + 1024;                                      // slack to align the base to 1024 bytes
    return L;
}
// misc area (int offsets): item counts [4], items [4][kChainMaxItems], positions,
// 1/rms per token, per-warp attention (max, sum) for 16 head rows
constexpr int kMiCnt = 0, kMiItems = 4, kMiPos = kMiItems + 4 * kChainMaxItems, kMiRinv = kMiPos + 8,
              kMiNch = kMiRinv + 8, kMiMl = kMiNch + 8;
static_assert((kMiMl + kCW * 16 * 2) * 4 <= 2048, "misc area below the layer records");

// ---- attention items ---------------------------------------------------------------------
//
// Items are (shard r, sequence b < T, KV head kh, key chunk c) in that order.
// Sequence b holds len_b = min(pos_b + 1, max_kv) keys, split into chunks of
// cs_b keys (a multiple of 16, at most ck, about even).

__device__ __forceinline__ void att_split(int len, int ck, int& nch, int& cs) {
    if (len <= 0) {
        nch = 0;
        cs = ck;
        return;
    }
    const int n0 = (len + ck - 1) / ck;
    cs = (((len + n0 - 1) / n0) + 15) & ~15;
    if (cs > ck) cs = ck;
    nch = (len + cs - 1) / cs;
}
__device__ __forceinline__ int att_len(const ChainArgs& A, int pos) { return min(max(pos + 1, 0), A.max_kv); }

struct AttItem {
    int r, b, kh, c, k0, nk, len;
};
__device__ __forceinline__ int att_count(const ChainArgs& A, const int* pos) {
    int per_r = 0;
    #pragma unroll 1
    for (int b = 0; b < A.T; ++b) {
        int nch, cs;
        att_split(att_len(A, pos[b]), A.ck, nch, cs);
        per_r += nch * A.hkv_s;
    }
    return per_r * A.N;
}
__device__ __forceinline__ AttItem att_item(const ChainArgs& A, const int* pos, int i) {
    int per_r = 0;
    #pragma unroll 1
    for (int b = 0; b < A.T; ++b) {
        int nch, cs;
        att_split(att_len(A, pos[b]), A.ck, nch, cs);
        per_r += nch * A.hkv_s;
    }
    AttItem it;
    it.r = i / per_r;
    int rem = i - it.r * per_r;
    #pragma unroll 1
    for (int b = 0; b < A.T; ++b) {
        const int len = att_len(A, pos[b]);
        int nch, cs;
        att_split(len, A.ck, nch, cs);
        if (rem < nch * A.hkv_s) {
            it.b = b;
            it.kh = rem / nch;
            it.c = rem - it.kh * nch;
            it.k0 = it.c * cs;
            it.nk = min(cs, len - it.k0);
            it.len = len;
            return it;
        }
        rem -= nch * A.hkv_s;
    }
    it.b = it.kh = it.c = it.k0 = it.nk = it.len = 0;   // not reached for i < att_count
    return it;
}

// ---- producer --------------------------------------------------------------------------
//
// One thread issues every copy of the CTA, in the order the consumers use
// them: per layer the QKV items, the attention tiles, the o_proj items, the
// gate/up items, the down items. Weight copies start before the preceding
// kernel has finished (they do not depend on it); KV tiles after it. One loop
// serves every projection step (the geometry is chosen at run time), so the
// issuing code is small.
// Copy k of the CTA into its ring slot once the slot is free: one box, or
// two boxes half a slot apart (tm2). False if the wait gave up.
__device__ __forceinline__ bool prod_put(const CRing& R, uint32_t k, const CUtensorMap* tm, int y, int z, uint32_t bytes,
                                      const CUtensorMap* tm2, int z2, uint64_t pol, int* status) {
    const int s = (int)(k % (uint32_t)R.ns);
    if (k >= (uint32_t)R.ns && !mbar_wait(&R.empty[s], (k / R.ns - 1) & 1, R.abort, status)) return false;
    unsigned char* dst = R.base + (size_t)s * kChainSlot;
    mbar_arrive_expect_tx(&R.full[s], bytes);
    tma_load_3d_hint(dst, tm, 0, y, z, &R.full[s], pol);
    if (tm2) tma_load_3d_hint(dst + kChainSlot / 2, tm2, 0, y, z2, &R.full[s], pol);
    return true;
}

// the projection phase of step s of a layer (steps: QKV, attention, o_proj, gate/up, down)
__device__ __forceinline__ int step_phase(int s) { return s == 0 ? PH_QKV : s == 2 ? PH_O : s == 3 ? PH_GU : PH_D; }

__device__ __forceinline__ void chain_producer(const ChainArgs& A, const CRing& R, const int* misc) {
    const uint64_t pol = l2_evict_first_policy();
    const int* cnt = misc + kMiCnt;
    const int* items = misc + kMiItems;
    uint32_t k = 0;
    bool ok = true;
    int pos[kTMax];
    bool have_pos = false;
    const int N = A.N;
    #pragma unroll 1
    for (int l = 0; l < A.L && ok; ++l) {
        const CUtensorMap* M = A.maps + (size_t)l * kChainMaps * N;   // [kind][shard]
        #pragma unroll 1
        for (int s = 0; s < 5 && ok; ++s) {
            if (s == 1) {
                if (!have_pos) {
                    pdl_wait();                                   // KV caches and positions of the preceding kernel
                    #pragma unroll 1
                    for (int b = 0; b < kTMax; ++b) pos[b] = b < A.T ? A.pos[b] : 0;
                    have_pos = true;
                }
                const int na = att_count(A, pos);
                const uint32_t bytes = (uint32_t)A.ck * A.d * 2;
                #pragma unroll 1
                for (int i = A.att_rank[blockIdx.x]; i < na && ok; i += A.grid) {
                    const AttItem a = att_item(A, pos, i);
                    const int row = (a.b * A.hkv_s + a.kh) * A.max_kv + a.k0;
                    #pragma unroll 1
                    for (int kv = 0; kv < 2 && ok; ++kv) {
                        ok = prod_put(R, k, M + (4 + kv) * N + a.r, 0, row, bytes, nullptr, 0, pol, A.status);
                        k += ok ? 1u : 0u;
                    }
                }
                continue;
            }
            const int ph = step_phase(s);
            const bool col = ph == PH_QKV || ph == PH_GU;          // items of one shard; else every shard's rows
            const int nsh = col ? 1 : N, nl = A.nl[ph], kc = A.kc[ph];
            const uint32_t bytes = (ph == PH_GU ? 2048u : 1024u) * kc;
            #pragma unroll 1
            for (int n = 0; n < cnt[ph] && ok; ++n) {
                const int it = items[ph * kChainMaxItems + n];
                const int r0 = col ? it >> 16 : 0, i = col ? it & 0xffff : it;
                #pragma unroll 1
                for (int r = r0; r < r0 + nsh && ok; ++r) {
                    const CUtensorMap* tm = M + ph * N + r;
                    #pragma unroll 1
                    for (int j = 0; j < nl && ok; ++j) {
                        ok = prod_put(R, k, tm, j * kc, 8 * i, bytes, ph == PH_GU ? tm : nullptr, A.F_s + 8 * i, pol,
                                      A.status);
                        k += ok ? 1u : 0u;
                    }
                }
            }
        }
    }
    // every copy issued has landed before this thread leaves (if the consumers
    // gave up, some were never waited for); bounded, independent of the abort flag
    volatile int no_abort = 0;
    const uint32_t first = k > (uint32_t)R.ns ? k - R.ns : 0u;
    #pragma unroll 1
    for (uint32_t q = first; q < k; ++q) mbar_wait(&R.full[q % R.ns], (q / R.ns) & 1, &no_abort, nullptr);
}

// ---- consumers ---------------------------------------------------------------------------

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_all;" ::: "memory"); }

constexpr int kLayOff = 2048;   // byte offset of the two ChainLayer copies in the misc area

// Per-CTA consumer state. Shared-memory regions are addressed from one base
// and the launch's offsets (kernel parameters), so no pointer stays live in a
// register across phases.
struct Ctx {
    unsigned char* sm;
    int o_misc, o_xin, o_xa, o_gam, o_att, o_stage, o_qs, o_res, o_part, o_carry, o_ring, ns, d;
    uint32_t k = 0;          // ring loads consumed
    int lb = 0;              // this layer's pointer record (0 or 1)
    __device__ __forceinline__ void init(unsigned char* base, const ChainArgs& A) {
        sm = base;
        o_misc = A.sm_misc;
        o_xin = A.sm_xin;
        o_xa = A.sm_xa;
        o_gam = A.sm_gam;
        o_att = A.sm_att;
        o_stage = A.sm_stage;
        o_qs = A.sm_qs;
        o_res = A.sm_res;
        o_part = A.sm_part;
        o_carry = A.sm_carry;
        o_ring = A.sm_ring;
        ns = A.n_slots;
        d = A.d;
    }
    __device__ __forceinline__ int* misc() const { return reinterpret_cast<int*>(sm + o_misc); }
    __device__ __forceinline__ float* xin() const { return reinterpret_cast<float*>(sm + o_xin); }
    __device__ __forceinline__ bf16* xa() const { return reinterpret_cast<bf16*>(sm + o_xa); }
    __device__ __forceinline__ float* gam() const { return reinterpret_cast<float*>(sm + o_gam); }
    __device__ __forceinline__ float* att() const { return reinterpret_cast<float*>(sm + o_att); }
    __device__ __forceinline__ float* stage() const { return reinterpret_cast<float*>(sm + o_stage); }
    __device__ __forceinline__ bf16* qs() const { return reinterpret_cast<bf16*>(sm + o_qs); }
    __device__ __forceinline__ bf16* knew() const { return reinterpret_cast<bf16*>(sm + o_qs + kPsBytes); }
    __device__ __forceinline__ bf16* vnew() const { return knew() + d; }
    __device__ __forceinline__ float* res() const { return reinterpret_cast<float*>(sm + o_res); }
    __device__ __forceinline__ float* part() const { return reinterpret_cast<float*>(sm + o_part); }
    __device__ __forceinline__ float* carry() const { return reinterpret_cast<float*>(sm + o_carry); }
    __device__ __forceinline__ const ChainLayer* lay() const {
        return reinterpret_cast<const ChainLayer*>(sm + o_misc + kLayOff) + lb;
    }
    __device__ __forceinline__ CRing ring() const {
        CRing R;
        R.full = reinterpret_cast<uint64_t*>(sm);
        R.empty = R.full + kChainMaxSlots;
        R.abort = reinterpret_cast<volatile int*>(R.empty + kChainMaxSlots);
        R.base = sm + o_ring;
        R.ns = ns;
        return R;
    }
    __device__ __forceinline__ volatile int* abort() const {
        return reinterpret_cast<volatile int*>(reinterpret_cast<uint64_t*>(sm) + 2 * kChainMaxSlots);
    }
};

// Measurement hook: %globaltimer when a phase's inputs have arrived (w = 0)
// and when its last output is stored (w = 1).
__device__ __forceinline__ void stamp(const ChainArgs& A, int l, int ph, int w) {
    if (A.stamps && threadIdx.x == 0) A.stamps[(((size_t)blockIdx.x * A.L + l) * 5 + ph) * 2 + w] = global_ns();
}

// Copies every shard's gamma into shared memory, [N][H] (asynchronously:
// call before a poll).
__device__ __forceinline__ void gammas_fetch(Ctx& C, const ChainArgs& A, const float* const* g) {
    const int H4 = A.H / 4;
    #pragma unroll 1
    for (int i = threadIdx.x; i < A.N * H4; i += kCT) {
        const int r = i / H4, e = i - r * H4;
        cp_async16(C.gam() + r * A.H + 4 * e, g[r] + 4 * e);
    }
    cp_commit();
}

// 1/rms of every token of xin (T x H, float32) into the misc area.
// (with a single token the warps' partial sums were stored while the vector was polled: have_part)
__device__ __forceinline__ void rms_stats(Ctx& C, const ChainArgs& A, bool have_part) {
    const int T = A.T, H = A.H, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float* xin = C.xin();
    float* part = C.att();                                // [token][warp] partial sums
    if (!have_part) {
        #pragma unroll 1
        for (int t = 0; t < T; ++t) {
            float sq = 0.f;
            #pragma unroll 1
            for (int k2 = threadIdx.x; k2 < H / 2; k2 += kCT) {
                const float2 xv = *reinterpret_cast<const float2*>(xin + t * H + 2 * k2);
                sq = fmaf(xv.x, xv.x, fmaf(xv.y, xv.y, sq));
            }
            sq = warp_sum(sq);
            if (lane == 0) part[t * kCW + warp] = sq;
        }
        csync();
    }
    if (threadIdx.x < T) {
        const float* pt = part + threadIdx.x * kCW;
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < kCW; ++w) a += pt[w];
        reinterpret_cast<float*>(C.misc())[kMiRinv + threadIdx.x] = rsqrtf(a * (1.0f / (float)H) + A.eps);
    }
    csync();
}

// The o_proj operand: every CTA with o_proj items combines the split-KV
// partials of all groups itself (chunks in order: running max, rescaled
// sums) into xa, [token][shard r's heads] bf16.
__device__ __forceinline__ bool combine_att(Ctx& C, const ChainArgs& A, unsigned ep) {
    const int tid = threadIdx.x, T = A.T, MB = A.max_batch, G = A.G, d = A.d, hk = A.hkv_s;
    const int* nch_t = C.misc() + kMiNch;
    const int nq = A.N * T * hk * G * (d / 4);
    bool ok = true;
    #pragma unroll 1
    for (int q = tid; q < nq; q += kCT) {
        const int e4 = q % (d / 4), rest = q / (d / 4), j = rest % G, rest2 = rest / G, kh = rest2 % hk;
        const int rt = rest2 / hk, t = rt % T, r = rt / T, n = nch_t[t];
        const int gi = (r * MB + t) * hk + kh;
        float M = -INFINITY, den = 0.f, num0 = 0.f, num1 = 0.f, num2 = 0.f, num3 = 0.f;
        int c0 = 0;
        // per chunk two double pairs: O's four values as bf16, then (max, sum)
        constexpr int kCh = 5;                         // chunks per round trip
        do {
            int off[2 * kCh];
            unsigned long long v[2 * kCh][2];
#pragma unroll
            for (int u = 0; u < 2 * kCh; ++u) off[u] = -1;
            const int nb = min(kCh, n - c0);
#pragma unroll
            for (int c = 0; c < kCh; ++c)
                if (c < nb) {
                    const int base = dp_off(A, A.fp + ((size_t)gi * A.maxch + c0 + c) * G * (d + 2));
                    off[2 * c] = base + (j * d + 4 * e4) / 4;
                    off[2 * c + 1] = base + (G * d / 2 + 2 * j) / 2;
                }
            ok = ll_wait2<2 * kCh>(A.cbase, off, v, ep, A, C.abort()) && ok;
#pragma unroll
            for (int c = 0; c < kCh; ++c)
                if (c < nb) {
                    const float mc = ll_val(v[2 * c + 1][0]), Mn = fmaxf(M, mc);
                    const float fa = ex2_approx(M - Mn), fb = ex2_approx(mc - Mn);
                    const uint32_t o01 = (uint32_t)v[2 * c][0], o23 = (uint32_t)v[2 * c][1];
                    den = fmaf(den, fa, ll_val(v[2 * c + 1][1]) * fb);
                    num0 = fmaf(num0, fa, bf_lo(o01) * fb);
                    num1 = fmaf(num1, fa, bf_hi(o01) * fb);
                    num2 = fmaf(num2, fa, bf_lo(o23) * fb);
                    num3 = fmaf(num3, fa, bf_hi(o23) * fb);
                    M = Mn;
                }
            c0 += max(nb, 0);
        } while (c0 < n && ok);
        const float inv = den > 0.f ? 1.0f / den : 0.f;
        bf16* dst = C.xa() + (size_t)t * A.xa_stride + r * A.hq_s * d + (kh * G + j) * d + 4 * e4;
        *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(num0 * inv, num1 * inv);
        *reinterpret_cast<uint32_t*>(dst + 2) = pack_bf16x2(num2 * inv, num3 * inv);
    }
    return ok;
}

// ---- projection steps -------------------------------------------------------------------
//
// A step of a CTA holds cnt items of sl ring loads each (load js of an item:
// shard js / nl, K range js % nl), consumed in the producer's order. Load j is
// split into f K parts (f: the largest power of two with cnt * sl * f <= kCW,
// at least 1), so that a CTA with few loads still keeps every warp busy. Task
// q = j * f + part; tasks go to the warps in waves of kCW (task q to warp
// q % kCW). A task is one warp's share of a load: all its rows (8, or 16 for
// gate/up) over a range of 16-byte K units, lane l taking units l, l + 32,
// ...: the operand unit is loaded once and multiplied into every row, fp32
// sums per lane, then one transposing butterfly; the per-token partial sums
// go to part[warp]. After a wave every (item, token, row) folds its tasks'
// partials in task order: per shard the K parts and loads in order, the
// shards' sums in rank order ((p0 + p1) + p2) + ... An item that continues
// into the next wave leaves its state in carry.
//
// One copy of this code serves all four projection steps of every layer (the
// operand, geometry and epilogue are chosen at run time), so that the code a
// layer runs stays small.

// floor(a / b) for 0 <= a < 2^16 and 1 <= b <= 64, with rb = 1 / b rounded
// to float: (a + 1/2) / b lies at least 1/(2b) from an integer, and the
// float product errs by at most a 2^-7 of that, so truncation is exact.
__device__ __forceinline__ int qdiv(int a, float rb) { return (int)(((float)a + 0.5f) * rb); }

struct Phase {
    int cnt, sl, nl, nsh, f, lf, ntask;
    float rsl, rnl, rsb;    // 1 / sl, 1 / nl, 1 / (nl f)
};
__device__ __forceinline__ Phase make_phase(int cnt, int nsh, int nl) {
    Phase P;
    P.cnt = cnt;
    P.nsh = nsh;
    P.nl = nl;
    P.sl = nsh * nl;
    P.f = 1;
    P.lf = 0;
    while (cnt * P.sl * P.f * 2 <= kCW) {
        P.f *= 2;
        ++P.lf;
    }
    P.ntask = cnt * P.sl * P.f;
    P.rsl = 1.0f / (float)P.sl;
    P.rnl = 1.0f / (float)nl;
    P.rsb = 1.0f / (float)(nl * P.f);
    return P;
}

__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t cnt) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(cnt) : "memory");
}

// The step's input vector: the layer input x (step QKV) or the residual
// stream after attention (gate/up) into xin as float32, or every shard's
// SwiGLU outputs (down) into xa as bf16; then, for QKV and gate/up, 1/rms
// per token. Every CTA loads x and h, items or not: they are the residuals
// of the o_proj and down epilogues.
__device__ __forceinline__ bool step_input(Ctx& C, const ChainArgs& A, int l, int ph, unsigned ep) {
    const int T = A.T, H = A.H;
    bool ok = true;
    float sq = 0.f;                                      // this thread's sum of squares (one token)
    if (ph == PH_QKV && l == 0) {
        #pragma unroll 1
        for (int i = threadIdx.x; i < T * H / 2; i += kCT) {
            const float2 v = *reinterpret_cast<const float2*>(A.x + 2 * (size_t)i);
            *reinterpret_cast<float2*>(C.xin() + 2 * i) = v;
            sq = fmaf(v.x, v.x, fmaf(v.y, v.y, sq));
        }
    } else {
        const bool down = ph == PH_D;
        const unsigned long long* src = ph == PH_QKV ? A.fx : down ? A.fa : A.fh;
        const int cols = down ? A.N * A.F_s / 4 : H / 2;    // double pairs per token (down: 4 bf16 values each)
        ok = poll_space(A, T * cols, ep, C.abort(), [&](int i) { return dp_off(A, src) + i; },
            [&](int i, float a, float b) {
                if (down) {                              // [token][N F_s] bf16, four values a double pair
                    *reinterpret_cast<uint2*>(C.xa() + 4 * i) = make_uint2(__float_as_uint(a), __float_as_uint(b));
                } else {
                    *reinterpret_cast<float2*>(C.xin() + 2 * i) = make_float2(a, b);
                    sq = fmaf(a, a, fmaf(b, b, sq));
                }
            });
    }
    cp_wait();
    const bool one = T == 1 && ph != PH_D;
    if (one) {
        sq = warp_sum(sq);
        if ((threadIdx.x & 31) == 0) C.att()[threadIdx.x >> 5] = sq;
    }
    if (csync_or(!ok)) return false;
    if (ph != PH_D) rms_stats(C, A, one);
    return true;
}

__device__ __forceinline__ bool proj_step(Ctx& C, const ChainArgs& A, int l, unsigned ep, int ph) {
    const int cnt = C.misc()[kMiCnt + ph];
    if (csync_or(*C.abort())) return false;
    const int* items = C.misc() + kMiItems + ph * kChainMaxItems;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, T = A.T, MB = A.max_batch, H = A.H, N = A.N;
    const ChainLayer& Ly = *C.lay();
    const bool norm = ph == PH_QKV || ph == PH_GU;     // RMSNorm input: operand x * gamma_r, items of one shard
    const int sidx = ph == PH_QKV ? 0 : ph == PH_O ? 2 : ph == PH_GU ? 3 : 4;   // step (stamps)
    if ((ph == PH_O || ph == PH_D) && !cnt) return true;
    if (ph == PH_QKV) {                                  // biases into shared memory while the input is polled
        float* sbias = C.res();
        #pragma unroll 1
        for (int e = tid; e < 8 * cnt; e += kCT) {
            const int it = items[e >> 3], r = it >> 16, i = it & 0xffff;
            if (Ly.bqkv[r]) cp_async4(sbias + e, Ly.bqkv[r] + 8 * i + (e & 7));
            else sbias[e] = 0.f;
        }
    }
    if (norm) gammas_fetch(C, A, ph == PH_QKV ? Ly.g_attn : Ly.g_ffn);
    if (ph == PH_O) {
        const bool ok = combine_att(C, A, ep);
        if (csync_or(!ok)) return false;
    } else if (!step_input(C, A, l, ph, ep)) {
        return false;
    }
    stamp(A, l, sidx, 0);
    if (!cnt) return true;

    const int nsh = norm ? 1 : N, nl = A.nl[ph], kc = A.kc[ph];
    const int Ks = ph == PH_O ? A.hq_s * A.d : ph == PH_D ? A.F_s : H;   // operand columns per shard
    const int nch = Ks / 64, nbox = ph == PH_GU ? 2 : 1;
    const float* rinv = reinterpret_cast<const float*>(C.misc()) + kMiRinv;
    const CRing R = C.ring();
    const int xs = ph == PH_D ? N * A.F_s : A.xa_stride;   // the down operand's tokens are unpadded
    // the output of item n, token t, row: v0 the row's total (the gate row's for gate/up), v1 the up row's
    auto epilogue = [&](int n, int t, int row, float v0, float v1) {
        const int it = items[n];
        if (norm) {
            const int r = it >> 16, i = it & 0xffff;
            if (ph == PH_QKV) {
                ll_st(A.fq + (size_t)(r * MB + t) * A.qkv_rows + 8 * i + row, v0 * rinv[t] + C.res()[8 * n + row], ep);
            } else {
                const float gt = v0 * rinv[t], up = v1 * rinv[t];
                // rows 2j and 2j + 1 as one pair of bf16 values (the down operand is bf16 anyway): the row
                // pair sits in adjacent lanes of the fold, and the even one stores both
                const float v = gt / (1.0f + expf(-gt)) * up, nv = __shfl_down_sync(__activemask(), v, 1);
                if (!(row & 1)) {
                    const unsigned long long pv = ((unsigned long long)ep << 32) | pack_bf16x2(v, nv);
                    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(A.fa + ((size_t)(t * N + r) * A.F_s + 8 * i + row) / 2),
                                 "l"(pv) : "memory");
                }
            }
        } else {
            const int e = t * H + 8 * it + row;
            const float v = v0 + C.xin()[e];             // + the residual
            if (ph == PH_O) ll_st(A.fh + e, v, ep);
            else if (l == A.L - 1) A.y[e] = v;
            else ll_st(A.fx + e, v, ep + 1);
        }
    };
    if (nbox == 1 && T == 1 && cnt * nsh * nl <= 2) {
        // One token, one box per load and at most two loads (QKV, o_proj here): warp w computes
        // row w of every item over all its loads, in order (per shard the loads in K order, the
        // shards' sums in rank order), then releases them; lane 0 writes the output.
        const int sl = nsh * nl;
        #pragma unroll 1
        for (int n = 0; n < cnt; ++n) {
            const float* gam = C.gam() + (items[n] >> 16) * H;
            float tot = 0.f;
            #pragma unroll 1
            for (int r = 0; r < nsh; ++r) {
                float acc = 0.f;
                #pragma unroll 1
                for (int jj = 0; jj < nl; ++jj) {
                    const uint32_t k = C.k + (uint32_t)(n * sl + r * nl + jj);
                    const unsigned char* w = ring_wait(R, k, A.status);
                    const int nv = min(kc, nch - jj * kc), kb = jj * kc * 64;
                    #pragma unroll 1
                    for (int u = lane; u < nv * 8; u += 32) {
                        const int ch = u >> 3, u8 = u & 7, e = kb + 64 * ch + 8 * u8, line = warp * kc + ch;
                        float xf[8];
                        if (norm) {
                            const float4* xp = reinterpret_cast<const float4*>(C.xin() + e);
                            const float4* gp = reinterpret_cast<const float4*>(gam + e);
                            const float4 x0 = xp[0], x1 = xp[1], g0 = gp[0], g1 = gp[1];
                            xf[0] = x0.x * g0.x;
                            xf[1] = x0.y * g0.y;
                            xf[2] = x0.z * g0.z;
                            xf[3] = x0.w * g0.w;
                            xf[4] = x1.x * g1.x;
                            xf[5] = x1.y * g1.y;
                            xf[6] = x1.z * g1.z;
                            xf[7] = x1.w * g1.w;
                        } else {
                            const uint4 v = *reinterpret_cast<const uint4*>(C.xa() + r * Ks + e);
                            xf[0] = bf_lo(v.x);
                            xf[1] = bf_hi(v.x);
                            xf[2] = bf_lo(v.y);
                            xf[3] = bf_hi(v.y);
                            xf[4] = bf_lo(v.z);
                            xf[5] = bf_hi(v.z);
                            xf[6] = bf_lo(v.w);
                            xf[7] = bf_hi(v.w);
                        }
                        acc = dot8f(*reinterpret_cast<const uint4*>(w + (line << 7) + ((u8 ^ (line & 7)) << 4)), xf, acc);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&R.empty[k % R.ns]);
                }
                const float ps = warp_sum(acc);
                tot = r == 0 ? ps : tot + ps;
            }
            if (lane == 0) epilogue(n, 0, warp, tot, 0.f);
        }
        C.k += (uint32_t)(cnt * sl);
        stamp(A, l, sidx, 1);
        return true;
    }
    // Tasks over the loads (gate/up, and steps with more loads): partial sums folded in shared memory.
    const Phase P = make_phase(cnt, nsh, nl);
    const int per = P.sl * P.f;                          // tasks per item
    int wave = 0;
    #pragma unroll 1
    for (int w0 = 0; w0 < P.ntask; w0 += kCW, ++wave) {
        const int q = w0 + warp;
        if (q < P.ntask) {
            const int j = q >> P.lf, kp = q - (j << P.lf);
            const int n = qdiv(j, P.rsl), js = j - n * P.sl, r = qdiv(js, P.rnl), jj = js - r * nl;
            const int nv = min(kc, nch - jj * kc), U = nv * 8, u0 = (kp * U) >> P.lf, u1 = ((kp + 1) * U) >> P.lf;
            const uint32_t k = C.k + (uint32_t)j;
            const unsigned char* w = ring_wait(R, k, A.status);
            const int kb = jj * kc * 64;                 // the load's first operand column
            const float* gam = C.gam() + (items[n] >> 16) * H + kb;
            const bf16* xa0 = C.xa() + r * Ks + kb;
            float* part = C.part() + warp * kPartFloats;
            // a gate/up load holds a gate box and an up box of 8 rows each, both multiplied per operand unit
            #pragma unroll 1
            for (int t = 0; t < T; ++t) {
                float acc[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[i] = 0.f;
                #pragma unroll 1
                for (int u = u0 + lane; u < u1; u += 32) {
                    const int ch = u >> 3, u8 = u & 7, e = 64 * ch + 8 * u8;
                    float xf[8];
                    if (norm) {
                        const float4* xp = reinterpret_cast<const float4*>(C.xin() + t * H + kb + e);
                        const float4* gp = reinterpret_cast<const float4*>(gam + e);
                        const float4 x0 = xp[0], x1 = xp[1], g0 = gp[0], g1 = gp[1];
                        xf[0] = x0.x * g0.x;
                        xf[1] = x0.y * g0.y;
                        xf[2] = x0.z * g0.z;
                        xf[3] = x0.w * g0.w;
                        xf[4] = x1.x * g1.x;
                        xf[5] = x1.y * g1.y;
                        xf[6] = x1.z * g1.z;
                        xf[7] = x1.w * g1.w;
                    } else {
                        const uint4 v = *reinterpret_cast<const uint4*>(xa0 + (size_t)t * xs + e);
                        xf[0] = bf_lo(v.x);
                        xf[1] = bf_hi(v.x);
                        xf[2] = bf_lo(v.y);
                        xf[3] = bf_hi(v.y);
                        xf[4] = bf_lo(v.z);
                        xf[5] = bf_hi(v.z);
                        xf[6] = bf_lo(v.w);
                        xf[7] = bf_hi(v.w);
                    }
#pragma unroll
                    for (int row = 0; row < 8; ++row) {
                        const int line = row * kc + ch;
                        const unsigned char* wl = w + (line << 7) + ((u8 ^ (line & 7)) << 4);
                        acc[row] = dot8f(*reinterpret_cast<const uint4*>(wl), xf, acc[row]);
                        if (nbox == 2) acc[8 + row] = dot8f(*reinterpret_cast<const uint4*>(wl + kChainSlot / 2), xf, acc[8 + row]);
                    }
                }
                if (nbox == 2) {
                    const float v = lane_reduce<16>(acc);
                    if (!(lane & 1)) part[t * 16 + (lane >> 1)] = v;
                } else {
                    const float v = lane_reduce<8>(acc);
                    if (!(lane & 3)) part[t * 16 + (lane >> 2)] = v;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_cnt(&R.empty[k % R.ns], (uint32_t)(kCW / P.f));
        }
        csync();
        // fold the wave's partials; items that end in this wave run the epilogue
        const int qe = min(w0 + kCW, P.ntask);
        const int n0 = w0 / per, n1 = (qe - 1) / per;
        const float* cin = C.carry() + ((wave - 1) & 1) * (kTMax * 16);
        float* cout = C.carry() + (wave & 1) * (kTMax * 16);
        #pragma unroll 1
        for (int idx = tid; idx < (n1 - n0 + 1) * T * 8; idx += kCT) {
            const int nn = idx / (T * 8), rem = idx - nn * (T * 8), t = rem >> 3, row = rem & 7;
            const int n = n0 + nn, qa = max(n * per, w0), qb = min((n + 1) * per, qe);
            // c0: the current shard's sum (gate rows for gate/up), c1: the total of the
            // shards before it (up rows for gate/up); selects, not branches
            float c0 = 0.f, c1 = 0.f;
            if (qa > n * per) {
                c0 = cin[(t * 8 + row) * 2];
                c1 = cin[(t * 8 + row) * 2 + 1];
            }
            const float* pp = C.part() + (qa - w0) * kPartFloats + t * 16 + row;
            const int sb = nl * P.f;                     // tasks per shard
            int i = qa - n * per, sh = qdiv(i, P.rsb), k = i - sh * sb;
            #pragma unroll 4
            for (int qq = qa; qq < qb; ++qq, pp += kPartFloats) {
                const float v0 = pp[0], v1 = nbox == 2 ? pp[8] : 0.f;
                const bool start = k == 0;
                if (nbox == 2) {
                    c0 = start ? v0 : c0 + v0;
                    c1 = start ? v1 : c1 + v1;
                } else {
                    c1 = start && sh > 0 ? (sh == 1 ? c0 : c1 + c0) : c1;   // fold the finished shard, rank order
                    c0 = start ? v0 : c0 + v0;
                }
                const bool wrap = ++k == sb;
                k = wrap ? 0 : k;
                sh += wrap ? 1 : 0;
            }
            if (qb < (n + 1) * per) {
                cout[(t * 8 + row) * 2] = c0;
                cout[(t * 8 + row) * 2 + 1] = c1;
                continue;
            }
            epilogue(n, t, row, nsh > 1 ? c1 + c0 : c0, c1);
        }
        if (w0 + kCW < P.ntask) csync();                // the next wave overwrites the partials
    }
    C.k += (uint32_t)(P.ntask / P.f);
    stamp(A, l, sidx, 1);
    return true;
}

// Attention items of this CTA: RoPE of q and of the new key (rotate-half
// pairs (e, e + d/2) at angle pos * theta^(-2e/d)), the new K/V row written
// into the shared-memory tiles and into the shard's cache; then per warp its
// keys: scores q K^T (scaled, log2 units), online softmax, O = P V; the warps'
// (max, sum, O) merged into the chunk's partial.
__device__ __forceinline__ bool phase_att(Ctx& C, const ChainArgs& A, int l, unsigned ep) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int* pos = C.misc() + kMiPos;
    const int G = A.G, d = A.d, half = d >> 1, MB = A.max_batch, DC = d >> 6;
    const int na = att_count(A, pos);
    const ChainLayer& Ly = *C.lay();
    float* ml = reinterpret_cast<float*>(C.misc()) + kMiMl;
    float* st = C.stage();
    #pragma unroll 1
    for (int i = A.att_rank[blockIdx.x]; i < na; i += A.grid) {
        if (csync_or(*C.abort())) return false;
        const AttItem a = att_item(A, pos, i);
        const int pb = pos[a.b];
        const bool has_new = pb >= 0 && pb < A.max_kv && pb >= a.k0 && pb < a.k0 + a.nk;
        // the rotation of this position (table row) while q, k, v are polled
        float* rot = st + (G + 2) * d;                       // [d/2] (cos, sin)
        if (pb >= 0 && pb < A.max_kv)
            #pragma unroll 1
            for (int e = tid; e < half / 2; e += kCT) cp_async16(rot + 4 * e, A.rope + ((size_t)pb * half + 2 * e));
        cp_commit();
        // raw q (G heads), k and v of the group, as written by the QKV phase
        const unsigned long long* row = A.fq + (size_t)(a.r * MB + a.b) * A.qkv_rows;
        // three runs of double pairs: q of the group's G heads, then k, then v
        const int dpq = dp_off(A, row + a.kh * G * d), dpk = dp_off(A, row + (A.hq_s + a.kh) * d),
                  dpv = dp_off(A, row + (A.hq_s + A.hkv_s + a.kh) * d), nq2 = G * half, nk2 = nq2 + half;
        const bool ok = poll_space(A, (G + 2) * half, ep, C.abort(),
            [&](int p) { return p < nq2 ? dpq + p : p < nk2 ? dpk + (p - nq2) : dpv + (p - nk2); },
            [&](int p, float x0, float x1) { *reinterpret_cast<float2*>(st + 2 * p) = make_float2(x0, x1); });
        cp_wait();
        if (csync_or(!ok)) return false;
        if (i == A.att_rank[blockIdx.x]) stamp(A, l, 1, 0);
        const bool inrange = pb >= 0 && pb < A.max_kv;
        #pragma unroll 1
        for (int p = tid; p < (G + 1) * half; p += kCT) {
            const int hr = p / half, e = p - hr * half;
            const float x0 = st[hr * d + e], x1 = st[hr * d + e + half];
            const float cs = inrange ? rot[2 * e] : 1.f, sn = inrange ? rot[2 * e + 1] : 0.f;
            const float r0 = x0 * cs - x1 * sn, r1 = x0 * sn + x1 * cs;
            if (hr < G) {                                // q: rotated and scaled, bf16 tile rows 0..G-1
                C.qs()[hr * (d + 8) + e] = __float2bfloat16_rn(r0 * A.qscale);
                C.qs()[hr * (d + 8) + e + half] = __float2bfloat16_rn(r1 * A.qscale);
            } else {
                C.knew()[e] = __float2bfloat16_rn(r0);
                C.knew()[e + half] = __float2bfloat16_rn(r1);
            }
        }
        #pragma unroll 1
        for (int e = tid; e < d; e += kCT) C.vnew()[e] = __float2bfloat16_rn(st[(G + 1) * d + e]);
        csync();
        const uint32_t k0 = C.k;
        C.k += 2;
        unsigned char* Kt = ring_wait(C.ring(), k0, A.status);
        unsigned char* Vt = ring_wait(C.ring(), k0 + 1, A.status);
        if (has_new) {
            const int kr = pb - a.k0;
            #pragma unroll 1
            for (int e2 = tid; e2 < half; e2 += kCT) {     // bf16 pairs of the new row
                const int e = 2 * e2, line = kr * DC + (e >> 6);
                const int byte = line * 128 + ((((e & 63) >> 3) ^ (line & 7)) << 4) + (e & 7) * 2;
                const uint32_t kv = *reinterpret_cast<const uint32_t*>(C.knew() + e);
                const uint32_t vv = *reinterpret_cast<const uint32_t*>(C.vnew() + e);
                *reinterpret_cast<uint32_t*>(Kt + byte) = kv;
                *reinterpret_cast<uint32_t*>(Vt + byte) = vv;
                const size_t crow = ((size_t)(a.b * A.hkv_s + a.kh) * A.max_kv + pb) * d + e;
                *reinterpret_cast<uint32_t*>(reinterpret_cast<bf16*>(Ly.kc[a.r]) + crow) = kv;
                *reinterpret_cast<uint32_t*>(reinterpret_cast<bf16*>(Ly.vc[a.r]) + crow) = vv;
            }
            // generic-proxy writes into a slot the next copy (async proxy) will overwrite
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        csync();
        // tensor cores: warp w takes keys 16w..16w+15 of the tile. S = q K^T
        // (q rows = heads, 16 with zero rows >= G), masked online softmax per
        // head row, O = P V with V read transposed by ldmatrix.
        const int nw = min(A.ck / 16, (a.nk + 15) / 16);   // warps holding keys
        if (warp < nw) {
            const int g = lane >> 2, t = lane & 3, qst = d + 8;
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
            const bf16* qr = C.qs() + g * qst + 2 * t;
            #pragma unroll 1
            for (int kk = 0; kk < d / 16; ++kk) {
                const uint32_t a0 = lds32(qr + 16 * kk), a2 = lds32(qr + 16 * kk + 8);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int key = 16 * warp + 8 * nt + g, line = key * DC + (kk >> 2);
                    const unsigned char* ln = Kt + line * 128 + 4 * t;
                    const uint32_t b0 = lds32(ln + (((2 * (kk & 3)) ^ (line & 7)) << 4));
                    const uint32_t b1 = lds32(ln + (((2 * (kk & 3) + 1) ^ (line & 7)) << 4));
                    mma_bf16_16816(nt ? s1 : s0, a0, 0u, a2, 0u, b0, b1);
                }
            }
            const int kb = 16 * warp + 2 * t;
            const bool v00 = kb < a.nk, v01 = kb + 1 < a.nk, v10 = kb + 8 < a.nk, v11 = kb + 9 < a.nk;
            float mx = fmaxf(fmaxf(v00 ? s0[0] : -INFINITY, v01 ? s0[1] : -INFINITY),
                             fmaxf(v10 ? s1[0] : -INFINITY, v11 ? s1[1] : -INFINITY));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float p00 = v00 ? ex2_approx(s0[0] - mx) : 0.f, p01 = v01 ? ex2_approx(s0[1] - mx) : 0.f;
            const float p10 = v10 ? ex2_approx(s1[0] - mx) : 0.f, p11 = v11 ? ex2_approx(s1[1] - mx) : 0.f;
            float lsum = (p00 + p01) + (p10 + p11);
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
            const uint32_t pa0 = pack_bf16x2(p00, p01), pa2 = pack_bf16x2(p10, p11);
            const uint32_t vbase = smem_u32(Vt);
            const int mi = lane >> 3, rr = lane & 7;
            const int vkey = 16 * warp + (mi & 1) * 8 + rr;
            #pragma unroll 1
            for (int jj = 0; jj < d / 16; ++jj) {
                const int e0 = 16 * jj + (mi >> 1) * 8, line = vkey * DC + (e0 >> 6);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vbase + line * 128 + ((((e0 & 63) >> 3) ^ (line & 7)) << 4), b0, b1, b2, b3);
                float o0[4] = {0.f, 0.f, 0.f, 0.f}, o1[4] = {0.f, 0.f, 0.f, 0.f};
                mma_bf16_16816(o0, pa0, 0u, pa2, 0u, b0, b1);
                mma_bf16_16816(o1, pa0, 0u, pa2, 0u, b2, b3);
                if (g < G) {
                    float* dst = C.att() + (warp * G + g) * d + 16 * jj + 2 * t;
                    *reinterpret_cast<float2*>(dst) = make_float2(o0[0], o0[1]);
                    *reinterpret_cast<float2*>(dst + 8) = make_float2(o1[0], o1[1]);
                }
            }
            if (g < G && t == 0) {
                ml[(warp * 16 + g) * 2] = mx;
                ml[(warp * 16 + g) * 2 + 1] = lsum;
            }
        }
        ring_release(C.ring(), k0);
        ring_release(C.ring(), k0 + 1);
        csync();
        // merge the warps (fixed order) into the chunk partial: O (unnormalised), then (max, sum) per head.
        // First each head's chunk maximum and the warps' factors relative to it, then O two columns a thread.
        const int gi = (a.r * MB + a.b) * A.hkv_s + a.kh;
        unsigned long long* part = A.fp + ((size_t)gi * A.maxch + a.c) * G * (d + 2);
        float* fw = st;                                  // [warp][8 heads] (the staged q, k, v are consumed)
        if (tid < G) {
            float M = -INFINITY;
            #pragma unroll 1
            for (int w = 0; w < nw; ++w) M = fmaxf(M, ml[(w * 16 + tid) * 2]);
            float den = 0.f;
            #pragma unroll 1
            for (int w = 0; w < nw; ++w) {
                const float f = ex2_approx(ml[(w * 16 + tid) * 2] - M);
                fw[w * 8 + tid] = f;
                den = fmaf(f, ml[(w * 16 + tid) * 2 + 1], den);
            }
            ll_st(part + G * d / 2 + 2 * tid, M, ep);
            ll_st(part + G * d / 2 + 2 * tid + 1, den, ep);
        }
        csync();
        // O as bf16 (it feeds the bf16 o_proj operand): four values a thread, two to a pair
        const int lq = d == 128 ? 5 : 4;                 // log2(d / 4)
        #pragma unroll 1
        for (int idx = tid; idx < G * d / 4; idx += kCT) {
            const int j = idx >> lq, e = 4 * (idx - (j << lq));
            float4 nsum = make_float4(0.f, 0.f, 0.f, 0.f);
            #pragma unroll 1
            for (int w = 0; w < nw; ++w) {
                const float f = fw[w * 8 + j];
                const float4 o = *reinterpret_cast<const float4*>(C.att() + (w * G + j) * d + e);
                nsum.x = fmaf(f, o.x, nsum.x);
                nsum.y = fmaf(f, o.y, nsum.y);
                nsum.z = fmaf(f, o.z, nsum.z);
                nsum.w = fmaf(f, o.w, nsum.w);
            }
            const unsigned long long p0 = ((unsigned long long)ep << 32) | pack_bf16x2(nsum.x, nsum.y);
            const unsigned long long p1 = ((unsigned long long)ep << 32) | pack_bf16x2(nsum.z, nsum.w);
            asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(part + (j * d + e) / 2), "l"(p0), "l"(p1)
                         : "memory");
        }
        stamp(A, l, 1, 1);
    }
    return true;
}

__global__ void __launch_bounds__(kChainThreads, 1) chain_kernel(const __grid_constant__ ChainArgs A) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5;
    Ctx C;
    C.init(sm, A);
    const CRing R = C.ring();
    ChainLayer* lay = reinterpret_cast<ChainLayer*>(sm + A.sm_misc + kLayOff);
    if (tid == 0) {
        for (int s = 0; s < A.n_slots; ++s) {
            mbar_init(&R.full[s], 1);
            mbar_init(&R.empty[s], kCW);
        }
        *R.abort = 0;
        fence_mbar_init();
    }
    // this CTA's items of the projection phases (static tables)
    int* misc = C.misc();
    for (int p = 0; p < 4; ++p) {
        const int* st = A.tab + A.tab_off[p];
        const int a = st[blockIdx.x], n = st[blockIdx.x + 1] - a;
        if (tid == 0) misc[kMiCnt + p] = n;
        // QKV and gate/up items as (shard << 16) | row block
        const int per_r = p == PH_QKV ? A.qkv_rows / 8 : p == PH_GU ? A.F_s / 8 : 0;
        for (int i = tid; i < n; i += blockDim.x) {
            const int v = st[A.grid + 1 + a + i];
            misc[kMiItems + p * kChainMaxItems + i] = per_r ? (v / per_r) << 16 | (v % per_r) : v;
        }
    }
    // query rows >= G of the attention tile stay zero
    for (int i = tid; i < kPsBytes / 2; i += blockDim.x) C.qs()[i] = __float2bfloat16_rn(0.f);
    // layer 0's pointers
    for (int i = tid; i < (int)(sizeof(ChainLayer) / 8); i += blockDim.x)
        reinterpret_cast<unsigned long long*>(&lay[0])[i] = reinterpret_cast<const unsigned long long*>(A.layers)[i];
    __syncthreads();
    pdl_trigger();
    // Register split: the launch gives each of the 384 threads 168 registers
    // (64512). The third warpgroup (the copy-issuing warp and three idle
    // warps) keeps 40 each (5120), which leaves the consumers 232 each
    // (59392): 5120 + 59392 = 64512, so the increase is always satisfiable
    // (the launcher checks the launch's register count).
    if (warp >= kCW) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs) : "memory");
        if (warp == kCW && (tid & 31) == 0) chain_producer(A, R, misc);
        return;
    }
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsumerRegs) : "memory");
    pdl_wait();   // inputs, positions, caches and the launch counter of the preceding kernel
    const unsigned gen = *reinterpret_cast<volatile unsigned*>(A.gen);
    if (tid < kTMax) {
        const int p = tid < A.T ? A.pos[tid] : 0;
        misc[kMiPos + tid] = p;
        if (tid < A.T && (p < 0 || p >= A.max_kv)) set_status(A.status, TP_ERR_CAPACITY);
        int nch = 0, cs;
        if (tid < A.T) att_split(att_len(A, p), A.ck, nch, cs);
        misc[kMiNch + tid] = nch;
    }
    constexpr int kLayChunks = (int)(sizeof(ChainLayer) / 16);
    static_assert(sizeof(ChainLayer) % 16 == 0, "layer record copied in 16-byte pieces");
    for (int l = 0; l < A.L; ++l) {
        if (l > 0) asm volatile("cp.async.wait_all;" ::: "memory");
        csync();
        C.lb = l & 1;
        if (l + 1 < A.L && tid < kLayChunks) {
            cp_async16(reinterpret_cast<unsigned char*>(&lay[(l + 1) & 1]) + 16 * tid,
                       reinterpret_cast<const unsigned char*>(A.layers + l + 1) + 16 * tid);
            asm volatile("cp.async.commit_group;" ::: "memory");
        }
        const unsigned ep = gen * 256u + (unsigned)l + 1u;
        bool ok = true;
        #pragma unroll 1
        for (int st = 0; st < 5 && ok; ++st) ok = st == 1 ? phase_att(C, A, l, ep) : proj_step(C, A, l, ep, step_phase(st));
        if (!ok) break;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    csync();
    if (tid == 0) {
        // the last CTA to finish advances the launch counter (epochs of the next launch)
        __threadfence();
        const unsigned old = atomicAdd(A.done, 1u);
        if (old == (unsigned)A.grid - 1u) {
            *reinterpret_cast<volatile unsigned*>(A.done) = 0u;
            __threadfence();
            atomicAdd(A.gen, 1u);
        }
    }
}

}  // namespace

size_t chain_smem(ChainArgs& a) {
    const ChainSmem L = chain_layout(a.N, a.max_batch, a.H, a.xa_stride, a.d, a.n_slots);
    a.sm_misc = L.misc;
    a.sm_xin = L.xin;
    a.sm_xa = L.xa;
    a.sm_gam = L.gam;
    a.sm_att = L.att;
    a.sm_stage = L.stage;
    a.sm_qs = L.qs;
    a.sm_res = L.res;
    a.sm_part = L.part;
    a.sm_carry = L.carry;
    a.sm_ring = L.ring;
    return (size_t)L.total;
}

cudaError_t chain_map(const void* W, long K, long rows, int kc, int box_rows, CUtensorMap* out) {
    static std::mutex mu;
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (K % 64 || kc < 1 || kc > 256 || box_rows < 1 || box_rows > 256) return cudaErrorInvalidValue;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void**>(&encode),
                                                         12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || !encode) return e != cudaSuccess ? e : cudaErrorNotSupported;
    }
    cuuint64_t gdim[3] = {64u, (cuuint64_t)(K / 64), (cuuint64_t)rows};
    cuuint64_t gstride[2] = {128u, (cuuint64_t)K * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)kc, (cuuint32_t)box_rows};
    cuuint32_t estride[3] = {1u, 1u, 1u};
    CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(W), gdim, gstride, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

static_assert(kChainThreads == 3 * 128, "two consumer warpgroups and the producer's warpgroup");

cudaError_t launch_chain(const ChainArgs& a, size_t smem, cudaStream_t s) {
    static size_t configured = 0;
    static int launch_regs = -1;
    if (launch_regs < 0) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(chain_kernel));
        if (e != cudaSuccess) return e;
        launch_regs = fa.numRegs;
    }
    // the consumers' register increase waits for registers the launch holds:
    // refuse a build whose launch holds fewer than the split hands out
    if (kChainThreads * launch_regs < 128 * kProducerRegs + 256 * kConsumerRegs) return cudaErrorInvalidConfiguration;
    if (smem > configured) {
        cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(chain_kernel),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid);
    cfg.blockDim = dim3(kChainThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    // One CTA per SM, every SM taken: once the preceding kernel's CTAs have
    // left, the whole grid is resident, which the consumers' polls rely on
    // (bounded: a grid that could not become resident ends with
    // TP_ERR_TIMEOUT). Programmatic serialization lets the weight copies start
    // on SMs the preceding kernel has already left.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    ChainArgs A = a;
    void* args[] = {&A};
    cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(chain_kernel), args);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace tpk
