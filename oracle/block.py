"""Float64 reference of the tensor-parallel block, its sharding rules and the
parameter gather. See the package docstring for scope and sources.

Notation: H hidden, Hq / Hkv query / key-value heads, d head_dim, F FFN
intermediate, N tensor-parallel degree (logical shards). Per-shard sizes are
Hq' = Hq/N, Hkv' = Hkv/N, F' = F/N. Weights are ``[out, in]``; a linear layer
is ``y = x @ W.T``.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# storage types
# ---------------------------------------------------------------------------


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64. A bfloat16 is the top half
    of a float32, so widening is exact."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def to_f64(a: np.ndarray) -> np.ndarray:
    """Stored tensor -> float64. ``uint16`` arrays are bfloat16 bit patterns."""
    if a.dtype == np.uint16:
        return bf16_to_f64(a)
    return np.asarray(a, dtype=np.float64)


def layer_f64(layer: dict) -> dict:
    return {k: to_f64(v) for k, v in layer.items()}


# ---------------------------------------------------------------------------
# the unsharded block's operations
# ---------------------------------------------------------------------------


def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """``x / sqrt(mean(x^2) + eps) * gamma`` over the last axis."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * gamma


def rope(u: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half rotary embedding.

    ``u`` is ``[tokens, heads, d]``, ``positions`` is ``[tokens]``. For
    ``i < d/2`` the pair ``(u_i, u_{i+d/2})`` is rotated by the angle
    ``p * theta^(-2i/d)``.
    """
    d = u.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / d)
    ang = positions.astype(np.float64)[:, None] * inv_freq[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = u[..., :half], u[..., half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def silu(z: np.ndarray) -> np.ndarray:
    """``z / (1 + exp(-z))``."""
    return z / (1.0 + np.exp(-z))


def softmax(s: np.ndarray, axis: int = -1) -> np.ndarray:
    m = np.max(s, axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
              q_pos: np.ndarray) -> np.ndarray:
    """Grouped-query attention of one sequence.

    ``q`` is ``[Sq, Hq, d]`` at positions ``q_pos`` ``[Sq]``; ``k`` and ``v``
    are ``[Lk, Hkv, d]`` for positions ``0..Lk-1``. Query head ``h`` reads
    key/value head ``h // (Hq/Hkv)``. Key ``j`` is visible to a query at
    position ``p`` iff ``j <= p`` (causal, diagonal included). Scores are
    scaled by ``1/sqrt(d)``. Returns ``[Sq, Hq, d]``.
    """
    Sq, Hq, d = q.shape
    Lk, Hkv, _ = k.shape
    group = Hq // Hkv
    visible = np.arange(Lk)[None, :] <= q_pos[:, None]          # [Sq, Lk]
    out = np.empty_like(q)
    for h in range(Hq):
        g = h // group
        s = (q[:, h, :] @ k[:, g, :].T) / np.sqrt(d)             # [Sq, Lk]
        s = np.where(visible, s, -np.inf)
        out[:, h, :] = softmax(s, axis=-1) @ v[:, g, :]
    return out


def swiglu_ffn(n: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray,
               w_down: np.ndarray) -> np.ndarray:
    """``(silu(n @ Wg.T) * (n @ Wu.T)) @ Wd.T``."""
    return (silu(n @ w_gate.T) * (n @ w_up.T)) @ w_down.T


# ---------------------------------------------------------------------------
# tp = 1: the unsharded pre-norm block
#   h = x + Attn(RMSNorm(x)),  y = h + FFN(RMSNorm(h))
# ---------------------------------------------------------------------------


def _positions(pos: np.ndarray, S: int) -> np.ndarray:
    """Positions of the S new tokens of every sequence: ``pos[b] + t``."""
    return (pos[:, None].astype(np.int64) + np.arange(S)[None, :])


def attn_half_tp1(L: dict, x: np.ndarray, k_cache: np.ndarray,
                  v_cache: np.ndarray, pos: np.ndarray, S: int, cfg) -> np.ndarray:
    """Attention half of the unsharded block.

    ``x`` is ``[B*S, H]`` (sequence-major), caches are ``[B, Hkv, Lmax, d]``
    float64 and are updated in place at positions ``pos[b]..pos[b]+S-1``
    (the cache stores rotated keys). Returns ``h = x + o @ Wo.T``.
    """
    B = pos.shape[0]
    Hq, Hkv, d = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    n = rmsnorm(x, L["gamma_attn"], cfg.eps)
    q = n @ L["wq"].T
    k = n @ L["wk"].T
    v = n @ L["wv"].T
    if "bq" in L:
        q, k, v = q + L["bq"], k + L["bk"], v + L["bv"]
    P = _positions(pos, S)
    o = np.empty((B * S, Hq * d))
    for b in range(B):
        rows = slice(b * S, (b + 1) * S)
        qb = rope(q[rows].reshape(S, Hq, d), P[b], cfg.rope_theta)
        kb = rope(k[rows].reshape(S, Hkv, d), P[b], cfg.rope_theta)
        vb = v[rows].reshape(S, Hkv, d)
        k_cache[b][:, P[b], :] = kb.transpose(1, 0, 2)
        v_cache[b][:, P[b], :] = vb.transpose(1, 0, 2)
        Lk = int(P[b, -1]) + 1
        kk = k_cache[b, :, :Lk, :].transpose(1, 0, 2)
        vv = v_cache[b, :, :Lk, :].transpose(1, 0, 2)
        o[rows] = attention(qb, kk, vv, P[b]).reshape(S, Hq * d)
    return x + o @ L["wo"].T


def ffn_half_tp1(L: dict, h: np.ndarray, cfg) -> np.ndarray:
    n2 = rmsnorm(h, L["gamma_ffn"], cfg.eps)
    return h + swiglu_ffn(n2, L["w_gate"], L["w_up"], L["w_down"])


def block_tp1(L: dict, x, k_cache, v_cache, pos, S, cfg) -> np.ndarray:
    h = attn_half_tp1(L, x, k_cache, v_cache, pos, S, cfg)
    return ffn_half_tp1(L, h, cfg)


# ---------------------------------------------------------------------------
# sharding rules (column-parallel rows, row-parallel columns, fused rows,
# replicated tensors, vocab padding) and the parameter gather
# ---------------------------------------------------------------------------

REPLICATED = "replicated"
COLWISE = "colwise"            # column-parallel: output dim (dim 0) split
ROWWISE = "rowwise"            # row-parallel: input dim (dim 1) split
FUSED_QKV = "fused_qkv"
FUSED_GATE_UP = "fused_gate_up"
PACKED_COLWISE = "packed_colwise"
VOCAB_PARALLEL = "vocab_parallel"


def check_divisible(cfg, N: int) -> None:
    """Heads, KV heads and the FFN width must divide by the TP degree
    ("Multi-GPU & Multi-Node", Requirements & constraints, Divisibility)."""
    for name in ("n_heads", "n_kv_heads", "ffn", "expert_ffn"):
        val = getattr(cfg, name, 0)
        if val and val % N:
            raise ValueError(f"{name}={val} is not divisible by tp={N}")


def shard_rows(W: np.ndarray, N: int) -> list:
    """Column-parallel: shard r holds output rows ``[r*out/N, (r+1)*out/N)``."""
    R = W.shape[0] // N
    return [W[r * R:(r + 1) * R].copy() for r in range(N)]


def shard_cols(W: np.ndarray, N: int) -> list:
    """Row-parallel: shard r holds input columns ``[r*in/N, (r+1)*in/N)``."""
    C = W.shape[1] // N
    return [W[:, r * C:(r + 1) * C].copy() for r in range(N)]


def shard_fused(segments: list, N: int) -> list:
    """A fused column-parallel weight made of stacked segments (e.g. Q, K, V)
    is sharded segment by segment: shard r is ``[seg0_r; seg1_r; ...]``."""
    parts = [shard_rows(s, N) for s in segments]
    return [np.concatenate([p[r] for p in parts], axis=0) for r in range(N)]


def vocab_padded(org_vocab: int, N: int) -> int:
    """Padded vocabulary: ``org_vocab`` rounded up to a multiple of 64*N, so
    each shard holds a multiple of 64 rows (Qwen2.5-0.5B: 151936 rows split
    75968 per shard at tp=2, as the gather-on-read PR's Problem reports)."""
    m = 64 * N
    return (org_vocab + m - 1) // m * m


def shard_vocab(W: np.ndarray, N: int, fill=np.nan) -> list:
    """Vocab-parallel head: pad rows to ``vocab_padded`` (padding rows at the
    tail, contents ``fill``), then split rows equally."""
    V, C = W.shape
    Vp = vocab_padded(V, N)
    P = np.full((Vp, C), fill, dtype=W.dtype)
    P[:V] = W
    return shard_rows(P, N)


def gather_param(shards: list, kind: str, org_vocab: int | None = None) -> np.ndarray:
    """All-gather of a sharded parameter (the gather-on-read PR, Change).

    * replicated (no shard stamp, e.g. a row-parallel bias): passes through;
    * colwise: rows concatenated in rank order;
    * rowwise: columns concatenated in rank order;
    * fused (qkv, gate_up, packed colwise): rows concatenated in rank order,
      i.e. grouped by rank -- not the unsharded segment order;
    * vocab-parallel: rows concatenated, then cut to ``org_vocab``.

    The result is a new array; the shards are not modified.
    """
    if kind == REPLICATED:
        return shards[0].copy()
    if kind in (COLWISE, FUSED_QKV, FUSED_GATE_UP, PACKED_COLWISE):
        return np.concatenate(shards, axis=0)
    if kind == ROWWISE:
        return np.concatenate(shards, axis=1)
    if kind == VOCAB_PARALLEL:
        return np.concatenate(shards, axis=0)[:org_vocab].copy()
    raise ValueError(kind)


def fused_gather_permutation(seg_rows: list, N: int) -> np.ndarray:
    """Row permutation taking the unsharded fused weight ``[seg0; seg1; ...]``
    to its rank-grouped gather: ``gathered[i] == unsharded[perm[i]]``."""
    starts = np.cumsum([0] + list(seg_rows))[:-1]
    perm = []
    for r in range(N):
        for s0, n in zip(starts, seg_rows):
            R = n // N
            perm.extend(range(s0 + r * R, s0 + (r + 1) * R))
    return np.asarray(perm, dtype=np.int64)


def shard_layer(L: dict, cfg, N: int) -> list:
    """Per-shard tensors of one dense block.

    Column-parallel: Q, K, V (and their biases) and gate, up are split on the
    output dim and fused per shard as ``[q_r; k_r; v_r]`` and
    ``[gate_r; up_r]``. Row-parallel: o_proj and down_proj are split on the
    input dim. Norm gammas are replicated ("Multi-GPU & Multi-Node", How
    tensor parallelism works: steps 1 and 3, and the replicated norms
    paragraph).
    """
    check_divisible(cfg, N)
    qkv = shard_fused([L["wq"], L["wk"], L["wv"]], N)
    gu = shard_fused([L["w_gate"], L["w_up"]], N)
    wo = shard_cols(L["wo"], N)
    wd = shard_cols(L["w_down"], N)
    if "bq" in L:
        bqkv = shard_fused([L["bq"][:, None], L["bk"][:, None], L["bv"][:, None]], N)
        bqkv = [b[:, 0] for b in bqkv]
    else:
        bqkv = [None] * N
    return [{
        "wqkv": qkv[r], "bqkv": bqkv[r], "wo": wo[r], "wgu": gu[r], "wd": wd[r],
        "gamma_attn": L["gamma_attn"].copy(), "gamma_ffn": L["gamma_ffn"].copy(),
    } for r in range(N)]


def shard_kv_cache(cache: np.ndarray, N: int) -> list:
    """Shard r owns KV heads ``[r*Hkv', (r+1)*Hkv')`` of ``[B, Hkv, L, d]``."""
    Hs = cache.shape[1] // N
    return [cache[:, r * Hs:(r + 1) * Hs].copy() for r in range(N)]


# ---------------------------------------------------------------------------
# tp = N: per-shard compute and the rank-ordered reduction
# ---------------------------------------------------------------------------


def reduce_rank_order(partials: list) -> np.ndarray:
    """Sum of the N row-parallel partials in rank order,
    ``((p0 + p1) + p2) + ...`` -- the single-device form of the all-reduce
    (TP-runtime issue, Problem and Collective backend abstraction: the local
    reduce and the copy-and-reduce fallback)."""
    acc = partials[0].copy()
    for p in partials[1:]:
        acc = acc + p
    return acc


def row_parallel_linear(x_shards: list, w_shards: list) -> np.ndarray:
    """Row-parallel linear: shard r computes ``x_r @ W_r.T`` over its slice of
    the input dim; the partials are reduced in rank order."""
    return reduce_rank_order([xs @ ws.T for xs, ws in zip(x_shards, w_shards)])


def attn_half_tpN(shards: list, x, k_caches: list, v_caches: list, pos, S, cfg, N):
    """Attention half with N logical shards ("Multi-GPU & Multi-Node", How
    tensor parallelism works, steps 1-3): each shard normalises the replicated
    ``x`` with its own copy of gamma, projects its slice of heads, rotates,
    appends to its own KV cache, attends over its own heads, and multiplies
    by its column slice of o_proj; ``h = x + sum_r partial_r`` in rank order."""
    B = pos.shape[0]
    Hq_s, Hkv_s, d = cfg.n_heads // N, cfg.n_kv_heads // N, cfg.head_dim
    P = _positions(pos, S)
    partials = []
    for r in range(N):
        Sr = shards[r]
        n = rmsnorm(x, Sr["gamma_attn"], cfg.eps)
        qkv = n @ Sr["wqkv"].T
        if Sr["bqkv"] is not None:
            qkv = qkv + Sr["bqkv"]
        q = qkv[:, :Hq_s * d]
        k = qkv[:, Hq_s * d:(Hq_s + Hkv_s) * d]
        v = qkv[:, (Hq_s + Hkv_s) * d:]
        o = np.empty((B * S, Hq_s * d))
        kc, vc = k_caches[r], v_caches[r]
        for b in range(B):
            rows = slice(b * S, (b + 1) * S)
            qb = rope(q[rows].reshape(S, Hq_s, d), P[b], cfg.rope_theta)
            kb = rope(k[rows].reshape(S, Hkv_s, d), P[b], cfg.rope_theta)
            vb = v[rows].reshape(S, Hkv_s, d)
            kc[b][:, P[b], :] = kb.transpose(1, 0, 2)
            vc[b][:, P[b], :] = vb.transpose(1, 0, 2)
            Lk = int(P[b, -1]) + 1
            o[rows] = attention(qb, kc[b, :, :Lk].transpose(1, 0, 2),
                                vc[b, :, :Lk].transpose(1, 0, 2), P[b]).reshape(S, Hq_s * d)
        partials.append(o @ Sr["wo"].T)
    return x + reduce_rank_order(partials)


def ffn_half_tpN(shards: list, h, cfg, N):
    """FFN half with N logical shards: gate/up column-parallel, SwiGLU per
    shard, down row-parallel, rank-ordered reduce, residual added last."""
    Fs = cfg.ffn // N
    partials = []
    for r in range(N):
        Sr = shards[r]
        n2 = rmsnorm(h, Sr["gamma_ffn"], cfg.eps)
        gu = n2 @ Sr["wgu"].T
        a = silu(gu[:, :Fs]) * gu[:, Fs:]
        partials.append(a @ Sr["wd"].T)
    return h + reduce_rank_order(partials)


def block_tpN(shards, x, k_caches, v_caches, pos, S, cfg, N):
    h = attn_half_tpN(shards, x, k_caches, v_caches, pos, S, cfg, N)
    return ffn_half_tpN(shards, h, cfg, N)


def block_rows_tpN(shards, x, k_caches, v_caches, pos, S, cfg, N, rows):
    """Selected rows of ``block_tpN``'s output, computing only what they
    depend on, for checks at sizes where the whole block is too slow here.

    Row ``t`` belongs to sequence ``b = t // S`` at position
    ``pos[b] + t % S``; causal attention makes it depend on the cached prefix
    of that sequence and on the keys and values of the sequence's new tokens
    up to ``t`` only. Per shard the operations are those of ``attn_half_tpN``
    (norm, projection, bias, rotation, attention, o_proj partial) restricted
    to those tokens, followed by the rank-ordered reduce, the residual and
    ``ffn_half_tpN`` on the selected rows. The caches passed in are not
    modified. Returns ``(y_rows [len(rows), H], rows)`` with rows sorted.
    """
    rows = np.array(sorted(set(int(t) for t in rows)), dtype=np.int64)
    Hq_s, Hkv_s, d = cfg.n_heads // N, cfg.n_kv_heads // N, cfg.head_dim
    P = _positions(pos, S)
    h_rows = np.empty((rows.size, x.shape[1]))
    for b in sorted(set((rows // S).tolist())):
        sel = np.nonzero(rows // S == b)[0]
        local = rows[sel] - b * S                       # token indices within the sequence
        upto = int(local.max()) + 1
        toks = slice(b * S, b * S + upto)
        Pb = P[b, :upto]
        partials = []
        for r in range(N):
            Sr = shards[r]
            n = rmsnorm(x[toks], Sr["gamma_attn"], cfg.eps)
            # the q rows of the fused projection only for the selected tokens,
            # the k and v rows for every token up to the last selected one
            W, bias = Sr["wqkv"], Sr["bqkv"]
            nq = Hq_s * d
            q = n[local] @ W[:nq].T
            kv = n @ W[nq:].T
            if bias is not None:
                q = q + bias[:nq]
                kv = kv + bias[nq:]
            q = rope(q.reshape(local.size, Hq_s, d), Pb[local], cfg.rope_theta)
            k = rope(kv[:, :Hkv_s * d].reshape(upto, Hkv_s, d), Pb, cfg.rope_theta)
            v = kv[:, Hkv_s * d:].reshape(upto, Hkv_s, d)
            kc = k_caches[r][b].copy()
            vc = v_caches[r][b].copy()
            kc[:, Pb, :] = k.transpose(1, 0, 2)
            vc[:, Pb, :] = v.transpose(1, 0, 2)
            Lk = int(Pb[-1]) + 1
            o = attention(q, kc[:, :Lk].transpose(1, 0, 2), vc[:, :Lk].transpose(1, 0, 2), Pb[local])
            partials.append(o.reshape(local.size, Hq_s * d) @ Sr["wo"].T)
        h_rows[sel] = x[rows[sel]] + reduce_rank_order(partials)
    return ffn_half_tpN(shards, h_rows, cfg, N), rows


# ---------------------------------------------------------------------------
# logits over the vocab-parallel head
# ---------------------------------------------------------------------------


def lm_head_logits(h: np.ndarray, gamma: np.ndarray, W: np.ndarray, eps: float) -> np.ndarray:
    """Logits of the final hidden state over the unpadded head ``W``
    ``[org_vocab, H]``: ``RMSNorm(h) @ W.T``. The norm is replicated ("Multi-GPU
    & Multi-Node", How tensor parallelism works); the head is the gathered
    vocab-parallel parameter (the gather-on-read PR, Change)."""
    return rmsnorm(h, gamma, eps) @ W.T


def lm_head_logits_tpN(h: np.ndarray, gamma: np.ndarray, head_shards: list, org_vocab: int,
                       eps: float) -> np.ndarray:
    """Vocab-parallel logits: shard r computes the logits of its rows of the
    padded head (column-parallel over the vocabulary), the shards' logits are
    concatenated in rank order and the padding columns (rows >= org_vocab of
    the head) are dropped, as the vocab-parallel gather drops its rows."""
    n = rmsnorm(h, gamma, eps)
    return np.concatenate([n @ Wr.T for Wr in head_shards], axis=1)[:, :org_vocab]


# ---------------------------------------------------------------------------
# MoE feed-forward block ("Multi-GPU & Multi-Node", Supported architectures:
# the router is replicated; experts are either sliced -- each shard holds 1/tp
# of every expert -- or placed whole, 1/tp of the experts per shard)
# ---------------------------------------------------------------------------


def router_topk(logits: np.ndarray, k: int):
    """Softmax over all experts, the k largest probabilities (ties to the
    lower expert id), renormalised to sum to one. Returns ``ids [T, k]``
    (int32, in descending-probability order) and ``w [T, k]``."""
    p = softmax(np.asarray(logits, dtype=np.float64), axis=-1)
    T, E = p.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k))
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-p[t, e], e))[:k]
        ids[t] = order
        w[t] = p[t, order] / np.sum(p[t, order])
    return ids, w


def bucket_by_expert(ids: np.ndarray, n_experts: int):
    """Stable grouping of the ``(token, slot)`` pairs by expert id.

    Returns ``offsets [E+1]`` and ``perm [T*k]``: the flat indices
    ``t*k + j`` of expert e's pairs are ``perm[offsets[e]:offsets[e+1]]``, in
    increasing flat index."""
    flat = ids.reshape(-1)
    counts = np.array([np.sum(flat == e) for e in range(n_experts)], dtype=np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    perm = np.concatenate([np.nonzero(flat == e)[0] for e in range(n_experts)]).astype(np.int32)
    return offsets, perm


def moe_ffn_tp1(x, gamma, e_gate, e_up, e_down, logits, eps, k):
    """``y_t = x_t + sum_j w_tj * SwiGLU_{e_tj}(RMSNorm(x)_t)``, j in order."""
    n = rmsnorm(x, gamma, eps)
    ids, w = router_topk(logits, k)
    acc = np.zeros_like(x)
    for j in range(k):
        c = np.empty_like(x)
        for e in np.unique(ids[:, j]):
            t = np.nonzero(ids[:, j] == e)[0]
            c[t] = swiglu_ffn(n[t], e_gate[e], e_up[e], e_down[e])
        acc = acc + w[:, j:j + 1] * c
    return x + acc


def shard_experts(e_gate, e_up, e_down, N):
    """Expert slicing: for every expert, shard r holds gate and up rows and
    down columns ``[r*Fe', (r+1)*Fe')``, fused as ``egu_r [E, 2Fe', H]``
    (gate rows then up rows) and ``ed_r [E, H, Fe']``."""
    Fe = e_gate.shape[1]
    Fs = Fe // N
    out = []
    for r in range(N):
        sl = slice(r * Fs, (r + 1) * Fs)
        egu = np.concatenate([e_gate[:, sl, :], e_up[:, sl, :]], axis=1)
        out.append({"egu": egu, "ed": e_down[:, :, sl].copy()})
    return out


def moe_ffn_tpN(shards, gammas, x, logits, eps, k, N):
    """Expert-sliced MoE FFN: the router is replicated; shard r computes, for
    every token, ``sum_j w_tj * SwiGLU`` of its slices of the chosen experts;
    the shards' partials are reduced in rank order and added to ``x``."""
    ids, w = router_topk(logits, k)
    partials = []
    for r in range(N):
        egu, ed = shards[r]["egu"], shards[r]["ed"]
        Fs = ed.shape[2]
        n = rmsnorm(x, gammas[r], eps)
        acc = np.zeros_like(x)
        for j in range(k):
            c = np.empty_like(x)
            for e in np.unique(ids[:, j]):
                t = np.nonzero(ids[:, j] == e)[0]
                gu = n[t] @ egu[e].T
                c[t] = (silu(gu[:, :Fs]) * gu[:, Fs:]) @ ed[e].T
            acc = acc + w[:, j:j + 1] * c
        partials.append(acc)
    return x + reduce_rank_order(partials)


def shard_experts_ep(e_gate, e_up, e_down, N):
    """Expert parallelism: shard r holds the whole experts
    ``[r*E/N, (r+1)*E/N)``, fused as ``egu_r [E/N, 2Fe, H]`` (gate rows then up
    rows) and ``ed_r [E/N, H, Fe]``; ``first`` is its first expert id. E must
    divide by N (the pages' divisibility rule, Requirements & constraints)."""
    E = e_gate.shape[0]
    if E % N:
        raise ValueError(f"{E} experts do not divide over {N} shards")
    per = E // N
    out = []
    for r in range(N):
        sl = slice(r * per, (r + 1) * per)
        out.append({"egu": np.concatenate([e_gate[sl], e_up[sl]], axis=1), "ed": e_down[sl].copy(),
                    "first": r * per})
    return out


def moe_ffn_ep_partials(shards, gammas, x, logits, eps, k):
    """Per-shard partials of the expert-parallel MoE FFN: shard r sums, over the
    choices j in order, ``w_tj * SwiGLU_e(RMSNorm_r(x)_t)`` for the chosen
    experts e it holds; a choice held elsewhere adds nothing on shard r."""
    ids, w = router_topk(logits, k)
    partials = []
    for r, sh in enumerate(shards):
        egu, ed, e0 = sh["egu"], sh["ed"], sh["first"]
        per, Fe = egu.shape[0], ed.shape[2]
        n = rmsnorm(x, gammas[r], eps)
        acc = np.zeros_like(x)
        for j in range(k):
            c = np.zeros_like(x)
            for e in np.unique(ids[:, j]):
                if not e0 <= e < e0 + per:
                    continue
                t = np.nonzero(ids[:, j] == e)[0]
                gu = n[t] @ egu[e - e0].T
                c[t] = (silu(gu[:, :Fe]) * gu[:, Fe:]) @ ed[e - e0].T
            acc = acc + w[:, j:j + 1] * c
        partials.append(acc)
    return partials


def moe_ffn_ep_tpN(shards, gammas, x, logits, eps, k):
    """Expert-parallel MoE FFN: the shards' partials reduced in rank order and
    added to ``x`` -- the same reduce point as expert slicing."""
    return x + reduce_rank_order(moe_ffn_ep_partials(shards, gammas, x, logits, eps, k))


# ---------------------------------------------------------------------------
# helpers for parity tests on large workloads (sampled outputs)
# ---------------------------------------------------------------------------


def relerr(gpu: np.ndarray, ref: np.ndarray) -> float:
    """``max|gpu - ref| / max|ref|`` (normwise infinity relative error)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(gpu - ref)) / (den if den > 0 else 1.0))


def relerr_elementwise(gpu: np.ndarray, ref: np.ndarray, floor: float = 1e-6) -> float:
    """``max_i |gpu_i - ref_i| / max(|ref_i|, floor * max|ref|)``: the
    element-wise relative error, a diagnostic reported beside the normwise
    figure (a small localised error can hide under the normwise one; the
    floor keeps entries near zero from dominating)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    top = np.max(np.abs(ref)) if ref.size else 0.0
    den = np.maximum(np.abs(ref), floor * (top if top > 0 else 1.0))
    return float(np.max(np.abs(gpu - ref) / den)) if ref.size else 0.0
