"""Pins of the CPU oracle to things other than itself.

Each test checks an oracle function against a closed form, a library routine
(torch float64 on the CPU), brute force on tiny inputs, or an invariant the
pages state. They are chosen so that a dropped term, a wrong sign or index, or
a transposed operand in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TINY = synth.scaled(synth.WORKLOADS["tiny_llama_fp32_tp2"], hidden=32, n_heads=16,
                    n_kv_heads=8, head_dim=8, ffn=64, kv_len=5, batch=2, org_vocab=0)


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


# ------------------------------------------------------------------ storage


def test_bf16_decode_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x4049], dtype=np.uint16)
    got = O.bf16_to_f64(bits)
    assert got.tolist() == [1.0, -2.0, 1.0078125, 0.0, -0.0, 3.140625]


def test_bf16_rounding_of_generator_is_nearest_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0).
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20], dtype=np.float32)
    got = O.bf16_to_f64(synth.round_to_bf16_bits(x))
    assert got.tolist() == [1.0, 1.015625, 1.0078125]


# ------------------------------------------------------------------ RMSNorm


def test_rmsnorm_constant_vector_closed_form():
    eps = 1e-6
    for c in (3.0, -0.5, 1e-3):
        x = np.full((1, 16), c)
        got = O.rmsnorm(x, np.ones(16), eps)
        want = math.copysign(1.0, c) / math.sqrt(1.0 + eps / (c * c))
        assert np.allclose(got, want, rtol=1e-15, atol=0)


def test_rmsnorm_matches_torch_rms_norm():
    x = rng(1).standard_normal((5, 48))
    g = 1 + 0.1 * rng(2).standard_normal(48)
    want = F.rms_norm(torch.from_numpy(x), (48,), torch.from_numpy(g), eps=1e-5).numpy()
    assert np.allclose(O.rmsnorm(x, g, 1e-5), want, rtol=1e-13, atol=1e-15)


def test_rmsnorm_scale_invariant_without_eps():
    x = rng(3).standard_normal((3, 20))
    g = rng(4).standard_normal(20)
    assert np.allclose(O.rmsnorm(7.5 * x, g, 0.0), O.rmsnorm(x, g, 0.0), rtol=1e-14)


# ------------------------------------------------------------------ RoPE


def test_rope_position_zero_is_identity():
    u = rng(5).standard_normal((3, 2, 16))
    assert np.array_equal(O.rope(u, np.zeros(3, dtype=np.int64), 1e4), u)


def test_rope_first_pair_closed_form():
    # i = 0 has frequency 1: (1, 0) at position p turns into (cos p, sin p).
    u = np.zeros((1, 1, 4))
    u[0, 0, 0] = 1.0
    got = O.rope(u, np.array([3]), 10000.0)
    assert np.allclose(got[0, 0], [math.cos(3), 0.0, math.sin(3), 0.0], atol=1e-15)
    # last pair i = 1 of d = 4 has frequency theta^(-1/2) = 0.01
    u = np.zeros((1, 1, 4))
    u[0, 0, 1] = 1.0
    got = O.rope(u, np.array([5]), 10000.0)
    assert np.allclose(got[0, 0], [0.0, math.cos(0.05), 0.0, math.sin(0.05)], atol=1e-15)


def test_rope_equals_complex_rotation():
    # (u_i + i u_{i+d/2}) * exp(i p theta^(-2i/d)) -- an independent formulation.
    d, theta = 32, 5e5
    u = rng(6).standard_normal((7, 3, d))
    pos = rng(7).integers(0, 4096, size=7)
    z = u[..., : d // 2] + 1j * u[..., d // 2:]
    freq = np.array([theta ** (-(2 * i) / d) for i in range(d // 2)])
    zr = z * np.exp(1j * pos[:, None, None] * freq[None, None, :])
    want = np.concatenate([zr.real, zr.imag], axis=-1)
    assert np.allclose(O.rope(u, pos, theta), want, rtol=0, atol=1e-12)


def test_rope_preserves_pair_norms_and_is_relative():
    d, theta = 16, 1e4
    q = rng(8).standard_normal((1, 1, d))
    k = rng(9).standard_normal((1, 1, d))
    qr = O.rope(q, np.array([37]), theta)
    n0 = q[..., :8] ** 2 + q[..., 8:] ** 2
    n1 = qr[..., :8] ** 2 + qr[..., 8:] ** 2
    assert np.allclose(n0, n1, rtol=1e-13)
    dots = [float(np.sum(O.rope(q, np.array([m]), theta) * O.rope(k, np.array([m - 11]), theta)))
            for m in (11, 40, 300)]
    assert np.allclose(dots, dots[0], rtol=1e-11)


# ------------------------------------------------------------------ attention


def _sdpa(q, k, v, causal):
    # torch library attention on [heads, S, d] in float64, GQA by repeating kv heads
    Hq, Hkv = q.shape[1], k.shape[1]
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
    o = F.scaled_dot_product_attention(qt, kt, vt, is_causal=causal)
    return o.permute(1, 0, 2).numpy()


def test_attention_decode_matches_torch_sdpa_gqa():
    q = rng(10).standard_normal((1, 8, 16))
    k = rng(11).standard_normal((9, 2, 16))
    v = rng(12).standard_normal((9, 2, 16))
    got = O.attention(q, k, v, np.array([8]))
    assert np.allclose(got, _sdpa(q, k, v, False), rtol=1e-12, atol=1e-14)


def test_attention_prefill_causal_matches_torch_sdpa():
    q = rng(13).standard_normal((6, 4, 8))
    k = rng(14).standard_normal((6, 2, 8))
    v = rng(15).standard_normal((6, 2, 8))
    got = O.attention(q, k, v, np.arange(6))
    assert np.allclose(got, _sdpa(q, k, v, True), rtol=1e-12, atol=1e-14)


def test_attention_special_cases():
    d = 8
    v = rng(16).standard_normal((5, 1, d))
    q = rng(17).standard_normal((1, 2, d))
    # one visible key: output is that value row
    out = O.attention(q, rng(18).standard_normal((5, 1, d)), v, np.array([0]))
    assert np.allclose(out[0, 0], v[0, 0]) and np.allclose(out[0, 1], v[0, 0])
    # identical keys: output is the mean of the visible values
    k = np.repeat(rng(19).standard_normal((1, 1, d)), 5, axis=0)
    out = O.attention(q, k, v, np.array([4]))
    assert np.allclose(out[0, 0], v[:, 0].mean(axis=0), rtol=1e-13)
    # one key aligned with a huge query: output is that key's value row
    k = np.zeros((5, 1, d))
    k[3, 0, 0] = 1.0
    qq = np.zeros((1, 1, d))
    qq[0, 0, 0] = 1e4
    out = O.attention(qq, k, v, np.array([4]))
    assert np.allclose(out[0, 0], v[3, 0], atol=1e-12)


def test_attention_is_invariant_to_split_kv_chunking():
    # Flash-decoding combine: per-chunk (max, sum, unnormalised output) merged
    # with log-sum-exp weights equals the whole-sequence softmax.
    d, L = 16, 37
    q = rng(20).standard_normal((1, 1, d))
    k = rng(21).standard_normal((L, 1, d))
    v = rng(22).standard_normal((L, 1, d))
    whole = O.attention(q, k, v, np.array([L - 1]))[0, 0]
    s = (k[:, 0] @ q[0, 0]) / math.sqrt(d)
    parts = []
    for c0 in range(0, L, 10):
        sc = s[c0:c0 + 10]
        m = sc.max()
        e = np.exp(sc - m)
        parts.append((m, e.sum(), e @ v[c0:c0 + 10, 0]))
    M = max(p[0] for p in parts)
    den = sum(l * math.exp(m - M) for m, l, _ in parts)
    num = sum(o * math.exp(m - M) for m, _, o in parts)
    assert np.allclose(num / den, whole, rtol=1e-13)


# ------------------------------------------------------------------ SwiGLU


def test_silu_matches_torch_and_limits():
    z = np.linspace(-30, 30, 121)
    assert np.allclose(O.silu(z), F.silu(torch.from_numpy(z)).numpy(), rtol=1e-14, atol=1e-300)
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert abs(O.silu(np.array([60.0]))[0] - 60.0) < 1e-20


def test_ffn_half_zero_down_is_identity():
    cfg = TINY
    L = {"gamma_ffn": np.ones(cfg.hidden), "w_gate": rng(23).standard_normal((cfg.ffn, cfg.hidden)),
         "w_up": rng(24).standard_normal((cfg.ffn, cfg.hidden)), "w_down": np.zeros((cfg.hidden, cfg.ffn))}
    h = rng(25).standard_normal((3, cfg.hidden))
    assert np.array_equal(O.ffn_half_tp1(L, h, cfg), h)


# ------------------------------------------------------------------ row-parallel reduce


def test_row_parallel_partials_sum_to_unsharded_matmul_exactly():
    # Dyadic integers: every sum is exact in float64, so the rank-ordered sum
    # of the partials must equal the brute-force product bit for bit.
    x = synth.dyadic((3, 16), 30)
    W = synth.dyadic((5, 16), 31)
    brute = np.array([[sum(int(x[t, k]) * int(W[o, k]) for k in range(16)) for o in range(5)]
                      for t in range(3)], dtype=np.float64)
    for N in (1, 2, 4, 8):
        got = O.row_parallel_linear(np.split(x, N, axis=1), O.shard_cols(W, N))
        assert np.array_equal(got, brute), N


def test_reduce_is_in_rank_order():
    # ((p0 + p1) + p2) differs from p0 + (p1 + p2) in float64 for these values.
    p = [np.array([1.0]), np.array([1e-16]), np.array([1e-16])]
    assert O.reduce_rank_order(p)[0] == (1.0 + 1e-16) + 1e-16
    assert O.reduce_rank_order(p)[0] != 1.0 + (1e-16 + 1e-16)


# ------------------------------------------------------------------ whole block


def _tiny_inputs(cfg, seed, bias):
    r = rng(seed)
    H, Hq, Hkv, d, Fw = cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn
    L = {"gamma_attn": 1 + 0.1 * r.standard_normal(H), "wq": 0.2 * r.standard_normal((Hq * d, H)),
         "wk": 0.2 * r.standard_normal((Hkv * d, H)), "wv": 0.2 * r.standard_normal((Hkv * d, H)),
         "wo": 0.2 * r.standard_normal((H, Hq * d)), "gamma_ffn": 1 + 0.1 * r.standard_normal(H),
         "w_gate": 0.2 * r.standard_normal((Fw, H)), "w_up": 0.2 * r.standard_normal((Fw, H)),
         "w_down": 0.2 * r.standard_normal((H, Fw))}
    if bias:
        L["bq"] = 0.1 * r.standard_normal(Hq * d)
        L["bk"] = 0.1 * r.standard_normal(Hkv * d)
        L["bv"] = 0.1 * r.standard_normal(Hkv * d)
    return L


def _torch_block(L, x, kc, vc, pos, S, cfg):
    """The same block assembled from torch library routines (rms_norm, linear,
    scaled_dot_product_attention, silu) with RoPE as a complex rotation."""
    t = lambda a: torch.from_numpy(np.asarray(a))
    B = len(pos)
    Hq, Hkv, d, H = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.hidden
    xt = t(x)
    n = F.rms_norm(xt, (H,), t(L["gamma_attn"]), eps=cfg.eps)
    q = F.linear(n, t(L["wq"]), t(L["bq"]) if "bq" in L else None)
    k = F.linear(n, t(L["wk"]), t(L["bk"]) if "bk" in L else None)
    v = F.linear(n, t(L["wv"]), t(L["bv"]) if "bv" in L else None)
    freq = torch.tensor([cfg.rope_theta ** (-(2 * i) / d) for i in range(d // 2)], dtype=torch.float64)

    def rot(u, p):
        z = torch.complex(u[..., : d // 2], u[..., d // 2:])
        z = z * torch.polar(torch.ones_like(freq), p[:, None, None].double() * freq)
        return torch.cat([z.real, z.imag], dim=-1)

    kc, vc = t(kc).clone(), t(vc).clone()
    outs = []
    for b in range(B):
        p = torch.arange(S) + int(pos[b])
        qb = rot(q[b * S:(b + 1) * S].reshape(S, Hq, d), p)
        kb = rot(k[b * S:(b + 1) * S].reshape(S, Hkv, d), p)
        kc[b, :, p] = kb.permute(1, 0, 2)
        vc[b, :, p] = v[b * S:(b + 1) * S].reshape(S, Hkv, d).permute(1, 0, 2)
        Lk = int(pos[b]) + S
        mask = torch.arange(Lk)[None, :] <= p[:, None]
        o = F.scaled_dot_product_attention(
            qb.permute(1, 0, 2), kc[b, :, :Lk].repeat_interleave(Hq // Hkv, 0),
            vc[b, :, :Lk].repeat_interleave(Hq // Hkv, 0), attn_mask=mask)
        outs.append(o.permute(1, 0, 2).reshape(S, Hq * d))
    h = xt + F.linear(torch.cat(outs), t(L["wo"]))
    n2 = F.rms_norm(h, (H,), t(L["gamma_ffn"]), eps=cfg.eps)
    y = h + F.linear(F.silu(F.linear(n2, t(L["w_gate"]))) * F.linear(n2, t(L["w_up"])), t(L["w_down"]))
    return y.numpy(), kc.numpy(), vc.numpy()


@pytest.mark.parametrize("S,bias", [(1, False), (1, True), (4, True)])
def test_block_tp1_matches_torch_library_assembly(S, bias):
    cfg = TINY
    L = _tiny_inputs(cfg, 40 + S, bias)
    B = 2
    Lmax = cfg.kv_len + S
    kc = rng(50).standard_normal((B, cfg.n_kv_heads, Lmax, cfg.head_dim))
    vc = rng(51).standard_normal((B, cfg.n_kv_heads, Lmax, cfg.head_dim))
    pos = np.array([cfg.kv_len, cfg.kv_len - 2], dtype=np.int32)
    x = rng(52).standard_normal((B * S, cfg.hidden))
    want, wk, wv = _torch_block(L, x, kc, vc, pos, S, cfg)
    k2, v2 = kc.copy(), vc.copy()
    got = O.block_tp1(L, x, k2, v2, pos, S, cfg)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    assert np.allclose(k2, wk, atol=1e-13) and np.allclose(v2, wv, atol=1e-13)


@pytest.mark.parametrize("N", [1, 2, 4, 8])
@pytest.mark.parametrize("S", [1, 3])
def test_block_tpN_equals_tp1(N, S):
    # "every rank ends the block holding the identical hidden state" -- the
    # sharded block re-associates the row-parallel sums only.
    cfg = TINY
    L = _tiny_inputs(cfg, 60 + N, True)
    B = 2
    Lmax = cfg.kv_len + S
    kc = rng(61).standard_normal((B, cfg.n_kv_heads, Lmax, cfg.head_dim))
    vc = rng(62).standard_normal((B, cfg.n_kv_heads, Lmax, cfg.head_dim))
    pos = np.array([cfg.kv_len, 1], dtype=np.int32)
    x = rng(63).standard_normal((B * S, cfg.hidden))
    k1, v1 = kc.copy(), vc.copy()
    ref = O.block_tp1(L, x, k1, v1, pos, S, cfg)
    shards = O.shard_layer(L, cfg, N)
    ks, vs = O.shard_kv_cache(kc, N), O.shard_kv_cache(vc, N)
    got = O.block_tpN(shards, x, ks, vs, pos, S, cfg, N)
    assert O.relerr(got, ref) < 1e-12
    assert np.allclose(np.concatenate(ks, axis=1), k1, atol=1e-12)
    assert np.allclose(np.concatenate(vs, axis=1), v1, atol=1e-12)


@pytest.mark.parametrize("N", [1, 2, 4])
def test_block_rows_tpN_matches_torch_assembly_on_selected_rows(N):
    # The row-sampled form used for checks at full size: the rows it returns
    # must be the torch library block's rows (causal prefill with a cached
    # prefix, rows from both sequences, first and last tokens included), and
    # the caches it is given must stay untouched.
    cfg = TINY
    S, B = 6, 2
    L = _tiny_inputs(cfg, 80 + N, True)
    Lmax = cfg.kv_len + S
    kc = rng(81).standard_normal((B, cfg.n_kv_heads, Lmax, cfg.head_dim))
    vc = rng(82).standard_normal((B, cfg.n_kv_heads, Lmax, cfg.head_dim))
    pos = np.array([cfg.kv_len, 2], dtype=np.int32)
    x = rng(83).standard_normal((B * S, cfg.hidden))
    want, _, _ = _torch_block(L, x, kc, vc, pos, S, cfg)
    shards = O.shard_layer(L, cfg, N)
    ks, vs = O.shard_kv_cache(kc, N), O.shard_kv_cache(vc, N)
    ks0, vs0 = [k.copy() for k in ks], [v.copy() for v in vs]
    rows = [11, 0, 3, 6, 7, 5, 3]
    got, order = O.block_rows_tpN(shards, x, ks, vs, pos, S, cfg, N, rows)
    assert order.tolist() == sorted(set(rows))
    assert np.allclose(got, want[order], rtol=1e-12, atol=1e-12)
    assert all(np.array_equal(a, b) for a, b in zip(ks + vs, ks0 + vs0))


def test_block_tpN_detects_a_wrong_shard_index():
    # A plausible mistake -- a shard using its neighbour's o_proj slice -- must
    # change the answer (the invariant above would catch it).
    cfg = TINY
    L = _tiny_inputs(cfg, 70, False)
    pos = np.array([cfg.kv_len], dtype=np.int32)
    kc = rng(71).standard_normal((1, cfg.n_kv_heads, cfg.kv_len + 1, cfg.head_dim))
    vc = rng(72).standard_normal((1, cfg.n_kv_heads, cfg.kv_len + 1, cfg.head_dim))
    x = rng(73).standard_normal((1, cfg.hidden))
    shards = O.shard_layer(L, cfg, 2)
    shards[0]["wo"], shards[1]["wo"] = shards[1]["wo"], shards[0]["wo"]
    ref = O.block_tp1(L, x, kc.copy(), vc.copy(), pos, 1, cfg)
    got = O.block_tpN(shards, x, O.shard_kv_cache(kc, 2), O.shard_kv_cache(vc, 2), pos, 1, cfg, 2)
    assert O.relerr(got, ref) > 1e-3


@pytest.mark.parametrize("N", [1, 2, 4])
def test_kv_cache_shards_are_the_kv_heads_of_the_shards_q_heads(N):
    # The shards concatenate back to the cache along the head axis, and the KV
    # heads a shard holds are exactly those its q heads read under GQA (q head
    # j reads KV head j // (Hq / Hkv)), found here by brute force over the heads.
    B, Hq, Hkv, Lk, d = 2, 16, 4, 5, 3
    cache = rng(81).standard_normal((B, Hkv, Lk, d))
    shards = O.shard_kv_cache(cache, N)
    assert np.array_equal(np.concatenate(shards, axis=1), cache)
    for r, sh in enumerate(shards):
        q_heads = range(r * Hq // N, (r + 1) * Hq // N)
        needed = sorted({j // (Hq // Hkv) for j in q_heads})
        assert np.array_equal(sh, cache[:, needed])


def test_divisibility_rule():
    with pytest.raises(ValueError):
        O.check_divisible(synth.WORKLOADS["qwen25_05b_decode_tp2"], 4)  # 14 heads, 2 kv heads
    O.check_divisible(synth.WORKLOADS["llama3_8b_prefill_tp8"], 8)


# ------------------------------------------------------------------ gather


def test_gather_roundtrips_are_exact_and_shards_unchanged():
    W = rng(80).standard_normal((24, 16))
    for N in (1, 2, 4, 8):
        for kind, shard in ((O.COLWISE, O.shard_rows), (O.ROWWISE, O.shard_cols)):
            s = shard(W, N)
            before = [a.copy() for a in s]
            g = O.gather_param(s, kind)
            assert np.array_equal(g, W)
            g[0, 0] = 123.0  # the gathered tensor is a copy
            assert all(np.array_equal(a, b) for a, b in zip(s, before))
        b = rng(81).standard_normal(16)
        assert np.array_equal(O.gather_param([b] * N, O.REPLICATED), b)


def test_fused_gather_is_rank_grouped_row_multiset():
    Hq, Hkv, d, H = 4, 2, 3, 5
    Wq, Wk, Wv = (rng(82 + i).standard_normal((n * d, H)) for i, n in enumerate((Hq, Hkv, Hkv)))
    full = np.concatenate([Wq, Wk, Wv])
    for N in (1, 2):
        g = O.gather_param(O.shard_fused([Wq, Wk, Wv], N), O.FUSED_QKV)
        # equal as a row multiset
        key = lambda a: sorted(map(tuple, a))
        assert key(g) == key(full)
        # and the exact rank-grouped permutation
        perm = O.fused_gather_permutation([Hq * d, Hkv * d, Hkv * d], N)
        assert np.array_equal(g, full[perm])
        if N == 2:
            assert not np.array_equal(g, full)
            # shard 0 is [q_0; k_0; v_0]
            assert np.array_equal(g[:Hq * d // 2], Wq[:Hq * d // 2])
            assert np.array_equal(g[Hq * d // 2:Hq * d // 2 + Hkv * d // 2], Wk[:Hkv * d // 2])
        # x @ gathered.T equals the concatenation of the shards' outputs
        x = rng(90).standard_normal((2, H))
        outs = np.concatenate([x @ s.T for s in O.shard_fused([Wq, Wk, Wv], N)], axis=1)
        assert np.allclose(x @ g.T, outs, rtol=1e-15)


def test_vocab_parallel_golden():
    spec = json.load(open(os.path.join(GOLDEN, "vocab_sharding.json")))
    back = spec["check_row_from_end"]
    for case in spec["cases"]:
        V, N = case["org_vocab"], case["tp"]
        assert O.vocab_padded(V, N) // N == case["rows_per_shard"]
        assert O.vocab_padded(V, N) - V == case["padding_rows"]
    # small stand-in with the same structure as the 1000-row head
    W = rng(91).standard_normal((1000, 8))
    s = O.shard_vocab(W, 2)
    assert [a.shape[0] for a in s] == [512, 512]
    assert np.isnan(s[1][512 - 24:]).all() and not np.isnan(s[1][:512 - 24]).any()
    g = O.gather_param(s, O.VOCAB_PARALLEL, org_vocab=1000)
    assert g.shape == (1000, 8)
    assert np.array_equal(g[1000 - back], W[1000 - back])   # lives on the last shard
    assert np.array_equal(g, W)


# ------------------------------------------------------------------ MoE


def test_router_topk_against_torch_topk_and_closed_form():
    logits = rng(100).standard_normal((50, 64))
    ids, w = O.router_topk(logits, 4)
    tv, ti = torch.topk(torch.softmax(torch.from_numpy(logits), -1), 4, dim=-1)
    assert np.array_equal(ids, ti.numpy())
    # renormalised top-k probabilities == softmax over the top-k logits
    top_logits = np.take_along_axis(logits, ids.astype(np.int64), axis=1)
    assert np.allclose(w, torch.softmax(torch.from_numpy(top_logits), -1).numpy(), rtol=1e-13)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=1e-15)


def test_router_ties_go_to_lower_expert():
    ids, w = O.router_topk(np.zeros((2, 8)), 3)
    assert ids.tolist() == [[0, 1, 2], [0, 1, 2]]
    assert np.allclose(w, 1 / 3)


def test_bucketing_is_a_stable_permutation():
    ids = rng(101).integers(0, 16, size=(40, 4)).astype(np.int32)
    off, perm = O.bucket_by_expert(ids, 16)
    assert off[0] == 0 and off[-1] == 160
    assert sorted(perm.tolist()) == list(range(160))
    flat = ids.reshape(-1)
    for e in range(16):
        seg = perm[off[e]:off[e + 1]]
        assert (flat[seg] == e).all() and (np.diff(seg) > 0).all()
        assert len(seg) == np.sum(flat == e)


def _moe_inputs(seed, T=12, H=16, E=6, Fe=8):
    r = rng(seed)
    return (r.standard_normal((T, H)), 1 + 0.1 * r.standard_normal(H),
            0.3 * r.standard_normal((E, Fe, H)), 0.3 * r.standard_normal((E, Fe, H)),
            0.3 * r.standard_normal((E, H, Fe)), r.standard_normal((T, E)))


def test_moe_single_expert_equals_dense_swiglu():
    x, g, eg, eu, ed, logits = _moe_inputs(110)
    logits[:, :] = -50.0
    logits[:, 3] = 50.0
    y = O.moe_ffn_tp1(x, g, eg, eu, ed, logits, 1e-5, 1)
    n = O.rmsnorm(x, g, 1e-5)
    dense = (F.silu(torch.from_numpy(n @ eg[3].T)).numpy() * (n @ eu[3].T)) @ ed[3].T
    assert np.allclose(y, x + dense, rtol=1e-13, atol=1e-13)


def test_expert_slices_sum_to_unsliced_expert():
    x, g, eg, eu, ed, _ = _moe_inputs(111)
    n = O.rmsnorm(x, g, 1e-5)
    full = O.swiglu_ffn(n, eg[2], eu[2], ed[2])
    for N in (2, 4, 8):
        sh = O.shard_experts(eg, eu, ed, N)
        parts = []
        for s in sh:
            Fs = s["ed"].shape[2]
            gu = n @ s["egu"][2].T
            parts.append((O.silu(gu[:, :Fs]) * gu[:, Fs:]) @ s["ed"][2].T)
        assert O.relerr(O.reduce_rank_order(parts), full) < 1e-14


@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_moe_tpN_equals_tp1(N):
    x, g, eg, eu, ed, logits = _moe_inputs(112 + N)
    ref = O.moe_ffn_tp1(x, g, eg, eu, ed, logits, 1e-5, 4)
    got = O.moe_ffn_tpN(O.shard_experts(eg, eu, ed, N), [g] * N, x, logits, 1e-5, 4, N)
    assert O.relerr(got, ref) < 1e-13


def test_moe_matches_dense_per_token_loop():
    # Brute force: every token, every chosen expert, by explicit loops.
    x, g, eg, eu, ed, logits = _moe_inputs(120, T=5)
    y = O.moe_ffn_tp1(x, g, eg, eu, ed, logits, 1e-5, 2)
    n = O.rmsnorm(x, g, 1e-5)
    p = torch.softmax(torch.from_numpy(logits), -1).numpy()
    for t in range(5):
        top = np.argsort(-p[t], kind="stable")[:2]
        acc = np.zeros(16)
        for e in top:
            a = F.silu(torch.from_numpy(eg[e] @ n[t])).numpy() * (eu[e] @ n[t])
            acc += p[t, e] / p[t, top].sum() * (ed[e] @ a)
        assert np.allclose(y[t], x[t] + acc, rtol=1e-13, atol=1e-13)


# ---- MoE with expert parallelism (whole experts per shard) ------------------------


@pytest.mark.parametrize("N", [1, 2, 3, 6])
def test_moe_ep_equals_tp1(N):
    # whole experts placed on shards, partials reduced in rank order: the
    # unsharded MoE block up to rounding
    x, g, eg, eu, ed, logits = _moe_inputs(130 + N)
    ref = O.moe_ffn_tp1(x, g, eg, eu, ed, logits, 1e-5, 4)
    got = O.moe_ffn_ep_tpN(O.shard_experts_ep(eg, eu, ed, N), [g] * N, x, logits, 1e-5, 4)
    assert O.relerr(got, ref) < 1e-13


def test_moe_ep_equals_expert_slicing():
    x, g, eg, eu, ed, logits = _moe_inputs(140)
    ep = O.moe_ffn_ep_tpN(O.shard_experts_ep(eg, eu, ed, 2), [g] * 2, x, logits, 1e-5, 3)
    sl = O.moe_ffn_tpN(O.shard_experts(eg, eu, ed, 2), [g] * 2, x, logits, 1e-5, 3, 2)
    assert O.relerr(ep, sl) < 1e-13


def test_moe_ep_partials_stay_on_the_owner():
    # every token picks experts 0 and 1, both on shard 0 of 3: the other
    # shards add exactly nothing, and shard 0's partial is the whole MoE term
    x, g, eg, eu, ed, logits = _moe_inputs(141)
    logits[:, :2] += 40.0
    parts = O.moe_ffn_ep_partials(O.shard_experts_ep(eg, eu, ed, 3), [g] * 3, x, logits, 1e-5, 2)
    assert not parts[1].any() and not parts[2].any()
    ref = O.moe_ffn_tp1(x, g, eg, eu, ed, logits, 1e-5, 2) - x
    assert O.relerr(parts[0], ref) < 1e-13
    # and a choice of shard 2's expert lands on shard 2 only
    logits[0, 5] += 200.0
    parts = O.moe_ffn_ep_partials(O.shard_experts_ep(eg, eu, ed, 3), [g] * 3, x, logits, 1e-5, 2)
    assert not parts[1].any() and parts[2][0].any() and not parts[2][1:].any()


def test_moe_ep_shards_regroup_to_the_experts():
    _, _, eg, eu, ed, _ = _moe_inputs(142)
    sh = O.shard_experts_ep(eg, eu, ed, 3)
    assert [s["first"] for s in sh] == [0, 2, 4]
    egu = np.concatenate([s["egu"] for s in sh])
    assert np.array_equal(egu[:, :8], eg) and np.array_equal(egu[:, 8:], eu)
    assert np.array_equal(np.concatenate([s["ed"] for s in sh]), ed)


def test_moe_ep_rejects_indivisible_expert_count():
    _, _, eg, eu, ed, _ = _moe_inputs(143)
    with pytest.raises(ValueError):
        O.shard_experts_ep(eg, eu, ed, 4)


# ---- lens / logits over the vocab-parallel head ---------------------------------


def test_lm_head_identity_head_gives_the_closed_form_norm():
    # head rows = unit vectors, h = a constant c, gamma = 1: every logit is
    # RMSNorm(c) = sign(c) / sqrt(1 + eps / c^2), whatever the row
    H, V, eps = 64, 40, 1e-6
    W = np.eye(H)[:V]
    for c in (-2.5, 0.75, 3.0):
        h = np.full((2, H), c)
        logits = O.lm_head_logits(h, np.ones(H), W, eps)
        assert logits.shape == (2, V)
        assert np.allclose(logits, math.copysign(1.0, c) / math.sqrt(1.0 + eps / (c * c)), rtol=1e-15)


def test_lm_head_identity_head_picks_normalised_columns():
    # with unit-vector rows, logit i is column i of RMSNorm(h) (the head's
    # orientation: logits = n @ W.T, not W @ n)
    H, V, eps = 32, 20, 1e-6
    h = rng(71).standard_normal((3, H))
    g = rng(72).uniform(0.5, 1.5, H)
    perm = rng(73).permutation(H)[:V]
    W = np.eye(H)[perm]
    n = h / np.sqrt((h * h).mean(-1, keepdims=True) + eps) * g
    assert np.allclose(O.lm_head_logits(h, g, W, eps), n[:, perm], rtol=1e-14, atol=0)


@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_lm_head_vocab_parallel_equals_unsharded_and_drops_padding(N):
    H, V, eps = 64, 1000, 1e-5           # 1000 rows: padded to a multiple of 64 N, padding on the last shard
    h = rng(81).standard_normal((2, H))
    g = rng(82).uniform(0.5, 1.5, H)
    W = rng(83).standard_normal((V, H)) * 0.02
    shards = O.shard_vocab(W, N)          # padding rows are NaN: any leak shows up
    assert sum(s.shape[0] for s in shards) == O.vocab_padded(V, N)
    tpN = O.lm_head_logits_tpN(h, g, shards, V, eps)
    assert tpN.shape == (2, V) and np.isfinite(tpN).all()
    ref = O.lm_head_logits(h, g, W, eps)
    assert np.allclose(tpN, ref, rtol=1e-12, atol=1e-14)
    # the last real row lives on the last shard (the cross-shard index of the gather)
    last = O.rmsnorm(h, g, eps) @ W[V - 1]
    assert np.allclose(tpN[:, V - 1], last, rtol=1e-12)


def test_lm_head_matches_torch():
    H, V, eps = 96, 300, 1e-6
    h = rng(91).standard_normal((4, H))
    g = rng(92).uniform(0.5, 1.5, H)
    W = rng(93).standard_normal((V, H))
    t = F.linear(F.rms_norm(torch.from_numpy(h), (H,), torch.from_numpy(g), eps), torch.from_numpy(W)).numpy()
    assert np.allclose(O.lm_head_logits(h, g, W, eps), t, rtol=1e-12, atol=1e-12)


def test_elementwise_error_sees_what_the_normwise_error_hides():
    # the survey's o16 diagnostic: per-entry error relative to the entry, with
    # a floor of 1e-6 of the largest magnitude for entries near zero
    ref = np.array([1000.0, 1.0])
    gpu = np.array([1000.0, 1.5])
    assert O.relerr(gpu, ref) == pytest.approx(0.5 / 1000.0)
    assert O.relerr_elementwise(gpu, ref) == pytest.approx(0.5)
    # an exact zero in ref is measured against the floor, not divided by zero
    assert O.relerr_elementwise(np.array([1.0, 1e-7]), np.array([1.0, 0.0])) == pytest.approx(0.1)
    # sign errors count in full; equal arrays give 0
    assert O.relerr_elementwise(np.array([-2.0, 4.0]), np.array([2.0, 4.0])) == pytest.approx(2.0)
    assert O.relerr_elementwise(ref, ref) == 0.0
    # never below the normwise figure
    rng = np.random.default_rng(0)
    a = rng.standard_normal(1000)
    b = a + 1e-3 * rng.standard_normal(1000)
    assert O.relerr_elementwise(b, a) >= O.relerr(b, a)
