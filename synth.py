"""Seeded synthetic inputs for the tensor-parallel block workloads.

This module is the one piece shared by the CPU oracle and the CUDA path. It
only draws random numbers and rounds them to the storage type; it holds none
of the block's arithmetic (no norm, projection, attention, sharding or
reduction).

Every tensor is produced in a fixed order from ``numpy.random.Generator
(PCG64(seed))``. Floating-point draws are made in float32 and then rounded to
the storage type: float32 values are kept as they are, bfloat16 values are
rounded to nearest-even and returned as their raw ``uint16`` bit patterns.

Shapes follow PyTorch's ``nn.Linear`` convention, weights ``[out, in]`` so that
``y = x @ W.T`` (the convention used by "Gather tensor-parallel sharded
parameters on read in a trace", section Change, fused-weights bullet).

The five workloads are synthetic stand-ins shaped like the models the pages
measure: a tiny Llama block, a Qwen2.5-0.5B-shaped 24-layer decoder, a
Llama-3-8B-shaped block in decode and in prefill, and an expert-sliced MoE
feed-forward block.
"""
from __future__ import annotations

import dataclasses
import numpy as np

F32 = "f32"
BF16 = "bf16"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    eps: float
    rope_theta: float
    dtype: str                # storage type of weights and KV cache
    tp: int                   # number of logical tensor-parallel shards
    batch: int                # sequences
    tokens_per_seq: int       # 1 for decode, S for prefill
    kv_len: int               # cached positions before the step
    seed: int
    n_layers: int = 1
    qkv_bias: bool = False
    org_vocab: int = 0        # lm_head rows before padding (0: no head)
    n_experts: int = 0
    top_k: int = 0
    expert_ffn: int = 0
    expert_parallel: int = 0  # MoE sharding: 0 expert slicing, 1 whole experts per shard
    mode: str = "decode"      # decode | prefill | moe_ffn

    @property
    def tokens(self) -> int:
        return self.batch * self.tokens_per_seq

    @property
    def max_kv(self) -> int:
        return self.kv_len + self.tokens_per_seq


WORKLOADS = {
    # Tiny Llama block, fp32, tp=2, batch-1 decode over 16 cached positions,
    # plus an lm_head of 1000 rows padded to 1024 for the gather.
    "tiny_llama_fp32_tp2": Workload(
        name="tiny_llama_fp32_tp2", hidden=256, n_heads=4, n_kv_heads=2,
        head_dim=64, ffn=512, eps=1e-6, rope_theta=1e4, dtype=F32, tp=2,
        batch=1, tokens_per_seq=1, kv_len=16, seed=0, org_vocab=1000),
    # Qwen2.5-0.5B-shaped 24-layer decoder, bf16, tp=2, batch-1 decode, KV 512.
    "qwen25_05b_decode_tp2": Workload(
        name="qwen25_05b_decode_tp2", hidden=896, n_heads=14, n_kv_heads=2,
        head_dim=64, ffn=4864, eps=1e-6, rope_theta=1e6, dtype=BF16, tp=2,
        batch=1, tokens_per_seq=1, kv_len=512, seed=1, n_layers=24,
        qkv_bias=True, org_vocab=151936),
    # Llama-3-8B-shaped block, decode, bf16, tp=4, batch 8, KV 2048.
    "llama3_8b_decode_tp4": Workload(
        name="llama3_8b_decode_tp4", hidden=4096, n_heads=32, n_kv_heads=8,
        head_dim=128, ffn=14336, eps=1e-5, rope_theta=5e5, dtype=BF16, tp=4,
        batch=8, tokens_per_seq=1, kv_len=2048, seed=2),
    # Llama-3-8B-shaped block, causal prefill, bf16, tp=8, 4 x 2048 tokens.
    "llama3_8b_prefill_tp8": Workload(
        name="llama3_8b_prefill_tp8", hidden=4096, n_heads=32, n_kv_heads=8,
        head_dim=128, ffn=14336, eps=1e-5, rope_theta=5e5, dtype=BF16, tp=8,
        batch=4, tokens_per_seq=2048, kv_len=0, seed=3, mode="prefill"),
    # Expert-sliced MoE feed-forward block, bf16, tp=4, 256 decode tokens.
    "moe_expert_slice_tp4": Workload(
        name="moe_expert_slice_tp4", hidden=2048, n_heads=0, n_kv_heads=0,
        head_dim=0, ffn=0, eps=1e-5, rope_theta=0.0, dtype=BF16, tp=4,
        batch=256, tokens_per_seq=1, kv_len=0, seed=4, n_experts=64, top_k=4,
        expert_ffn=1024, mode="moe_ffn"),
    # The same MoE block with expert parallelism: 16 whole experts per shard.
    "moe_expert_parallel_tp4": Workload(
        name="moe_expert_parallel_tp4", hidden=2048, n_heads=0, n_kv_heads=0,
        head_dim=0, ffn=0, eps=1e-5, rope_theta=0.0, dtype=BF16, tp=4,
        batch=256, tokens_per_seq=1, kv_len=0, seed=4, n_experts=64, top_k=4,
        expert_ffn=1024, expert_parallel=1, mode="moe_ffn"),
}


def scaled(w: Workload, **changes) -> Workload:
    """A copy of ``w`` with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(w, **changes)


def round_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest, ties to even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_as_f32(bits: np.ndarray) -> np.ndarray:
    """Decode raw bfloat16 bit patterns to float32 (exact widening)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


class _Draw:
    def __init__(self, seed: int):
        self.rng = np.random.Generator(np.random.PCG64(seed))

    def normal(self, shape, std=1.0, mean=0.0) -> np.ndarray:
        a = self.rng.standard_normal(size=shape, dtype=np.float32)
        if std != 1.0:
            a *= np.float32(std)
        if mean != 0.0:
            a += np.float32(mean)
        return a

    def stored(self, shape, dtype, std=1.0, mean=0.0) -> np.ndarray:
        a = self.normal(shape, std, mean)
        return round_to_bf16_bits(a) if dtype == BF16 else a


def _layer(d: _Draw, w: Workload) -> dict:
    H, Hq, Hkv, hd, F = w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.ffn
    t = {}
    t["gamma_attn"] = d.normal((H,), 0.02, 1.0)
    t["wq"] = d.stored((Hq * hd, H), w.dtype, 0.02)
    t["wk"] = d.stored((Hkv * hd, H), w.dtype, 0.02)
    t["wv"] = d.stored((Hkv * hd, H), w.dtype, 0.02)
    if w.qkv_bias:
        t["bq"] = d.normal((Hq * hd,), 0.02)
        t["bk"] = d.normal((Hkv * hd,), 0.02)
        t["bv"] = d.normal((Hkv * hd,), 0.02)
    t["wo"] = d.stored((H, Hq * hd), w.dtype, 0.02)
    t["gamma_ffn"] = d.normal((H,), 0.02, 1.0)
    t["w_gate"] = d.stored((F, H), w.dtype, 0.02)
    t["w_up"] = d.stored((F, H), w.dtype, 0.02)
    t["w_down"] = d.stored((H, F), w.dtype, 0.02)
    return t


def make_inputs(w: Workload, with_head: bool = True) -> dict:
    """All tensors of one workload, drawn in a fixed order.

    Returns a dict with ``layers`` (a list of per-layer weight dicts), ``x``
    (the hidden state entering the block, float32 ``[tokens, hidden]``, values
    already representable in the storage type), ``k_cache`` / ``v_cache``
    (per layer, ``[batch, kv_heads, kv_len, head_dim]`` in the storage type:
    keys are taken as already rotated), ``pos`` (``int32 [batch]``, the first
    new position of each sequence), and where present ``lm_head``
    (``[org_vocab, hidden]``) with the final norm's ``gamma_final``, or the
    MoE tensors.
    """
    d = _Draw(w.seed)
    out = {"workload": w}
    if w.mode == "moe_ffn":
        H, E, Fe = w.hidden, w.n_experts, w.expert_ffn
        out["gamma_ffn"] = d.normal((H,), 0.02, 1.0)
        out["e_gate"] = d.stored((E, Fe, H), w.dtype, 0.02)
        out["e_up"] = d.stored((E, Fe, H), w.dtype, 0.02)
        out["e_down"] = d.stored((E, H, Fe), w.dtype, 0.02)
        xs = d.stored((w.tokens, H), w.dtype, 1.0)
        out["x"] = bf16_bits_as_f32(xs) if w.dtype == BF16 else xs
        out["router_logits"] = d.normal((w.tokens, E), 1.0)
        return out
    out["layers"] = [_layer(d, w) for _ in range(w.n_layers)]
    xs = d.stored((w.tokens, w.hidden), w.dtype, 1.0)
    out["x"] = bf16_bits_as_f32(xs) if w.dtype == BF16 else xs
    kv_shape = (w.batch, w.n_kv_heads, w.kv_len, w.head_dim)
    out["k_cache"], out["v_cache"] = [], []
    for _ in range(w.n_layers):
        out["k_cache"].append(d.stored(kv_shape, w.dtype, 1.0))
        out["v_cache"].append(d.stored(kv_shape, w.dtype, 1.0))
    out["pos"] = np.full((w.batch,), w.kv_len, dtype=np.int32)
    if with_head and w.org_vocab:
        out["lm_head"] = d.stored((w.org_vocab, w.hidden), w.dtype, 0.02)
        out["gamma_final"] = d.normal((w.hidden,), 0.02, 1.0)     # the final norm before the head
    return out


def dyadic(shape, seed: int, lo: int = -4, hi: int = 4, scale_log2: int = 0):
    """Small integers times a power of two: every sum and product of such
    values stays exact in float64 (used for brute-force exactness checks)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(lo, hi + 1, size=shape).astype(np.float64) * (2.0 ** scale_log2)
