"""Test-side drivers of the CPU oracle on a workload's seeded inputs."""
import numpy as np

import oracle as O


def full_cache(stored: np.ndarray, max_kv: int) -> np.ndarray:
    c = O.to_f64(stored)
    B, Hkv, L, d = c.shape
    out = np.zeros((B, Hkv, max_kv, d))
    out[:, :, :L] = c
    return out


def dense_tpN(inputs: dict, max_kv: int, n_layers: int | None = None):
    """Sharded oracle block(s): returns (y, [(k_cache, v_cache) per layer])
    with caches gathered back to ``[B, Hkv, max_kv, d]``."""
    w = inputs["workload"]
    N = w.tp
    x = np.asarray(inputs["x"], dtype=np.float64)
    pos = inputs["pos"]
    layers = inputs["layers"][:n_layers] if n_layers else inputs["layers"]
    caches = []
    for i, L in enumerate(layers):
        shards = O.shard_layer(O.layer_f64(L), w, N)
        ks = O.shard_kv_cache(full_cache(inputs["k_cache"][i], max_kv), N)
        vs = O.shard_kv_cache(full_cache(inputs["v_cache"][i], max_kv), N)
        x = O.block_tpN(shards, x, ks, vs, pos, w.tokens_per_seq, w, N)
        caches.append((np.concatenate(ks, axis=1), np.concatenate(vs, axis=1)))
    return x, caches


def dense_tp1(inputs: dict, max_kv: int, n_layers: int | None = None):
    w = inputs["workload"]
    x = np.asarray(inputs["x"], dtype=np.float64)
    layers = inputs["layers"][:n_layers] if n_layers else inputs["layers"]
    for i, L in enumerate(layers):
        kc = full_cache(inputs["k_cache"][i], max_kv)
        vc = full_cache(inputs["v_cache"][i], max_kv)
        x = O.block_tp1(O.layer_f64(L), x, kc, vc, inputs["pos"], w.tokens_per_seq, w)
    return x


def moe_tpN(inputs: dict):
    w = inputs["workload"]
    N = w.tp
    eg, eu, ed = (O.to_f64(inputs[k]) for k in ("e_gate", "e_up", "e_down"))
    g = O.to_f64(inputs["gamma_ffn"])
    x = np.asarray(inputs["x"], dtype=np.float64)
    if getattr(w, "expert_parallel", 0):                 # whole experts per shard
        return O.moe_ffn_ep_tpN(O.shard_experts_ep(eg, eu, ed, N), [g] * N, x, inputs["router_logits"], w.eps,
                                w.top_k)
    shards = O.shard_experts(eg, eu, ed, N)
    return O.moe_ffn_tpN(shards, [g] * N, x, inputs["router_logits"], w.eps, w.top_k, N)
