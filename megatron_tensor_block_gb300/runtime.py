"""Device-memory owner around the C ABI: allocates the per-shard buffers, KV
caches and workspace a plan asks for (with torch, used only as an
allocator), shards full weights through ``tp_shard_weights`` and chains
layers through ``tp_block_forward``. All computation is in the library."""
from __future__ import annotations

import numpy as np

from . import binding as B


def _torch():
    import torch
    return torch


def to_device(a: np.ndarray, device="cuda"):
    """Uploads a stored tensor; ``uint16`` arrays are bfloat16 bit patterns."""
    torch = _torch()
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def desc_of(w, max_kv: int | None = None, max_batch: int | None = None, max_tokens: int | None = None) -> dict:
    """``tp_model_desc`` fields for a workload description."""
    return dict(hidden=w.hidden, n_heads=w.n_heads, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, ffn=w.ffn,
                n_experts=w.n_experts, top_k=w.top_k, expert_ffn=w.expert_ffn, org_vocab=w.org_vocab,
                eps=w.eps, rope_theta=w.rope_theta, dtype=B.TP_BF16 if w.dtype == "bf16" else B.TP_F32,
                has_qkv_bias=int(w.qkv_bias), max_batch=max_batch or w.batch,
                max_tokens=max_tokens or w.tokens, max_kv=max_kv or max(w.max_kv, 1),
                expert_parallel=int(getattr(w, "expert_parallel", 0)))


class Workspace:
    def __init__(self, plan: B.Plan, info: dict, device="cuda", stream=None):
        torch = _torch()
        self.nbytes = int(info["workspace_bytes"])
        self.buf = torch.empty(max(self.nbytes, 256), dtype=torch.uint8, device=device)
        B.tp_workspace_init(plan, self.buf, self.nbytes, stream)

    def status(self, stream=None) -> int:
        return B.tp_get_device_status(self.buf, stream)


class ShardedLayer:
    """One block's shard tensors (and KV caches), built on the device."""

    def __init__(self, plan, info, w, layer: dict | None, device="cuda", moe: dict | None = None):
        torch = _torch()
        N = w.tp
        dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        es = 2 if w.dtype == "bf16" else 4
        H = w.hidden

        def buf(nbytes, dtype=dt):
            n = nbytes // (2 if dtype == torch.bfloat16 else 4)
            return torch.empty(n, dtype=dtype, device=device)

        self.full = {}
        self.shards = {k: [] for k in ("wqkv", "bqkv", "wo", "wgu", "wd", "gamma_attn", "gamma_ffn", "egu", "ed")}
        if layer is not None:
            for k, v in layer.items():
                self.full[k] = to_device(v, device)
            for r in range(N):
                self.shards["wqkv"].append(buf(info["wqkv_bytes"]))
                self.shards["bqkv"].append(buf(info["bqkv_bytes"], torch.float32) if info["bqkv_bytes"] else None)
                self.shards["wo"].append(buf(info["wo_bytes"]))
                self.shards["wgu"].append(buf(info["wgu_bytes"]))
                self.shards["wd"].append(buf(info["wd_bytes"]))
                self.shards["gamma_attn"].append(buf(info["gamma_bytes"], torch.float32))
                self.shards["gamma_ffn"].append(buf(info["gamma_bytes"], torch.float32))
            if not w.qkv_bias:
                self.shards["bqkv"] = []
        if moe is not None:
            for k in ("e_gate", "e_up", "e_down", "gamma_ffn"):
                self.full[k] = to_device(moe[k], device)
            for r in range(N):
                self.shards["egu"].append(buf(info["egu_bytes"]))
                self.shards["ed"].append(buf(info["ed_bytes"]))
                self.shards["gamma_ffn"].append(buf(info["gamma_bytes"], torch.float32))
        B.tp_shard_weights(plan, self.full, self.shards)
        del es, H

    def drop_full(self):
        """Frees the unsharded copies (only the shards are used by forward)."""
        self.full = {}


class KVCache:
    """Per-shard caches ``[max_batch][Hkv'][max_kv][d]`` filled from the full
    cache ``[B][Hkv][L][d]`` by ``tp_shard_kv`` (contiguous KV-head groups)."""

    def __init__(self, w, k_full: np.ndarray | None, v_full: np.ndarray | None, max_kv: int, max_batch: int,
                 device="cuda", plan: B.Plan | None = None):
        torch = _torch()
        N = w.tp
        dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        Hs = w.n_kv_heads // N
        self.k = [torch.zeros(max_batch, Hs, max_kv, w.head_dim, dtype=dt, device=device) for _ in range(N)]
        self.v = [torch.zeros(max_batch, Hs, max_kv, w.head_dim, dtype=dt, device=device) for _ in range(N)]
        if k_full is not None and k_full.shape[2] > 0:
            if plan is None:
                raise ValueError("KVCache: filling the shards from a full cache needs the plan")
            kf, vf = to_device(k_full, device), to_device(v_full, device)
            B.tp_shard_kv(plan, kf, vf, kf.shape[0], kf.shape[2], (self.k, self.v))

    def full(self):
        """Concatenation of the shards' caches over the KV-head dim."""
        torch = _torch()
        return torch.cat(self.k, dim=1), torch.cat(self.v, dim=1)


class Model:
    """A stack of tensor-parallel blocks of one workload on one device."""

    def __init__(self, inputs: dict, device="cuda", max_kv: int | None = None, keep_full: bool = False,
                 share_norm: bool = False):
        """``share_norm``: point every shard at shard 0's copy of each
        replicated norm gamma (the copies hold the same values), so that the
        prefill path forms one normalised copy of the activations instead of
        one per shard."""
        torch = _torch()
        w = inputs["workload"]
        self.w = w
        self.device = device
        self.max_batch = w.batch
        self.max_kv = max_kv or w.max_kv
        self.plan = B.tp_plan(desc_of(w, max_kv=self.max_kv), w.tp)
        self.info = B.tp_plan_get_info(self.plan)
        self.ws = Workspace(self.plan, self.info, device)
        self.layers, self.caches = [], []
        if w.mode == "moe_ffn":
            self.layers.append(ShardedLayer(self.plan, self.info, w, None, device, moe=inputs))
            self.router_logits = to_device(inputs["router_logits"], device)
        else:
            for i, L in enumerate(inputs["layers"]):
                self.layers.append(ShardedLayer(self.plan, self.info, w, L, device))
                self.caches.append(KVCache(w, inputs["k_cache"][i], inputs["v_cache"][i], self.max_kv,
                                           self.max_batch, device, plan=self.plan))
            self.pos = torch.from_numpy(inputs["pos"]).to(device)
        if share_norm:
            for l in self.layers:
                for k in ("gamma_attn", "gamma_ffn"):
                    if l.shards.get(k):
                        l.shards[k] = [l.shards[k][0]] * len(l.shards[k])
        if not keep_full:
            for l in self.layers:
                l.drop_full()
        self.x = to_device(inputs["x"], device)
        self.y = torch.empty_like(self.x)
        self.tmp = torch.empty_like(self.x) if len(self.layers) > 1 else None

    @property
    def mode(self) -> int:
        return {"decode": B.TP_MODE_DECODE, "prefill": B.TP_MODE_PREFILL, "moe_ffn": B.TP_MODE_MOE_FFN}[self.w.mode]

    def stack(self):
        """The decode layers as one ``tp_stack_t`` (created on first use)."""
        if getattr(self, "_stack", None) is None:
            self._stack = B.tp_stack_create(self.plan, [L.shards for L in self.layers],
                                            [(c.k, c.v) for c in self.caches])
        return self._stack

    def forward_stack(self, x=None, y=None, stream=None):
        """Decode through every layer in one launch (``tp_stack_decode``)."""
        x = self.x if x is None else x
        y = self.y if y is None else y
        B.tp_stack_decode(self.stack(), x, y, self.pos, self.w.batch, self.ws.buf, self.ws.nbytes, stream)
        return y

    def forward(self, x=None, y=None, stream=None):
        """Runs every layer; returns the output tensor."""
        x = self.x if x is None else x
        y = self.y if y is None else y
        w = self.w
        n = len(self.layers)
        cur = x
        for i, L in enumerate(self.layers):
            # ping-pong between y and tmp so the last layer writes y
            out = y if (n - 1 - i) % 2 == 0 else self.tmp
            kv = (self.caches[i].k, self.caches[i].v) if self.caches else None
            B.tp_block_forward(self.plan, L.shards, kv, cur, out, getattr(self, "pos", None), w.batch,
                               w.tokens_per_seq, self.mode, getattr(self, "router_logits", None), self.ws.buf,
                               self.ws.nbytes, stream)
            cur = out
        return y
