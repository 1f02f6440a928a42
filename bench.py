"""Benchmark of the tensor-parallel block on GB300.

Workload (default): Llama-3-8B-shaped block decode, bf16 weights, 4 logical
tensor-parallel shards, batch 8, KV length 2048 -- one step is one pass of the
whole block (fused RMSNorm + column-parallel QKV + RoPE + KV append,
split-KV GQA attention, row-parallel o_proj with rank-ordered reduction,
RMSNorm + column-parallel gate/up + SwiGLU, row-parallel down_proj with
rank-ordered reduction) for the 8 new tokens.

Other workloads (`--workload`): the Llama-3-8B-shaped tp=8 prefill of 4 x
2048 tokens (tensor-core bound: reported in TFLOP/s against the bf16 peak),
the 24-layer Qwen2.5-0.5B-shaped decode, and the expert-sliced MoE
feed-forward block (256 tokens, 64 experts, top-4).

`python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
[--workload NAME]` prints one JSON line (rank 0). Under torchrun every rank
runs an independent replica on its own GPU (the path has no cross-GPU
exchange); the timed region is bracketed by a barrier and device
synchronisation and the slowest rank's time is reported. `--impl reference`
times the CPU oracle on the host.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
os.environ.setdefault("OMP_NUM_THREADS", str(os.cpu_count() or 1))
os.environ.setdefault("OPENBLAS_NUM_THREADS", os.environ["OMP_NUM_THREADS"])

import numpy as np  # noqa: E402

import synth  # noqa: E402

FWD_PER_GRAPH = 32                 # forwards captured per CUDA graph in the timed region

METRIC = "TP-block decode tokens/s + HBM GB/s (% of ~8 TB/s peak) on 1 GB300"
METRICS = {
    "decode": METRIC,
    "prefill": "TP-block prefill tokens/s + bf16 tensor TFLOP/s (% of dense peak) on 1 GB300",
    "moe": "MoE expert-sliced FFN tokens/s + HBM GB/s on 1 GB300",
    "moe_ep": "MoE expert-parallel FFN tokens/s + HBM GB/s on 1 GB300",
}
DEFAULT_WORKLOAD = "llama3_8b_decode_tp4"
WORKLOAD_KIND = {"llama3_8b_decode_tp4": "decode", "qwen25_05b_decode_tp2": "decode",
                 "llama3_8b_prefill_tp8": "prefill", "moe_expert_slice_tp4": "moe", "moe_expert_parallel_tp4": "moe"}
STAGES = {
    "decode": ["qkv_rope", "attention", "o_proj_reduce", "gate_up_swiglu", "down_reduce"],
    "prefill": ["qkv_rope", "attention", "o_proj_reduce", "gate_up_swiglu", "down_reduce"],
    "moe": ["route_bucket", "expert_gate_up", "expert_down", "combine"],
}
DOMINANT = {"decode": "gate_up_swiglu", "prefill": "gate_up_swiglu", "moe": "expert_gate_up"}
# phases of the one-launch bf16 decode step (tp_profile_phases)
STEP_PHASES = ["norm", "qkv_rope", "attention_combine", "o_proj_reduce", "gate_up_swiglu", "down_reduce"]
# each phase is reported as its streaming part and its finishing part (finishes + barrier)
STEP_INTERVALS = [f"{ph}{part}" for ph in STEP_PHASES for part in ("", "/finish")]
# the committed ncu summary of each dominant kernel and the source it was taken on
PROFILE = {"decode": ("decode_step_llama3_8b_decode.md", "kernels_decode.cu"),
           "prefill": ("tc_gateup_llama3_8b_prefill.md", "kernels_prefill.cu"),
           "moe": ("moe_gemm_expert_slice.md", "kernels_moe.cu"),
           "stack": ("chain_qwen25_05b_decode.md", "kernels_chain.cu")}
LAUNCHES_PER_LAYER = {"decode": 1, "prefill": 8, "moe": 6}
L2_BYTES = 129e6


def stage_bytes(w) -> dict:
    """Algorithmic HBM bytes per launch of each decode kernel: every weight
    and KV element read once, new K/V and activations written once."""
    es = 2 if w.dtype == "bf16" else 4
    H, Hq, Hkv, d, F, T = w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.ffn, w.tokens
    L = w.kv_len
    qkv_rows = (Hq + 2 * Hkv) * d
    return {
        "qkv_rope": qkv_rows * H * es + T * H * 4 + T * Hq * d * 4 + 2 * T * Hkv * d * es,
        "attention": 2 * w.batch * Hkv * (L + 1) * d * es + T * Hq * d * 4 + T * Hq * d * es,
        "o_proj_reduce": H * Hq * d * es + T * Hq * d * es + 2 * T * H * 4,
        "gate_up_swiglu": 2 * F * H * es + T * H * 4 + T * F * es,
        "down_reduce": H * F * es + T * F * es + 2 * T * H * 4,
    }


def step_bytes(w) -> int:
    """Bytes the method must move per decode step: weights + KV read once."""
    es = 2 if w.dtype == "bf16" else 4
    H, Hq, Hkv, d, F = w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.ffn
    weights = (H * (Hq + 2 * Hkv) * d + H * Hq * d + 3 * H * F) * es
    kv = 2 * w.batch * Hkv * (w.kv_len + 1) * d * es
    return weights * w.n_layers + kv * w.n_layers


def prefill_flops(w) -> dict:
    """Algorithmic FLOPs per launch of each prefill stage (2 per multiply-add;
    causal attention counts each query's visible keys only)."""
    H, Hq, Hkv, d, F, T, S = w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.ffn, w.tokens, w.tokens_per_seq
    L = w.kv_len
    keys = w.batch * (S * L + S * (S + 1) // 2)          # sum over queries of visible keys
    return {
        "qkv_rope": 2 * T * H * (Hq + 2 * Hkv) * d,
        "attention": 4 * d * Hq * keys,
        "o_proj_reduce": 2 * T * Hq * d * H,
        "gate_up_swiglu": 2 * T * H * 2 * F,
        "down_reduce": 2 * T * F * H,
    }


def moe_bytes(inputs) -> dict:
    """Algorithmic HBM bytes of the expert GEMMs: the weights of every expert
    that receives at least one token, read once, plus the routed activations
    (top-k of the logits; ties to the lower expert id, as the router does)."""
    w = inputs["workload"]
    lg = np.asarray(inputs["router_logits"])
    ids = np.argsort(-lg, axis=1, kind="stable")[:, :w.top_k]
    hit = np.unique(ids).size
    es, H, Fe, ns = 2, w.hidden, w.expert_ffn, w.tokens * w.top_k
    return {"expert_gate_up": hit * 2 * Fe * H * es + w.tp * ns * H * es + ns * Fe * es,
            "expert_down": hit * H * Fe * es + ns * Fe * es + w.tp * ns * H * 4,
            "experts_hit": hit}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return {"hbm": float(j["hbm_gbs"]), "tensor_burst": float(j["bf16_tflops"]),
                "tensor_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), "kind": "measured"}
    return {"hbm": 6800.0, "tensor_burst": 1900.0, "tensor_sustained": 1700.0, "kind": "fallback"}


def traffic_fields(kind: str) -> dict:
    """`traffic` (DRAM bytes per launch of the dominant kernel) and where it
    comes from: the committed ncu summary of that kernel, used only if it was
    taken on the current kernel source; null otherwise."""
    name, src_name = PROFILE[kind]
    v = kernel_traffic(kind)
    src = (f"profiles/{name}: dram__bytes_read.sum + dram__bytes_write.sum of one ncu capture, taken on the "
           f"current {src_name}" if v is not None else
           f"none: no ncu capture of the current {src_name} (profiles/{name} predates it)")
    return {"traffic": v, "traffic_source": src}


def kernel_traffic(kind: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    name, src_name = PROFILE[kind]
    f = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(f):
        return None
    txt = open(f).read()
    m1 = re.search(r"dram_bytes_per_launch:\s*([0-9.]+)", txt)
    m2 = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", txt)
    if not (m1 and m2):
        return None
    src = os.path.join(ROOT, "megatron_tensor_block_gb300", "csrc", src_name)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    return float(m1.group(1)) if sha.startswith(m2.group(1)) else None


class Clocks:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle legs
# ---------------------------------------------------------------------------


class OracleLeg:
    """The CPU oracle on a bounded sample of a workload. Setup (float64
    shards and caches) is untimed; `step()` processes one sample unit and
    returns the tokens it covered."""

    def __init__(self, inputs):
        import oracle as O
        self.O = O
        self.inputs = inputs
        w = self.w = inputs["workload"]
        self.kind = WORKLOAD_KIND.get(w.name, "decode")
        self.i = 0
        if self.kind == "moe":
            eg, eu, ed = (O.to_f64(inputs[k]) for k in ("e_gate", "e_up", "e_down"))
            self.ep = bool(w.expert_parallel)
            self.shards = (O.shard_experts_ep if self.ep else O.shard_experts)(eg, eu, ed, w.tp)
            self.gammas = [O.to_f64(inputs["gamma_ffn"])] * w.tp
            self.x = np.asarray(inputs["x"], dtype=np.float64)
            self.chunk = 16
            return
        self.layers = [O.shard_layer(O.layer_f64(L), w, w.tp) for L in inputs["layers"]]
        kc = np.zeros((w.batch, w.n_kv_heads, w.max_kv, w.head_dim))
        vc = np.zeros_like(kc)
        self.caches = []
        for li in range(len(inputs["layers"])):
            k, v = kc.copy(), vc.copy()
            k[:, :, :w.kv_len] = O.to_f64(inputs["k_cache"][li])
            v[:, :, :w.kv_len] = O.to_f64(inputs["v_cache"][li])
            self.caches.append((O.shard_kv_cache(k, w.tp), O.shard_kv_cache(v, w.tp)))
        self.x = np.asarray(inputs["x"], dtype=np.float64)
        self.chunk = 64 if self.kind == "prefill" else 1

    def describe(self) -> str:
        if self.kind == "moe":
            return (f"{self.chunk}-token slices of the {self.w.tokens} routed tokens through the float64 numpy "
                    f"oracle's {'expert-parallel' if self.ep else 'expert-sliced'} MoE block (tp={self.w.tp})")
        if self.kind == "prefill":
            return (f"the first {self.chunk} prompt tokens (positions 0..{self.chunk - 1}) of one sequence through "
                    f"the float64 numpy oracle's sharded block (tp={self.w.tp}), repeated; the full workload is "
                    f"{self.w.batch} x {self.w.tokens_per_seq} tokens with longer causal spans")
        return (f"single-token decode steps (one sequence each, round-robin over the batch of {self.w.batch}) "
                f"through the float64 numpy oracle's sharded block ({self.w.n_layers} layer(s))")

    def step(self) -> int:
        O, w = self.O, self.w
        if self.kind == "moe":
            t0 = (self.i * self.chunk) % w.tokens
            self.i += 1
            sl = slice(t0, t0 + self.chunk)
            if self.ep:
                O.moe_ffn_ep_tpN(self.shards, self.gammas, self.x[sl], self.inputs["router_logits"][sl], w.eps,
                                 w.top_k)
            else:
                O.moe_ffn_tpN(self.shards, self.gammas, self.x[sl], self.inputs["router_logits"][sl], w.eps,
                              w.top_k, w.tp)
            return self.chunk
        if self.kind == "prefill":
            x = self.x[:self.chunk]
            pos = np.zeros(1, dtype=np.int32)
            for shards, (ks, vs) in zip(self.layers, self.caches):
                x = O.block_tpN(shards, x, [k[:1] for k in ks], [v[:1] for v in vs], pos, self.chunk, w, w.tp)
            return self.chunk
        b = self.i % w.batch
        self.i += 1
        x = self.x[b:b + 1]
        pos = self.inputs["pos"][b:b + 1]
        for shards, (ks, vs) in zip(self.layers, self.caches):
            x = O.block_tpN(shards, x, [k[b:b + 1] for k in ks], [v[b:b + 1] for v in vs], pos, 1, w, w.tp)
        return 1


def lens_timing(w, stream, peak: float, n: int = 50) -> dict:
    """Logits of the final hidden state over the vocab-parallel head (the
    lens), timed alone on a head of the workload's shape: one launch reads
    the whole head (larger than L2, so no flush between launches)."""
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import desc_of, to_device
    hi = synth.make_inputs(synth.scaled(w, n_layers=1))
    plan = tb.tp_plan(desc_of(w), w.tp)
    info = tb.tp_plan_get_info(plan)
    V, H = hi["lm_head"].shape
    full = to_device(hi["lm_head"])
    shards = [torch.empty(info["vocab_rows_shard"], H, dtype=full.dtype, device="cuda") for _ in range(w.tp)]
    tb.tp_shard_param(plan, tb.TP_PARAM_VOCAB_PARALLEL, full, V, H, tb.TP_BF16, shards)
    del full
    x = to_device(hi["x"])
    g = to_device(hi["gamma_final"].astype(np.float32))
    out = torch.empty(w.tokens * V, dtype=torch.float32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(3):
            tb.tp_lm_head_forward(plan, shards, g, x, w.tokens, out, None, stream)
        e0.record(stream)
        for _ in range(n):
            tb.tp_lm_head_forward(plan, shards, g, x, w.tokens, out, None, stream)
        e1.record(stream)
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / n
    nbytes = info["vocab_rows_shard"] * w.tp * H * 2
    gbs = nbytes / (us / 1e6) / 1e9
    return {"kernel": "lm_head_kernel (tp_lm_head_forward)", "us": us, "algorithmic_bytes": nbytes, "gbs": gbs,
            "frac_of_peak": gbs / peak, "launches": n}


def cpu_model() -> str:
    """The host CPU's model name (lscpu on Arm hosts, /proc/cpuinfo elsewhere)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_rate(inputs, budget_s: float) -> dict:
    """Tokens per second of the oracle leg over about `budget_s` seconds."""
    leg = OracleLeg(inputs)
    leg.step()                                           # warm
    n, tok, t0 = 0, 0, time.perf_counter()
    while True:
        tok += leg.step()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 4096:
            break
    out = {"value": tok / el, "unit": "tokens/s", "steps": n, "seconds": el,
           "sample": f"{n} x " + leg.describe() + "; weights pre-sharded to float64 outside the timing"}
    if leg.kind == "prefill":
        out["extrapolation"] = prefill_extrapolation(leg, el / n)
    return out


def prefill_extrapolation(leg, s_per_sample: float) -> dict:
    """The whole prefill step's oracle time, extrapolated from the sample by
    FLOPs: the sample is `chunk` prompt tokens at positions 0..chunk-1 of one
    sequence, so its linear FLOPs scale with tokens and its attention FLOPs
    with the visible keys."""
    w = leg.w
    full = sum(prefill_flops(w).values())
    sample = sum(prefill_flops(synth.scaled(w, batch=1, tokens_per_seq=leg.chunk, kv_len=0)).values())
    return {"method": "sample seconds x (full-step FLOPs / sample FLOPs)", "sample_flops": sample,
            "full_step_flops": full, "full_step_s": s_per_sample * full / sample,
            "tokens_per_s": w.tokens / (s_per_sample * full / sample)}


def cpu_baseline(inputs, budget_s: float = 15.0) -> dict:
    """The oracle as it stands, on the host: all cores in this process (the
    reported value), then one thread in a child process (BLAS threads are
    fixed when numpy loads)."""
    w = inputs["workload"]
    allc = oracle_rate(inputs, budget_s)
    out = {"value": allc["value"], "unit": "tokens/s", "cores": int(os.environ["OMP_NUM_THREADS"]),
           "kind": "oracle", "cpu_model": cpu_model(), "sample": allc["sample"]}
    if "extrapolation" in allc:
        out["extrapolation"] = allc["extrapolation"]
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--cpu-leg", "--workload", w.name,
                            "--cpu-budget", str(budget_s / 2)], env=env, capture_output=True, text=True,
                           timeout=300)
        one = json.loads(r.stdout.strip().splitlines()[-1])
        out["single_thread"] = {"value": one["value"], "unit": "tokens/s", "cores": 1, "sample": one["sample"]}
    except (OSError, subprocess.SubprocessError, ValueError, IndexError, KeyError) as e:
        out["single_thread"] = {"value": None, "error": f"{type(e).__name__}: {e}"[:200]}
    return out


def run_cpu_leg(args):
    """Child process of cpu_baseline: the oracle leg with this process's
    thread settings, as one JSON line."""
    w = synth.WORKLOADS[args.workload]
    r = oracle_rate(synth.make_inputs(w, with_head=False), args.cpu_budget)
    r["threads"] = int(os.environ.get("OMP_NUM_THREADS", "0"))
    print(json.dumps(r), flush=True)


def config_of(w) -> dict:
    kind = WORKLOAD_KIND[w.name]
    c = {"workload": w.name, "tp_logical_shards": w.tp, "hidden": w.hidden}
    if kind == "moe":
        c.update(tokens=w.tokens, experts=w.n_experts, top_k=w.top_k, expert_ffn=w.expert_ffn)
    else:
        c.update(batch=w.batch, tokens_per_seq=w.tokens_per_seq, kv_len=w.kv_len, layers=w.n_layers,
                 heads=[w.n_heads, w.n_kv_heads], head_dim=w.head_dim, ffn=w.ffn)
    return c


def run_reference(args, world, rank):
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    kind = WORKLOAD_KIND[w.name]
    inputs = synth.make_inputs(w, with_head=False)
    leg = OracleLeg(inputs)
    for _ in range(args.warmup):
        leg.step()
    budget = 120.0
    t0 = time.perf_counter()
    n, tok = 0, 0
    for _ in range(args.steps):
        tok += leg.step()
        n += 1
        if time.perf_counter() - t0 > budget:
            break
    el = time.perf_counter() - t0
    value = tok / el
    cores = int(os.environ["OMP_NUM_THREADS"])
    sample = (f"each step is {leg.describe()}; {n} of {args.steps} requested steps fit the {budget:.0f} s bound")
    cpu = {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
           "sample": sample}
    if leg.kind == "prefill":
        cpu["extrapolation"] = prefill_extrapolation(leg, el / max(n, 1))
    line = {"impl": "reference", "metric": METRICS["moe_ep" if getattr(w, "expert_parallel", 0) else kind], "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": n, "steps_requested": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / max(n, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w),
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------


def graph_timing(fwd, stream, steps: int, warmup: int, local: int, world: int):
    """Device-resident timing of `steps` forwards: forwards are captured
    FWD_PER_GRAPH to a CUDA graph, so consecutive launches overlap through
    programmatic dependent launch as they would inside a model's graph (a
    dependency between two graph launches is a full serialisation); a
    one-forward graph covers a remainder. Returns the slowest rank's
    milliseconds, the forwards per graph and the clock record of the timed
    region (barrier and device synchronisation on both sides)."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(3):
            fwd(stream=stream)
    stream.synchronize()
    per = max(1, min(FWD_PER_GRAPH, steps))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(per):
            fwd(stream=stream)
    graph1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph1, stream=stream):
        fwd(stream=stream)
    for _ in range(max(warmup, 3)):
        graph.replay()
        graph1.replay()
    torch.cuda.synchronize()
    clocks = Clocks(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(steps // per):
            graph.replay()
        for _ in range(steps % per):
            graph1.replay()
        ev1.record(stream)
    ev1.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    return max_over_ranks(ev0.elapsed_time(ev1), world), per, clk


# workloads measured beside the headline in the default run, with the number
# of forwards that fill about a second of device time
SIDE_WORKLOADS = {"llama3_8b_prefill_tp8": 2.7, "moe_expert_slice_tp4": 0.2, "moe_expert_parallel_tp4": 0.18}


def side_measure(name: str, args, local: int) -> dict:
    """Device-resident measurement of another workload, reported as a key of
    the headline line: the same graph timing as the headline over about a
    second of forwards (so the clock record has samples under load), then
    events around each stage of 200 more forwards, and the roofline of the
    dominant stage."""
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import Model
    w = synth.WORKLOADS[name]
    kind = WORKLOAD_KIND[name]
    inputs = synth.make_inputs(w, with_head=False)
    model = Model(inputs, share_norm=True)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    steps = max(args.steps, int(1000.0 / SIDE_WORKLOADS[name]))
    t_ms, per, clk = graph_timing(model.forward, stream, steps, args.warmup, local, 1)
    assert model.ws.status() == 0, f"{name}: device status after the timed region"
    ms_step = t_ms / steps
    stages = STAGES[kind]
    n_prof = 200
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(n_prof)]
    for row in evs:
        for e in row:
            e.record(stream)
    stream.synchronize()
    with torch.cuda.stream(stream):
        for i in range(n_prof):
            tb.tp_profile_stages(model.plan, evs[i])
            model.forward(stream=stream)
        tb.tp_profile_stages(model.plan, None)
    torch.cuda.synchronize()
    stage_ms = {st: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n_prof))
                for j, st in enumerate(stages)}
    pk = peaks()
    dom = DOMINANT[kind]
    out = {"workload": name, "config": config_of(w), "steps": steps, "ms_per_step": ms_step,
           "tokens_per_s": w.tokens * steps / (t_ms / 1e3), "stages_us": {k: 1e3 * v for k, v in stage_ms.items()},
           "launch": f"CUDA graph of {per} forwards, replayed; stage times from 200 forwards with events "
                     f"between the stages (programmatic overlap off)", "clocks": clk}
    if kind == "prefill":
        fl = prefill_flops(w)
        step_tf = sum(fl.values()) / (ms_step / 1e3) / 1e12
        dom_tf = fl[dom] / (stage_ms[dom] / 1e3) / 1e12
        out.update(step_flops=sum(fl.values()), step_tflops=step_tf,
                   frac_of_burst=step_tf / pk["tensor_burst"], frac_of_sustained=step_tf / pk["tensor_sustained"],
                   frac_of_nominal_2250=step_tf / 2250.0,
                   roofline={"bound": "tensor", "kernel": dom, "achieved": dom_tf, "peak": pk["tensor_sustained"],
                             "unit": "TFLOP/s", "frac": dom_tf / pk["tensor_sustained"],
                             "peak_kind": pk["kind"] + " bf16 dense, sustained", "algorithmic_flops": fl[dom]},
                   stage_tflops={k: fl[k] / (stage_ms[k] / 1e3) / 1e12 for k in stages})
    else:
        mb = moe_bytes(inputs)
        sb = mb["expert_gate_up"] + mb["expert_down"]
        gbs = sb / (ms_step / 1e3) / 1e9
        dom_gbs = mb[dom] / (stage_ms[dom] / 1e3) / 1e9
        out.update(step_bytes=sb, step_gbs=gbs, frac_of_peak=gbs / pk["hbm"], experts_hit=mb["experts_hit"],
                   roofline={"bound": "hbm", "kernel": dom, "achieved": dom_gbs, "peak": pk["hbm"], "unit": "GB/s",
                             "frac": dom_gbs / pk["hbm"], "peak_kind": pk["kind"] + " copy bandwidth",
                             "algorithmic_bytes": mb[dom]})
    del model
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def run_ours(args, world, rank, local):
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import Model

    torch.cuda.set_device(local)
    w = synth.WORKLOADS[args.workload]
    kind = WORKLOAD_KIND[w.name]
    stages = STAGES[kind]
    inputs = synth.make_inputs(w, with_head=False)
    # replicated norm gammas: one tensor shared by the shards (prefill and MoE
    # form one normalised copy; decode reads it per shard either way)
    model = Model(inputs, share_norm=(kind in ("prefill", "moe")))
    # several decode layers: all of them in one launch per token
    stacked = kind == "decode" and w.dtype == "bf16" and w.n_layers > 1 and not args.per_layer
    fwd = model.forward_stack if stacked else model.forward
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    t_ms, per, clk = graph_timing(fwd, stream, args.steps, args.warmup, local, world)
    assert model.ws.status() == 0, "device status after the timed region"
    ms_step = t_ms / args.steps
    tokens_step = w.tokens
    value = tokens_step * args.steps * world / (t_ms / 1e3)

    # ---- per-kernel durations: events around each launch, on the launching stream
    step_kernel = kind == "decode" and w.dtype == "bf16" and not stacked   # one persistent launch per layer
    n_prof = max(1, min(args.steps, 2000 if kind != "prefill" else 200))
    n_ev = 2 if (step_kernel or stacked) else len(stages) + 1
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(n_prof)]
    for row in evs:          # torch creates events lazily: record once so the raw handles exist
        for e in row:
            e.record(stream)
    stream.synchronize()
    phases = []
    with torch.cuda.stream(stream):
        for i in range(n_prof):
            if stacked:
                evs[i][0].record(stream)
                fwd(stream=stream)
                evs[i][1].record(stream)
                continue
            tb.tp_profile_stages(model.plan, evs[i])
            model.forward(stream=stream)
            if step_kernel and i % 10 == 0:
                phases.append(tb.tp_profile_phases(model.plan, len(STEP_INTERVALS), stream, median=True))
        tb.tp_profile_stages(model.plan, None)
    torch.cuda.synchronize()
    stage_ms = {}
    if stacked:
        kernel_ms = statistics.mean(evs[i][0].elapsed_time(evs[i][1]) for i in range(n_prof))
        stage_ms["all_layers"] = kernel_ms
    elif step_kernel:
        stages = STEP_INTERVALS
        for j, name in enumerate(stages):
            stage_ms[name] = statistics.mean(ph[0][j] for ph in phases) / 1e3
        median_us = {name: statistics.mean(ph[1][j] for ph in phases) for j, name in enumerate(stages)}
        kernel_ms = statistics.mean(evs[i][0].elapsed_time(evs[i][1]) for i in range(n_prof))
    else:
        for j, name in enumerate(stages):
            ts = [evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n_prof)]
            stage_ms[name] = statistics.mean(ts)
    pk = peaks()
    dom = DOMINANT[kind]
    dom_ms = stage_ms.get(dom)
    extra = {}
    if stacked:
        # back-to-back launches of the one multi-layer kernel: its average
        # launch duration in the timed region is the step time
        sb = step_bytes(w)
        achieved = sb / (ms_step / 1e3) / 1e9
        peak = pk["hbm"]
        roof = {"bound": "hbm", "kernel": f"chain_kernel (all {w.n_layers} layers in one persistent launch)",
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_kind": pk["kind"] + " copy bandwidth", "algorithmic_bytes": sb, "launch_us": ms_step * 1e3,
                "launch_us_isolated": kernel_ms * 1e3, **traffic_fields("stack")}
        extra["hbm"] = {"step_bytes": sb, "step_gbs": achieved, "frac_of_peak": achieved / peak,
                        "frac_of_8000": achieved / 8000.0, "peak_gbs": peak, "peak_kind": pk["kind"]}
        l2_note = f"inputs larger than L2 ({sb / 1e6:.1f} MB read per step vs 129 MB L2)"
    elif step_kernel:
        # the timed region is back-to-back launches of this one kernel (one per
        # layer): its average launch duration there is the step time per layer
        sb = step_bytes(w) // max(w.n_layers, 1)            # one launch = one layer
        launch_ms = ms_step / max(w.n_layers, 1)
        achieved = sb / (launch_ms / 1e3) / 1e9
        peak = pk["hbm"]
        roof = {"bound": "hbm", "kernel": "decode_step_kernel (one persistent launch per layer)", "achieved": achieved,
                "peak": peak, "unit": "GB/s", "frac": achieved / peak, "peak_kind": pk["kind"] + " copy bandwidth",
                "algorithmic_bytes": sb, "launch_us": launch_ms * 1e3,
                "launch_us_isolated": kernel_ms * 1e3, **traffic_fields(kind)}
        if w.n_layers > 1:
            roof["note"] = "phase times of the last layer of each profiled step"
        step_gbs = step_bytes(w) / (ms_step / 1e3) / 1e9
        extra["hbm"] = {"step_bytes": step_bytes(w), "step_gbs": step_gbs, "frac_of_peak": step_gbs / peak,
                        "frac_of_8000": step_gbs / 8000.0, "peak_gbs": peak, "peak_kind": pk["kind"]}
        extra["phase_median_arrival_us"] = median_us
        l2_note = f"inputs larger than L2 ({step_bytes(w) / 1e6:.1f} MB read per step vs 129 MB L2)"
    elif kind == "prefill":
        fl = prefill_flops(w)
        achieved = fl[dom] / (dom_ms / 1e3) / 1e12
        peak = pk["tensor_sustained"]
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_kind": pk["kind"] + " bf16 dense, sustained (kernel timed inside "
                "a long loop of steps)", "algorithmic_flops": fl[dom], **traffic_fields(kind)}
        step_tf = sum(fl.values()) / (ms_step / 1e3) / 1e12
        extra["tensor"] = {"step_flops": sum(fl.values()), "step_tflops": step_tf, "frac_of_peak": step_tf / peak,
                           "peak_tflops": peak, "stage_tflops": {k: fl[k] / (stage_ms[k] / 1e3) / 1e12
                                                                 for k in stages}}
        l2_note = f"inputs larger than L2 ({w.tokens * w.hidden * 4 / 1e6:.0f} MB activations, weights " \
                  f"{(sum(fl.values()) - fl['attention']) / (2 * w.tokens) * 2 / 1e6:.0f} MB per step vs 129 MB L2)"
    elif kind == "moe":
        mb = moe_bytes(inputs)
        achieved = mb[dom] / (dom_ms / 1e3) / 1e9
        peak = pk["hbm"]
        roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_kind": pk["kind"], "algorithmic_bytes": mb[dom],
                **traffic_fields(kind)}
        sb = mb["expert_gate_up"] + mb["expert_down"]
        step_gbs = sb / (ms_step / 1e3) / 1e9
        extra["hbm"] = {"step_bytes": sb, "step_gbs": step_gbs, "frac_of_peak": step_gbs / peak, "peak_gbs": peak,
                        "experts_hit": mb["experts_hit"]}
        l2_note = f"inputs larger than L2 ({sb / 1e6:.0f} MB of expert weights read per step vs 129 MB L2)"
    else:                                   # fp32 decode: separate launches
        sb = stage_bytes(w)
        achieved = sb[dom] / (dom_ms / 1e3) / 1e9
        peak = pk["hbm"]
        roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_kind": pk["kind"], "algorithmic_bytes": sb[dom],
                **traffic_fields(kind)}
        if w.n_layers > 1:
            roof["note"] = "stage times of the last layer of each step"
        step_gbs = step_bytes(w) / (ms_step / 1e3) / 1e9
        extra["hbm"] = {"step_bytes": step_bytes(w), "step_gbs": step_gbs, "frac_of_peak": step_gbs / peak,
                        "frac_of_8000": step_gbs / 8000.0, "peak_gbs": peak, "peak_kind": pk["kind"]}
        l2_note = f"inputs larger than L2 ({step_bytes(w) / 1e6:.1f} MB read per step vs 129 MB L2)"

    if roof.get("traffic") and roof.get("launch_us"):
        # the DRAM rate implied by the captured traffic (steady state: L2 may still hold part of the previous
        # step's reads, so this can sit below the algorithmic rate)
        roof["traffic_gbs"] = roof["traffic"] / (roof["launch_us"] * 1e-6) / 1e9
        roof["traffic_frac"] = roof["traffic_gbs"] / roof["peak"]
    if kind == "decode" and w.dtype == "bf16" and w.org_vocab:
        extra["lens"] = lens_timing(w, stream, pk["hbm"])   # reported beside the block, not in its time

    # ---- end to end through the public API: pinned host inputs -> device, forward, y -> pinned host.
    # As a serving loop would: inputs and outputs double-buffered, step i+1's input copy and step i's
    # output copy on their own streams beside the kernels, ordered by events (a buffer is refilled
    # only after the kernel two steps back has read it, and y only after its copy-out).
    x_host = torch.from_numpy(np.ascontiguousarray(inputs["x"])).pin_memory()
    y_hosts = [torch.empty_like(x_host).pin_memory() for _ in range(2)]
    if kind == "moe":
        in_attr, in_host = "router_logits", torch.from_numpy(np.ascontiguousarray(inputs["router_logits"])).pin_memory()
    else:
        in_attr, in_host = "pos", torch.from_numpy(inputs["pos"]).pin_memory()
    in_orig = getattr(model, in_attr)
    xs = [model.x, torch.empty_like(model.x)]
    ys = [model.y, torch.empty_like(model.y)]
    ins = [in_orig, torch.empty_like(in_orig)]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    k_done = [torch.cuda.Event() for _ in range(2)]
    h_done = [torch.cuda.Event() for _ in range(2)]
    o_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(h2d):
            if i >= 2:
                h2d.wait_event(k_done[b])               # kernel i - 2 has read these buffers
            xs[b].copy_(x_host, non_blocking=True)
            ins[b].copy_(in_host, non_blocking=True)
            h_done[b].record(h2d)
        stream.wait_event(h_done[b])
        if i >= 2:
            stream.wait_event(o_done[b])                # y of step i - 2 has been copied out
        setattr(model, in_attr, ins[b])
        fwd(x=xs[b], y=ys[b], stream=stream)
        k_done[b].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(k_done[b])
            y_hosts[b].copy_(ys[b], non_blocking=True)
            o_done[b].record(d2h)

    def e2e_run(n, e0=None, e1=None):
        if e0 is not None:
            e0.record(stream)
            h2d.wait_event(e0)
        for i in range(n):
            e2e_step(i)
        stream.wait_event(o_done[(n - 1) % 2])
        if e1 is not None:
            e1.record(stream)

    e2e_run(3)
    torch.cuda.synchronize()
    barrier(world)
    # enough steps that the pipeline's fill and drain (one input copy before the first kernel, one output
    # copy after the last) do not dominate a short run; the count is reported with the figure
    e2e_steps = max(args.steps, 200) if kind != "prefill" else max(1, min(args.steps, 100))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(e2e_steps, e0, e1)
    e1.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    setattr(model, in_attr, in_orig)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = tokens_step * e2e_steps * world / (e2e_ms / 1e3)
    assert model.ws.status() == 0
    assert torch.equal(y_hosts[(e2e_steps - 1) % 2], ys[(e2e_steps - 1) % 2].cpu())

    config = config_of(w)
    config.update({"parallelism": f"{w.tp} logical TP shards per GPU; replicas across GPUs", "l2": l2_note,
                   "launch": f"CUDA graph of {per} forwards (programmatic dependent launch between them), "
                             f"replayed; a one-forward graph for a remainder"})
    line = {
        "metric": METRICS["moe_ep" if getattr(w, "expert_parallel", 0) else kind], "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": config,
        **extra,
        "stages_us": {k: 1e3 * v for k, v in stage_ms.items()},
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "tokens/s",
                "h2d_bytes_per_step": x_host.numel() * 4 + in_host.numel() * in_host.element_size(),
                "d2h_bytes_per_step": y_hosts[0].numel() * 4, "steps": e2e_steps,
                "overlap": "inputs and outputs double-buffered; copies on their own streams beside the kernels",
                "path": ("tp_stack_decode" if stacked else "tp_block_forward") + " via the ctypes binding"},
        "gpu_launches": args.steps if stacked else
        (LAUNCHES_PER_LAYER[kind] if w.dtype == "bf16" else 5) * max(w.n_layers, 1) * args.steps,
        "clocks": clk,
    }
    if world == 1 and args.workload == DEFAULT_WORKLOAD and not args.no_side:
        # the other measured configurations, device-timed, beside the headline
        for name in SIDE_WORKLOADS:
            line[WORKLOAD_KIND[name] if not synth.WORKLOADS[name].expert_parallel else "moe_ep"] = \
                side_measure(name, args, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inputs)
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOAD_KIND))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side", action="store_true",
                    help="default workload only: skip the prefill and MoE measurements reported beside it")
    ap.add_argument("--cpu-leg", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-budget", type=float, default=10.0, help=argparse.SUPPRESS)
    ap.add_argument("--per-layer", action="store_true",
                    help="multi-layer decode: one launch per layer (tp_block_forward) instead of one launch per "
                         "token for all layers (tp_stack_decode)")
    args = ap.parse_args()
    if args.cpu_leg:
        run_cpu_leg(args)
        return
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
