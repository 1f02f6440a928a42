"""Benchmark of the tensor-parallel block decode step on GB300.

Workload (default): Llama-3-8B-shaped block, bf16 weights, 4 logical
tensor-parallel shards, batch 8, KV length 2048 -- one step is one pass of the
whole block (fused RMSNorm + column-parallel QKV + RoPE + KV append,
split-KV GQA attention, row-parallel o_proj with rank-ordered reduction,
RMSNorm + column-parallel gate/up + SwiGLU, row-parallel down_proj with
rank-ordered reduction) for the 8 new tokens.

`python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]`
prints one JSON line (rank 0). Under torchrun every rank runs an independent
replica on its own GPU (the path has no cross-GPU exchange); the timed region
is bracketed by a barrier and device synchronisation and the slowest rank's
time is reported. `--impl reference` times the CPU oracle on the host.
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

METRIC = "TP-block decode tokens/s + HBM GB/s (% of ~8 TB/s peak) on 1 GB300"
DEFAULT_WORKLOAD = "llama3_8b_decode_tp4"
STAGES = ["qkv_rope", "attention", "o_proj_reduce", "gate_up_swiglu", "down_reduce"]
DOMINANT = "gate_up_swiglu"
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
    """Bytes the method must move per step: weights + KV read once."""
    es = 2 if w.dtype == "bf16" else 4
    H, Hq, Hkv, d, F = w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.ffn
    weights = (H * (Hq + 2 * Hkv) * d + H * Hq * d + 3 * H * F) * es
    kv = 2 * w.batch * Hkv * (w.kv_len + 1) * d * es
    return weights + kv


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_traffic(name: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    f = os.path.join(ROOT, "profiles", f"{name}_llama3_8b_decode.md")
    if not os.path.exists(f):
        return None
    txt = open(f).read()
    m1 = re.search(r"dram_bytes_per_launch:\s*([0-9.]+)", txt)
    m2 = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", txt)
    if not (m1 and m2):
        return None
    src = os.path.join(ROOT, "megatron_tensor_block_gb300", "csrc", "kernels_decode.cu")
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


def oracle_setup(inputs):
    """Untimed setup of the oracle: float64 shards and caches."""
    import oracle as O
    w = inputs["workload"]
    L = inputs["layers"][0]
    shards = O.shard_layer(O.layer_f64(L), w, w.tp)
    kc = np.zeros((w.batch, w.n_kv_heads, w.max_kv, w.head_dim))
    vc = np.zeros_like(kc)
    kc[:, :, :w.kv_len] = O.to_f64(inputs["k_cache"][0])
    vc[:, :, :w.kv_len] = O.to_f64(inputs["v_cache"][0])
    return shards, O.shard_kv_cache(kc, w.tp), O.shard_kv_cache(vc, w.tp)


def oracle_step(inputs, setup, b: int):
    """One decode token of sequence b through the oracle's sharded block."""
    import oracle as O
    w = inputs["workload"]
    shards, ks, vs = setup
    x = np.asarray(inputs["x"][b:b + 1], dtype=np.float64)
    pos = inputs["pos"][b:b + 1]
    kb = [k[b:b + 1] for k in ks]
    vb = [v[b:b + 1] for v in vs]
    return O.block_tpN(shards, x, kb, vb, pos, 1, w, w.tp)


def cpu_baseline(inputs, budget_s: float = 20.0) -> dict:
    setup = oracle_setup(inputs)
    oracle_step(inputs, setup, 0)                        # warm
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_step(inputs, setup, n % inputs["workload"].batch)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 4096:
            break
    return {"value": n / el, "unit": "tokens/s", "cores": int(os.environ["OMP_NUM_THREADS"]), "kind": "oracle",
            "sample": f"{n} single-token decode steps (one sequence each, round-robin over the batch) of the "
                      f"float64 numpy oracle's sharded block, weights pre-sharded to float64 outside the timing"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    inputs = synth.make_inputs(w, with_head=False)
    setup = oracle_setup(inputs)
    for i in range(args.warmup):
        oracle_step(inputs, setup, i % w.batch)
    budget = 120.0
    t0 = time.perf_counter()
    n = 0
    for i in range(args.steps):
        oracle_step(inputs, setup, i % w.batch)
        n += 1
        if time.perf_counter() - t0 > budget:
            break
    el = time.perf_counter() - t0
    value = n / el
    cores = int(os.environ["OMP_NUM_THREADS"])
    sample = (f"each step is one decode token of one sequence (round-robin over the batch of {w.batch}) through the "
              f"float64 numpy oracle's sharded block; {n} of {args.steps} requested steps fit the {budget:.0f} s bound")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": n, "steps_requested": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / max(n, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "tp_logical_shards": w.tp, "batch": w.batch, "kv_len": w.kv_len,
                       "hidden": w.hidden, "heads": [w.n_heads, w.n_kv_heads], "head_dim": w.head_dim,
                       "ffn": w.ffn},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------


def run_ours(args, world, rank, local):
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import Model

    torch.cuda.set_device(local)
    w = synth.WORKLOADS[args.workload]
    inputs = synth.make_inputs(w, with_head=False)
    model = Model(inputs)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    # ---- device-resident timing: one step = one forward, replayed from a CUDA graph
    with torch.cuda.stream(stream):
        for _ in range(3):
            model.forward()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        model.forward()
    for _ in range(max(args.warmup, 3)):
        graph.replay()
    torch.cuda.synchronize()
    assert model.ws.status() == 0, "device status after warm-up"

    clocks = Clocks(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    t_ms = ev0.elapsed_time(ev1)
    t_ms = max_over_ranks(t_ms, world)
    ms_step = t_ms / args.steps
    tokens_step = w.tokens
    value = tokens_step * args.steps * world / (t_ms / 1e3)

    # ---- per-kernel durations: stage events around each launch over K' steps
    n_prof = min(args.steps, 2000)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(STAGES) + 1)] for _ in range(n_prof)]
    for row in evs:          # torch creates events lazily: record once so the raw handles exist
        for e in row:
            e.record(stream)
    stream.synchronize()
    with torch.cuda.stream(stream):
        for i in range(n_prof):
            tb.tp_profile_stages(model.plan, evs[i])
            model.forward(stream=stream)
        tb.tp_profile_stages(model.plan, None)
    torch.cuda.synchronize()
    stage_ms = {}
    for j, name in enumerate(STAGES):
        ts = [evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n_prof)]
        stage_ms[name] = statistics.mean(ts)
    sb = stage_bytes(w)
    peak, peak_kind = peaks()
    dom_ms = stage_ms[DOMINANT]
    achieved = sb[DOMINANT] / (dom_ms / 1e3) / 1e9
    step_gbs = step_bytes(w) / (ms_step / 1e3) / 1e9

    # ---- end to end through the public API: pinned host x -> device, forward, y -> pinned host
    x_host = torch.from_numpy(np.ascontiguousarray(inputs["x"])).pin_memory()
    y_host = torch.empty_like(x_host).pin_memory()
    pos_host = torch.from_numpy(inputs["pos"]).pin_memory()
    with torch.cuda.stream(stream):
        for _ in range(3):
            model.x.copy_(x_host, non_blocking=True)
            model.pos.copy_(pos_host, non_blocking=True)
            model.forward(stream=stream)
            y_host.copy_(model.y, non_blocking=True)
    stream.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            model.x.copy_(x_host, non_blocking=True)
            model.pos.copy_(pos_host, non_blocking=True)
            model.forward(stream=stream)
            y_host.copy_(model.y, non_blocking=True)
        e1.record(stream)
    e1.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = tokens_step * args.steps * world / (e2e_ms / 1e3)
    assert model.ws.status() == 0

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": w.name, "tp_logical_shards": w.tp, "batch": w.batch, "kv_len": w.kv_len,
                   "hidden": w.hidden, "heads": [w.n_heads, w.n_kv_heads], "head_dim": w.head_dim, "ffn": w.ffn,
                   "parallelism": f"{w.tp} logical TP shards per GPU; replicas across GPUs",
                   "l2": f"inputs larger than L2 ({step_bytes(w) / 1e6:.1f} MB read per step vs 129 MB L2)",
                   "launch": "CUDA graph of one forward, replayed per step"},
        "hbm": {"step_bytes": step_bytes(w), "step_gbs": step_gbs, "frac_of_peak": step_gbs / peak,
                "frac_of_8000": step_gbs / 8000.0, "peak_gbs": peak, "peak_kind": peak_kind},
        "stages_us": {k: 1e3 * v for k, v in stage_ms.items()},
        "roofline": {"bound": "hbm", "kernel": DOMINANT, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind, "algorithmic_bytes": sb[DOMINANT],
                     "traffic": kernel_traffic("gemv_swiglu")},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": x_host.numel() * 4 + pos_host.numel() * 4,
                "d2h_bytes_per_step": y_host.numel() * 4, "path": "tp_block_forward via the ctypes binding"},
        "gpu_launches": (9 if w.dtype == "bf16" else 5) * args.steps,
        "clocks": clk,
    }
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
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=["llama3_8b_decode_tp4"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
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
