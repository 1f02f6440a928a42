"""Host-side logic of bench.py's multi-rank mode on CPU (gloo, world size 2):
every rank runs its own replica; the timed region is bracketed by barriers and
the slowest rank's time is reported; only rank 0 prints."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import json, os, sys
sys.path.insert(0, os.environ["ROOT"])
import bench
world, rank, local = bench.dist_setup()
bench.barrier(world)
t = bench.max_over_ranks(1.0 + rank * 2.5, world)
print(json.dumps({"rank": rank, "world": world, "max": t}), flush=True)
class A: pass
a = A(); a.workload = "moe_expert_slice_tp4"; a.warmup = 0; a.steps = 1; a.gpus = world
if rank != 0:
    bench.run_reference(a, world, rank)      # ranks other than 0 return without work or output
import torch.distributed as dist
dist.destroy_process_group()
"""


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_two_rank_barrier_and_max_over_ranks():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, ROOT=ROOT, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", _CHILD], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append([json.loads(l) for l in out.splitlines() if l.startswith("{")])
    for r, lines in enumerate(outs):
        assert len(lines) == 1, lines              # rank 1 printed nothing from run_reference
        assert lines[0]["rank"] == r and lines[0]["world"] == 2
        assert lines[0]["max"] == pytest.approx(3.5)


def test_workload_table_covers_every_measured_workload():
    sys.path.insert(0, ROOT)
    import bench
    import synth
    for name, kind in bench.WORKLOAD_KIND.items():
        assert name in synth.WORKLOADS
        assert kind in bench.STAGES and kind in bench.METRICS and bench.DOMINANT[kind] in bench.STAGES[kind]
    # the decode line's metric names its two figures: tokens/s and HBM bandwidth against the nominal peak
    assert bench.METRICS["decode"] == "TP-block decode tokens/s + HBM GB/s (% of ~8 TB/s peak) on 1 GB300"
    w = synth.WORKLOADS["llama3_8b_prefill_tp8"]
    fl = bench.prefill_flops(w)
    assert abs(sum(fl.values()) / 1e12 - 3.711) < 0.01       # linear 3.573 T + causal attention 0.137 T
    assert abs(bench.step_bytes(synth.WORKLOADS["llama3_8b_decode_tp4"]) / 1e6 - 503.3) < 0.1
