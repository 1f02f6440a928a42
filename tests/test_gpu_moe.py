"""MoE feed-forward block, expert slicing and expert parallelism (whole
experts per shard): the CUDA path against the oracle.

Routing and bucketing are integer results and must match bit for bit (the
top-k choice is made on the given float32 logits on both sides); the block
output must be within the bf16 tolerance 2e-2 (normwise max relative)."""
import numpy as np
import pytest

import oracle as O
from tests import _parity as P
import synth
from tests import _oracle_runs as R

pytestmark = pytest.mark.gpu
MOE = synth.WORKLOADS["moe_expert_slice_tp4"]


def _skewed(w, seed):
    """Inputs whose routing piles many tokens onto a few experts (several
    32-slot passes) and leaves others empty."""
    inp = synth.make_inputs(w)
    rng = np.random.Generator(np.random.PCG64(seed))
    lg = inp["router_logits"]
    heavy = rng.random(w.tokens) < 0.8
    lg[heavy, 3] += 6.0
    lg[:, w.n_experts - 1] -= 20.0          # never chosen
    return inp


# per-expert slot counts around the expert GEMM's 8-slot boxes and 32-slot passes
PASS_COUNTS = [1, 7, 8, 9, 15, 16, 17, 31, 32, 33, 48, 63, 64, 65, 0, 2]


def _counts(w, counts, seed):
    """Top-1 inputs whose routing gives expert e exactly counts[e] tokens (in a
    seeded random token order)."""
    assert w.top_k == 1 and len(counts) == w.n_experts and sum(counts) == w.tokens
    inp = synth.make_inputs(w)
    rng = np.random.Generator(np.random.PCG64(seed))
    owner = rng.permutation(np.repeat(np.arange(w.n_experts), counts))
    inp["router_logits"][np.arange(w.tokens), owner] += 20.0
    return inp


CASES = {
    "moe_expert_slice_tp4": lambda: synth.make_inputs(MOE),
    "moe_small_tp2_skewed_ragged": lambda: _skewed(
        synth.scaled(MOE, hidden=512, n_experts=16, top_k=2, expert_ffn=512, tp=2, batch=90, seed=41), 5),
    "moe_small_tp1_top1": lambda: synth.make_inputs(
        synth.scaled(MOE, hidden=256, n_experts=8, top_k=1, expert_ffn=256, tp=1, batch=9, seed=42)),
    # expert parallelism: the full-size shape with 16 whole experts per shard
    "moe_ep_tp4": lambda: synth.make_inputs(synth.scaled(MOE, expert_parallel=1, seed=43)),
    # expert parallelism with most tokens on expert 3 (shard 0) and the last expert never chosen
    "moe_ep_small_tp2_skewed_ragged": lambda: _skewed(
        synth.scaled(MOE, hidden=512, n_experts=16, top_k=2, expert_ffn=512, tp=2, batch=90, seed=44,
                     expert_parallel=1), 6),
    # expert slot counts at and around the 8-slot box and 32-slot pass boundaries (and an empty expert)
    "moe_pass_boundaries_tp2": lambda: _counts(
        synth.scaled(MOE, hidden=256, n_experts=16, top_k=1, expert_ffn=512, tp=2, batch=sum(PASS_COUNTS), seed=46),
        PASS_COUNTS, 7),
    "moe_ep_pass_boundaries_tp2": lambda: _counts(
        synth.scaled(MOE, hidden=256, n_experts=16, top_k=1, expert_ffn=256, tp=2, batch=sum(PASS_COUNTS), seed=47,
                     expert_parallel=1), PASS_COUNTS, 8),
    # expert parallelism over 8 shards, 2 experts each
    "moe_ep_tp8": lambda: synth.make_inputs(
        synth.scaled(MOE, hidden=512, n_experts=16, top_k=4, expert_ffn=256, tp=8, batch=33, seed=45,
                     expert_parallel=1)),
}


def _ws_int(m, offset, n):
    import torch
    return m.ws.buf[offset:offset + 4 * n].view(torch.int32).cpu().numpy()


@pytest.mark.parametrize("case", list(CASES))
def test_moe_block_matches_oracle(gpu_lib, case):
    import torch
    from megatron_tensor_block_gb300.runtime import Model
    inputs = CASES[case]()
    w = inputs["workload"]
    m = Model(inputs)
    y = m.forward()
    torch.cuda.synchronize()
    assert m.ws.status() == 0
    # routing and bucketing, bit-exact
    ids, wts = O.router_topk(inputs["router_logits"], w.top_k)
    offsets, perm = O.bucket_by_expert(ids, w.n_experts)
    n = w.tokens * w.top_k
    assert np.array_equal(_ws_int(m, m.info["moe_ids_offset"], n), ids.reshape(-1))
    assert np.array_equal(_ws_int(m, m.info["moe_bucket_offset"], w.n_experts + 1), offsets)
    assert np.array_equal(_ws_int(m, m.info["moe_perm_offset"], n), perm)
    # block output
    ref = R.moe_tpN(inputs)
    err = P.err(y.double().cpu().numpy(), ref)
    assert err <= 2e-2, err


@pytest.mark.parametrize("case", ["moe_small_tp2_skewed_ragged", "moe_ep_small_tp2_skewed_ragged"])
def test_moe_is_deterministic(gpu_lib, case):
    import torch
    from megatron_tensor_block_gb300.runtime import Model
    m = Model(CASES[case]())
    a = m.forward().clone()
    b = m.forward().clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("case", ["moe_expert_slice_tp4", "moe_small_tp2_skewed_ragged"])
def test_moe_shared_gamma_gives_identical_bytes(gpu_lib, case):
    # Every shard pointing at one gamma tensor: one normalised copy of the
    # slots' activations serves all shards; same values, so the same bytes.
    import torch
    from megatron_tensor_block_gb300.runtime import Model
    inputs = CASES[case]()
    m1 = Model(inputs)
    y1 = m1.forward().clone()
    m2 = Model(inputs, share_norm=True)
    y2 = m2.forward().clone()
    torch.cuda.synchronize()
    assert m1.ws.status() == 0 and m2.ws.status() == 0
    assert torch.equal(y1, y2)
