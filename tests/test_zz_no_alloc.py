"""The allocation-free decode entry point.

Some callers cannot allocate device memory -- code running while a CUDA graph
is captured, plug-ins whose host program owns all device memory, loops that
cannot afford an allocation's synchronisation -- so the library offers a
decode forward whose scratch lives in a static device array it owns. These
tests call it through the C ABI. Each case makes two calls in a row on
DIFFERENT inputs (new x, new per-sequence positions): a piece of the first
call left in the shared array must not count for the second. Each call's
output is compared with the oracle and, byte for byte, with the
workspace-based ``tp_block_forward`` on the same inputs, and the array's
status word is read back. This file is collected last on purpose: it must
pass after the other tests (the static array keeps earlier calls' contents)
as well as alone in a fresh process.
"""
import numpy as np
import pytest

import oracle as O
from tests import _parity as P
import synth
from tests import _oracle_runs as R

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}
LLAMA = synth.WORKLOADS["llama3_8b_decode_tp4"]
CASES = {
    "llama3_8b_decode_tp4": LLAMA,
    "tiny_llama_fp32_tp2": synth.WORKLOADS["tiny_llama_fp32_tp2"],
    "llama_shape_small_tp2_b5": synth.scaled(LLAMA, hidden=1024, n_heads=16, n_kv_heads=4, ffn=2048, tp=2,
                                             batch=5, kv_len=300, seed=31),
}


def _second_inputs(inputs, seed):
    """Same weights and caches; a new x and new positions inside the cached
    range (each sequence attends over a shorter, ragged prefix)."""
    w = inputs["workload"]
    rng = np.random.default_rng(seed)
    out = dict(inputs)
    x = rng.standard_normal(inputs["x"].shape).astype(np.float32)
    out["x"] = x
    L = max(w.kv_len, 1)
    out["pos"] = rng.integers(0, L, size=w.batch).astype(np.int32) if w.kv_len > 0 else inputs["pos"].copy()
    return out


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_decode_two_calls_on_different_inputs(gpu_lib, name):
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import Model
    w = CASES[name]
    first = synth.make_inputs(w, with_head=False)
    m = Model(first)
    kv = (m.caches[0].k, m.caches[0].v)
    for i, inputs in enumerate((first, _second_inputs(first, seed=900 + len(name)))):
        x = torch.from_numpy(inputs["x"]).to("cuda")
        pos = torch.from_numpy(inputs["pos"]).to("cuda")
        y_ws = torch.empty_like(x)
        m.pos.copy_(pos)
        m.forward(x=x, y=y_ws)                  # existing entry point, caller workspace
        y = torch.full_like(x, float("nan"))
        tb.tp_block_forward_noalloc(m.plan, m.layers[0].shards, kv, x, y, pos, w.batch)
        assert tb.tp_noalloc_status() == 0
        torch.cuda.synchronize()
        assert m.ws.status() == 0
        assert torch.equal(y, y_ws), f"call {i}: differs from tp_block_forward on the same inputs"
        ref, _ = R.dense_tpN(inputs, m.max_kv)
        got = y.double().cpu().numpy()
        assert np.isfinite(got).all()
        err = P.err(got, ref)
        assert err <= TOL[w.dtype], f"call {i}: relative error {err}"


def test_noalloc_decode_on_a_prefill_sized_plan(gpu_lib):
    # a plan sized for 8192-token prefill still decodes through the static
    # array: the decode footprint does not depend on max_tokens
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import Model, desc_of
    w = synth.scaled(LLAMA, hidden=1024, n_heads=16, n_kv_heads=4, ffn=2048, tp=4, batch=3, kv_len=100, seed=33)
    inputs = synth.make_inputs(w, with_head=False)
    m = Model(inputs)
    big = tb.tp_plan(desc_of(w, max_kv=m.max_kv, max_tokens=8192), w.tp)
    assert tb.tp_plan_get_info(big)["noalloc_scratch_bytes"] == m.info["noalloc_scratch_bytes"]
    y_ws = m.forward().clone()
    y = torch.full_like(m.x, float("nan"))
    tb.tp_block_forward_noalloc(big, m.layers[0].shards, (m.caches[0].k, m.caches[0].v), m.x, y, m.pos, w.batch)
    assert tb.tp_noalloc_status() == 0
    torch.cuda.synchronize()
    assert torch.equal(y, y_ws)


def test_noalloc_status_reports_a_position_past_capacity(gpu_lib):
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import Model
    w = CASES["llama_shape_small_tp2_b5"]
    m = Model(synth.make_inputs(w, with_head=False))
    k_before = m.caches[0].k[0].clone()
    pos = torch.full_like(m.pos, m.max_kv)      # one past the last slot: skipped and flagged
    y = torch.empty_like(m.x)
    tb.tp_block_forward_noalloc(m.plan, m.layers[0].shards, (m.caches[0].k, m.caches[0].v), m.x, y, pos,
                                w.batch)
    assert tb.tp_noalloc_status() == tb.binding.TP_ERR_CAPACITY
    assert torch.equal(k_before, m.caches[0].k[0])
    # the next call clears the status word
    tb.tp_block_forward_noalloc(m.plan, m.layers[0].shards, (m.caches[0].k, m.caches[0].v), m.x, y, m.pos,
                                w.batch)
    assert tb.tp_noalloc_status() == 0


def test_noalloc_rejects_plans_beyond_the_static_array(gpu_lib):
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import desc_of
    plan = tb.tp_plan(desc_of(LLAMA, max_kv=200000), LLAMA.tp)   # the split-KV partials alone exceed 16 MiB
    assert tb.tp_plan_get_info(plan)["noalloc_scratch_bytes"] > tb.binding.TP_NOALLOC_SCRATCH_BYTES
    x = torch.zeros(LLAMA.batch, LLAMA.hidden, device="cuda")
    y = torch.empty_like(x)
    pos = torch.zeros(LLAMA.batch, dtype=torch.int32, device="cuda")
    with pytest.raises(tb.TpError) as e:
        tb.tp_block_forward_noalloc(plan, {}, ([0] * LLAMA.tp, [0] * LLAMA.tp), x, y, pos, LLAMA.batch)
    assert e.value.status == tb.binding.TP_ERR_CAPACITY
    assert "static array" in str(e.value)
