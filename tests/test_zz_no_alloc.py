"""The allocation-free decode entry point.

Some callers cannot allocate device memory -- code running while a CUDA graph
is captured, plug-ins whose host program owns all device memory, loops that
cannot afford an allocation's synchronisation -- so the library offers a
decode forward whose scratch lives in a static device array it owns. These
tests call it through the C ABI and check that two calls in a row give the
same result as the workspace-based ``tp_block_forward``. This file is
collected last on purpose: it must pass after the other tests (the static
array keeps earlier calls' contents) as well as alone in a fresh process.
"""
import numpy as np
import pytest

import oracle as O
import synth

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}
CASES = {
    "llama3_8b_decode_tp4": synth.WORKLOADS["llama3_8b_decode_tp4"],
    "tiny_llama_fp32_tp2": synth.WORKLOADS["tiny_llama_fp32_tp2"],
    "llama_shape_small_tp2_b5": synth.scaled(synth.WORKLOADS["llama3_8b_decode_tp4"], hidden=1024, n_heads=16,
                                             n_kv_heads=4, ffn=2048, tp=2, batch=5, kv_len=300, seed=31),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_decode_matches_workspace_decode_twice(gpu_lib, name):
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import Model
    w = CASES[name]
    m = Model(synth.make_inputs(w, with_head=False))
    y_ref = m.forward().clone()                 # existing entry point, caller workspace
    torch.cuda.synchronize()
    ref = y_ref.double().cpu().numpy()
    kv = (m.caches[0].k, m.caches[0].v)
    for _ in range(2):
        y = torch.full_like(m.x, float("nan"))
        tb.tp_block_forward_noalloc(m.plan, m.layers[0].shards, kv, m.x, y, m.pos, w.batch)
        torch.cuda.synchronize()
        got = y.double().cpu().numpy()
        assert np.isfinite(got).all()
        assert O.relerr(got, ref) <= TOL[w.dtype]
        assert torch.equal(y, y_ref)            # same kernels, same order: identical bytes


def test_noalloc_rejects_plans_beyond_the_static_array(gpu_lib):
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import desc_of
    w = synth.WORKLOADS["llama3_8b_decode_tp4"]
    plan = tb.tp_plan(desc_of(w, max_kv=200000), w.tp)     # the split-KV partials alone exceed 16 MiB
    x = torch.zeros(w.batch, w.hidden, device="cuda")
    y = torch.empty_like(x)
    pos = torch.zeros(w.batch, dtype=torch.int32, device="cuda")
    with pytest.raises(tb.TpError) as e:
        tb.tp_block_forward_noalloc(plan, {}, ([0] * w.tp, [0] * w.tp), x, y, pos, w.batch)
    assert e.value.status == tb.binding.TP_ERR_CAPACITY
    assert "static array" in str(e.value)
