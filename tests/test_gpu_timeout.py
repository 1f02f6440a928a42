"""A bounded device wait that runs out ("feat: multi-GPU tensor-parallel
runtime ...", Acceptance criteria: no silent wrong results).

Every wait of the one-launch decode step gives up after 1 s and records
TP_ERR_TIMEOUT. The test hook tp_debug_withhold_arrival makes each grid
barrier of a launch wait for one arrival more than the grid makes -- as if
one CTA were lost -- without faulting, trapping or spinning unbounded: the
launch must end (every CTA leaving through its abort path), report
TP_ERR_TIMEOUT in the workspace status word, and, after the workspace is
re-initialised, the next forward must match the oracle and the output of a
forward made before the failure, byte for byte.
"""
import time

import numpy as np
import pytest

import synth
from tests import _oracle_runs as R
from tests import _parity as P

pytestmark = pytest.mark.gpu


def test_a_withheld_barrier_arrival_times_out_and_the_workspace_recovers(gpu_lib):
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import Model
    w = synth.scaled(synth.WORKLOADS["llama3_8b_decode_tp4"], hidden=1024, n_heads=16, n_kv_heads=4, ffn=2048,
                     batch=3, kv_len=300, seed=41)
    inputs = synth.make_inputs(w, with_head=False)
    m = Model(inputs)
    y0 = m.forward().clone()
    torch.cuda.synchronize()
    assert m.ws.status() == 0

    tb.tp_debug_withhold_arrival(m.plan, True)
    try:
        t0 = time.monotonic()
        m.forward()
        torch.cuda.synchronize()                # the launch ends: its waits are bounded
        took = time.monotonic() - t0
    finally:
        tb.tp_debug_withhold_arrival(m.plan, False)
    assert m.ws.status() == tb.binding.TP_ERR_TIMEOUT
    assert 0.9 < took < 30.0, took              # about one wait limit per CTA, not a hang

    # the context is still usable; the re-initialised workspace gives the right answer again
    tb.tp_workspace_init(m.plan, m.ws.buf, m.ws.nbytes)
    y = m.forward()
    torch.cuda.synchronize()
    assert m.ws.status() == 0
    assert torch.equal(y, y0)
    ref, _ = R.dense_tpN(inputs, m.max_kv)
    got = y.double().cpu().numpy()
    assert np.isfinite(got).all()
    assert P.err(got, ref) <= 2e-2
