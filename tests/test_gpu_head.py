"""Logits of the final hidden state over the vocab-parallel head
(tp_lm_head_forward) against the oracle's RMSNorm(h) @ W.T over the unpadded
head, element by element (normwise max relative error), through the C ABI.

Tolerance 2e-2: the norm's operand x * gamma is rounded to bf16 for the
products, which accumulate in float32 (the bf16 configurations' bound)."""
import numpy as np
import pytest

import oracle as O
from tests import _parity as P
import synth

pytestmark = pytest.mark.gpu

TOL = 2e-2
QWEN = synth.WORKLOADS["qwen25_05b_decode_tp2"]
LLAMA = synth.WORKLOADS["llama3_8b_decode_tp4"]

CASES = {
    # the Qwen2.5-0.5B-shaped head: 151936 rows, 75968 per shard, no padding, one token
    "qwen_head_full_tp2": synth.scaled(QWEN, n_layers=1),
    # 1000 rows padded to 1024 over 4 shards (the last shard's 24 tail rows are padding), 3 tokens
    "padded_tp4_t3": synth.scaled(QWEN, hidden=448, n_heads=8, n_kv_heads=4, ffn=1024, tp=4, batch=3,
                                  n_layers=1, org_vocab=1000, seed=31),
    # 8 shards, 8 tokens, a stage range that crosses shard boundaries
    "tp8_t8": synth.scaled(LLAMA, hidden=1024, n_heads=16, n_kv_heads=8, ffn=2048, tp=8, batch=8, kv_len=4,
                           n_layers=1, org_vocab=5003, seed=32),
}


def _setup(w):
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import desc_of, to_device
    inputs = synth.make_inputs(w)
    head = inputs["lm_head"]
    plan = tb.tp_plan(desc_of(w), w.tp)
    info = tb.tp_plan_get_info(plan)
    V, Hd = head.shape
    R = info["vocab_rows_shard"]
    full = to_device(head)
    shards = [torch.empty(R, Hd, dtype=full.dtype, device="cuda") for _ in range(w.tp)]
    tb.tp_shard_param(plan, tb.TP_PARAM_VOCAB_PARALLEL, full, V, Hd, tb.TP_BF16, shards)
    x = to_device(inputs["x"])
    gamma = to_device(inputs["gamma_final"].astype(np.float32))
    return inputs, plan, shards, x, gamma


def _logits(plan, shards, x, gamma, T, V):
    import torch
    import megatron_tensor_block_gb300 as tb
    guard = 64
    buf = torch.full((T * V + guard,), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tp_lm_head_forward(plan, shards, gamma, x, T, buf, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    out = buf.cpu().numpy()
    assert np.isnan(out[T * V:]).all(), "wrote past the logits (a padding row leaked)"
    return out[:T * V].reshape(T, V).astype(np.float64)


@pytest.mark.parametrize("case", list(CASES))
def test_lm_head_matches_oracle(gpu_lib, case):
    w = CASES[case]
    inputs, plan, shards, x, gamma = _setup(w)
    V = w.org_vocab
    got = _logits(plan, shards, x, gamma, w.tokens, V)
    h = np.asarray(inputs["x"], dtype=np.float64)
    g = np.asarray(inputs["gamma_final"], dtype=np.float64)
    ref = O.lm_head_logits(h, g, O.to_f64(inputs["lm_head"]), w.eps)
    err = P.err(got, ref)
    assert err <= TOL, err
    # the last real row sits on the last shard: the cross-shard index of the gather
    assert P.err(got[:, V - 1:], ref[:, V - 1:]) <= TOL


def test_lm_head_is_deterministic(gpu_lib):
    w = CASES["padded_tp4_t3"]
    _, plan, shards, x, gamma = _setup(w)
    a = _logits(plan, shards, x, gamma, w.tokens, w.org_vocab)
    b = _logits(plan, shards, x, gamma, w.tokens, w.org_vocab)
    assert np.array_equal(a, b)


def test_lm_head_rejects_bad_arguments(gpu_lib):
    import torch
    import megatron_tensor_block_gb300 as tb
    w = CASES["padded_tp4_t3"]
    _, plan, shards, x, gamma = _setup(w)
    out = torch.empty(9 * w.org_vocab, dtype=torch.float32, device="cuda")
    with pytest.raises(tb.TpError) as e:
        tb.tp_lm_head_forward(plan, shards, gamma, x, 9, out)          # more than 8 tokens
    assert e.value.status == tb.binding.TP_ERR_SHAPE
    with pytest.raises(tb.TpError) as e:
        tb.tp_lm_head_forward(plan, shards[:-1] + [None], gamma, x, 1, out)
    assert e.value.status == tb.binding.TP_ERR_NULL
