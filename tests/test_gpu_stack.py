"""Several decode blocks in one launch (tp_stack_decode) against the CPU
oracle's chained blocks, element by element (normwise max relative error),
through the C ABI, plus the K/V rows each layer appends.

Tolerance 2e-2 (bf16 storage, float32 accumulation), as for one block."""
import numpy as np
import pytest

import oracle as O
from tests import _parity as P
import synth
from tests import _oracle_runs as R

pytestmark = pytest.mark.gpu

TOL = 2e-2
LLAMA = synth.WORKLOADS["llama3_8b_decode_tp4"]
QWEN = synth.WORKLOADS["qwen25_05b_decode_tp2"]

CASES = {
    # head_dim 64, 7 query heads per KV head, biases, 3 layers, 301 keys:
    # three uneven key chunks, the new key in the last
    "qwen_shape_3_layers_kv300": synth.scaled(QWEN, hidden=448, n_heads=14, n_kv_heads=2, ffn=1024, batch=1,
                                              kv_len=300, n_layers=3, seed=21, org_vocab=0),
    # head_dim 128, tp 4, 3 sequences, 2 layers, 200 keys (4 chunks of 64)
    "llama_shape_tp4_b3_2_layers": synth.scaled(LLAMA, hidden=1024, n_heads=16, n_kv_heads=4, ffn=2048, batch=3,
                                                kv_len=200, n_layers=2, seed=22),
    # empty caches: one key per sequence, 8 sequences
    "qwen_shape_empty_cache_b8": synth.scaled(QWEN, hidden=448, n_heads=14, n_kv_heads=2, ffn=1024, batch=8,
                                              kv_len=0, n_layers=2, seed=23, org_vocab=0),
    # tp 1: the unsharded block, 2 layers, keys exactly one tile (128)
    "qwen_shape_tp1": synth.scaled(QWEN, hidden=256, n_heads=4, n_kv_heads=1, ffn=512, tp=1, batch=2,
                                   kv_len=127, n_layers=2, seed=24, org_vocab=0),
    # tp 8, one KV head and two query heads per shard, head_dim 128, a full batch of 8, 129 keys in chunks of 48, 48, 33
    "llama_shape_tp8_b8": synth.scaled(LLAMA, hidden=1024, n_heads=16, n_kv_heads=8, ffn=2048, tp=8, batch=8,
                                       kv_len=128, n_layers=1, seed=25),
}


def _model(inputs):
    from megatron_tensor_block_gb300.runtime import Model
    return Model(inputs)


def _run_stack(m):
    import torch
    y = m.forward_stack()
    torch.cuda.synchronize()
    assert m.ws.status() == 0
    return y.double().cpu().numpy()


@pytest.mark.parametrize("case", list(CASES))
def test_stack_matches_oracle(gpu_lib, case):
    w = CASES[case]
    inputs = synth.make_inputs(w)
    m = _model(inputs)
    y = _run_stack(m)
    ref, caches = R.dense_tpN(inputs, m.max_kv)
    err = P.err(y, ref)
    assert err <= TOL, err
    pos = inputs["pos"]
    for layer in range(w.n_layers):
        k, v = m.caches[layer].full()
        kk = np.stack([k[b, :, pos[b]].double().cpu().numpy() for b in range(len(pos))])
        vv = np.stack([v[b, :, pos[b]].double().cpu().numpy() for b in range(len(pos))])
        rk = np.stack([caches[layer][0][b, :, pos[b]] for b in range(len(pos))])
        rv = np.stack([caches[layer][1][b, :, pos[b]] for b in range(len(pos))])
        assert P.err(kk, rk) <= TOL and P.err(vv, rv) <= TOL, layer
        # nothing else in the cache moved
        old = R.full_cache(inputs["k_cache"][layer], m.max_kv)
        kn = k.double().cpu().numpy()
        for b in range(len(pos)):
            kn[b, :, pos[b]] = old[b, :, pos[b]]
        assert np.array_equal(kn, old), layer


def test_stack_qwen25_24_layers_full_size(gpu_lib):
    inputs = synth.make_inputs(QWEN, with_head=False)
    m = _model(inputs)
    y = _run_stack(m)
    ref, _ = R.dense_tpN(inputs, m.max_kv)
    err = P.err(y, ref)
    assert err <= TOL, err


def test_stack_agrees_with_per_layer_launches(gpu_lib):
    import torch
    inputs = synth.make_inputs(CASES["llama_shape_tp4_b3_2_layers"])
    m = _model(inputs)
    y_stack = m.forward_stack().clone()
    y_layers = m.forward().clone()
    torch.cuda.synchronize()
    a, b = y_stack.double().cpu().numpy(), y_layers.double().cpu().numpy()
    assert P.err(a, b) <= TOL


def test_stack_is_deterministic_across_launches(gpu_lib):
    import torch
    inputs = synth.make_inputs(CASES["qwen_shape_3_layers_kv300"])
    m = _model(inputs)
    ys = [m.forward_stack().clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert m.ws.status() == 0
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[1], ys[2])


def test_stack_in_cuda_graph(gpu_lib):
    import torch
    inputs = synth.make_inputs(CASES["qwen_shape_3_layers_kv300"])
    m = _model(inputs)
    ref = m.forward_stack().clone()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(4):
            m.forward_stack(stream=s)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert m.ws.status() == 0
    assert torch.equal(m.y, ref)


def test_stack_position_past_capacity_is_reported(gpu_lib):
    import torch
    import megatron_tensor_block_gb300 as tb
    inputs = synth.make_inputs(CASES["qwen_shape_tp1"])
    m = _model(inputs)
    k_before = [c.k[0].clone() for c in m.caches]
    m.pos.fill_(m.max_kv)
    m.forward_stack()
    torch.cuda.synchronize()
    assert m.ws.status() == tb.binding.TP_ERR_CAPACITY
    for c, kb in zip(m.caches, k_before):
        assert torch.equal(kb, c.k[0])


def test_stack_shares_a_workspace_with_per_layer_launches(gpu_lib):
    import torch
    inputs = synth.make_inputs(CASES["qwen_shape_3_layers_kv300"])
    m = _model(inputs)
    a = m.forward_stack().clone()
    b = m.forward().clone()                  # the other mode writes the shared data region
    c = m.forward_stack().clone()
    torch.cuda.synchronize()
    assert m.ws.status() == 0
    assert torch.equal(a, c)
    assert P.err(a.double().cpu().numpy(), b.double().cpu().numpy()) <= TOL


def test_stack_many_launches_keep_their_epochs(gpu_lib):
    import torch
    inputs = synth.make_inputs(CASES["qwen_shape_tp1"])
    m = _model(inputs)
    ref = m.forward_stack().clone()
    for _ in range(300):                     # the launch counter advances once per launch
        m.forward_stack()
    torch.cuda.synchronize()
    assert m.ws.status() == 0
    assert torch.equal(m.y, ref)


RAGGED = {
    # per-sequence positions (ragged KV lengths), each attending over its own keys 0..pos[b]
    "llama_shape_tp4_b3_2_layers": [200, 5, 130],
    "llama_shape_tp8_b8": [128, 0, 64, 127, 1, 99, 3, 50],
}


@pytest.mark.parametrize("case", list(RAGGED))
def test_stack_ragged_positions_match_oracle(gpu_lib, case):
    w = CASES[case]
    inputs = synth.make_inputs(w)
    inputs["pos"] = np.array(RAGGED[case], dtype=np.int32)
    m = _model(inputs)
    y = _run_stack(m)
    ref, caches = R.dense_tpN(inputs, m.max_kv)
    assert P.err(y, ref) <= TOL
    k, _ = m.caches[0].full()
    pos = inputs["pos"]
    kk = np.stack([k[b, :, pos[b]].double().cpu().numpy() for b in range(len(pos))])
    rk = np.stack([caches[0][0][b, :, pos[b]] for b in range(len(pos))])
    assert P.err(kk, rk) <= TOL
