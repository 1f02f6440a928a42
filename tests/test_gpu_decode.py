"""Decode parity: the CUDA block against the CPU oracle on the same seeded
inputs, element by element (normwise max relative error), through the C ABI.

Tolerances: 1e-5 for fp32 storage, 2e-2 for bf16 storage with fp32
accumulation (the workload text's bounds)."""
import numpy as np
import pytest

import oracle as O
from tests import _parity as P
import synth
from tests import _oracle_runs as R

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}
LLAMA = synth.WORKLOADS["llama3_8b_decode_tp4"]
QWEN = synth.WORKLOADS["qwen25_05b_decode_tp2"]
TINY = synth.WORKLOADS["tiny_llama_fp32_tp2"]

CASES = {
    "tiny_fp32_tp2": TINY,
    # several tiles per shard, a ragged last KV chunk (301 keys), 3 of 8 sequences
    "llama_shape_small_tp4_b3": synth.scaled(LLAMA, hidden=1024, n_heads=16, n_kv_heads=4, ffn=2048,
                                             batch=3, kv_len=300, seed=11),
    # head_dim 64, GQA group 7 (Qwen-like), biases, 8 sequences, empty cache
    "qwen_shape_small_tp2_empty_cache": synth.scaled(QWEN, hidden=448, n_heads=14, n_kv_heads=2,
                                                     ffn=1024, batch=8, kv_len=0, n_layers=1, seed=12,
                                                     org_vocab=0),
    # tp=8, one KV head per shard, one sequence, KV exactly one chunk
    "llama_shape_tp8_b1": synth.scaled(LLAMA, hidden=1024, n_heads=16, n_kv_heads=8, ffn=2048, tp=8,
                                       batch=1, kv_len=255, seed=13),
    # tp=1 degenerates to the unsharded block
    "llama_shape_tp1": synth.scaled(LLAMA, hidden=512, n_heads=8, n_kv_heads=2, ffn=1024, tp=1,
                                    batch=2, kv_len=40, seed=14),
    # 160 QKV tiles, more than there are SMs: two per CTA on the first 80, so the key split gives the
    # other CTAs the larger share; 8 query heads per KV head, 2 sequences, ragged last key block
    "qkv_tiles_exceed_sms_tp4": synth.scaled(LLAMA, hidden=1024, n_heads=64, n_kv_heads=8, ffn=1024, tp=4,
                                             batch=2, kv_len=100, seed=15),
}


def _run(gpu_lib, inputs, **kw):
    import torch
    from megatron_tensor_block_gb300.runtime import Model
    m = Model(inputs, **kw)
    y = m.forward()
    torch.cuda.synchronize()
    assert m.ws.status() == 0
    return m, y.double().cpu().numpy()


def _cache_at_new_positions(m, layer, inputs):
    k, v = m.caches[layer].full()
    pos = inputs["pos"]
    kk = np.stack([k[b, :, pos[b]].double().cpu().numpy() for b in range(len(pos))])
    vv = np.stack([v[b, :, pos[b]].double().cpu().numpy() for b in range(len(pos))])
    return kk, vv


@pytest.mark.parametrize("case", list(CASES))
def test_decode_block_matches_oracle(gpu_lib, case):
    w = CASES[case]
    inputs = synth.make_inputs(w)
    m, y = _run(gpu_lib, inputs)
    ref, caches = R.dense_tpN(inputs, m.max_kv)
    err = P.err(y, ref)
    assert err <= TOL[w.dtype], err
    # the new K (rotated) and V rows written to each shard's cache
    kk, vv = _cache_at_new_positions(m, 0, inputs)
    pos = inputs["pos"]
    rk = np.stack([caches[0][0][b, :, pos[b]] for b in range(len(pos))])
    rv = np.stack([caches[0][1][b, :, pos[b]] for b in range(len(pos))])
    assert P.err(kk, rk) <= TOL[w.dtype] and P.err(vv, rv) <= TOL[w.dtype]
    # and nothing else in the caches moved
    k, v = m.caches[0].full()
    old = R.full_cache(inputs["k_cache"][0], m.max_kv)
    kn = k.double().cpu().numpy()
    for b in range(len(pos)):
        kn[b, :, pos[b]] = old[b, :, pos[b]]
    assert np.array_equal(kn, old)


def test_decode_tpN_equals_unsharded_block(gpu_lib):
    w = CASES["llama_shape_small_tp4_b3"]
    inputs = synth.make_inputs(w)
    m, y = _run(gpu_lib, inputs)
    assert P.err(y, R.dense_tp1(inputs, m.max_kv)) <= TOL[w.dtype]


def test_decode_llama3_8b_full_size(gpu_lib):
    inputs = synth.make_inputs(LLAMA)
    m, y = _run(gpu_lib, inputs)
    ref, _ = R.dense_tpN(inputs, m.max_kv)
    err = P.err(y, ref)
    assert err <= TOL["bf16"], err


def test_decode_qwen25_24_layers_full_size(gpu_lib):
    inputs = synth.make_inputs(QWEN, with_head=False)
    m, y = _run(gpu_lib, inputs)
    ref, _ = R.dense_tpN(inputs, m.max_kv)
    err = P.err(y, ref)
    assert err <= TOL["bf16"], err


def test_decode_is_deterministic(gpu_lib):
    import torch
    from megatron_tensor_block_gb300.runtime import Model
    inputs = synth.make_inputs(CASES["llama_shape_small_tp4_b3"])
    m = Model(inputs)
    y1 = m.forward().clone()
    y2 = m.forward().clone()
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_decode_many_launches_keep_their_epochs(gpu_lib):
    # split down tiles are combined from (value, epoch) pieces: every launch
    # has its own epoch, so a piece left by an earlier launch never counts
    import torch
    from megatron_tensor_block_gb300.runtime import Model
    inputs = synth.make_inputs(CASES["llama_shape_small_tp4_b3"])
    m = Model(inputs)
    ref = m.forward().clone()
    for _ in range(200):
        m.forward()
    torch.cuda.synchronize()
    assert m.ws.status() == 0
    assert torch.equal(m.y, ref)


def test_decode_position_past_capacity_is_reported(gpu_lib):
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import Model
    inputs = synth.make_inputs(CASES["llama_shape_tp1"])
    m = Model(inputs)
    k_before = m.caches[0].k[0].clone()
    m.pos.fill_(m.max_kv)          # one past the last slot: the kernels skip the write and flag it
    m.forward()
    torch.cuda.synchronize()
    assert m.ws.status() == tb.binding.TP_ERR_CAPACITY
    assert torch.equal(k_before, m.caches[0].k[0])


def test_decode_ragged_positions_match_oracle(gpu_lib):
    # every sequence at its own position: ragged KV lengths (300, 0 and 151 cached keys before the step)
    w = CASES["llama_shape_small_tp4_b3"]
    inputs = synth.make_inputs(w)
    inputs["pos"] = np.array([300, 0, 151], dtype=np.int32)
    m, y = _run(gpu_lib, inputs)
    ref, _ = R.dense_tpN(inputs, m.max_kv)
    assert P.err(y, ref) <= TOL[w.dtype]
