"""Prefill parity: the tensor-core block (tcgen05 projections, causal
attention) against the CPU oracle on the same seeded inputs, through the C
ABI. Small cases compare every output element and every cache row written;
the full Llama-3-8B-shaped tp=8 prefill (4 x 2048 tokens) compares sampled
rows, which the oracle forms one by one from what they depend on.

Tolerance: normwise max relative error 2e-2 (bf16 storage, fp32
accumulation)."""
import numpy as np
import pytest

import oracle as O
from tests import _parity as P
import synth
from tests import _oracle_runs as R

pytestmark = pytest.mark.gpu

TOL = 2e-2
PRE = synth.WORKLOADS["llama3_8b_prefill_tp8"]

CASES = {
    # ragged everything: 2 x 130 tokens (three 128-row tiles, the last with 4
    # rows; query blocks of 64 with a 2-row tail), a 70-token cached prefix
    "llama_shape_tp2_ragged_prefix": synth.scaled(PRE, hidden=512, n_heads=8, n_kv_heads=2, ffn=1024, tp=2,
                                                  batch=2, tokens_per_seq=130, kv_len=70, seed=21),
    # head_dim 64, GQA group 7, q/k/v biases, 576 fused QKV rows (a ragged
    # 256-column tile), F' = 576 (a ragged gate/up tile), H = 896 (7 tiles)
    "qwen_shape_tp2_bias": synth.scaled(PRE, hidden=896, n_heads=14, n_kv_heads=2, head_dim=64, ffn=1152,
                                        tp=2, batch=1, tokens_per_seq=200, kv_len=0, qkv_bias=True,
                                        rope_theta=1e6, eps=1e-6, seed=22),
    # tp=8 with one KV head per shard, three sequences of one query block
    "llama_shape_tp8_b3": synth.scaled(PRE, hidden=1024, n_heads=16, n_kv_heads=8, ffn=2048, tp=8,
                                       batch=3, tokens_per_seq=64, kv_len=0, seed=23),
    # tp=1 is the unsharded block; a single token per sequence
    "llama_shape_tp1_s1": synth.scaled(PRE, hidden=512, n_heads=8, n_kv_heads=2, ffn=1024, tp=1,
                                       batch=2, tokens_per_seq=1, kv_len=33, seed=24),
}


def _run(inputs, **kw):
    import torch
    from megatron_tensor_block_gb300.runtime import Model
    m = Model(inputs, **kw)
    y = m.forward()
    torch.cuda.synchronize()
    assert m.ws.status() == 0
    return m, y.double().cpu().numpy()


@pytest.mark.parametrize("case", list(CASES))
def test_prefill_block_matches_oracle(gpu_lib, case):
    w = CASES[case]
    inputs = synth.make_inputs(w, with_head=False)
    m, y = _run(inputs)
    ref, caches = R.dense_tpN(inputs, m.max_kv)
    err = P.err(y, ref)
    assert err <= TOL, err
    # every cache row the block wrote (rotated K, V), and nothing else moved
    k, v = (t.double().cpu().numpy() for t in m.caches[0].full())
    S, pos = w.tokens_per_seq, inputs["pos"]
    for b in range(w.batch):
        new = slice(int(pos[b]), int(pos[b]) + S)
        assert P.err(k[b, :, new], caches[0][0][b, :, new]) <= TOL
        assert P.err(v[b, :, new], caches[0][1][b, :, new]) <= TOL
    old_k = R.full_cache(inputs["k_cache"][0], m.max_kv)
    for b in range(w.batch):
        k[b, :, int(pos[b]):int(pos[b]) + S] = old_k[b, :, int(pos[b]):int(pos[b]) + S]
    assert np.array_equal(k, old_k)


def test_prefill_shared_gamma_gives_identical_bytes(gpu_lib):
    # One normalised copy for all shards (shared gamma pointer) or one per
    # shard: the same values, so the same bytes.
    import torch
    w = CASES["llama_shape_tp2_ragged_prefix"]
    inputs = synth.make_inputs(w, with_head=False)
    m1, _ = _run(inputs)
    m2, _ = _run(inputs, share_norm=True)
    assert torch.equal(m1.y, m2.y)


def test_prefill_is_deterministic(gpu_lib):
    import torch
    from megatron_tensor_block_gb300.runtime import Model
    w = CASES["llama_shape_tp8_b3"]
    m = Model(synth.make_inputs(w, with_head=False))
    y1 = m.forward().clone()
    y2 = m.forward().clone()            # the caches now hold the same rows again
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_prefill_past_capacity_sets_status(gpu_lib):
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import Model
    w = synth.scaled(PRE, hidden=512, n_heads=8, n_kv_heads=2, ffn=1024, tp=2, batch=1, tokens_per_seq=64,
                     kv_len=40, seed=25)
    m = Model(synth.make_inputs(w, with_head=False), max_kv=80)     # positions 40..103 > 79
    m.forward()
    torch.cuda.synchronize()
    assert m.ws.status() == tb.binding.TP_ERR_CAPACITY


def test_prefill_rejects_fp32_plans(gpu_lib):
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import Model
    w = synth.scaled(synth.WORKLOADS["tiny_llama_fp32_tp2"], tokens_per_seq=4, kv_len=4, org_vocab=0)
    m = Model(synth.make_inputs(w, with_head=False))
    with pytest.raises(tb.TpError) as e:
        tb.tp_block_forward(m.plan, m.layers[0].shards, (m.caches[0].k, m.caches[0].v), m.x, m.y, m.pos,
                            w.batch, 4, tb.TP_MODE_PREFILL, None, m.ws.buf, m.ws.nbytes)
    assert e.value.status == tb.binding.TP_ERR_UNSUPPORTED
    torch.cuda.synchronize()


def test_full_llama3_8b_prefill_tp8_sampled_rows(gpu_lib):
    # The configuration the prefill throughput is measured on, in the same
    # launch configuration (shared gamma copies); rows at tile and query-block
    # edges of the first and last sequences.
    w = PRE
    inputs = synth.make_inputs(w, with_head=False)
    m, y = _run(inputs, share_norm=True)
    S = w.tokens_per_seq
    # every sequence's last token, tile and query-block edges, and 64 seeded-random rows
    rows = [b * S + S - 1 for b in range(w.batch)] + [0, 1, 63, 64, 127, 128, 3 * S, 3 * S + 129, 4 * S - 2]
    rows += np.random.Generator(np.random.PCG64(2024)).integers(0, w.tokens, 64).tolist()
    L = O.layer_f64(inputs["layers"][0])
    shards = O.shard_layer(L, w, w.tp)
    ks = O.shard_kv_cache(R.full_cache(inputs["k_cache"][0], m.max_kv), w.tp)
    vs = O.shard_kv_cache(R.full_cache(inputs["v_cache"][0], m.max_kv), w.tp)
    ref, order = O.block_rows_tpN(shards, np.asarray(inputs["x"], dtype=np.float64), ks, vs, inputs["pos"], S, w,
                                  w.tp, rows)
    err = P.err(y[order], ref)
    assert err <= TOL, err
    assert np.isfinite(y).all()
