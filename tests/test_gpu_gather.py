"""Sharding and gathering through the C ABI: bit-exact against the oracle's
sharding rules and gather, on the workloads' parameters.

Checks follow the gather-on-read PR's Verification section: row-parallel
weights gather back equal to the unsharded tensor, fused column weights equal
as a row multiset (and exactly the rank-grouped order), the lm_head has the
full vocabulary with row vocab-5 equal to the reference row, and the shards
are unchanged by the gather."""
import numpy as np
import pytest

import oracle as O
import synth

pytestmark = pytest.mark.gpu


def _np(t):
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _dtype_code(a):
    import megatron_tensor_block_gb300 as tb
    return tb.TP_BF16 if a.dtype == np.uint16 else tb.TP_F32


def _plan(w):
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import desc_of
    return tb.tp_plan(desc_of(w), w.tp)


@pytest.mark.parametrize("name", ["tiny_llama_fp32_tp2", "qwen25_05b_decode_tp2"])
def test_lm_head_vocab_parallel_roundtrip(gpu_lib, name):
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import to_device
    w = synth.WORKLOADS[name]
    head = synth.make_inputs(synth.scaled(w, n_layers=1))["lm_head"]
    plan = _plan(w)
    info = tb.tp_plan_get_info(plan)
    V, Hd = head.shape
    R = info["vocab_rows_shard"]
    full = to_device(head)
    shards = [torch.empty(R, Hd, dtype=full.dtype, device="cuda") for _ in range(w.tp)]
    dt = _dtype_code(head)
    tb.tp_shard_param(plan, tb.TP_PARAM_VOCAB_PARALLEL, full, V, Hd, dt, shards)
    # shard contents: the oracle's rule, padding rows at the tail of the last shard (zeros here)
    ref = O.shard_vocab(head, w.tp, fill=0)
    for r in range(w.tp):
        assert np.array_equal(_np(shards[r]), ref[r])
    before = [s.clone() for s in shards]
    out = torch.full((V, Hd), float("nan"), dtype=full.dtype, device="cuda")
    tb.tp_gather_param(plan, tb.TP_PARAM_VOCAB_PARALLEL, shards, R, Hd, dt, out)
    torch.cuda.synchronize()
    got = _np(out)
    assert got.shape == (w.org_vocab, Hd)
    assert np.array_equal(got, head)
    assert np.array_equal(got[V - 5], head[V - 5])
    assert np.array_equal(got, O.gather_param([_np(s) for s in shards], O.VOCAB_PARALLEL, org_vocab=V))
    assert all(torch.equal(a, b) for a, b in zip(shards, before))


def test_fused_and_row_parallel_gathers_qwen_layer(gpu_lib):
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import Model
    w = synth.scaled(synth.WORKLOADS["qwen25_05b_decode_tp2"], n_layers=1, org_vocab=0)
    inputs = synth.make_inputs(w)
    m = Model(inputs, keep_full=True)
    L = inputs["layers"][0]
    sh = m.layers[0].shards
    info = m.info
    H, N = w.hidden, w.tp
    oshards = O.shard_layer({k: v for k, v in L.items()}, w, N)

    def gather(kind, tensors, rows, cols):
        out = torch.empty(rows * (N if kind != tb.TP_PARAM_ROWWISE else 1),
                          cols * (N if kind == tb.TP_PARAM_ROWWISE else 1), dtype=tensors[0].dtype, device="cuda")
        tb.tp_gather_param(m.plan, kind, tensors, rows, cols, tb.TP_BF16 if tensors[0].dtype == torch.bfloat16
                           else tb.TP_F32, out)
        return _np(out)

    # the device shards are the oracle's shards, bit for bit
    for r in range(N):
        assert np.array_equal(_np(sh["wqkv"][r]).reshape(-1, H), oshards[r]["wqkv"])
        assert np.array_equal(_np(sh["wo"][r]).reshape(H, -1), oshards[r]["wo"])
        assert np.array_equal(_np(sh["wgu"][r]).reshape(-1, H), oshards[r]["wgu"])
        assert np.array_equal(_np(sh["wd"][r]).reshape(H, -1), oshards[r]["wd"])
        assert np.array_equal(_np(sh["bqkv"][r]), oshards[r]["bqkv"])
    qkv_rows = info["qkv_rows"]
    g = gather(tb.TP_PARAM_FUSED_QKV, [t.view(qkv_rows, H) for t in sh["wqkv"]], qkv_rows, H)
    full = np.concatenate([L["wq"], L["wk"], L["wv"]])
    assert sorted(map(bytes, g)) == sorted(map(bytes, full))                      # row multiset
    perm = O.fused_gather_permutation([w.n_heads * w.head_dim, w.n_kv_heads * w.head_dim,
                                       w.n_kv_heads * w.head_dim], N)
    assert np.array_equal(g, full[perm])                                           # rank-grouped order
    Fs = info["ffn_shard"]
    g = gather(tb.TP_PARAM_FUSED_GATE_UP, [t.view(2 * Fs, H) for t in sh["wgu"]], 2 * Fs, H)
    assert np.array_equal(g, np.concatenate([L["w_gate"], L["w_up"]])[O.fused_gather_permutation([w.ffn, w.ffn], N)])
    # row-parallel weights gather back to the tp=1 tensors exactly
    hq = info["hq_shard"] * w.head_dim
    assert np.array_equal(gather(tb.TP_PARAM_ROWWISE, [t.view(H, hq) for t in sh["wo"]], H, hq), L["wo"])
    assert np.array_equal(gather(tb.TP_PARAM_ROWWISE, [t.view(H, Fs) for t in sh["wd"]], H, Fs), L["w_down"])
    # replicated: the norm weight
    assert np.array_equal(gather(tb.TP_PARAM_REPLICATED, [t.view(1, H) for t in sh["gamma_attn"]], 1, H)[0],
                          L["gamma_attn"])
    # column-parallel bias
    b = gather(tb.TP_PARAM_FUSED_QKV, [t.view(qkv_rows, 1) for t in sh["bqkv"]], qkv_rows, 1)[:, 0]
    assert np.array_equal(b, np.concatenate([L["bq"], L["bk"], L["bv"]])[perm])


@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_unaligned_shapes_take_the_element_path(gpu_lib, N):
    import torch
    import megatron_tensor_block_gb300 as tb
    w = synth.scaled(synth.WORKLOADS["llama3_8b_decode_tp4"], tp=N, org_vocab=37 * N - 3)
    plan = _plan(w)
    rng = np.random.Generator(np.random.PCG64(5))
    a = rng.standard_normal((6, 3 * N)).astype(np.float32)          # 12-byte rows per shard
    src = torch.from_numpy(a).cuda()
    sh = [torch.empty(6, 3, device="cuda") for _ in range(N)]
    tb.tp_shard_param(plan, tb.TP_PARAM_ROWWISE, src, 6, 3 * N, tb.TP_F32, sh)
    out = torch.empty(6, 3 * N, device="cuda")
    tb.tp_gather_param(plan, tb.TP_PARAM_ROWWISE, sh, 6, 3, tb.TP_F32, out)
    assert np.array_equal(out.cpu().numpy(), a)
    assert all(np.array_equal(s.cpu().numpy(), o) for s, o in zip(sh, O.shard_cols(a, N)))
    # vocab-parallel with a ragged last shard, bf16, odd width
    V, Hd = w.org_vocab, 5
    head = synth.round_to_bf16_bits(rng.standard_normal((V, Hd)).astype(np.float32))
    from megatron_tensor_block_gb300.runtime import to_device
    R = tb.tp_plan_get_info(plan)["vocab_rows_shard"]
    vs = [torch.empty(R, Hd, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    tb.tp_shard_param(plan, tb.TP_PARAM_VOCAB_PARALLEL, to_device(head), V, Hd, tb.TP_BF16, vs)
    out = torch.empty(V, Hd, dtype=torch.bfloat16, device="cuda")
    tb.tp_gather_param(plan, tb.TP_PARAM_VOCAB_PARALLEL, vs, R, Hd, tb.TP_BF16, out)
    assert np.array_equal(_np(out), head)


def test_reduce_partials_rank_order(gpu_lib):
    import torch
    import megatron_tensor_block_gb300 as tb
    w = synth.scaled(synth.WORKLOADS["llama3_8b_decode_tp4"], hidden=256)
    plan = _plan(w)
    N, M, H = 4, 5, 256
    # dyadic values: every fp32 sum is exact, so the result must match bit for bit
    p = synth.dyadic((N, M, H), 7, scale_log2=-3).astype(np.float32)
    res = synth.dyadic((M, H), 8).astype(np.float32)
    bias = synth.dyadic((H,), 9, scale_log2=-1).astype(np.float32)
    out = torch.empty(M, H, device="cuda")
    tb.tp_reduce_partials(plan, torch.from_numpy(p).cuda(), torch.from_numpy(res).cuda(),
                          torch.from_numpy(bias).cuda(), out, M)
    want = res + O.reduce_rank_order([p[r].astype(np.float64) for r in range(N)]) + bias
    assert np.array_equal(out.cpu().numpy().astype(np.float64), want)
    # general values: within fp32 rounding of the float64 reduction
    p = np.random.Generator(np.random.PCG64(3)).standard_normal((N, M, H)).astype(np.float32)
    tb.tp_reduce_partials(plan, torch.from_numpy(p).cuda(), None, None, out, M)
    assert O.relerr(out.cpu().numpy(), O.reduce_rank_order([p[r].astype(np.float64) for r in range(N)])) < 1e-6


@pytest.mark.parametrize("case", [
    dict(N=4, heads=(32, 8), d=128, B=8, L=2048, max_kv=2049, max_batch=8, dtype="bf16"),   # Llama-3-8B shape
    dict(N=2, heads=(14, 2), d=64, B=1, L=512, max_kv=513, max_batch=1, dtype="bf16"),      # Qwen shape
    dict(N=8, heads=(16, 8), d=64, B=3, L=37, max_kv=64, max_batch=5, dtype="f32"),         # ragged, partial batch
    dict(N=1, heads=(8, 2), d=128, B=2, L=1, max_kv=3, max_batch=2, dtype="f32"),
])
def test_kv_cache_placement_matches_the_oracle(gpu_lib, case):
    # each shard's cache holds its contiguous group of KV heads ("Multi-GPU &
    # Multi-Node", How tensor parallelism works, step 2), bit for bit; the
    # positions past L and the sequences past B stay as they were
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import desc_of, to_device
    N, (Hq, Hkv), d = case["N"], case["heads"], case["d"]
    w = synth.scaled(synth.WORKLOADS["llama3_8b_decode_tp4"], hidden=512, n_heads=Hq, n_kv_heads=Hkv, head_dim=d,
                     ffn=512 * N, tp=N, batch=case["max_batch"], kv_len=case["max_kv"] - 1, dtype=case["dtype"])
    plan = tb.tp_plan(desc_of(w, max_kv=case["max_kv"], max_batch=case["max_batch"]), N)
    rng = np.random.Generator(np.random.PCG64(77 + N))
    B, L = case["B"], case["L"]
    full = [rng.standard_normal((B, Hkv, L, d)).astype(np.float32) for _ in range(2)]
    if case["dtype"] == "bf16":
        full = [synth.round_to_bf16_bits(a) for a in full]
    dt = torch.bfloat16 if case["dtype"] == "bf16" else torch.float32
    shape = (case["max_batch"], Hkv // N, case["max_kv"], d)
    k = [torch.full(shape, 7.0, dtype=dt, device="cuda") for _ in range(N)]
    v = [torch.full(shape, -3.0, dtype=dt, device="cuda") for _ in range(N)]
    kf, vf = (to_device(a) for a in full)
    tb.tp_shard_kv(plan, kf, vf, B, L, (k, v))
    torch.cuda.synchronize()
    for src, dst, sentinel in ((full[0], k, 7.0), (full[1], v, -3.0)):
        ref = O.shard_kv_cache(src, N)
        for r in range(N):
            got = _np(dst[r])
            assert np.array_equal(got[:B, :, :L], ref[r]), f"shard {r}"
            rest = dst[r].float().cpu().numpy()
            assert (rest[:, :, L:] == sentinel).all() and (rest[B:] == sentinel).all()
