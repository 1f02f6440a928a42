"""Every parameter kind through ``tp_shard_param`` and ``tp_gather_param``,
bit for bit against the oracle's sharding rules and gather ("Gather
tensor-parallel sharded parameters on read in a trace", Change and
Verification): replicated, column-parallel, row-parallel, the fused QKV and
gate/up kinds with the plan's segments and with explicit ones, and a packed
column-parallel tensor of uneven segments. Each kind runs at tp 1, 2, 4 and
8, in float32 and bfloat16, with 16-byte aligned rows (the vector copy path)
and with odd widths (the element path).

Besides equality with the oracle on both sides (shards, gathered tensor), the
checks are the page's: a round trip gives the unsharded tensor back for the
plain kinds, fused kinds come back as the unsharded rows permuted into rank
groups (equal as a row multiset), and the gather leaves the shards unchanged.
"""
import numpy as np
import pytest

import oracle as O
import synth

pytestmark = pytest.mark.gpu

LLAMA = synth.WORKLOADS["llama3_8b_decode_tp4"]


def _np(t):
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _plan(N):
    # head_dim 64, 8 q / 8 kv heads and F = 512: divisible for every tp up to 8
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import desc_of
    w = synth.scaled(LLAMA, hidden=256, n_heads=8, n_kv_heads=8, head_dim=64, ffn=512, tp=N, batch=1, kv_len=4)
    return w, tb.tp_plan(desc_of(w), N)


def _tensor(rng, rows, cols, dtype):
    a = rng.standard_normal((rows, cols)).astype(np.float32)
    return synth.round_to_bf16_bits(a) if dtype == "bf16" else a


def _kinds(w, N):
    """(name, kind code, oracle kind, rows, segments passed, segment rows the oracle uses)."""
    import megatron_tensor_block_gb300 as tb
    q, kv, F = w.n_heads * w.head_dim, w.n_kv_heads * w.head_dim, w.ffn
    packed = [3 * N, 5 * N, N]                           # uneven segments, each divisible by tp
    return [
        ("replicated", tb.TP_PARAM_REPLICATED, O.REPLICATED, 7, None, None),
        ("colwise", tb.TP_PARAM_COLWISE, O.COLWISE, 6 * N, None, None),
        ("rowwise", tb.TP_PARAM_ROWWISE, O.ROWWISE, 5, None, None),
        ("fused_qkv_plan", tb.TP_PARAM_FUSED_QKV, O.FUSED_QKV, q + 2 * kv, None, [q, kv, kv]),
        ("fused_qkv_explicit", tb.TP_PARAM_FUSED_QKV, O.FUSED_QKV, 4 * N + 2 * N, [4 * N, N, N], [4 * N, N, N]),
        ("fused_gate_up_plan", tb.TP_PARAM_FUSED_GATE_UP, O.FUSED_GATE_UP, 2 * F, None, [F, F]),
        ("fused_gate_up_explicit", tb.TP_PARAM_FUSED_GATE_UP, O.FUSED_GATE_UP, 4 * N, [2 * N, 2 * N], [2 * N, 2 * N]),
        ("packed_colwise", tb.TP_PARAM_PACKED_COLWISE, O.PACKED_COLWISE, sum(packed), packed, packed),
    ]


def _oracle_shards(kind, a, N, segs):
    if kind == O.REPLICATED:
        return [a.copy() for _ in range(N)]
    if kind == O.COLWISE:
        return O.shard_rows(a, N)
    if kind == O.ROWWISE:
        return O.shard_cols(a, N)
    starts = np.cumsum([0] + segs)
    return O.shard_fused([a[s:e] for s, e in zip(starts[:-1], starts[1:])], N)


@pytest.mark.parametrize("aligned", [True, False], ids=["aligned", "unaligned"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_every_kind_shards_and_gathers_like_the_oracle(gpu_lib, N, dtype, aligned):
    import torch
    import megatron_tensor_block_gb300 as tb
    from megatron_tensor_block_gb300.runtime import to_device
    w, plan = _plan(N)
    code = tb.TP_BF16 if dtype == "bf16" else tb.TP_F32
    rng = np.random.Generator(np.random.PCG64(1000 + 10 * N + (dtype == "bf16") + 2 * aligned))
    for name, kind, okind, rows, segs, osegs in _kinds(w, N):
        # per-shard widths: 64 (128 or 256-byte rows) or odd (rows not 16-byte aligned)
        cw = 64 if aligned else 3
        cols = cw * N if kind == tb.TP_PARAM_ROWWISE else (cw if aligned else 5)
        a = _tensor(rng, rows, cols, dtype)
        ref = _oracle_shards(okind, a, N, osegs)
        full = to_device(a)
        shards = [torch.full(r.shape, float("nan"), dtype=full.dtype, device="cuda") for r in ref]
        tb.tp_shard_param(plan, kind, full, rows, cols, code, shards, segments=segs)
        got = [_np(s) for s in shards]
        for r in range(N):
            assert np.array_equal(got[r], ref[r]), f"{name}: shard {r} differs from the oracle's"
        rs, cs = ref[0].shape
        out_shape = {O.REPLICATED: (rs, cs), O.ROWWISE: (rs, N * cs)}.get(okind, (N * rs, cs))
        before = [s.clone() for s in shards]
        out = torch.full(out_shape, float("nan"), dtype=full.dtype, device="cuda")
        tb.tp_gather_param(plan, kind, shards, rs, cs, code, out)
        torch.cuda.synchronize()
        g = _np(out)
        assert np.array_equal(g, O.gather_param(ref, okind)), f"{name}: gather differs from the oracle's"
        if okind in (O.REPLICATED, O.COLWISE, O.ROWWISE):
            assert np.array_equal(g, a), f"{name}: round trip is not exact"
        else:
            assert sorted(map(bytes, g)) == sorted(map(bytes, a)), f"{name}: not the same row multiset"
            assert np.array_equal(g, a[O.fused_gather_permutation(osegs, N)]), f"{name}: not rank-grouped"
        assert all(torch.equal(x, y) for x, y in zip(shards, before)), f"{name}: the gather changed a shard"


def test_fused_kinds_reject_segments_that_do_not_divide(gpu_lib):
    import torch
    import megatron_tensor_block_gb300 as tb
    w, plan = _plan(4)
    a = torch.zeros(12, 8, device="cuda")
    sh = [torch.empty(3, 8, device="cuda") for _ in range(4)]
    with pytest.raises(tb.TpError) as e:
        tb.tp_shard_param(plan, tb.TP_PARAM_PACKED_COLWISE, a, 12, 8, tb.TP_F32, sh, segments=[6, 6])
    assert e.value.status == tb.binding.TP_ERR_SHAPE
    with pytest.raises(tb.TpError) as e:
        tb.tp_shard_param(plan, tb.TP_PARAM_PACKED_COLWISE, a, 12, 8, tb.TP_F32, sh, segments=[4, 4])
    assert e.value.status == tb.binding.TP_ERR_SHAPE             # segments sum to 8, not 12
    with pytest.raises(tb.TpError) as e:
        tb.tp_shard_param(plan, tb.TP_PARAM_PACKED_COLWISE, a, 12, 8, tb.TP_F32, sh)
    assert e.value.status == tb.binding.TP_ERR_INVALID_ARG       # packed kinds need their segments
