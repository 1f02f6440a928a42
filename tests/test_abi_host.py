"""Host-side checks of the C ABI (no GPU needed): the library loads and
exports every declared entry point, plans validate as the pages require, and
launching calls fail loudly without an sm_103 device."""
import ctypes
import json
import os
import re

import pytest

import synth
import megatron_tensor_block_gb300 as tb
from megatron_tensor_block_gb300 import binding as B
from megatron_tensor_block_gb300.runtime import desc_of

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tp_block.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tp_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = tb.load()
    names = declared_functions()
    assert "tp_block_forward" in names and "tp_gather_param" in names
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_version():
    assert tb.tp_version() == 1


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_every_workload_plans(name):
    w = synth.WORKLOADS[name]
    plan = tb.tp_plan(desc_of(w), w.tp)
    info = tb.tp_plan_get_info(plan)
    assert info["tp"] == w.tp
    assert info["workspace_bytes"] > 0
    assert info["weight_bytes_total"] == w.tp * info["weight_bytes_shard"]


def test_plan_shapes_llama3_8b_decode():
    w = synth.WORKLOADS["llama3_8b_decode_tp4"]
    info = tb.tp_plan_get_info(tb.tp_plan(desc_of(w), 4))
    assert (info["hq_shard"], info["hkv_shard"], info["ffn_shard"], info["qkv_rows"]) == (8, 2, 3584, 1536)
    assert info["wqkv_bytes"] == 1536 * 4096 * 2
    assert info["wgu_bytes"] == 7168 * 4096 * 2 and info["wd_bytes"] == 4096 * 3584 * 2
    # every shard holds 1/tp of the projection weights
    total = 2 * (4096 * 4096 * 2 + 2 * 1024 * 4096 + 3 * 14336 * 4096)
    assert info["weight_bytes_total"] == total


def test_reduce_points_golden():
    g = json.load(open(os.path.join(GOLDEN, "reduce_points.json")))
    w = synth.WORKLOADS["llama3_8b_decode_tp4"]
    assert tb.tp_plan_get_info(tb.tp_plan(desc_of(w), 4))["reduce_points"] == g["dense_block_reduce_points"]
    m = synth.WORKLOADS["moe_expert_slice_tp4"]
    assert tb.tp_plan_get_info(tb.tp_plan(desc_of(m), 4))["reduce_points"] == g["moe_ffn_block_reduce_points"]
    # the GLM-5.2 numbers: two all-reduces per layer at hidden 6144, tp 3
    glm = synth.scaled(w, hidden=g["glm_hidden"], n_heads=48, n_kv_heads=6, ffn=12288, tp=g["glm_tp"])
    assert tb.tp_plan_get_info(tb.tp_plan(desc_of(glm), g["glm_tp"]))["reduce_points"] * g["glm_layers"] == 156


def test_vocab_rows_golden():
    spec = json.load(open(os.path.join(GOLDEN, "vocab_sharding.json")))
    base = synth.WORKLOADS["qwen25_05b_decode_tp2"]
    for case in spec["cases"]:
        w = synth.scaled(base, org_vocab=case["org_vocab"], tp=case["tp"])
        info = tb.tp_plan_get_info(tb.tp_plan(desc_of(w), case["tp"]))
        assert info["vocab_rows_shard"] == case["rows_per_shard"]
        assert info["vocab_padded"] - case["org_vocab"] == case["padding_rows"]


def _status(desc, tp):
    try:
        tb.tp_plan(desc, tp)
        return 0
    except tb.TpError as e:
        return e.status


def test_plan_rejects_invalid_inputs_with_clear_errors():
    w = synth.WORKLOADS["qwen25_05b_decode_tp2"]
    d = desc_of(w)
    assert _status(d, 4) == B.TP_ERR_INDIVISIBLE            # 14 heads, 2 kv heads, tp 4
    assert "not divisible" in tb.tp_last_error()
    assert _status(d, 0) == B.TP_ERR_INVALID_ARG
    assert _status(d, 9) == B.TP_ERR_INVALID_ARG
    assert _status(dict(d, n_heads=15, n_kv_heads=2), 1) == B.TP_ERR_INVALID_ARG
    assert _status(dict(d, head_dim=96), 2) == B.TP_ERR_UNSUPPORTED
    assert _status(dict(d, dtype=7), 2) == B.TP_ERR_INVALID_ARG
    assert _status(dict(d, ffn=4864 + 2), 2) == B.TP_ERR_UNSUPPORTED   # divisible by 2, F/2 not a multiple of 64
    assert _status(dict(d, ffn=4863), 2) == B.TP_ERR_INDIVISIBLE
    m = desc_of(synth.WORKLOADS["moe_expert_slice_tp4"])
    assert _status(dict(m, top_k=65), 4) == B.TP_ERR_INVALID_ARG
    assert _status(dict(m, expert_ffn=1022), 4) == B.TP_ERR_INDIVISIBLE
    # expert parallelism: whole experts per shard, so the expert count must divide
    assert _status(dict(m, expert_parallel=1, n_experts=62), 4) == B.TP_ERR_INDIVISIBLE
    assert _status(dict(m, expert_parallel=2), 4) == B.TP_ERR_INVALID_ARG
    assert _status(dict(d, expert_parallel=1), 2) == B.TP_ERR_INVALID_ARG      # no experts
    assert _status(dict(m, reserved0=1), 4) == B.TP_ERR_INVALID_ARG
    assert _status(d, 2) == 0 and tb.tp_last_error() == ""


def test_expert_parallel_plan_holds_whole_experts():
    # the same bytes per shard as expert slicing: E/N whole experts instead of
    # 1/N of every expert
    m = desc_of(synth.WORKLOADS["moe_expert_slice_tp4"])
    sl = tb.tp_plan_get_info(tb.tp_plan(m, 4))
    ep = tb.tp_plan_get_info(tb.tp_plan(dict(m, expert_parallel=1), 4))
    assert (sl["experts_shard"], sl["expert_ffn_shard"]) == (64, 256)
    assert (ep["experts_shard"], ep["expert_ffn_shard"]) == (16, 1024)
    assert ep["egu_bytes"] == sl["egu_bytes"] == 16 * 2 * 1024 * 2048 * 2
    assert ep["ed_bytes"] == sl["ed_bytes"]


def test_describe_reports_one_nth_of_the_weights():
    w = synth.WORKLOADS["llama3_8b_decode_tp4"]
    s = tb.tp_plan_describe(tb.tp_plan(desc_of(w), 4))
    assert "4 logical shards" in s and "= 0.2500 of" in s and "2 reductions per block" in s


def test_launching_calls_need_an_sm103_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    w = synth.WORKLOADS["tiny_llama_fp32_tp2"]
    plan = tb.tp_plan(desc_of(w), 2)
    info = tb.tp_plan_get_info(plan)
    with pytest.raises(tb.TpError) as e:
        # the pointer is never dereferenced: the device check fails first
        tb.tp_workspace_init(plan, 4096, info["workspace_bytes"], stream=0)
    assert e.value.status == B.TP_ERR_UNSUPPORTED


def test_argument_errors_precede_any_launch():
    w = synth.WORKLOADS["tiny_llama_fp32_tp2"]
    plan = tb.tp_plan(desc_of(w), 2)
    info = tb.tp_plan_get_info(plan)
    with pytest.raises(tb.TpError) as e:
        tb.tp_workspace_init(plan, 4096, info["workspace_bytes"] - 1, stream=0)
    assert e.value.status == B.TP_ERR_CAPACITY
    with pytest.raises(tb.TpError) as e:
        tb.tp_workspace_init(plan, 4100, info["workspace_bytes"], stream=0)
    assert e.value.status == B.TP_ERR_ALIGN
    with pytest.raises(tb.TpError) as e:
        tb.tp_gather_param(plan, B.TP_PARAM_VOCAB_PARALLEL, [4096, 8192], 400, 256, B.TP_F32, 4096, stream=0)
    assert e.value.status == B.TP_ERR_SHAPE          # org_vocab 1000 > 2 x 400 rows
    with pytest.raises(tb.TpError) as e:
        tb.tp_gather_param(plan, 17, [4096, 8192], 512, 256, B.TP_F32, 4096, stream=0)
    assert e.value.status == B.TP_ERR_INVALID_ARG
    with pytest.raises(tb.TpError) as e:
        tb.tp_block_forward(plan, {}, None, 4096, 4096, 0, 1, 1, B.TP_MODE_DECODE, None, 8192,
                            info["workspace_bytes"], stream=0)
    assert e.value.status == B.TP_ERR_INVALID_ARG    # y aliases x
    with pytest.raises(tb.TpError) as e:
        tb.tp_block_forward(plan, {}, None, 4096, 8192, 0, 2, 1, B.TP_MODE_DECODE, None, 16384,
                            info["workspace_bytes"], stream=0)
    assert e.value.status == B.TP_ERR_SHAPE          # B above max_batch


def test_noalloc_footprint_covers_the_piece_buffer_and_ignores_max_tokens():
    # the no-alloc decode uses control words, decode buffers and the down
    # pieces' pair buffer; prefill/MoE buffers (sized by max_tokens) are not
    # part of it
    w = synth.WORKLOADS["llama3_8b_decode_tp4"]
    small = tb.tp_plan_get_info(tb.tp_plan(desc_of(w), 4))
    big = tb.tp_plan_get_info(tb.tp_plan(desc_of(w, max_tokens=8192), 4))
    assert small["noalloc_scratch_bytes"] == big["noalloc_scratch_bytes"]
    assert 0 < small["noalloc_scratch_bytes"] <= B.TP_NOALLOC_SCRATCH_BYTES
    assert big["workspace_bytes"] > B.TP_NOALLOC_SCRATCH_BYTES     # the whole workspace would not fit
    # down pieces: 64 output tiles x 4 shards x 2 slots x 64 rows x 8 tokens x 8 bytes = 1 MiB
    assert small["noalloc_scratch_bytes"] >= 64 * 4 * 2 * 64 * 8 * 8
    moe = tb.tp_plan_get_info(tb.tp_plan(desc_of(synth.WORKLOADS["moe_expert_slice_tp4"]), 4))
    assert moe["noalloc_scratch_bytes"] == 0


def test_noalloc_rejects_an_oversized_plan_before_any_launch():
    w = synth.WORKLOADS["llama3_8b_decode_tp4"]
    plan = tb.tp_plan(desc_of(w, max_kv=200000), 4)
    assert tb.tp_plan_get_info(plan)["noalloc_scratch_bytes"] > B.TP_NOALLOC_SCRATCH_BYTES
    # the pointers are never dereferenced: the capacity check comes first
    with pytest.raises(tb.TpError) as e:
        tb.tp_block_forward_noalloc(plan, {}, ([0] * 4, [0] * 4), 4096, 8192, 16384, w.batch, stream=0)
    assert e.value.status == B.TP_ERR_CAPACITY
    assert "static array" in str(e.value)


def test_kv_placement_argument_errors_precede_any_launch():
    w = synth.WORKLOADS["llama3_8b_decode_tp4"]
    plan = tb.tp_plan(desc_of(w), 4)
    kv = ([4096] * 4, [8192] * 4)
    with pytest.raises(tb.TpError) as e:
        tb.tp_shard_kv(plan, 4096, 8192, 9, 10, kv, stream=0)
    assert e.value.status == B.TP_ERR_SHAPE                  # B above max_batch
    with pytest.raises(tb.TpError) as e:
        tb.tp_shard_kv(plan, 4096, 8192, 8, w.max_kv + 1, kv, stream=0)
    assert e.value.status == B.TP_ERR_CAPACITY               # L above max_kv
    with pytest.raises(tb.TpError) as e:
        tb.tp_shard_kv(plan, 4096, 8192, 8, 10, ([4096] * 3 + [0], [8192] * 4), stream=0)
    assert e.value.status == B.TP_ERR_NULL
    moe = tb.tp_plan(desc_of(synth.WORKLOADS["moe_expert_slice_tp4"]), 4)
    with pytest.raises(tb.TpError) as e:
        tb.tp_shard_kv(moe, 4096, 8192, 8, 10, kv, stream=0)
    assert e.value.status == B.TP_ERR_INVALID_ARG


def test_withhold_hook_is_off_by_default_and_validates():
    w = synth.WORKLOADS["llama3_8b_decode_tp4"]
    plan = tb.tp_plan(desc_of(w), 4)
    tb.tp_debug_withhold_arrival(plan, True)
    tb.tp_debug_withhold_arrival(plan, False)
    assert tb.load().tp_debug_withhold_arrival(plan.handle, 2) == B.TP_ERR_INVALID_ARG
    assert tb.load().tp_debug_withhold_arrival(None, 1) == B.TP_ERR_NULL
