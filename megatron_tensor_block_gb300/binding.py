"""ctypes binding of ``include/tp_block.h``: the same entry points under the
same names, argument marshalling only. Tensors may be passed as integers
(device addresses) or as objects with ``data_ptr()`` (torch tensors);
streams as integers, ``torch.cuda.Stream`` objects or ``None`` (torch's
current stream). A non-zero status raises :class:`TpError` with the library's
message. Every computation happens in the CUDA library; if it is missing, the
import of the library fails loudly.
"""
from __future__ import annotations

import ctypes as C
import os

from . import build as _build

TP_MAX_SHARDS = 8
TP_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024

TP_OK = 0
TP_ERR_INVALID_ARG = -1
TP_ERR_INDIVISIBLE = -2
TP_ERR_UNSUPPORTED = -3
TP_ERR_NULL = -4
TP_ERR_ALIGN = -5
TP_ERR_SHAPE = -6
TP_ERR_CAPACITY = -7
TP_ERR_CUDA = -8
TP_ERR_TIMEOUT = -9
STATUS_NAMES = {0: "TP_OK", -1: "TP_ERR_INVALID_ARG", -2: "TP_ERR_INDIVISIBLE", -3: "TP_ERR_UNSUPPORTED",
                -4: "TP_ERR_NULL", -5: "TP_ERR_ALIGN", -6: "TP_ERR_SHAPE", -7: "TP_ERR_CAPACITY",
                -8: "TP_ERR_CUDA", -9: "TP_ERR_TIMEOUT"}

TP_F32, TP_BF16 = 0, 1
TP_MODE_DECODE, TP_MODE_PREFILL, TP_MODE_MOE_FFN = 0, 1, 2
(TP_PARAM_REPLICATED, TP_PARAM_COLWISE, TP_PARAM_ROWWISE, TP_PARAM_FUSED_QKV, TP_PARAM_FUSED_GATE_UP,
 TP_PARAM_PACKED_COLWISE, TP_PARAM_VOCAB_PARALLEL) = range(7)

_P8 = C.c_void_p * TP_MAX_SHARDS


class tp_model_desc(C.Structure):
    _fields_ = [("hidden", C.c_int64), ("n_heads", C.c_int64), ("n_kv_heads", C.c_int64),
                ("head_dim", C.c_int64), ("ffn", C.c_int64), ("n_experts", C.c_int64),
                ("top_k", C.c_int64), ("expert_ffn", C.c_int64), ("org_vocab", C.c_int64),
                ("eps", C.c_double), ("rope_theta", C.c_double), ("dtype", C.c_int32),
                ("has_qkv_bias", C.c_int32), ("max_batch", C.c_int64), ("max_tokens", C.c_int64),
                ("max_kv", C.c_int64), ("expert_parallel", C.c_int32), ("reserved0", C.c_int32)]


class tp_plan_info(C.Structure):
    _fields_ = [("tp", C.c_int32), ("reduce_points", C.c_int32)] + [
        (n, C.c_int64) for n in (
            "hq_shard", "hkv_shard", "ffn_shard", "expert_ffn_shard", "qkv_rows", "vocab_padded",
            "vocab_rows_shard", "wqkv_bytes", "bqkv_bytes", "wo_bytes", "wgu_bytes", "wd_bytes",
            "gamma_bytes", "egu_bytes", "ed_bytes", "kv_cache_bytes", "lm_head_bytes", "workspace_bytes",
            "weight_bytes_shard", "weight_bytes_total", "moe_ids_offset", "moe_bucket_offset",
            "moe_perm_offset", "experts_shard", "noalloc_scratch_bytes")]


class tp_block_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "wq", "wk", "wv", "bq", "bk", "bv", "wo", "w_gate", "w_up", "w_down", "gamma_attn", "gamma_ffn",
        "e_gate", "e_up", "e_down")]


class tp_shard_set(C.Structure):
    _fields_ = [(n, _P8) for n in ("wqkv", "bqkv", "wo", "wgu", "wd", "gamma_attn", "gamma_ffn", "egu", "ed")]


class tp_kv_set(C.Structure):
    _fields_ = [("k", _P8), ("v", _P8)]


class TpError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def load(path: str | None = None) -> C.CDLL:
    """Loads (building first if needed) the CUDA library."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = _build.LIB
        if not os.path.exists(path) or _build.is_stale():
            _build.build()
    lib = C.CDLL(path)
    P, I32, I64, VP = C.c_void_p, C.c_int32, C.c_int64, C.c_void_p
    sig = {
        "tp_plan": (I32, [C.POINTER(tp_model_desc), I32, C.POINTER(P)]),
        "tp_plan_destroy": (None, [P]),
        "tp_plan_get_info": (I32, [P, C.POINTER(tp_plan_info)]),
        "tp_plan_describe": (I32, [P, C.c_char_p, C.c_size_t]),
        "tp_shard_weights": (I32, [P, C.POINTER(tp_block_weights), C.POINTER(tp_shard_set), VP]),
        "tp_shard_param": (I32, [P, I32, VP, I64, I64, I32, C.POINTER(I64), I32, C.POINTER(VP), VP]),
        "tp_gather_param": (I32, [P, I32, C.POINTER(VP), I64, I64, I32, VP, VP]),
        "tp_shard_kv": (I32, [P, VP, VP, I64, I64, C.POINTER(tp_kv_set), VP]),
        "tp_workspace_init": (I32, [P, VP, C.c_size_t, VP]),
        "tp_block_forward": (I32, [P, C.POINTER(tp_shard_set), C.POINTER(tp_kv_set), VP, VP, VP, I32, I32,
                                   I32, VP, VP, C.c_size_t, VP]),
        "tp_block_forward_noalloc": (I32, [P, C.POINTER(tp_shard_set), C.POINTER(tp_kv_set), VP, VP, VP, I32,
                                           VP]),
        "tp_noalloc_status": (I32, [C.POINTER(I32), VP]),
        "tp_stack_create": (I32, [P, I32, C.POINTER(tp_shard_set), C.POINTER(tp_kv_set), C.POINTER(P)]),
        "tp_stack_destroy": (None, [P]),
        "tp_stack_ctas": (I32, [P]),
        "tp_stack_set_stamps": (I32, [P, VP, I32]),
        "tp_stack_decode": (I32, [P, VP, VP, VP, I32, VP, C.c_size_t, VP]),
        "tp_lm_head_forward": (I32, [P, C.POINTER(VP), VP, VP, I32, VP, VP, VP]),
        "tp_reduce_partials": (I32, [P, VP, VP, VP, VP, I64, VP]),
        "tp_get_device_status": (I32, [VP, C.POINTER(I32), VP]),
        "tp_gemm_bf16": (I32, [VP, VP, VP, I64, I64, I64, VP, VP]),
        "tp_gemm_bf16_kn": (I32, [VP, VP, VP, I64, I64, I64, VP, VP]),
        "tp_profile_stages": (I32, [P, C.POINTER(VP), I32]),
        "tp_profile_phases": (I32, [P, C.POINTER(C.c_double), C.POINTER(C.c_double), I32, VP]),
        "tp_profile_phase_stamps": (I32, [P, C.POINTER(C.c_uint64), I32, VP]),
        "tp_debug_withhold_arrival": (I32, [P, I32]),
        "tp_last_error": (C.c_char_p, []),
        "tp_version": (I32, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(status: int) -> None:
    if status != TP_OK:
        raise TpError(status, _lib.tp_last_error().decode())


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


class Plan:
    """Owns a ``tp_plan_t``; destroyed with the object."""

    def __init__(self, handle: int):
        self.handle = handle

    def __del__(self):
        if self.handle and _lib is not None:
            _lib.tp_plan_destroy(self.handle)
            self.handle = None


def tp_plan(desc, tp: int) -> Plan:
    lib = load()
    if isinstance(desc, dict):
        desc = tp_model_desc(**desc)
    h = C.c_void_p()
    _check(lib.tp_plan(C.byref(desc), int(tp), C.byref(h)))
    return Plan(h.value)


def tp_plan_get_info(plan: Plan) -> dict:
    info = tp_plan_info()
    _check(load().tp_plan_get_info(plan.handle, C.byref(info)))
    return {n: getattr(info, n) for n, _ in tp_plan_info._fields_}


def tp_plan_describe(plan: Plan) -> str:
    buf = C.create_string_buffer(1024)
    _check(load().tp_plan_describe(plan.handle, buf, len(buf)))
    return buf.value.decode()


def _shard_set(d: dict) -> tp_shard_set:
    s = tp_shard_set()
    for name, _ in tp_shard_set._fields_:
        arr = getattr(s, name)
        for r, t in enumerate(d.get(name) or []):
            arr[r] = _ptr(t)
    return s


def _kv_set(k: list, v: list) -> tp_kv_set:
    s = tp_kv_set()
    for r, t in enumerate(k):
        s.k[r] = _ptr(t)
    for r, t in enumerate(v):
        s.v[r] = _ptr(t)
    return s


def tp_shard_weights(plan: Plan, full: dict, out: dict, stream=None) -> None:
    fw = tp_block_weights(**{n: _ptr(full.get(n)) for n, _ in tp_block_weights._fields_})
    _check(load().tp_shard_weights(plan.handle, C.byref(fw), C.byref(_shard_set(out)), _stream(stream)))


def tp_shard_param(plan: Plan, kind: int, full, rows: int, cols: int, dtype: int, shards_out: list,
                   segments=None, stream=None) -> None:
    arr = (C.c_void_p * len(shards_out))(*[_ptr(t) for t in shards_out])
    seg = (C.c_int64 * len(segments))(*segments) if segments else None
    _check(load().tp_shard_param(plan.handle, kind, _ptr(full), rows, cols, dtype, seg,
                                 len(segments) if segments else 0, arr, _stream(stream)))


def tp_gather_param(plan: Plan, kind: int, shards: list, rows_per_shard: int, cols_per_shard: int,
                    dtype: int, out, stream=None) -> None:
    arr = (C.c_void_p * len(shards))(*[_ptr(t) for t in shards])
    _check(load().tp_gather_param(plan.handle, kind, arr, rows_per_shard, cols_per_shard, dtype,
                                  _ptr(out), _stream(stream)))


def tp_shard_kv(plan: Plan, k_full, v_full, B: int, L: int, kv: tuple, stream=None) -> None:
    """Copies full ``[B, Hkv, L, d]`` caches into the shards' caches ``kv = (k_list, v_list)``."""
    kvs = _kv_set(*kv)
    _check(load().tp_shard_kv(plan.handle, _ptr(k_full), _ptr(v_full), B, L, C.byref(kvs), _stream(stream)))


def tp_workspace_init(plan: Plan, workspace, nbytes: int, stream=None) -> None:
    _check(load().tp_workspace_init(plan.handle, _ptr(workspace), nbytes, _stream(stream)))


def tp_block_forward(plan: Plan, shards: dict, kv: tuple, x, y, pos, B: int, T_per_seq: int, mode: int,
                     router_logits, workspace, nbytes: int, stream=None) -> None:
    kvs = _kv_set(*kv) if kv is not None else None
    _check(load().tp_block_forward(plan.handle, C.byref(_shard_set(shards)),
                                   C.byref(kvs) if kvs is not None else None, _ptr(x), _ptr(y), _ptr(pos),
                                   B, T_per_seq, mode, _ptr(router_logits), _ptr(workspace), nbytes,
                                   _stream(stream)))


def tp_block_forward_noalloc(plan: Plan, shards: dict, kv: tuple, x, y, pos, B: int, stream=None) -> None:
    """Decode forward using the library's static scratch array instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    kvs = _kv_set(*kv)
    _check(load().tp_block_forward_noalloc(plan.handle, C.byref(_shard_set(shards)), C.byref(kvs), _ptr(x),
                                           _ptr(y), _ptr(pos), B, _stream(stream)))


def tp_noalloc_status(stream=None) -> int:
    """Status word of the static scratch array on the current device (the
    latest ``tp_block_forward_noalloc`` call's device-detected error, or 0)."""
    v = C.c_int32()
    _check(load().tp_noalloc_status(C.byref(v), _stream(stream)))
    return v.value


class Stack:
    """Owns a ``tp_stack_t`` (several decode blocks in one launch); keeps the
    plan alive and is destroyed with the object."""

    def __init__(self, handle: int, plan: Plan):
        self.handle = handle
        self.plan = plan

    def __del__(self):
        if self.handle and _lib is not None:
            _lib.tp_stack_destroy(self.handle)
            self.handle = None


def tp_stack_create(plan: Plan, layers: list, kvs: list) -> Stack:
    """``layers``: per layer a shard dict (as for tp_block_forward);
    ``kvs``: per layer a (k list, v list) pair."""
    n = len(layers)
    sets = (tp_shard_set * n)(*[_shard_set(d) for d in layers])
    kvset = (tp_kv_set * n)(*[_kv_set(*kv) for kv in kvs])
    h = C.c_void_p()
    _check(load().tp_stack_create(plan.handle, n, sets, kvset, C.byref(h)))
    return Stack(h.value, plan)


def tp_stack_ctas(stack: Stack) -> int:
    return int(load().tp_stack_ctas(stack.handle))


def tp_stack_set_stamps(stack: Stack, stamps, rows: int) -> None:
    """Measurement hook (``stamps``: zeroed device uint64 tensor of
    rows x layers x 5 x 2, or None to clear)."""
    _check(load().tp_stack_set_stamps(stack.handle, _ptr(stamps), rows))


def tp_stack_decode(stack: Stack, x, y, pos, B: int, workspace, nbytes: int, stream=None) -> None:
    _check(load().tp_stack_decode(stack.handle, _ptr(x), _ptr(y), _ptr(pos), B, _ptr(workspace), nbytes,
                                  _stream(stream)))


def tp_lm_head_forward(plan: Plan, head_shards: list, gamma, x, T: int, logits, device_status=None,
                       stream=None) -> None:
    """Logits of the final hidden state over the vocab-parallel head."""
    arr = (C.c_void_p * len(head_shards))(*[_ptr(t) for t in head_shards])
    _check(load().tp_lm_head_forward(plan.handle, arr, _ptr(gamma), _ptr(x), T, _ptr(logits),
                                     _ptr(device_status), _stream(stream)))


def tp_reduce_partials(plan: Plan, partials, residual, bias, out, M: int, stream=None) -> None:
    _check(load().tp_reduce_partials(plan.handle, _ptr(partials), _ptr(residual), _ptr(bias), _ptr(out), M,
                                     _stream(stream)))


def tp_gemm_bf16(A, B, C, M: int, N: int, K: int, device_status=None, stream=None) -> None:
    """C[M, N] = A[M, K] @ B[N, K].T on the tensor cores (bf16 in, float32 out)."""
    _check(load().tp_gemm_bf16(_ptr(A), _ptr(B), _ptr(C), M, N, K, _ptr(device_status), _stream(stream)))


def tp_gemm_bf16_kn(A, B, C, M: int, N: int, K: int, device_status=None, stream=None) -> None:
    """C[M, N] = A[M, K] @ B[K, N] on the tensor cores (B N-contiguous)."""
    _check(load().tp_gemm_bf16_kn(_ptr(A), _ptr(B), _ptr(C), M, N, K, _ptr(device_status), _stream(stream)))


def tp_debug_withhold_arrival(plan: Plan, on: bool) -> None:
    """Test hook: the plan's decode launches wait for one grid-barrier
    arrival too many, so their bounded waits run out (TP_ERR_TIMEOUT)."""
    _check(load().tp_debug_withhold_arrival(plan.handle, 1 if on else 0))


def tp_get_device_status(workspace, stream=None) -> int:
    v = C.c_int32()
    _check(load().tp_get_device_status(_ptr(workspace), C.byref(v), _stream(stream)))
    return v.value


def tp_profile_stages(plan: Plan, events) -> None:
    """``events``: list of ``torch.cuda.Event`` (or raw cudaEvent_t ints), or None to clear."""
    if not events:
        _check(load().tp_profile_stages(plan.handle, None, 0))
        return
    raw = [e if isinstance(e, int) else e.cuda_event for e in events]
    arr = (C.c_void_p * len(raw))(*raw)
    _check(load().tp_profile_stages(plan.handle, arr, len(raw)))


def tp_profile_phase_stamps(plan: Plan, rows: int, stream=None) -> list:
    """Raw per-CTA timestamps (ns) of the last profiled bf16 decode step: rows x 13."""
    arr = (C.c_uint64 * (rows * 13))()
    _check(load().tp_profile_phase_stamps(plan.handle, arr, rows, _stream(stream)))
    return [list(arr[i * 13:(i + 1) * 13]) for i in range(rows)]


def tp_profile_phases(plan: Plan, n: int = 9, stream=None, median: bool = False):
    """Phase durations (us) of the last profiled bf16 decode step; with
    ``median`` also the durations to the median CTA's arrival."""
    arr = (C.c_double * n)()
    med = (C.c_double * n)() if median else None
    _check(load().tp_profile_phases(plan.handle, arr, med, n, _stream(stream)))
    return (list(arr), list(med)) if median else list(arr)


def tp_last_error() -> str:
    return load().tp_last_error().decode()


def tp_version() -> int:
    return load().tp_version()
