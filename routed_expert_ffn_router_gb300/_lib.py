"""ctypes binding of libmoe_gb300.so (include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. Tensors are passed as raw device pointers (`data_ptr()`), streams as
their `cuda_stream` handle. There is no fallback: if the library is missing or
a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe_gb300.so")

MOE_OK, MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, \
    MOE_ERR_TIMEOUT, MOE_ERR_DEVICE = range(7)
MOE_F32, MOE_BF16 = 0, 1

# names of every entry point declared in include/moe.h
EXPORTS = ("moe_router_logits", "moe_route", "moe_permute", "moe_expert_ffn", "moe_layer_forward",
           "moe_workspace_bytes", "moe_workspace_init", "moe_read_status", "moe_status_str",
           "moe_last_launch_count", "moe_profile_enable", "moe_profile_collect",
           "moe_profile_forget", "moe_profile_totals", "moe_profile_kind_name",
           "moe_expert_ffn_static", "moe_static_read_status", "moe_cache_state_bytes", "moe_cache_init",
           "moe_cache_set_resident", "moe_cache_observe", "moe_cache_observe_layers",
           "moe_cache_observe_counts", "moe_cache_observe_device",
           "moe_cache_advance",
           "moe_cache_rebalance", "moe_cache_slot_map", "moe_cache_heat",
           "moe_cache_swapped_total", "moe_cache_profile_write", "moe_cache_profile_load",
           "moe_trace_write", "moe_trace_read", "moe_mailbox_create", "moe_mailbox_destroy",
           "moe_mailbox_pairs", "moe_mailbox_compute", "moe_mailbox_inject", "moe_mailbox_add",
           "moe_decode_stack_plan_bytes", "moe_decode_stack_prepare",
           "moe_decode_stack_prepare_routed", "moe_decode_stack")


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {code})")
        self.code = code


class moe_qmat(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p)]


class moe_layer_desc(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("S", ctypes.c_int32),
                ("gate", moe_qmat), ("up", moe_qmat), ("down", moe_qmat),
                ("shared_I", ctypes.c_int32),
                ("shared_gate", moe_qmat), ("shared_up", moe_qmat), ("shared_down", moe_qmat),
                ("pick_counts", ctypes.c_void_p), ("pick_max_rows", ctypes.c_int32)]


class moe_layer_io(ctypes.Structure):
    _fields_ = [("logits", ctypes.c_void_p), ("x", ctypes.c_void_p), ("slot_map", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("ids", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("miss_ids", ctypes.c_void_p), ("n_miss", ctypes.c_void_p)]


class moe_cache_params(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("half_life_tokens", ctypes.c_double),
                ("round_every_tokens", ctypes.c_int32), ("max_swaps", ctypes.c_int32),
                ("fill_every_tokens", ctypes.c_int32), ("max_fills", ctypes.c_int32),
                ("in_ratio", ctypes.c_double), ("in_picks", ctypes.c_double),
                ("max_window_tokens", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class moe_cache_swap(ctypes.Structure):
    _fields_ = [("layer", ctypes.c_int32), ("slot", ctypes.c_int32),
                ("expert_in", ctypes.c_int32), ("expert_out", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load the library (built by build.py / __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it first with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(path)
        P, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        D = ctypes.POINTER(moe_layer_desc)
        sig = {
            "moe_router_logits": ([P, i32, P, i32, i32, i32, P, P], i32),
            "moe_route": ([P, i32, i32, i32, P, P, P, P], i32),
            "moe_permute": ([P, i32, i32, i32, P, i32, P, P, P, P, P, P, sz, P], i32),
            "moe_expert_ffn": ([D, P, i32, i32, P, P, P, P, P, P, P, sz, P], i32),
            "moe_layer_forward": ([D, P, P, i32, i32, P, P, P, P, P, P, P, sz, P], i32),
            "moe_workspace_bytes": ([D, i32], sz),
            "moe_workspace_init": ([P, sz, P], i32),
            "moe_read_status": ([P, P, ctypes.POINTER(ctypes.c_int32)], i32),
            "moe_status_str": ([i32], ctypes.c_char_p),
            "moe_last_launch_count": ([], ctypes.c_int32),
            "moe_profile_enable": ([ctypes.c_int32], i32),
            "moe_profile_collect": ([], i32),
            "moe_profile_forget": ([], i32),
            "moe_profile_totals": ([ctypes.c_int32, ctypes.POINTER(ctypes.c_double),
                                    ctypes.POINTER(ctypes.c_int64)], i32),
            "moe_profile_kind_name": ([ctypes.c_int32], ctypes.c_char_p),
            "moe_expert_ffn_static": ([D, P, i32, i32, P, P, P, P, P, P, P], i32),
            "moe_static_read_status": ([P, ctypes.POINTER(ctypes.c_int32)], i32),
            "moe_decode_stack_plan_bytes": ([ctypes.c_int32], sz),
            "moe_decode_stack_prepare": ([D, ctypes.POINTER(moe_layer_io), ctypes.c_int32,
                                          ctypes.c_int32, P, sz, P, sz, P], i32),
            "moe_decode_stack_prepare_routed": ([D, ctypes.POINTER(moe_layer_io), P, ctypes.c_int32,
                                                 ctypes.c_int32, P, sz, P, sz, P], i32),
            "moe_decode_stack": ([P, ctypes.c_int32, ctypes.c_int32, P, sz, P], i32),
            "moe_cache_state_bytes": ([ctypes.POINTER(moe_cache_params), P], sz),
            "moe_cache_init": ([P, sz, ctypes.POINTER(moe_cache_params), P], i32),
            "moe_cache_set_resident": ([P, ctypes.c_int32, P, ctypes.c_int32], i32),
            "moe_cache_observe": ([P, ctypes.c_int32, P, ctypes.c_int32, ctypes.c_int32], i32),
            "moe_cache_observe_layers": ([P, P, ctypes.c_int32, ctypes.c_int32], i32),
            "moe_cache_observe_counts": ([P, P], i32),
            "moe_cache_observe_device": ([P, P, P], i32),
            "moe_cache_advance": ([P, ctypes.c_int32, P, ctypes.c_int32], ctypes.c_int32),
            "moe_cache_rebalance": ([P, ctypes.c_int32, P, ctypes.c_int32], ctypes.c_int32),
            "moe_cache_slot_map": ([P, ctypes.c_int32, P], i32),
            "moe_cache_heat": ([P, ctypes.c_int32, P], i32),
            "moe_cache_swapped_total": ([P], ctypes.c_int64),
            "moe_cache_profile_write": ([P, P, ctypes.c_int64], ctypes.c_int64),
            "moe_cache_profile_load": ([P, P, ctypes.c_int64], i32),
            "moe_trace_write": ([ctypes.c_int32, P, P, ctypes.c_int32, ctypes.c_int32, P, ctypes.c_int64],
                                ctypes.c_int64),
            "moe_trace_read": ([P, ctypes.c_int64, P, P, P, P, ctypes.c_int32, ctypes.c_int64], ctypes.c_int64),
            "moe_mailbox_create": ([ctypes.c_int32, ctypes.c_int32], P),
            "moe_mailbox_destroy": ([P], None),
            "moe_mailbox_pairs": ([P, ctypes.c_int32, ctypes.c_int32, P, ctypes.c_int32, P, ctypes.c_int32],
                                  ctypes.c_int32),
            "moe_mailbox_compute": ([P, D, P, i32, ctypes.c_int32, P, P, P, ctypes.c_int32, P], i32),
            "moe_mailbox_inject": ([P, ctypes.c_int32], i32),
            "moe_mailbox_add": ([P, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P, P],
                                i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
        return L


def status_str(code: int) -> str:
    return load().moe_status_str(int(code)).decode()


def _check(fn: str, code: int):
    if code != MOE_OK:
        raise MoeError(fn, code, status_str(code))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


# --------------------------------------------------------------------------- calls
def moe_router_logits(x, x_dtype, wg, T, H, E, logits, stream=None):
    _check("moe_router_logits", load().moe_router_logits(_ptr(x), x_dtype, _ptr(wg), T, H, E,
                                                         _ptr(logits), _stream(stream)))


def moe_route(logits, T, E, k, ids, w, status=None, stream=None):
    _check("moe_route", load().moe_route(_ptr(logits), T, E, k, _ptr(ids), _ptr(w), _ptr(status),
                                         _stream(stream)))


def moe_permute(ids, T, E, k, slot_map, S, offsets, sorted_pair, pair_pos, miss_ids, n_miss,
                ws, ws_bytes, stream=None):
    _check("moe_permute", load().moe_permute(
        _ptr(ids), T, E, k, _ptr(slot_map), S, _ptr(offsets), _ptr(sorted_pair), _ptr(pair_pos),
        _ptr(miss_ids), _ptr(n_miss), _ptr(ws), ws_bytes, _stream(stream)))


def moe_expert_ffn(desc, x, x_dtype, T, ids, w, slot_map, y, miss_ids, n_miss, ws, ws_bytes,
                   stream=None):
    _check("moe_expert_ffn", load().moe_expert_ffn(
        ctypes.byref(desc), _ptr(x), x_dtype, T, _ptr(ids), _ptr(w), _ptr(slot_map), _ptr(y),
        _ptr(miss_ids), _ptr(n_miss), _ptr(ws), ws_bytes, _stream(stream)))


def moe_expert_ffn_static(desc, x, x_dtype, T, ids, w, slot_map, y, miss_ids, n_miss, stream=None):
    """moe_expert_ffn without a workspace argument: for callers that cannot
    allocate device memory (the library's own fixed 16 MiB scratch is used)."""
    _check("moe_expert_ffn_static", load().moe_expert_ffn_static(
        ctypes.byref(desc), _ptr(x), x_dtype, T, _ptr(ids), _ptr(w), _ptr(slot_map), _ptr(y),
        _ptr(miss_ids), _ptr(n_miss), _stream(stream)))


def moe_static_read_status(stream=None):
    """-> (moe_status code, raw device status bits) of the last
    moe_expert_ffn_static call on the current device. Synchronises the stream."""
    out = ctypes.c_int32(0)
    code = load().moe_static_read_status(_stream(stream), ctypes.byref(out))
    if code == MOE_ERR_CUDA:
        raise MoeError("moe_static_read_status", code, status_str(code))
    return code, int(out.value)


def moe_layer_forward(desc, logits, x, x_dtype, T, slot_map, y, ids, w, miss_ids, n_miss, ws,
                      ws_bytes, stream=None):
    _check("moe_layer_forward", load().moe_layer_forward(
        ctypes.byref(desc), _ptr(logits), _ptr(x), x_dtype, T, _ptr(slot_map), _ptr(y), _ptr(ids),
        _ptr(w), _ptr(miss_ids), _ptr(n_miss), _ptr(ws), ws_bytes, _stream(stream)))


def moe_decode_stack_plan_bytes(n_layers: int) -> int:
    return int(load().moe_decode_stack_plan_bytes(n_layers))


def moe_decode_stack_prepare(descs, ios, T, plan, plan_bytes, ws, ws_bytes, stream=None):
    """descs: sequence of moe_layer_desc; ios: sequence of moe_layer_io (device pointers)."""
    n = len(descs)
    D = (moe_layer_desc * n)(*descs)
    IO = (moe_layer_io * n)(*ios)
    _check("moe_decode_stack_prepare",
           load().moe_decode_stack_prepare(D, IO, n, T, _ptr(plan), plan_bytes, _ptr(ws), ws_bytes,
                                           _stream(stream)))


def moe_decode_stack_prepare_routed(descs, ios, router_w, T, plan, plan_bytes, ws, ws_bytes,
                                    stream=None):
    """router_w: sequence of device tensors (or pointers), one [E][H] bf16 per layer."""
    n = len(descs)
    D = (moe_layer_desc * n)(*descs)
    IO = (moe_layer_io * n)(*ios)
    W = (ctypes.c_void_p * n)(*[_ptr(w) for w in router_w])
    _check("moe_decode_stack_prepare_routed",
           load().moe_decode_stack_prepare_routed(D, IO, W, n, T, _ptr(plan), plan_bytes, _ptr(ws),
                                                  ws_bytes, _stream(stream)))


def moe_decode_stack(plan, n_layers, T, ws, ws_bytes, stream=None):
    _check("moe_decode_stack",
           load().moe_decode_stack(_ptr(plan), n_layers, T, _ptr(ws), ws_bytes, _stream(stream)))


def moe_workspace_bytes(desc, T) -> int:
    return int(load().moe_workspace_bytes(ctypes.byref(desc), T))


def moe_workspace_init(ws, ws_bytes, stream=None):
    _check("moe_workspace_init", load().moe_workspace_init(_ptr(ws), ws_bytes, _stream(stream)))


def moe_read_status(ws, stream=None):
    """-> (moe_status code, raw device status bits). Synchronises the stream."""
    out = ctypes.c_int32(0)
    code = load().moe_read_status(_ptr(ws), _stream(stream), ctypes.byref(out))
    if code == MOE_ERR_CUDA:
        _check("moe_read_status", code)
    return code, int(out.value)


def moe_last_launch_count() -> int:
    return int(load().moe_last_launch_count())


def moe_profile_enable(max_launches: int):
    _check("moe_profile_enable", load().moe_profile_enable(int(max_launches)))


def moe_profile_collect():
    _check("moe_profile_collect", load().moe_profile_collect())


def moe_profile_forget():
    _check("moe_profile_forget", load().moe_profile_forget())


def moe_profile_totals() -> dict:
    """{kernel kind name: (total ms, launches)} of the timing collected so far."""
    L = load()
    out = {}
    kind = 0
    while True:
        name = L.moe_profile_kind_name(kind).decode()
        if not name:
            return out
        ms, n = ctypes.c_double(0), ctypes.c_int64(0)
        _check("moe_profile_totals", L.moe_profile_totals(kind, ctypes.byref(ms), ctypes.byref(n)))
        out[name] = (ms.value, n.value)
        kind += 1
