"""The C-ABI library loads, exports every entry point of include/moe.h, and
rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

from routed_expert_ffn_router_gb300 import _lib
from routed_expert_ffn_router_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return _lib.load()


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), f"{n} declared in moe.h but not exported"
    assert set(names) == set(_lib.EXPORTS)


def test_status_strings(lib):
    for code in range(7):
        assert _lib.status_str(code)
    assert _lib.status_str(99) == "unknown status"


def _desc(H=256, I=128, E=8, k=2, S=8, shared_I=0, ptr=4096):
    d = _lib.moe_layer_desc()
    d.H, d.I, d.E, d.k, d.S, d.shared_I = H, I, E, k, S, shared_I
    for f in ("gate", "up", "down", "shared_gate", "shared_up", "shared_down"):
        setattr(d, f, _lib.moe_qmat(ptr, ptr))
    return d


@pytest.mark.parametrize("kw,code", [
    (dict(E=0), _lib.MOE_ERR_INVALID),
    (dict(E=1025, k=2), _lib.MOE_ERR_UNSUPPORTED),
    (dict(k=33, E=64), _lib.MOE_ERR_UNSUPPORTED),
    (dict(k=9, E=8), _lib.MOE_ERR_UNSUPPORTED),
    (dict(H=200), _lib.MOE_ERR_UNSUPPORTED),
    (dict(I=64), _lib.MOE_ERR_INVALID),
    (dict(S=0), _lib.MOE_ERR_INVALID),
    (dict(ptr=4097), _lib.MOE_ERR_INVALID),
    (dict(ptr=0), _lib.MOE_ERR_INVALID),
    (dict(shared_I=96), _lib.MOE_ERR_UNSUPPORTED),
])
def test_desc_validation(lib, kw, code):
    d = _desc(**kw)
    assert lib.moe_workspace_bytes(ctypes.byref(d), 4) == 0
    rc = lib.moe_expert_ffn(ctypes.byref(d), 4096, 1, 4, 4096, 4096, None, 4096, 4096, 4096, 4096,
                            1 << 30, None)
    assert rc == code


def test_workspace_checks(lib):
    d = _desc()
    need = lib.moe_workspace_bytes(ctypes.byref(d), 4)
    assert need > 0
    assert lib.moe_workspace_bytes(ctypes.byref(d), 64) > need
    # too small, misaligned, null
    assert lib.moe_expert_ffn(ctypes.byref(d), 4096, 1, 4, 4096, 4096, None, 4096, 4096, 4096, 4096,
                              need - 1, None) == _lib.MOE_ERR_WORKSPACE
    assert lib.moe_expert_ffn(ctypes.byref(d), 4096, 1, 4, 4096, 4096, None, 4096, 4096, 4096,
                              4096 + 16, need, None) == _lib.MOE_ERR_WORKSPACE
    assert lib.moe_expert_ffn(ctypes.byref(d), 4096, 1, 4, 4096, 4096, None, 4096, 4096, 4096, None,
                              need, None) == _lib.MOE_ERR_WORKSPACE
    # a bad dtype, a negative T, missing miss-list buffers
    assert lib.moe_expert_ffn(ctypes.byref(d), 4096, 7, 4, 4096, 4096, None, 4096, 4096, 4096, 4096,
                              need, None) == _lib.MOE_ERR_INVALID
    assert lib.moe_expert_ffn(ctypes.byref(d), 4096, 1, -1, 4096, 4096, None, 4096, 4096, 4096, 4096,
                              need, None) == _lib.MOE_ERR_INVALID
    assert lib.moe_expert_ffn(ctypes.byref(d), 4096, 1, 4, 4096, 4096, None, 4096, None, 4096, 4096,
                              need, None) == _lib.MOE_ERR_INVALID


def test_route_and_permute_validation(lib):
    assert lib.moe_route(4096, 4, 0, 1, 4096, 4096, None, None) == _lib.MOE_ERR_INVALID
    assert lib.moe_route(4096, 4, 8, 9, 4096, 4096, None, None) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_route(4096, -1, 8, 2, 4096, 4096, None, None) == _lib.MOE_ERR_INVALID
    assert lib.moe_route(None, 4, 8, 2, 4096, 4096, None, None) == _lib.MOE_ERR_INVALID
    assert lib.moe_route(None, 0, 8, 2, None, None, None, None) == _lib.MOE_OK  # T = 0: no-op
    assert lib.moe_permute(4096, 4, 8, 2, None, 0, 4096, 4096, 4096, 4096, 4096, 4096, 1 << 20,
                           None) == _lib.MOE_ERR_INVALID
    assert lib.moe_permute(4096, 4, 8, 2, None, 8, 4096, 4096, 4096, 4096, 4096, None, 1 << 20,
                           None) == _lib.MOE_ERR_WORKSPACE


def test_workspace_grows_with_T(lib):
    d = _desc(H=2048, I=768, E=128, k=8, S=128, shared_I=768)
    prev = 0
    for T in (0, 1, 8, 16, 64, 2048):
        n = lib.moe_workspace_bytes(ctypes.byref(d), T)
        assert n >= prev and n % 256 == 0
        prev = n


def test_static_entry_point_host_checks(lib):
    # the fixed-scratch entry point refuses, before touching the device, a
    # layer whose workspace exceeds its 16 MiB array, and reports bad
    # descriptions like the workspace entry point does
    big = _desc(H=2048, I=512, E=512, k=10, S=512, shared_I=512)
    assert lib.moe_workspace_bytes(ctypes.byref(big), 2048) > (16 << 20)
    assert lib.moe_expert_ffn_static(ctypes.byref(big), 4096, 1, 2048, 4096, 4096, None, 4096,
                                     4096, 4096, None) == _lib.MOE_ERR_UNSUPPORTED
    for kw, code in ((dict(E=0), _lib.MOE_ERR_INVALID), (dict(H=200), _lib.MOE_ERR_UNSUPPORTED),
                     (dict(ptr=4097), _lib.MOE_ERR_INVALID)):
        d = _desc(**kw)
        assert lib.moe_expert_ffn_static(ctypes.byref(d), 4096, 1, 4, 4096, 4096, None, 4096,
                                         4096, 4096, None) == code
    d = _desc()
    assert lib.moe_expert_ffn_static(ctypes.byref(d), 4096, 1, -1, 4096, 4096, None, 4096, 4096,
                                     4096, None) == _lib.MOE_ERR_INVALID


@pytest.mark.parametrize("entry", ["moe_expert_ffn", "moe_layer_forward"])
def test_separate_path_h_limit_is_reported_before_any_launch(lib, entry):
    # T <= 16 with H = 12288 (> 8192) cannot take the one-launch decode kernel
    # and is no prefill chunk: the separate-kernel path would need more than
    # 227 KB of shared memory per CTA, so the call is refused up front
    d = _desc(H=12288, I=128, E=8, k=2, S=8)
    need = lib.moe_workspace_bytes(ctypes.byref(d), 4)
    assert need > 0
    if entry == "moe_expert_ffn":
        rc = lib.moe_expert_ffn(ctypes.byref(d), 4096, 1, 4, 4096, 4096, None, 4096, 4096, 4096,
                                4096, need, None)
    else:
        rc = lib.moe_layer_forward(ctypes.byref(d), 4096, 4096, 1, 4, None, 4096, 4096, 4096, 4096,
                                   4096, 4096, need, None)
    assert rc == _lib.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("entry", ["moe_expert_ffn", "moe_layer_forward"])
@pytest.mark.parametrize("kw,T,dtype", [
    (dict(), 70000, 1),                                    # rows beyond a grid dimension
    (dict(E=1024, k=32, S=1024), 65535, 0),                # fp32 x: too many 16-row work units
])
def test_row_and_unit_limits_are_reported_before_any_launch(lib, entry, kw, T, dtype):
    d = _desc(**kw)
    need = lib.moe_workspace_bytes(ctypes.byref(d), T)
    assert need > 0
    if entry == "moe_expert_ffn":
        rc = lib.moe_expert_ffn(ctypes.byref(d), 4096, dtype, T, 4096, 4096, None, 4096, 4096,
                                4096, 4096, need, None)
    else:
        rc = lib.moe_layer_forward(ctypes.byref(d), 4096, 4096, dtype, T, None, 4096, 4096, 4096,
                                   4096, 4096, 4096, need, None)
    assert rc == _lib.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("T", [4, 20])
def test_layer_forward_checks_x_and_y_before_routing(lib, T):
    # a missing or misaligned activation or output is reported before the
    # routing launch, on the decode and the chunk paths alike
    d = _desc()
    need = lib.moe_workspace_bytes(ctypes.byref(d), T)
    for x, y in ((None, 4096), (4096, None), (4104, 4096), (4096, 4104)):
        rc = lib.moe_layer_forward(ctypes.byref(d), 4096, x, 1, T, None, y, 4096, 4096, 4096, 4096,
                                   4096, need, None)
        assert rc == _lib.MOE_ERR_INVALID, (x, y)


def test_pair_and_logit_counts_beyond_int32_are_refused(lib):
    T = 1 << 26  # T * k = 2^31 pairs at k = 32
    d = _desc(E=64, k=32, S=64)
    assert lib.moe_workspace_bytes(ctypes.byref(d), T) == 0
    assert lib.moe_permute(4096, T, 64, 32, None, 64, 4096, 4096, 4096, 4096, 4096, 4096, 1 << 40,
                           None) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_expert_ffn(ctypes.byref(d), 4096, 1, T, 4096, 4096, None, 4096, 4096, 4096,
                              4096, 1 << 40, None) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_layer_forward(ctypes.byref(d), 4096, 4096, 1, T, None, 4096, 4096, 4096, 4096,
                                 4096, 4096, 1 << 40, None) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_expert_ffn_static(ctypes.byref(d), 4096, 1, T, 4096, 4096, None, 4096, 4096,
                                     4096, None) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_router_logits(4096, 0, 4096, 1 << 22, 128, 1024, 4096,
                                 None) == _lib.MOE_ERR_UNSUPPORTED


def test_decode_stack_host_checks(lib):
    # the plan size covers 1 .. 124 layers (the cross-CTA counters of each
    # layer have a cache line of their own in the workspace head)
    assert lib.moe_decode_stack_plan_bytes(0) == 0
    assert lib.moe_decode_stack_plan_bytes(125) == 0
    one = lib.moe_decode_stack_plan_bytes(1)
    assert one > 0 and one % 64 == 0
    assert lib.moe_decode_stack_plan_bytes(48) == 48 * one
    d = (_lib.moe_layer_desc * 2)(_desc(), _desc())
    io = (_lib.moe_layer_io * 2)(_lib.moe_layer_io(*([4096] * 8)), _lib.moe_layer_io(*([4096] * 8)))
    ws = 1 << 20
    # argument errors return before anything touches the device
    assert lib.moe_decode_stack_prepare(None, io, 2, 4, 4096, one * 2, ws, 1 << 20, None) == _lib.MOE_ERR_INVALID
    assert lib.moe_decode_stack_prepare(d, None, 2, 4, 4096, one * 2, ws, 1 << 20, None) == _lib.MOE_ERR_INVALID
    assert lib.moe_decode_stack_prepare(d, io, 0, 4, 4096, one * 2, ws, 1 << 20, None) == _lib.MOE_ERR_INVALID
    assert lib.moe_decode_stack_prepare(d, io, 2, 0, 4096, one * 2, ws, 1 << 20, None) == _lib.MOE_ERR_INVALID
    assert lib.moe_decode_stack_prepare(d, io, 125, 4, 4096, one * 125, ws, 1 << 20, None) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_decode_stack_prepare(d, io, 2, 4, 4096, one, ws, 1 << 20, None) == _lib.MOE_ERR_INVALID
    assert lib.moe_decode_stack_prepare(d, io, 2, 4, 4096 + 32, one * 2, ws, 1 << 20, None) == _lib.MOE_ERR_INVALID
    assert lib.moe_decode_stack(None, 2, 4, ws, 1 << 20, None) == _lib.MOE_ERR_INVALID
    assert lib.moe_decode_stack(4096, 2, 17, ws, 1 << 20, None) == _lib.MOE_ERR_INVALID
    assert lib.moe_decode_stack(4096, 125, 4, ws, 1 << 20, None) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_decode_stack(4096, 2, 4, ws + 8, 1 << 20, None) == _lib.MOE_ERR_WORKSPACE
    assert lib.moe_decode_stack(4096, 2, 4, ws, 1024, None) == _lib.MOE_ERR_WORKSPACE
