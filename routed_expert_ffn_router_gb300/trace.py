"""Routing traces (libmoe_gb300.so, moe_trace_*): dump a layer's routing as the
pages' trace records and read them back. Marshalling only."""
from __future__ import annotations

import ctypes

import numpy as np

from . import _lib


def encode(layer: int, ids, w=None) -> bytes:
    """Records of one layer's tokens; ids/w: host arrays [T][k] (w None: weights 0)."""
    L = _lib.load()
    a = np.ascontiguousarray(np.asarray(ids, np.int32))
    T, k = a.shape
    wp = None
    if w is not None:
        wa = np.ascontiguousarray(np.asarray(w, np.float32))
        assert wa.shape == a.shape
        wp = wa.ctypes.data
    n = L.moe_trace_write(layer, a.ctypes.data, wp, T, k, None, 0)
    if n < 0:
        raise ValueError("invalid routing")
    buf = (ctypes.c_uint8 * max(n, 1))()
    if L.moe_trace_write(layer, a.ctypes.data, wp, T, k, buf, n) != n:
        raise ValueError("trace write failed")
    return bytes(buf)[:n]


def decode(data: bytes, k_max: int = 32):
    """-> (layer [R], k [R], ids [R][k_max], w [R][k_max]) of every record."""
    L = _lib.load()
    src = (ctypes.c_uint8 * max(len(data), 1)).from_buffer_copy(data or b"\0")
    R = L.moe_trace_read(src, len(data), None, None, None, None, k_max, 0)
    if R < 0:
        raise ValueError("malformed routing trace")
    layer = np.empty(R, np.int32)
    kk = np.empty(R, np.int32)
    ids = np.empty((R, k_max), np.int32)
    w = np.empty((R, k_max), np.float32)
    if R and L.moe_trace_read(src, len(data), layer.ctypes.data, kk.ctypes.data, ids.ctypes.data,
                              w.ctypes.data, k_max, R) != R:
        raise ValueError("malformed routing trace")
    return layer, kk, ids, w
