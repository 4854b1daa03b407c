"""Python face of the CPU oracle (moe_oracle.c).

TEST INFRASTRUCTURE ONLY: tests/, the smoke check and the CPU-baseline leg of
bench.py may import this package; the library package must not. The oracle is
plain single-threaded float64 C; this module only builds it and marshals numpy
arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no fused multiply-add)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
                               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class OrcLayer(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("S", ctypes.c_int32), ("shared_I", ctypes.c_int32)] + [
        (n, ctypes.c_void_p) for n in ("gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s",
                                       "sh_gate_q", "sh_up_q", "sh_down_q",
                                       "sh_gate_s", "sh_up_s", "sh_down_s")]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32 = ctypes.c_int
            L.orc_half_to_double.argtypes = [ctypes.c_uint16]
            L.orc_half_to_double.restype = ctypes.c_double
            L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.orc_bf16_to_double.restype = ctypes.c_double
            L.orc_weight.argtypes = [P, P, i32, i32, i32]
            L.orc_weight.restype = ctypes.c_double
            L.orc_router_logits.argtypes = [P, P, i32, i32, i32, P]
            L.orc_router_logits.restype = None
            L.orc_route.argtypes = [P, i32, i32, i32, P, P, P]
            L.orc_route.restype = i32
            L.orc_permute.argtypes = [P, i32, i32, i32, P, P, P, P, P, P]
            L.orc_permute.restype = i32
            L.orc_expert_h.argtypes = [ctypes.POINTER(OrcLayer), P, i32, i32, i32, P]
            L.orc_expert_h.restype = None
            L.orc_layer_rows.argtypes = [ctypes.POINTER(OrcLayer), P, i32, P, P, P, i32, P, P]
            L.orc_layer_rows.restype = i32
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _np(t, dtype=None):
    """torch tensor or array -> contiguous numpy array on the host."""
    if t is None:
        return None
    if hasattr(t, "detach"):
        t = t.detach().cpu().numpy()
    a = np.ascontiguousarray(t)
    return a if dtype is None else np.ascontiguousarray(a.view(dtype) if a.dtype.itemsize ==
                                                        np.dtype(dtype).itemsize else a.astype(dtype))


# ---------------------------------------------------------------------------
def half_to_double(bits: int) -> float:
    return lib().orc_half_to_double(int(bits) & 0xFFFF)


def bf16_to_double(bits: int) -> float:
    return lib().orc_bf16_to_double(int(bits) & 0xFFFF)


def weight(q, s, K: int, r: int, c: int) -> float:
    q = _np(q, np.uint8)
    s = _np(s, np.uint16)
    return lib().orc_weight(_p(q), _p(s), K, r, c)


def router_logits(x, wg):
    x = _np(x, np.float32)
    wg = _np(wg, np.float32)
    T, H = x.shape
    E = wg.shape[1]
    out = np.empty((T, E), np.float32)
    lib().orc_router_logits(_p(x), _p(wg), T, H, E, _p(out))
    return out


def route(logits, k: int):
    """-> ids int32 [T,k], w float32 [T,k], w_exact float64 [T,k]."""
    lg = _np(logits, np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    we = np.empty((T, k), np.float64)
    rc = lib().orc_route(_p(lg), T, E, k, _p(ids), _p(w), _p(we))
    if rc != 0:
        raise ValueError(f"non-finite logit in row {rc - 1}")
    return ids, w, we


def permute(ids, E: int, slot_map=None):
    ids = _np(ids, np.int32)
    T, k = ids.shape
    P = T * k
    off = np.empty(E + 1, np.int32)
    sp = np.empty(max(P, 1), np.int32)
    pp = np.empty(max(P, 1), np.int32)
    miss = np.empty(E, np.int32)
    nm = np.zeros(1, np.int32)
    sm = _np(slot_map, np.int32)
    rc = lib().orc_permute(_p(ids), T, E, k, _p(sm), _p(off), _p(sp), _p(pp), _p(miss), _p(nm))
    if rc != 0:
        raise ValueError("expert id out of range")
    return dict(offsets=off, sorted_pair=sp[:P], pair_pos=pp[:P], miss_ids=miss[:nm[0]],
                n_miss=int(nm[0]))


class Layer:
    """Host copies of one layer's weight pool, viewed by the oracle."""

    def __init__(self, inp):
        cfg = inp.cfg
        self.cfg = cfg
        self.keep = {}
        names = ("gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s")
        arrs = {}
        for n in names:
            arrs[n] = _np(getattr(inp, n), np.uint8 if n.endswith("_q") else np.uint16)
        sh = {}
        if inp.sh is not None:
            for n in names:
                sh[n] = _np(inp.sh[n], np.uint8 if n.endswith("_q") else np.uint16)
        self.keep = dict(arrs)
        self.keep.update({"sh_" + n: v for n, v in sh.items()})
        st = OrcLayer(cfg.H, cfg.I, cfg.E, cfg.k, inp.S, cfg.shared_I if inp.sh is not None else 0)
        for n in names:
            setattr(st, n, _p(arrs[n]).value)
            if sh:
                setattr(st, "sh_" + n, _p(sh[n]).value)
        self.st = st
        self.x = _np(inp.x, np.uint16 if inp.x_is_bf16 else np.float32)
        self.x_is_bf16 = inp.x_is_bf16
        self.slot_map = _np(inp.slot_map, np.int32)

    def rows(self, ids, w, rows=None, slot_map="default", x=None):
        """y (float64 [len(rows), H]) for the listed rows (default: all)."""
        ids = _np(ids, np.int32)
        w = _np(w, np.float32)
        T = ids.shape[0]
        rows = np.arange(T, dtype=np.int32) if rows is None else np.asarray(rows, np.int32)
        sm = self.slot_map if isinstance(slot_map, str) else _np(slot_map, np.int32)
        xx = self.x if x is None else x
        y = np.empty((len(rows), self.cfg.H), np.float64)
        rc = lib().orc_layer_rows(ctypes.byref(self.st), _p(xx), int(self.x_is_bf16), _p(ids),
                                  _p(w), _p(sm), len(rows), _p(rows), _p(y))
        if rc != 0:
            raise ValueError("slot out of range")
        return y

    def expert_h(self, t: int, slot: int):
        h = np.empty(self.cfg.I, np.float64)
        lib().orc_expert_h(ctypes.byref(self.st), _p(self.x), int(self.x_is_bf16), t, slot, _p(h))
        return h
