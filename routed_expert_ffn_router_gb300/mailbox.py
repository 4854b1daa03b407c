"""The mailbox (libmoe_gb300.so, moe_mailbox_*): the experts a layer's slot
map does not hold, computed by host threads from the host copy of every expert
and added to the layer output on the GPU in a fixed order.

`Mailbox` owns the library's thread pool and marshals arguments; the expert
arithmetic runs in the library (host code) and the sum in its kernel.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _lib
from .layer import make_desc


class Mailbox:
    def __init__(self, store, n_threads: int = 4, timeout_ms: int = 10000):
        """store: a layer's weights for every expert in HOST memory (the six
        [E][...] tensors gate_q ... down_s of a synth.LayerInputs), slot = id."""
        self.L = _lib.load()
        self.store = store
        self.cfg = store.cfg
        self.desc = make_desc(store)
        self.desc.S = self.cfg.E
        self.mb = self.L.moe_mailbox_create(int(n_threads), int(timeout_ms))
        if not self.mb:
            raise ValueError("invalid mailbox arguments")

    def close(self):
        if self.mb:
            self.L.moe_mailbox_destroy(self.mb)
            self.mb = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def pairs(self, ids, slot_map) -> np.ndarray:
        """Pairs p = t*k + j (ascending) whose expert the slot map does not hold."""
        ids = np.ascontiguousarray(np.asarray(ids, np.int32))
        sm = np.ascontiguousarray(np.asarray(slot_map, np.int32))
        T, k = ids.shape
        n = self.L.moe_mailbox_pairs(ids.ctypes.data, T, k, sm.ctypes.data, len(sm), None, 0)
        if n < 0:
            raise _lib.MoeError("moe_mailbox_pairs", _lib.MOE_ERR_INVALID, "invalid argument")
        out = np.empty(max(n, 1), np.int32)
        n2 = self.L.moe_mailbox_pairs(ids.ctypes.data, T, k, sm.ctypes.data, len(sm), out.ctypes.data, n)
        if n2 != n:
            raise _lib.MoeError("moe_mailbox_pairs", _lib.MOE_ERR_INVALID, "invalid argument")
        return out[:n]

    def compute(self, x, ids, w, pairs) -> np.ndarray:
        """partial [len(pairs)][H] fp32 (host) for the listed pairs."""
        cfg = self.cfg
        xh = x.contiguous() if isinstance(x, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(x))
        ids = np.ascontiguousarray(np.asarray(ids, np.int32))
        w = np.ascontiguousarray(np.asarray(w, np.float32))
        pairs = np.ascontiguousarray(np.asarray(pairs, np.int32))
        T = ids.shape[0]
        part = np.empty((max(len(pairs), 1), cfg.H), np.float32)
        dt = _lib.MOE_BF16 if cfg.x_dtype == "bf16" else _lib.MOE_F32
        _lib._check("moe_mailbox_compute", self.L.moe_mailbox_compute(
            self.mb, ctypes.byref(self.desc), ctypes.c_void_p(xh.data_ptr()), dt, T, ids.ctypes.data,
            w.ctypes.data, pairs.ctypes.data, len(pairs), part.ctypes.data))
        return part[:len(pairs)]

    def inject(self, mode: int):
        """Failure injection on the host: the next job stalls (1) or is lost (2)."""
        _lib._check("moe_mailbox_inject", self.L.moe_mailbox_inject(self.mb, int(mode)))

    @staticmethod
    def add(partial, pairs, T: int, k: int, y, stream=None):
        """y[t] += the partials of row t in list order (device tensors)."""
        n = int(pairs.numel())
        _lib._check("moe_mailbox_add", _lib.load().moe_mailbox_add(
            ctypes.c_void_p(partial.data_ptr() if n else 0), ctypes.c_void_p(pairs.data_ptr() if n else 0),
            n, T, k, y.shape[1], ctypes.c_void_p(y.data_ptr()), _lib._stream(stream)))

    def forward(self, lay, logits, x, slot_map, stream=None):
        """One window: the GPU layer call over the held experts, the missed
        experts on the host threads, their partials added on the GPU."""
        out = lay.forward(logits, x, slot_map=slot_map, stream=stream)
        st = torch.cuda.current_stream() if stream is None else stream
        st.synchronize()
        ids = out["ids"].cpu().numpy()
        pairs = self.pairs(ids, slot_map.cpu().numpy())
        if len(pairs):
            part = self.compute(x.cpu(), ids, out["w"].cpu().numpy(), pairs)
            dev = out["y"].device
            pd = torch.from_numpy(part).to(dev)
            qd = torch.from_numpy(pairs).to(dev)
            self.add(pd, qd, x.shape[0], self.cfg.k, out["y"], stream=stream)
        out["mailbox_pairs"] = pairs
        return out
