"""The adaptive expert cache's host planner (libmoe_gb300.so, moe_cache_*).

`ExpertCache` owns the planner's host state buffer and marshals arguments; the
rules (heat with a half-life, fill and swap rounds, the hysteresis, the STRP
profile) run in the library. Each move it returns says: copy expert
`expert_in`'s codes and scales into pool slot `slot` of `layer` (evicting
`expert_out`, or -1 for a free slot), then use `slot_map(layer)` for the layer.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _lib
from ._lib import moe_cache_params, moe_cache_swap

# the values of the adaptive cache described by the pages
DEFAULTS = dict(half_life_tokens=350.0, round_every_tokens=32, max_swaps=64, fill_every_tokens=8,
                max_fills=128, in_ratio=1.5, in_picks=2.0, max_window_tokens=32)


def make_params(n_layers: int, n_experts: int, **kw) -> moe_cache_params:
    v = dict(DEFAULTS)
    v.update(kw)
    p = moe_cache_params()
    p.n_layers, p.n_experts = n_layers, n_experts
    for k, x in v.items():
        setattr(p, k, x)
    return p


class ExpertCache:
    def __init__(self, n_layers: int, n_experts: int, slots, **params):
        self.L = _lib.load()
        self.p = make_params(n_layers, n_experts, **params)
        self.slots = np.ascontiguousarray(np.broadcast_to(np.asarray(slots, np.int32), (n_layers,)))
        n = self.L.moe_cache_state_bytes(ctypes.byref(self.p), self.slots.ctypes.data)
        if n == 0:
            raise ValueError("invalid cache parameters or slot counts")
        self.state = np.zeros((n + 7) // 8, np.float64)  # 8-byte aligned host buffer
        _lib._check("moe_cache_init", self.L.moe_cache_init(self.state.ctypes.data, self.state.nbytes,
                                                          ctypes.byref(self.p), self.slots.ctypes.data))
        self.n_max = self.p.max_fills + self.p.max_swaps
        self._moves = (moe_cache_swap * max(self.n_max, 1))()

    def _st(self):
        return self.state.ctypes.data

    def set_resident(self, layer: int, experts):
        e = np.ascontiguousarray(np.asarray(experts, np.int32))
        _lib._check("moe_cache_set_resident",
                    self.L.moe_cache_set_resident(self._st(), layer, e.ctypes.data, len(e)))

    def observe(self, layer: int, ids):
        """One window's routing ids [T][k] (host) of one layer."""
        a = np.ascontiguousarray(np.asarray(ids, np.int32))
        T, k = a.shape
        _lib._check("moe_cache_observe", self.L.moe_cache_observe(self._st(), layer, a.ctypes.data, T, k))

    def observe_layers(self, ids):
        """One window's routing ids [n_layers][T][k] (host) of every layer."""
        a = np.ascontiguousarray(np.asarray(ids, np.int32))
        Ln, T, k = a.shape
        if Ln != self.p.n_layers:
            raise ValueError("ids must hold every layer")
        _lib._check("moe_cache_observe_layers",
                    self.L.moe_cache_observe_layers(self._st(), a.ctypes.data, T, k))

    def observe_counts(self, counts):
        """Picks counted elsewhere, host int32 [n_layers][E]."""
        a = np.ascontiguousarray(np.asarray(counts, np.int32))
        if a.shape != (self.p.n_layers, self.p.n_experts):
            raise ValueError("counts must be [n_layers][n_experts]")
        _lib._check("moe_cache_observe_counts", self.L.moe_cache_observe_counts(self._st(), a.ctypes.data))

    def observe_device(self, counts, stream=None):
        """The device pick counters (a device int32 tensor [n_layers][E], one
        layer's row per moe_layer_desc.pick_counts): read, cleared and added."""
        if tuple(counts.shape) != (self.p.n_layers, self.p.n_experts) or not counts.is_contiguous():
            raise ValueError("counts must be a contiguous [n_layers][n_experts] tensor")
        _lib._check("moe_cache_observe_device", self.L.moe_cache_observe_device(
            self._st(), ctypes.c_void_p(counts.data_ptr()), _lib._stream(stream)))

    def _out(self, n):
        if n < 0:
            raise _lib.MoeError("moe_cache", _lib.MOE_ERR_INVALID, "invalid argument")
        return [(m.layer, m.slot, m.expert_in, m.expert_out) for m in self._moves[:n]]

    def advance(self, n_tokens: int):
        """-> the moves of the rounds that came due (list of (layer, slot, in, out))."""
        return self._out(self.L.moe_cache_advance(self._st(), n_tokens, self._moves, self.n_max))

    def rebalance(self, max_swaps: int | None = None):
        m = self.p.max_swaps if max_swaps is None else max_swaps
        buf = (moe_cache_swap * max(m, 1))()
        n = self.L.moe_cache_rebalance(self._st(), m, buf, m)
        if n < 0:
            raise _lib.MoeError("moe_cache_rebalance", _lib.MOE_ERR_INVALID, "invalid argument")
        return [(x.layer, x.slot, x.expert_in, x.expert_out) for x in buf[:n]]

    def slot_map(self, layer: int) -> np.ndarray:
        out = np.empty(self.p.n_experts, np.int32)
        _lib._check("moe_cache_slot_map", self.L.moe_cache_slot_map(self._st(), layer, out.ctypes.data))
        return out

    def heat(self, layer: int) -> np.ndarray:
        out = np.empty(self.p.n_experts, np.float64)
        _lib._check("moe_cache_heat", self.L.moe_cache_heat(self._st(), layer, out.ctypes.data))
        return out

    def swapped_total(self) -> int:
        return int(self.L.moe_cache_swapped_total(self._st()))

    def profile_bytes(self) -> bytes:
        n = self.L.moe_cache_profile_write(self._st(), None, 0)
        buf = (ctypes.c_uint8 * n)()
        if self.L.moe_cache_profile_write(self._st(), buf, n) != n:
            raise _lib.MoeError("moe_cache_profile_write", _lib.MOE_ERR_INVALID, "write failed")
        return bytes(buf)

    def load_profile(self, data: bytes):
        buf = (ctypes.c_uint8 * len(data)).from_buffer_copy(data)
        _lib._check("moe_cache_profile_load", self.L.moe_cache_profile_load(self._st(), buf, len(data)))


POOL_TENSORS = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")


def copy_moves(pool, store, moves, layer=0):
    """Apply a round's moves of one layer: expert `expert_in`'s codes and scales
    from `store` (any object with the six [E][...] tensors gate_q ... down_s, e.g.
    pinned host memory) into slot `slot` of `pool` (the same six tensors with S
    slots, e.g. the device pool a layer reads). Copies are issued on the
    current stream; call between windows, then upload the layer's slot map."""
    for m_layer, slot, e_in, _ in moves:
        if m_layer != layer:
            continue
        for name in POOL_TENSORS:
            getattr(pool, name)[slot].copy_(getattr(store, name)[e_in], non_blocking=True)
