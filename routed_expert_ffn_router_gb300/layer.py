"""A thin owner of one layer's device buffers around the C ABI.

`MoeLayer` keeps a layer's weight pool (torch tensors on the GPU), its
`moe_layer_desc` and a workspace, and forwards calls to libmoe_gb300.so. It
does marshalling only: routing, permutation, dequantisation, the FFN and the
combine all run in the library's kernels.
"""
from __future__ import annotations

import torch

from . import _lib
from ._lib import MOE_BF16, MOE_F32, moe_layer_desc, moe_qmat


def _qm(q, s):
    return moe_qmat(q.data_ptr(), s.data_ptr())


def make_desc(inp) -> moe_layer_desc:
    """moe_layer_desc over the (device) pool tensors of a synth.LayerInputs."""
    cfg = inp.cfg
    d = moe_layer_desc()
    d.H, d.I, d.E, d.k, d.S = cfg.H, cfg.I, cfg.E, cfg.k, inp.S
    d.gate = _qm(inp.gate_q, inp.gate_s)
    d.up = _qm(inp.up_q, inp.up_s)
    d.down = _qm(inp.down_q, inp.down_s)
    if inp.sh is not None:
        d.shared_I = cfg.shared_I
        d.shared_gate = _qm(inp.sh["gate_q"], inp.sh["gate_s"])
        d.shared_up = _qm(inp.sh["up_q"], inp.sh["up_s"])
        d.shared_down = _qm(inp.sh["down_q"], inp.sh["down_s"])
    else:
        d.shared_I = 0
    return d


class MoeLayer:
    def __init__(self, inp, T_max: int, device="cuda"):
        self.inp = inp
        self.cfg = inp.cfg
        self.device = torch.device(device)
        self.desc = make_desc(inp)
        self.T_max = T_max
        self.ws_bytes = _lib.moe_workspace_bytes(self.desc, T_max)
        if self.ws_bytes == 0:
            raise ValueError("invalid layer description")
        self.ws = torch.empty(self.ws_bytes + 256, dtype=torch.uint8, device=self.device)
        off = (-self.ws.data_ptr()) % 256
        self.ws_ptr = self.ws.data_ptr() + off
        _lib.moe_workspace_init(self.ws_ptr, self.ws_bytes)
        self.x_dtype = MOE_BF16 if inp.x_is_bf16 else MOE_F32

    def alloc_outputs(self, T: int):
        cfg, dev = self.cfg, self.device
        return dict(
            y=torch.empty(T, cfg.H, dtype=torch.float32, device=dev),
            ids=torch.empty(T, cfg.k, dtype=torch.int32, device=dev),
            w=torch.empty(T, cfg.k, dtype=torch.float32, device=dev),
            miss_ids=torch.empty(cfg.E, dtype=torch.int32, device=dev),
            n_miss=torch.zeros(1, dtype=torch.int32, device=dev))

    def forward(self, logits, x, slot_map="default", out=None, stream=None):
        """route + expert FFN; returns the output dict (y, ids, w, miss_ids, n_miss)."""
        T = x.shape[0]
        assert T <= self.T_max
        out = self.alloc_outputs(T) if out is None else out
        sm = self.inp.slot_map if isinstance(slot_map, str) else slot_map
        _lib.moe_layer_forward(self.desc, logits, x, self.x_dtype, T, sm, out["y"], out["ids"],
                               out["w"], out["miss_ids"], out["n_miss"], self.ws_ptr,
                               self.ws_bytes, stream)
        return out

    def expert_ffn(self, x, ids, w, slot_map="default", out=None, stream=None):
        T = x.shape[0]
        assert T <= self.T_max
        out = self.alloc_outputs(T) if out is None else out
        sm = self.inp.slot_map if isinstance(slot_map, str) else slot_map
        _lib.moe_expert_ffn(self.desc, x, self.x_dtype, T, ids, w, sm, out["y"], out["miss_ids"],
                            out["n_miss"], self.ws_ptr, self.ws_bytes, stream)
        return out

    def status(self, stream=None):
        return _lib.moe_read_status(self.ws_ptr, stream)

    def clear_status(self, stream=None):
        _lib.moe_workspace_init(self.ws_ptr, self.ws_bytes, stream)


class DecodeStack:
    """Several layers' decode windows in one launch (moe_decode_stack): one
    workspace shared by the layers, a device plan of their kernel arguments
    and each layer's output buffers. Marshalling only.

    Unchained (router_w None): each layer routes the given logits[l] and runs
    on the given xs[l]. Chained (router_w: one [E][H] bf16 tensor per layer):
    the launch computes each layer's logits from its input into self.logits[l]
    and writes layer l + 1's input bf16(x_l + y_l) into self.xs[l + 1];
    xs[0] is the caller's input."""

    def __init__(self, layers, logits, xs, T: int, slot_maps=None, router_w=None, device="cuda"):
        self.device = torch.device(device)
        self.T = T
        self.L = len(layers)
        self.inps = list(layers)
        self.descs = [make_desc(inp) for inp in layers]
        self.router_w = None if router_w is None else list(router_w)
        if self.router_w is None:
            self.logits = list(logits)
            self.xs = list(xs)
        else:
            self.logits = [torch.empty(T, inp.cfg.E, dtype=torch.float32, device=self.device)
                           for inp in layers]
            H = layers[0].cfg.H
            self.xs = [xs[0]] + [torch.empty(T, H, dtype=torch.int16, device=self.device)
                                 for _ in range(self.L - 1)]
        # each layer's slot map (its LayerInputs' own unless given; None = all held)
        self.slot_maps = ([inp.slot_map for inp in layers] if slot_maps is None
                          else list(slot_maps))
        self.ws_bytes = max(_lib.moe_workspace_bytes(d, T) for d in self.descs)
        if self.ws_bytes == 0:
            raise ValueError("invalid layer description")
        self.ws = torch.empty(self.ws_bytes + 256, dtype=torch.uint8, device=self.device)
        self.ws_ptr = self.ws.data_ptr() + (-self.ws.data_ptr()) % 256
        _lib.moe_workspace_init(self.ws_ptr, self.ws_bytes)
        self.outs = []
        for inp in layers:
            cfg = inp.cfg
            self.outs.append(dict(
                y=torch.empty(T, cfg.H, dtype=torch.float32, device=self.device),
                ids=torch.empty(T, cfg.k, dtype=torch.int32, device=self.device),
                w=torch.empty(T, cfg.k, dtype=torch.float32, device=self.device),
                miss_ids=torch.empty(cfg.E, dtype=torch.int32, device=self.device),
                n_miss=torch.zeros(1, dtype=torch.int32, device=self.device)))
        ios = []
        for l in range(self.L):
            o = self.outs[l]
            sm = self.slot_maps[l]
            ios.append(_lib.moe_layer_io(self.logits[l].data_ptr(), self.xs[l].data_ptr(),
                                         None if sm is None else sm.data_ptr(), o["y"].data_ptr(),
                                         o["ids"].data_ptr(), o["w"].data_ptr(),
                                         o["miss_ids"].data_ptr(), o["n_miss"].data_ptr()))
        self.plan_bytes = _lib.moe_decode_stack_plan_bytes(self.L)
        if self.plan_bytes == 0:
            raise ValueError("unsupported number of layers")
        self.plan = torch.empty(self.plan_bytes + 64, dtype=torch.uint8, device=self.device)
        self.plan_ptr = self.plan.data_ptr() + (-self.plan.data_ptr()) % 64
        if self.router_w is None:
            _lib.moe_decode_stack_prepare(self.descs, ios, T, self.plan_ptr, self.plan_bytes,
                                          self.ws_ptr, self.ws_bytes)
        else:
            _lib.moe_decode_stack_prepare_routed(self.descs, ios, self.router_w, T, self.plan_ptr,
                                                 self.plan_bytes, self.ws_ptr, self.ws_bytes)

    def forward(self, stream=None):
        _lib.moe_decode_stack(self.plan_ptr, self.L, self.T, self.ws_ptr, self.ws_bytes, stream)
        return self.outs

    def status(self, stream=None):
        return _lib.moe_read_status(self.ws_ptr, stream)
