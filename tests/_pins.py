"""Independent checkers used to pin the oracle (tests only).

Everything here is written separately from oracle/moe_oracle.c, in a different
form: vectorised numpy dequantisation, a dense-then-mask evaluation of the whole
layer (every expert on every row, then masked by a dense routing matrix), silu
through tanh, hand-built identity-shaped weight pools.
"""
from __future__ import annotations

import os
import types

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line or "=" not in line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            nums = [float(v) for v in val.split()]
            out[key] = nums[0] if len(nums) == 1 else nums
    return out


def dequant_np(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """[..., rows, K/2] uint8 codes + [..., rows, K/32] fp16 bits -> float64 [..., rows, K]."""
    q = np.asarray(q, np.uint8)
    lo = (q & 0x0F).astype(np.int16)
    hi = (q >> 4).astype(np.int16)
    codes = np.stack([lo, hi], axis=-1).reshape(*q.shape[:-1], q.shape[-1] * 2)
    codes = np.where(codes >= 8, codes - 16, codes).astype(np.float64)
    scales = np.asarray(s).astype(np.uint16).view(np.float16).astype(np.float64)
    return codes * np.repeat(scales, 32, axis=-1)


def silu_tanh(z):
    return 0.5 * z * (1.0 + np.tanh(0.5 * z))


def x_float64(inp) -> np.ndarray:
    x = inp.x.detach().cpu().numpy()
    if inp.x_is_bf16:
        return (x.astype(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def dense_then_mask(inp, ids, w, slot_map="default"):
    """Every resident expert on every row, then y = R @ O with R the dense routing matrix."""
    cfg = inp.cfg
    x = x_float64(inp)
    T = x.shape[0]
    sm = inp.slot_map if isinstance(slot_map, str) else slot_map
    sm = None if sm is None else np.asarray(sm.cpu() if hasattr(sm, "cpu") else sm)
    R = np.zeros((T, cfg.E))
    for t in range(T):
        for j in range(cfg.k):
            e = int(ids[t, j])
            slot = e if sm is None else int(sm[e])
            if slot >= 0:
                R[t, e] = float(w[t, j])
    y = np.zeros((T, cfg.H))
    for e in range(cfg.E):
        slot = e if sm is None else int(sm[e])
        if slot < 0 or not R[:, e].any():
            # an expert no row selected contributes R[:, e] = 0; skip the product
            continue
        Wg = dequant_np(inp.gate_q[slot].numpy(), inp.gate_s[slot].numpy())
        Wu = dequant_np(inp.up_q[slot].numpy(), inp.up_s[slot].numpy())
        Wd = dequant_np(inp.down_q[slot].numpy(), inp.down_s[slot].numpy())
        O = (Wd @ (silu_tanh(Wg @ x.T) * (Wu @ x.T))).T  # [T, H] for every row
        y += R[:, e:e + 1] * O
    if inp.sh is not None:
        sh = {k: v.numpy() for k, v in inp.sh.items()}
        Wg = dequant_np(sh["gate_q"], sh["gate_s"])
        Wu = dequant_np(sh["up_q"], sh["up_s"])
        Wd = dequant_np(sh["down_q"], sh["down_s"])
        y += (Wd @ (silu_tanh(Wg @ x.T) * (Wu @ x.T))).T
    return y


# ---------------------------------------------------------------------------
# hand-built pools
# ---------------------------------------------------------------------------
def encode_codes(codes: np.ndarray) -> np.ndarray:
    """int codes in [-8, 7], [..., K] -> packed uint8 [..., K/2] (even column low)."""
    c = np.asarray(codes, np.int16) & 0xF
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def identity_pool(E, H, I, gate_mult, up_mult, down_mult, scale_bits=0x3C00):
    """gate/up/down = mult * Id (H = I), every fp16 scale the given bit pattern."""
    assert H == I
    eye = np.eye(H, dtype=np.int16)
    pool = {}
    for kind, mults, rows, K in (("gate", gate_mult, I, H), ("up", up_mult, I, H),
                                 ("down", down_mult, H, I)):
        pool[kind + "_q"] = torch.from_numpy(np.stack([encode_codes(m * eye) for m in mults]))
        pool[kind + "_s"] = torch.full((E, rows, K // 32), scale_bits, dtype=torch.int16)
    return pool


def fake_inputs(cfg, x_bits_or_f32, pool, S, sh=None, slot_map=None, logits=None):
    from routed_expert_ffn_router_gb300.synth import LayerInputs
    return LayerInputs(cfg=cfg, seed=0, logits=logits, x=x_bits_or_f32, wg=None,
                       rank=torch.arange(1, cfg.E + 1), slot_map=slot_map, S=S, sh=sh, **pool)


def as_namespace(**kw):
    return types.SimpleNamespace(**kw)
