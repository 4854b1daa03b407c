"""Seeded synthetic inputs for the routed-expert FFN of one MoE layer.

This module is the single source of input bytes for both the CUDA path and the
CPU oracle. It holds no arithmetic of the method itself (no routing, no
dequantisation, no FFN): it draws random numbers, encodes them into the stored
formats (bf16 activations, symmetric int4 blocks of 32 with an fp16 scale) and
lays them out in the weight-pool format both sides read.

Workload shapes follow the Strata pages: hidden 2048 ("split-serving", the
`n * 2048 f32 hidden rows` frame), 512 experts x 48 layers with top-10 routing
(SGLang port post, section 1), verify windows of at most 16 rows ("Windows of 16
rows"), 2,048-token prompt chunks ("PREFILL_HEAD_ALIAS"). Router logits carry a
per-expert Zipf popularity bias: a seeded permutation gives each expert a rank
r(e) in 1..E and the bias is -s*ln r(e), the log of the Zipf pmf up to a constant
that softmax ignores.

Weight-pool format (per matrix kind; rows x K with K the reduction length):
  q     uint8  [S][rows][K/2]   two int4 codes per byte, even column in the low
                                nibble, two's complement in [-8, 7]
  scale uint16 [S][rows][K/32]  IEEE binary16 bit pattern, one per 32 columns
gate/up: rows = I, K = H.   down: rows = H, K = I.   slot s holds one expert.

Random draws use torch generators (CPU for small cases, CUDA for the multi-GB
pools) so the same code serves both; a given (config, seed, device) is
reproducible. Order of draws: popularity permutation, logits noise, x, then the
expert weights slot by slot (gate, up, down), then the shared expert.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch


# --------------------------------------------------------------------------
# configurations
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class MoeConfig:
    name: str
    H: int            # hidden size
    I: int            # expert intermediate size
    E: int            # experts
    k: int            # top-k
    T: int            # rows in the window / chunk
    shared_I: int = 0  # intermediate of the always-on shared expert (0 = none)
    zipf_s: float = 0.0  # Zipf exponent of the logit popularity bias (0 = none)
    resident_frac: float = 1.0  # fraction of experts resident in the pool
    layers: int = 1
    x_dtype: str = "bf16"  # "f32" or "bf16"
    router_from_x: bool = False  # logits = x @ Wg (tiny case) instead of drawn
    w_std: float = 0.02
    wg_std: float = 0.05

    @property
    def pairs(self) -> int:
        return self.T * self.k

    @property
    def n_resident(self) -> int:
        # floor(frac * E + 0.5): round half up, 0.6 * 256 = 153.6 -> 154
        return int(math.floor(self.resident_frac * self.E + 0.5))

    def expert_bytes(self, inter: Optional[int] = None) -> int:
        inter = self.I if inter is None else inter
        return 3 * self.H * inter * 9 // 16  # 0.5 B code + 2/32 B scale per weight

    def with_T(self, T: int) -> "MoeConfig":
        return dataclasses.replace(self, T=T, name=f"{self.name}_T{T}")


TINY = MoeConfig("tiny", H=256, I=128, E=8, k=2, T=4, x_dtype="f32",
                 router_from_x=True)
DECODE_WINDOW = MoeConfig("decode_window", H=2048, I=768, E=128, k=8, T=8,
                          shared_I=768, zipf_s=1.1)
DECODE_48 = MoeConfig("decode48", H=2048, I=512, E=512, k=10, T=16,
                      zipf_s=1.0, layers=48)
EXPERT_CACHE = MoeConfig("expert_cache", H=4096, I=1536, E=256, k=8, T=16,
                         zipf_s=1.2, resident_frac=0.6)
PREFILL = MoeConfig("prefill", H=2048, I=512, E=512, k=10, T=2048,
                    shared_I=512, zipf_s=1.0)

CONFIGS = {c.name: c for c in (TINY, DECODE_WINDOW, DECODE_48, EXPERT_CACHE, PREFILL)}
DECODE48_WINDOWS = (1, 2, 4, 8, 16)


# --------------------------------------------------------------------------
# encodings (input preparation only; the path never quantises)
# --------------------------------------------------------------------------
def f32_to_bf16_bits(a: torch.Tensor) -> torch.Tensor:
    """fp32 -> bf16 bit pattern (uint16 stored in int16), round to nearest even."""
    return a.to(torch.bfloat16).view(torch.int16)


def quantize_int4_blocks(w: torch.Tensor):
    """Encode fp32 weights [rows, K] into int4 codes + fp16 scales (blocks of 32).

    Per block of 32 along K: amax = max|w|; scale = fp16_rne(amax / 7) with the
    division in fp32; code = clamp(round_half_even(w / float(scale)), -8, 7);
    an all-zero block gets scale 0 and codes 0.
    Returns (q uint8 [rows, K/2], scale_bits int16 [rows, K/32]).
    """
    rows, K = w.shape
    assert K % 32 == 0
    wb = w.reshape(rows, K // 32, 32).float()
    amax = wb.abs().amax(dim=2)
    scale_h = (amax / 7.0).to(torch.float16)
    sf = scale_h.float().unsqueeze(2)
    safe = torch.where(sf == 0, torch.ones_like(sf), sf)
    code = torch.round(wb / safe).clamp_(-8, 7)
    code = torch.where(sf == 0, torch.zeros_like(code), code)
    c = code.to(torch.int16).reshape(rows, K) & 0xF
    q = (c[:, 0::2] | (c[:, 1::2] << 4)).to(torch.uint8)
    return q, scale_h.view(torch.int16)


# --------------------------------------------------------------------------
# layer inputs
# --------------------------------------------------------------------------
@dataclasses.dataclass
class LayerInputs:
    cfg: MoeConfig
    seed: int
    logits: Optional[torch.Tensor]  # f32 [T, E] (None when the router runs from x)
    x: torch.Tensor                 # f32 [T, H] or bf16 bits int16 [T, H]
    wg: Optional[torch.Tensor]      # f32 [H, E] router weight (tiny case)
    rank: torch.Tensor              # int64 [E], popularity rank 1..E (1 = hottest)
    slot_map: Optional[torch.Tensor]  # int32 [E], -1 = not resident; None = identity
    S: int
    gate_q: torch.Tensor
    gate_s: torch.Tensor
    up_q: torch.Tensor
    up_s: torch.Tensor
    down_q: torch.Tensor
    down_s: torch.Tensor
    sh: Optional[dict]  # shared expert: gate_q, gate_s, up_q, up_s, down_q, down_s

    def to(self, device) -> "LayerInputs":
        mv = lambda t: None if t is None else t.to(device)
        sh = None if self.sh is None else {k: v.to(device) for k, v in self.sh.items()}
        return dataclasses.replace(
            self, logits=mv(self.logits), x=mv(self.x), wg=mv(self.wg), rank=mv(self.rank),
            slot_map=mv(self.slot_map), gate_q=mv(self.gate_q), gate_s=mv(self.gate_s),
            up_q=mv(self.up_q), up_s=mv(self.up_s), down_q=mv(self.down_q),
            down_s=mv(self.down_s), sh=sh)

    @property
    def x_is_bf16(self) -> bool:
        return self.cfg.x_dtype == "bf16"

    def pool_bytes(self) -> int:
        n = sum(t.numel() * t.element_size() for t in
                (self.gate_q, self.gate_s, self.up_q, self.up_s, self.down_q, self.down_s))
        if self.sh is not None:
            n += sum(t.numel() * t.element_size() for t in self.sh.values())
        return n


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _draw_expert(g, H, inter, std, device, n=1):
    """n experts' gate/up/down drawn and encoded; returns six stacked tensors."""
    out = {k: [] for k in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")}
    for _ in range(n):
        for kind, rows, K in (("gate", inter, H), ("up", inter, H), ("down", H, inter)):
            w = torch.randn(rows, K, generator=g, device=device, dtype=torch.float32) * std
            q, s = quantize_int4_blocks(w)
            out[kind + "_q"].append(q)
            out[kind + "_s"].append(s)
            del w
    return {k: torch.stack(v) for k, v in out.items()}


def make_layer(cfg: MoeConfig, seed: int = 0, device="cpu", layer: int = 0,
               T: Optional[int] = None) -> LayerInputs:
    """Draw one layer's inputs. `layer` selects an independent seed stream."""
    T = cfg.T if T is None else T
    g = _gen(seed * 1_000_003 + layer, device)
    E, H, I = cfg.E, cfg.H, cfg.I
    rank = torch.randperm(E, generator=g, device=device) + 1
    logits = wg = None
    if cfg.router_from_x:
        x = torch.randn(T, H, generator=g, device=device)
        wg = torch.randn(H, E, generator=g, device=device) * cfg.wg_std
    else:
        noise = torch.randn(T, E, generator=g, device=device)
        bias = -cfg.zipf_s * torch.log(rank.double()).float()
        logits = (noise + bias.unsqueeze(0)).contiguous()
        x = torch.randn(T, H, generator=g, device=device)
    if cfg.x_dtype == "bf16":
        x = f32_to_bf16_bits(x)
    # resident experts: the hottest n_resident by rank, slots in rank order
    if cfg.resident_frac < 1.0:
        nres = cfg.n_resident
        slot_map = torch.where(rank <= nres, rank - 1, torch.full_like(rank, -1)).to(torch.int32)
        S = nres
    else:
        slot_map = None
        S = E
    chunk = 32
    parts = []
    for s0 in range(0, S, chunk):
        parts.append(_draw_expert(g, H, I, cfg.w_std, device, n=min(chunk, S - s0)))
    pool = {k: torch.cat([p[k] for p in parts]).contiguous() for k in parts[0]}
    sh = None
    if cfg.shared_I:
        d = _draw_expert(g, H, cfg.shared_I, cfg.w_std, device, n=1)
        sh = {k: v[0].contiguous() for k, v in d.items()}
    return LayerInputs(cfg=cfg, seed=seed, logits=logits, x=x.contiguous(), wg=wg, rank=rank,
                       slot_map=slot_map, S=S, sh=sh, **pool)


def draw_windows(inp: LayerInputs, n: int, seed: int, device=None):
    """n more (logits, x) windows for the same layer: same popularity ranks, fresh
    noise and activations. Returns (logits [n, T, E] f32, x [n, T, H])."""
    cfg = inp.cfg
    device = inp.x.device if device is None else device
    T = inp.x.shape[0]
    g = _gen(seed * 7_919 + 17, device)
    bias = -cfg.zipf_s * torch.log(inp.rank.to(device).double()).float()
    logits = torch.randn(n, T, cfg.E, generator=g, device=device) + bias
    x = torch.randn(n, T, cfg.H, generator=g, device=device)
    if cfg.x_dtype == "bf16":
        x = f32_to_bf16_bits(x)
    return logits.contiguous(), x.contiguous()


def clone_pool(inp: LayerInputs) -> LayerInputs:
    """A copy of the layer with its own weight-pool buffers (same bytes)."""
    sh = None if inp.sh is None else {k: v.clone() for k, v in inp.sh.items()}
    return dataclasses.replace(inp, gate_q=inp.gate_q.clone(), gate_s=inp.gate_s.clone(),
                               up_q=inp.up_q.clone(), up_s=inp.up_s.clone(),
                               down_q=inp.down_q.clone(), down_s=inp.down_s.clone(), sh=sh)


def router_weights(cfg: MoeConfig, seed: int = 0, layer: int = 0, device="cpu") -> torch.Tensor:
    """A layer's router weights for a chained stack: [E][H] bf16 bit patterns
    (uint16), N(0, cfg.wg_std) rounded to bf16, from their own seed stream."""
    g = _gen(seed * 1_000_003 + layer + 500_009, device)
    w = torch.randn(cfg.E, cfg.H, generator=g, device=device) * cfg.wg_std
    return f32_to_bf16_bits(w).contiguous()


def random_slot_map(E: int, frac: float, seed: int) -> torch.Tensor:
    """Seeded random residency (used to exercise the miss path): slots in id order."""
    g = _gen(seed, "cpu")
    keep = torch.rand(E, generator=g) < frac
    slot = torch.cumsum(keep.to(torch.int64), 0) - 1
    return torch.where(keep, slot, torch.full_like(slot, -1)).to(torch.int32), int(keep.sum())


def random_logits(T: int, E: int, seed: int, zipf_s: float = 0.0, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    rank = torch.randperm(E, generator=g, device=device) + 1
    noise = torch.randn(T, E, generator=g, device=device)
    return (noise - zipf_s * torch.log(rank.double()).float().unsqueeze(0)).contiguous()


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 exactly (bit placement only)."""
    return (bits.astype(np.uint16).astype(np.uint32) << 16).view(np.float32)
