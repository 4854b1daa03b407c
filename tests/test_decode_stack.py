"""Several layers in one launch (moe_decode_stack) against one launch per layer
and against the CPU oracle.

Each layer of the stack runs the one-launch decode kernel's arithmetic on its
own buffers, so every layer's routing, miss list and y must equal, bit for
bit, what moe_layer_forward gives for that layer alone; and y within the
2e-3 gate of the oracle on the rows checked. Cases: the 48-layer shape
(hidden 2048, I 512, top-10) at windows of 1, 5 and 16 rows (both token-tile
widths of the kernel), the decode-window shape with its shared expert, a
slot map with misses in every layer, two calls in a row (the per-layer
counters reset), and a plan over more layers than any earlier call.
"""
import numpy as np
import pytest
import torch

import oracle
from routed_expert_ffn_router_gb300 import _lib, synth
from routed_expert_ffn_router_gb300 import build as libbuild
from routed_expert_ffn_router_gb300.layer import DecodeStack, MoeLayer

pytestmark = pytest.mark.gpu
TOL = 2e-3
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    libbuild.build()
    _lib.load()


def _layers(cfg, L, T, seed=0):
    return [synth.make_layer(cfg, seed, device=DEV, layer=l, T=T) for l in range(L)]


def _run_stack(layers, T):
    st = DecodeStack(layers, [l.logits for l in layers], [l.x for l in layers], T)
    outs = st.forward()
    torch.cuda.synchronize()
    code, bits = st.status()
    assert code == _lib.MOE_OK, f"device status {bits}"
    return st, [{k: v.clone() for k, v in o.items()} for o in outs]


def _assert_same_as_single(layers, outs, T):
    for l, inp in enumerate(layers):
        lay = MoeLayer(inp, T_max=T)
        ref = lay.forward(inp.logits, inp.x)
        torch.cuda.synchronize()
        assert lay.status()[0] == _lib.MOE_OK
        o = outs[l]
        assert torch.equal(o["ids"], ref["ids"]), f"layer {l}: ids"
        assert torch.equal(o["w"], ref["w"]), f"layer {l}: weights"
        n = int(ref["n_miss"].item())
        assert int(o["n_miss"].item()) == n, f"layer {l}: n_miss"
        assert torch.equal(o["miss_ids"][:n], ref["miss_ids"][:n]), f"layer {l}: miss ids"
        assert torch.equal(o["y"], ref["y"]), f"layer {l}: y differs from the one-layer launch"


def _check_oracle(inp_dev, out, rows):
    inp = inp_dev.to("cpu")
    ids = out["ids"].cpu().numpy()
    w = out["w"].cpu().numpy()
    y_ref = oracle.Layer(inp).rows(ids, w, rows=rows)
    y = out["y"].cpu().double().numpy()[rows]
    err = np.abs(y - y_ref).max()
    assert err <= TOL * np.abs(y_ref).max(), f"{err:.3e} vs {np.abs(y_ref).max():.3e}"
    o_ids, o_w, _ = oracle.route(inp.logits.numpy(), inp.cfg.k)
    assert np.array_equal(ids, o_ids)


@pytest.mark.parametrize("T", [1, 5, 16])
def test_stack_of_48_layer_shape_equals_one_launch_per_layer(T):
    cfg = synth.MoeConfig("stack48", H=2048, I=512, E=128, k=10, T=T, zipf_s=1.0)
    layers = _layers(cfg, 6, T, seed=2)
    _, outs = _run_stack(layers, T)
    _assert_same_as_single(layers, outs, T)
    _check_oracle(layers[0], outs[0], rows=list(range(min(T, 4))))


def test_stack_with_shared_expert():
    cfg = synth.MoeConfig("stack_dw", H=2048, I=768, E=128, k=8, T=8, shared_I=768, zipf_s=1.1)
    layers = _layers(cfg, 3, 8, seed=4)
    _, outs = _run_stack(layers, 8)
    _assert_same_as_single(layers, outs, 8)
    _check_oracle(layers[2], outs[2], rows=[0, 7])


def test_stack_with_slot_maps_and_misses():
    cfg = synth.MoeConfig("stack_ec", H=1024, I=512, E=64, k=8, T=12, zipf_s=1.2)
    layers = []
    for l in range(3):
        inp = synth.make_layer(cfg, 7, layer=l)
        smt, S = synth.random_slot_map(cfg.E, 0.6, seed=11 + l)
        keep = (smt >= 0).nonzero().flatten()
        for kname in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s"):
            setattr(inp, kname, getattr(inp, kname)[keep].contiguous())
        inp.S = S
        inp.slot_map = smt
        layers.append(inp.to(DEV))
    _, outs = _run_stack(layers, 12)
    assert all(int(o["n_miss"].item()) > 0 for o in outs)
    _assert_same_as_single(layers, outs, 12)
    _check_oracle(layers[1], outs[1], rows=[0, 5, 11])


def test_two_calls_in_a_row_and_a_longer_stack():
    cfg = synth.MoeConfig("stack_rep", H=2048, I=512, E=64, k=6, T=4, zipf_s=1.0)
    layers = _layers(cfg, 20, 4, seed=9)
    st, first = _run_stack(layers, 4)
    outs = st.forward()
    torch.cuda.synchronize()
    assert st.status()[0] == _lib.MOE_OK
    for a, b in zip(first, outs):
        assert torch.equal(a["y"], b["y"]) and torch.equal(a["w"], b["w"])
    _assert_same_as_single(layers[:3], first[:3], 4)
    _assert_same_as_single(layers[-2:], first[-2:], 4)
