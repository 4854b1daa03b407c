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


def _assert_weights_match(w_gpu, w_orc, w_exact):
    """Bitwise, except that a weight whose exact value sits at an fp32 rounding
    midpoint (within 2^-40 relative) may round to either neighbour."""
    w_gpu = np.asarray(w_gpu, np.float32)
    for idx in np.argwhere(w_gpu != w_orc):
        idx = tuple(idx)
        a, b = w_gpu[idx], w_orc[idx]
        assert abs(int(a.view(np.int32)) - int(b.view(np.int32))) == 1, (idx, a, b)
        mid = (float(a) + float(b)) / 2
        assert abs(w_exact[idx] - mid) <= 2.0 ** -40 * abs(mid), (idx, a, b, w_exact[idx])


def _bf16_rne(f32):
    """fp32 -> bf16 bit patterns, round to nearest even (finite values)."""
    u = np.ascontiguousarray(f32, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("T", [1, 8])
def test_routed_chained_stack_layer_by_layer(T):
    """The router in the launch and layers chained through the residual: each
    layer checked on the GPU's own input for that layer. Its logits against the
    oracle's router (float64, rounded once) to fp32 rounding of the sum; its
    routing bit for bit against the oracle's routing of the GPU logits; its y
    within the gate; the next layer's input bit for bit against
    bf16(x + y); and the whole layer bitwise equal to moe_layer_forward on
    the same logits and input."""
    cfg = synth.MoeConfig("stack_rt", H=2048, I=512, E=128, k=10, T=T)
    L = 5
    layers = _layers(cfg, L, T, seed=3)
    wr = [synth.router_weights(cfg, 3, layer=l, device=DEV) for l in range(L)]
    st = DecodeStack(layers, None, [layers[0].x] + [None] * (L - 1), T, router_w=wr)
    st.forward()
    torch.cuda.synchronize()
    code, bits = st.status()
    assert code == _lib.MOE_OK, f"device status {bits}"
    outs = st.outs
    for l in range(L):
        x_bits = st.xs[l].cpu().numpy().view(np.uint16)
        x_f32 = synth.bf16_bits_to_f32(x_bits)
        w_f32 = synth.bf16_bits_to_f32(wr[l].cpu().numpy().view(np.uint16))
        lg = st.logits[l].cpu().numpy()
        lo = oracle.router_logits(x_f32, np.ascontiguousarray(w_f32.T))
        assert np.abs(lg - lo).max() <= 1e-5 * np.abs(lo).max() + 1e-6, f"layer {l}: router logits"
        ids, w, we = oracle.route(lg, cfg.k)
        assert np.array_equal(outs[l]["ids"].cpu().numpy(), ids), f"layer {l}: ids"
        _assert_weights_match(outs[l]["w"].cpu().numpy(), w, we)
        inp = layers[l].to("cpu")
        y_ref = oracle.Layer(inp).rows(ids, w, x=x_bits)
        y = outs[l]["y"].cpu().double().numpy()
        err = np.abs(y - y_ref).max()
        assert err <= TOL * np.abs(y_ref).max(), f"layer {l}: {err:.3e}"
        if l + 1 < L:
            nxt = _bf16_rne(x_f32 + outs[l]["y"].cpu().numpy())
            assert np.array_equal(st.xs[l + 1].cpu().numpy().view(np.uint16), nxt), f"layer {l}: residual"
        # the same layer through one launch: bitwise
        lay = MoeLayer(layers[l], T_max=T)
        ref = lay.forward(st.logits[l], st.xs[l])
        torch.cuda.synchronize()
        assert torch.equal(ref["y"], outs[l]["y"]) and torch.equal(ref["w"], outs[l]["w"]), f"layer {l}"


def test_a_launch_that_differs_from_its_plan_runs_nothing():
    """moe_decode_stack with another layer count, row count or workspace than
    the plan's (here: more or fewer layers, 12 rows on a 4-row plan, 5 rows on
    it, a second workspace) ORs 16 into the status word of the workspace given
    and leaves every output untouched; the prepared launch then runs as usual."""
    cfg = synth.MoeConfig("stack_guard", H=1024, I=512, E=32, k=4, T=4, zipf_s=1.0)
    layers = _layers(cfg, 2, 4, seed=5)
    st = DecodeStack(layers, [l.logits for l in layers], [l.x for l in layers], 4)
    for o in st.outs:
        o["y"].fill_(7.0)
    for L, T in ((3, 4), (1, 4), (2, 12), (2, 5)):
        _lib.moe_workspace_init(st.ws_ptr, st.ws_bytes)
        _lib.moe_decode_stack(st.plan_ptr, L, T, st.ws_ptr, st.ws_bytes)
        torch.cuda.synchronize()
        code, bits = st.status()
        assert code == _lib.MOE_ERR_DEVICE and bits & 16, (L, T, code, bits)
        assert all(bool((o["y"] == 7.0).all()) for o in st.outs), (L, T)
    # another workspace than the plan's
    other = torch.empty(st.ws_bytes + 256, dtype=torch.uint8, device=DEV)
    optr = other.data_ptr() + (-other.data_ptr()) % 256
    _lib.moe_workspace_init(optr, st.ws_bytes)
    _lib.moe_decode_stack(st.plan_ptr, 2, 4, optr, st.ws_bytes)
    torch.cuda.synchronize()
    code, bits = _lib.moe_read_status(optr)
    assert code == _lib.MOE_ERR_DEVICE and bits & 16, (code, bits)
    assert all(bool((o["y"] == 7.0).all()) for o in st.outs)
    _lib.moe_workspace_init(st.ws_ptr, st.ws_bytes)
    outs = st.forward()
    torch.cuda.synchronize()
    assert st.status()[0] == _lib.MOE_OK
    _assert_same_as_single(layers, [{k: v.clone() for k, v in o.items()} for o in outs], 4)
