"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: closed forms,
library routines for special cases, hand-worked values (tests/golden), brute
force on small inputs, invariants. The plausible mistakes each one catches are
named in its docstring.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from routed_expert_ffn_router_gb300 import synth
from tests import _pins


# ---------------------------------------------------------------- formats
def test_half_decode_matches_numpy_for_every_pattern():
    """fp16 scale decode: every finite bit pattern equals numpy's float16 (catches
    a wrong exponent bias, subnormal handling or sign)."""
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    L = oracle.lib()
    got = np.array([L.orc_half_to_double(int(b)) for b in bits[::7]])
    r = ref[::7]
    fin = np.isfinite(r)
    assert np.array_equal(got[fin], r[fin])
    assert np.all(np.isinf(got[np.isinf(r)]))
    assert np.all(np.isnan(got[np.isnan(r)]))


def test_bf16_decode_is_top_half_of_fp32():
    vals = np.array([1.0, -2.5, 3.140625, 1e-30, -7e20, 0.0], np.float32)
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
    for v, b in zip(vals, bits):
        assert oracle.bf16_to_double(int(b)) == float(np.float32((np.uint32(b) << 16).view(np.float32)))


def test_dequant_closed_form_all_codes():
    """Dequant of a hand-packed block: codes -8..7 at both nibble positions, scale
    1.0 then 0.5 (catches a swapped nibble order or a wrong sign extension)."""
    codes = np.array([[c for c in range(-8, 8)] * 2], np.int16)  # 1 row, 32 cols
    q = _pins.encode_codes(codes)
    for sbits, sval in ((0x3C00, 1.0), (0x3800, 0.5), (0xC000, -2.0)):
        s = np.array([[sbits]], np.uint16)
        got = [oracle.weight(q, s, 32, 0, c) for c in range(32)]
        assert got == [sval * float(c) for c in codes[0]]


def test_dequant_block_index_and_row_stride():
    """Scale index c/32 and row stride K/2: a 2x64 matrix with four distinct scales."""
    rng = np.random.default_rng(1)
    codes = rng.integers(-8, 8, size=(2, 64)).astype(np.int16)
    q = _pins.encode_codes(codes)
    s = np.array([[0x3C00, 0x4000], [0x3400, 0x4400]], np.uint16)  # 1, 2 / 0.25, 4
    sv = np.array([[1.0, 2.0], [0.25, 4.0]])
    for r in range(2):
        for c in range(64):
            assert oracle.weight(q, s, 64, r, c) == sv[r, c // 32] * codes[r, c]


def test_quantiser_worked_block_and_round_trip_bound():
    """Worked block: amax = 7 gives scale 1.0 exactly, so codes are rint(w).
    Round trip on random weights: |w - deq(q(w))| <= scale/2 (+ fp32 slack)."""
    w = torch.tensor([[7.0, -3.4, 2.5, 3.5, -0.5, 1.49] + [0.0] * 26])
    q, s = synth.quantize_int4_blocks(w)
    assert int(s[0, 0]) & 0xFFFF == 0x3C00
    got = [oracle.weight(q.numpy(), s.numpy(), 32, 0, c) for c in range(6)]
    assert got == [7.0, -3.0, 2.0, 4.0, -0.0, 1.0]  # half-even: 2.5 -> 2, 3.5 -> 4, -0.5 -> -0
    g = torch.Generator().manual_seed(3)
    w = torch.randn(8, 256, generator=g) * 0.02
    q, s = synth.quantize_int4_blocks(w)
    deq = _pins.dequant_np(q.numpy(), s.numpy())
    sc = np.repeat(s.numpy().astype(np.uint16).view(np.float16).astype(np.float64), 32, axis=1)
    err = np.abs(deq - w.double().numpy())
    assert np.all(err <= sc / 2 * (1 + 1e-6) + 1e-12)
    # the oracle's scalar dequant agrees with the vectorised one everywhere
    for r in range(8):
        for c in range(0, 256, 5):
            assert oracle.weight(q.numpy(), s.numpy(), 256, r, c) == deq[r, c]


# ---------------------------------------------------------------- routing
def _brute_topk(l, k):
    order = sorted(range(len(l)), key=lambda e: (-float(l[e]), e))  # full stable sort
    return order[:k]


@pytest.mark.parametrize("E,k,seed", [(8, 2, 0), (16, 5, 1), (64, 10, 2), (7, 7, 3), (33, 1, 4)])
def test_topk_ids_match_full_sort(E, k, seed):
    """Ids equal a full sort by (-logit, id); logits quantised to force many ties."""
    rng = np.random.default_rng(seed)
    lg = (np.round(rng.normal(size=(12, E)) * 2) / 2).astype(np.float32)
    ids, w, we = oracle.route(lg, k)
    for t in range(12):
        assert list(ids[t]) == _brute_topk(lg[t], k)


def test_topk_tie_special_cases():
    ids, w, _ = oracle.route(np.zeros((1, 2), np.float32), 1)
    assert ids[0, 0] == 0 and w[0, 0] == 1.0
    ids, w, _ = oracle.route(np.full((1, 5), 3.0, np.float32), 3)
    assert list(ids[0]) == [0, 1, 2]
    assert np.all(w == np.float32(1 / 3))


def test_weights_hand_worked_two_experts():
    """E = 2, k = 2, logits (0, 1): ids (1, 0), w = (1/(1+e^-1), e^-1/(1+e^-1));
    equal logits give (0.5, 0.5) with ids (0, 1)."""
    g = _pins.read_golden("hand_worked_two_experts.txt")
    ids, w, we = oracle.route(np.array([g["row0_logits"], g["row1_logits"]], np.float32), 2)
    assert list(ids[0]) == [int(v) for v in g["row0_ids"]]
    assert list(ids[1]) == [int(v) for v in g["row1_ids"]]
    assert list(w[0]) == [np.float32(v) for v in g["row0_w_exact"]]
    assert list(w[1]) == [np.float32(v) for v in g["row1_w_exact"]]
    assert abs(we[0, 0] - 1 / (1 + math.exp(-1))) < 1e-16


def test_weights_k_equals_E_is_plain_softmax():
    """k = E: the renormalised weights are the plain softmax (scipy), in id order
    of the sorted logits."""
    rng = np.random.default_rng(5)
    lg = rng.normal(size=(6, 9)).astype(np.float32)
    ids, w, we = oracle.route(lg, 9)
    for t in range(6):
        sm = scipy.special.softmax(lg[t].astype(np.float64))
        assert np.allclose(we[t], sm[ids[t]], rtol=1e-14, atol=0)
        assert np.array_equal(w[t], sm[ids[t]].astype(np.float32))


def test_weights_invariants_on_skewed_logits():
    """Sum to one within k*2^-24, non-increasing along j, every weight > 0."""
    lg = synth.random_logits(64, 512, seed=11, zipf_s=1.0).numpy()
    ids, w, _ = oracle.route(lg, 10)
    s = w.astype(np.float64).sum(1)
    assert np.all(np.abs(s - 1) <= 10 * 2.0 ** -24)
    assert np.all(np.diff(w, axis=1) <= 0)
    assert np.all(w > 0)
    # softmax over all E divided by the top-k mass gives the same weights
    full = scipy.special.softmax(lg.astype(np.float64), axis=1)
    sel = np.take_along_axis(full, ids, 1)
    assert np.allclose(sel / sel.sum(1, keepdims=True), w, rtol=2e-7, atol=0)


def test_route_rejects_non_finite():
    lg = np.zeros((3, 4), np.float32)
    lg[1, 2] = np.nan
    with pytest.raises(ValueError):
        oracle.route(lg, 2)


def test_router_logits_tiny_against_numpy():
    inp = synth.make_layer(synth.TINY, 0)
    lg = oracle.router_logits(inp.x, inp.wg)
    ref = (inp.x.double().numpy() @ inp.wg.double().numpy()).astype(np.float32)
    # identical after one rounding, except at an fp32 rounding midpoint
    assert np.max(np.abs(lg.view(np.int32) - ref.view(np.int32))) <= 1


# ---------------------------------------------------------------- permutation
@pytest.mark.parametrize("T,E,k,seed", [(4, 8, 2, 0), (16, 512, 10, 1), (64, 128, 8, 2), (1, 4, 4, 3)])
def test_permutation_invariants(T, E, k, seed):
    lg = synth.random_logits(T, E, seed=seed, zipf_s=1.0).numpy()
    ids, _, _ = oracle.route(lg, k)
    pm = oracle.permute(ids, E)
    P = T * k
    sp, pp, off = pm["sorted_pair"], pm["pair_pos"], pm["offsets"]
    assert off[0] == 0 and off[E] == P
    assert np.array_equal(np.diff(off), np.bincount(ids.ravel(), minlength=E))
    assert np.array_equal(sp[pp], np.arange(P))          # bijection both ways
    assert np.array_equal(pp[sp], np.arange(P))
    flat = ids.ravel()
    for e in range(E):
        seg = sp[off[e]:off[e + 1]]
        assert np.all(flat[seg] == e)                      # grouped by expert
        assert np.all(np.diff(seg) > 0)                    # stable: p ascending
    assert pm["n_miss"] == 0


def test_miss_list_counts_distinct_experts():
    """Hits and misses count distinct experts per layer ("extended-strata-moe
    reference", C API): two rows sharing a missing expert give one miss."""
    ids = np.array([[3, 1], [3, 0], [2, 1]], np.int32)
    slot_map = np.array([0, -1, 1, -1], np.int32)
    pm = oracle.permute(ids, 4, slot_map)
    assert pm["n_miss"] == 2 and list(pm["miss_ids"]) == [1, 3]


# ---------------------------------------------------------------- FFN
def test_hand_worked_two_expert_layer():
    """Golden: identity-shaped int4 experts, x in {-1, 0, 1}; only silu is transcendental."""
    g = _pins.read_golden("hand_worked_two_experts.txt")
    H = I = 32
    cfg = synth.MoeConfig("hand", H=H, I=I, E=2, k=2, T=2, x_dtype="f32")
    pool = _pins.identity_pool(2, H, I, gate_mult=(1, 2), up_mult=(2, 1), down_mult=(1, 1))
    x = np.zeros((2, H), np.float32)
    for h in range(H):
        x[0, h] = (1, -1, 0)[h % 3]
        x[1, h] = (-1, 0, 1)[h % 3]
    inp = _pins.fake_inputs(cfg, torch.from_numpy(x), pool, S=2)
    ids, w, _ = oracle.route(np.array([g["row0_logits"], g["row1_logits"]], np.float32), 2)
    y = oracle.Layer(inp).rows(ids, w)
    w1, w0 = np.float64(np.float32(g["row0_w_exact"][0])), np.float64(np.float32(g["row0_w_exact"][1]))
    for h in range(H):
        xv = x[0, h]
        exp0 = {1: w1 * g["e1_p1"] + w0 * g["e0_p1"], -1: w1 * g["e1_m1"] + w0 * g["e0_m1"], 0: 0.0}[int(xv)]
        assert abs(y[0, h] - exp0) < 1e-14
        xv = x[1, h]
        exp1 = {1: g["row1_y_p1"], -1: g["row1_y_m1"], 0: 0.0}[int(xv)]
        assert abs(y[1, h] - exp1) < 1e-14
    assert abs(g["silu_1"] - 1 / (1 + math.exp(-1))) < 1e-16


def test_zero_gate_weights_leave_shared_only():
    """All routed gate codes zero: silu(0) = 0 so every routed expert adds 0 and y
    is the shared expert alone (catches a missing shared term or a stray bias)."""
    cfg = synth.MoeConfig("zg", H=128, I=128, E=4, k=2, T=3, shared_I=128, x_dtype="bf16")
    inp = synth.make_layer(cfg, seed=7)
    inp.gate_q.zero_()
    ids, w, _ = oracle.route(synth.random_logits(3, 4, seed=2).numpy(), 2)
    L = oracle.Layer(inp)
    y = L.rows(ids, w)
    sm_none = np.full(4, -1, np.int32)
    y_shared = L.rows(ids, w, slot_map=sm_none)
    assert np.array_equal(y, y_shared)
    assert np.abs(y).max() > 0


@pytest.mark.parametrize("name", ["tiny", "decode_window_small"])
def test_sparse_equals_dense_then_mask(name):
    """The sparse oracle equals the brute-force dense-then-mask layer to 1e-12
    relative (catches a wrong expert slot, a transposed matrix, a dropped weight
    or a missing shared expert)."""
    if name == "tiny":
        cfg = synth.TINY
        inp = synth.make_layer(cfg, 0)
        lg = oracle.router_logits(inp.x, inp.wg)
    else:
        cfg = synth.MoeConfig("dw_small", H=512, I=256, E=16, k=4, T=8, shared_I=128, zipf_s=1.1)
        inp = synth.make_layer(cfg, 0)
        lg = inp.logits.numpy()
    ids, w, _ = oracle.route(lg, cfg.k)
    y = oracle.Layer(inp).rows(ids, w)
    ref = _pins.dense_then_mask(inp, ids, w)
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_negative_control_one_corrupted_byte_fails_the_tolerance_gate():
    """Negative control (the pages prove a gate can go red by corrupting one byte):
    one bit of one byte of an fp16 scale in a routed expert's down matrix moves y
    far beyond the parity tolerance (2e-3 of max|y|) against the intact layer, while
    the brute-force check of the corrupted layer still holds (so the gate compares
    bytes, not the oracle with itself)."""
    cfg = synth.MoeConfig("nc", H=256, I=128, E=8, k=2, T=4, shared_I=128, zipf_s=1.0)
    inp = synth.make_layer(cfg, 3)
    ids, w, _ = oracle.route(inp.logits.numpy(), cfg.k)
    y = oracle.Layer(inp).rows(ids, w)
    bad = synth.clone_pool(inp)
    e = int(ids[0][0])
    b = bad.down_s.view(torch.uint8).view(cfg.E, cfg.H, cfg.I // 32, 2)
    b[e, 0, 0, 1] ^= 0x40                      # the high byte: the exponent's top bit
    y_bad = oracle.Layer(bad).rows(ids, w)
    assert np.abs(y_bad - y).max() > 2e-3 * np.abs(y).max()
    ref_bad = _pins.dense_then_mask(bad, ids, w)
    assert np.max(np.abs(y_bad - ref_bad)) <= 1e-12 * np.max(np.abs(ref_bad))


@pytest.mark.slow
def test_sparse_equals_dense_then_mask_decode_window_full():
    """Same brute-force check at the full decode-window size (H 2048, 128 experts)."""
    cfg = synth.DECODE_WINDOW
    inp = synth.make_layer(cfg, 0)
    ids, w, _ = oracle.route(inp.logits.numpy(), cfg.k)
    y = oracle.Layer(inp).rows(ids, w)
    ref = _pins.dense_then_mask(inp, ids, w)
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_slot_map_pins():
    """All resident == no slot map; none resident == shared only with every
    touched expert listed; y(resident set A) + y(complement) - shared == y(all)."""
    cfg = synth.MoeConfig("sm", H=256, I=128, E=12, k=3, T=5, shared_I=128, zipf_s=1.0)
    inp = synth.make_layer(cfg, 4)
    ids, w, _ = oracle.route(inp.logits.numpy(), cfg.k)
    L = oracle.Layer(inp)
    y_all = L.rows(ids, w)
    ident = np.arange(cfg.E, dtype=np.int32)
    assert np.array_equal(L.rows(ids, w, slot_map=ident), y_all)
    none = np.full(cfg.E, -1, np.int32)
    y_none = L.rows(ids, w, slot_map=none)
    pm = oracle.permute(ids, cfg.E, none)
    assert list(pm["miss_ids"]) == sorted(set(ids.ravel().tolist()))
    rng = np.random.default_rng(0)
    keep = rng.random(cfg.E) < 0.6
    a = np.where(keep, ident, -1).astype(np.int32)
    b = np.where(~keep, ident, -1).astype(np.int32)
    y_a = L.rows(ids, w, slot_map=a)
    y_b = L.rows(ids, w, slot_map=b)
    assert np.max(np.abs(y_a + y_b - y_none - y_all)) <= 1e-12 * np.abs(y_all).max()
    # the dense brute force agrees under a partial slot map as well
    ref = _pins.dense_then_mask(inp, ids, w, slot_map=torch.from_numpy(a))
    assert np.max(np.abs(y_a - ref)) <= 1e-12 * np.abs(ref).max()


def test_expert_h_is_the_swiglu_of_the_gate_and_up_rows():
    """orc_expert_h equals silu(Wg x) * (Wu x) from the vectorised dequant."""
    cfg = synth.MoeConfig("h", H=256, I=128, E=3, k=1, T=2, x_dtype="bf16")
    inp = synth.make_layer(cfg, 9)
    L = oracle.Layer(inp)
    x = _pins.x_float64(inp)
    Wg = _pins.dequant_np(inp.gate_q[2].numpy(), inp.gate_s[2].numpy())
    Wu = _pins.dequant_np(inp.up_q[2].numpy(), inp.up_s[2].numpy())
    ref = _pins.silu_tanh(Wg @ x[1]) * (Wu @ x[1])
    assert np.allclose(L.expert_h(1, 2), ref, rtol=1e-12, atol=1e-15)
