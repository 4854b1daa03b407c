"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Routing (ids, fp32 weights), the permutation and the miss list must match bit
for bit; layer outputs within max|y - y_oracle| <= 2e-3 * max|y_oracle| over the
rows checked. Full-size configurations are checked on every row the oracle can
afford and on sampled rows for the 2,048-token chunk.
"""
import hashlib

import numpy as np
import pytest
import torch

import oracle
from routed_expert_ffn_router_gb300 import _lib, synth
from routed_expert_ffn_router_gb300 import build as libbuild
from routed_expert_ffn_router_gb300.layer import MoeLayer

pytestmark = pytest.mark.gpu
TOL = 2e-3
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    libbuild.build()
    _lib.load()


def assert_weights_match(w_gpu, w_orc, w_exact):
    """Bitwise, except that a weight whose exact value sits at an fp32 rounding
    midpoint (within 2^-40 relative) may round to either neighbour."""
    w_gpu = np.asarray(w_gpu, np.float32)
    bad = np.argwhere(w_gpu != w_orc)
    for idx in bad:
        idx = tuple(idx)
        a, b = w_gpu[idx], w_orc[idx]
        assert abs(int(a.view(np.int32)) - int(b.view(np.int32))) == 1, (idx, a, b)
        mid = (float(a) + float(b)) / 2
        assert abs(w_exact[idx] - mid) <= 2.0 ** -40 * abs(mid), (idx, a, b, w_exact[idx])


def check_y(y_gpu, y_ref, tol=TOL, what=""):
    y_gpu = np.asarray(y_gpu, np.float64)
    err = np.abs(y_gpu - y_ref).max()
    scale = np.abs(y_ref).max()
    assert np.all(np.isfinite(y_gpu)), what
    assert err <= tol * scale, f"{what}: max|dy| = {err:.3e}, max|y| = {scale:.3e}, ratio {err / scale:.3e}"
    return err / scale


def gpu_route(logits_np, k):
    T, E = logits_np.shape
    lg = torch.from_numpy(np.ascontiguousarray(logits_np)).to(DEV)
    ids = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    _lib.moe_route(lg, T, E, k, ids, w, st)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), int(st.item())


# ---------------------------------------------------------------- router
@pytest.mark.parametrize("xbf16", [False, True])
def test_router_logits_bit_exact(xbf16):
    cfg = synth.TINY if not xbf16 else synth.MoeConfig("tb", H=256, I=128, E=8, k=2, T=4,
                                                       router_from_x=True)
    inp = synth.make_layer(cfg, 0)
    lg_ref = oracle.router_logits(synth.bf16_bits_to_f32(inp.x.numpy()) if xbf16 else inp.x, inp.wg)
    x = inp.x.to(DEV)
    wg = inp.wg.to(DEV)
    out = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=DEV)
    _lib.moe_router_logits(x, _lib.MOE_BF16 if xbf16 else _lib.MOE_F32, wg, cfg.T, cfg.H, cfg.E, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.int32), lg_ref.view(np.int32))


ROUTE_CASES = [("tiny", 4, 8, 2, 0.0), ("decode_window", 8, 128, 8, 1.1),
               ("decode48_T1", 1, 512, 10, 1.0), ("decode48_T16", 16, 512, 10, 1.0),
               ("expert_cache", 16, 256, 8, 1.2), ("prefill", 2048, 512, 10, 1.0),
               ("maxE_maxk", 64, 1024, 32, 0.5), ("k_eq_E", 9, 7, 7, 0.0), ("E1", 5, 1, 1, 0.0)]


@pytest.mark.parametrize("name,T,E,k,s", ROUTE_CASES)
def test_route_bit_exact(name, T, E, k, s):
    lg = synth.random_logits(T, E, seed=T * 7 + E, zipf_s=s).numpy()
    ids_o, w_o, we = oracle.route(lg, k)
    ids, w, st = gpu_route(lg, k)
    assert st == 0
    assert np.array_equal(ids, ids_o)
    assert_weights_match(w, w_o, we)


@pytest.mark.parametrize("sigma", [0.01, 1.0, 12.0, 40.0])
def test_route_weights_many_rows(sigma):
    """Weights of 40,000 rows against the float64 oracle, logits spread from
    nearly equal to differences past 80 (the float64 fallback)."""
    rng = np.random.default_rng(int(sigma * 100) + 1)
    lg = (rng.normal(size=(40000, 64)) * sigma).astype(np.float32)
    ids_o, w_o, we = oracle.route(lg, 8)
    ids, w, st = gpu_route(lg, 8)
    assert st == 0
    assert np.array_equal(ids, ids_o)
    assert_weights_match(w, w_o, we)


def test_route_ties_go_to_lower_id():
    rng = np.random.default_rng(3)
    lg = (np.round(rng.normal(size=(300, 64)) * 2) / 2).astype(np.float32)  # many exact ties
    lg[0] = 0.0
    lg[1, :] = -0.0
    lg[1, 10] = 0.0
    ids_o, w_o, we = oracle.route(lg, 10)
    ids, w, st = gpu_route(lg, 10)
    assert np.array_equal(ids, ids_o)
    assert list(ids[0]) == list(range(10))
    assert_weights_match(w, w_o, we)


def test_route_flags_non_finite():
    lg = synth.random_logits(4, 32, seed=1).numpy()
    lg[2, 5] = np.inf
    _, _, st = gpu_route(lg, 4)
    assert st & 1


# ---------------------------------------------------------------- permutation
def gpu_permute(ids_np, E, slot_map=None, S=None):
    T, k = ids_np.shape
    P = T * k
    ids = torch.from_numpy(np.ascontiguousarray(ids_np)).to(DEV)
    off = torch.full((E + 1,), -7, dtype=torch.int32, device=DEV)
    sp = torch.full((max(P, 1),), -7, dtype=torch.int32, device=DEV)
    pp = torch.full((max(P, 1),), -7, dtype=torch.int32, device=DEV)
    miss = torch.full((E,), -7, dtype=torch.int32, device=DEV)
    nm = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    ws_bytes = 1 << 22
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=DEV)
    sm = None if slot_map is None else torch.from_numpy(np.asarray(slot_map, np.int32)).to(DEV)
    _lib.moe_permute(ids, T, E, k, sm, E if S is None else S, off, sp, pp, miss, nm, ws, ws_bytes)
    torch.cuda.synchronize()
    n = int(nm.item())
    return dict(offsets=off.cpu().numpy(), sorted_pair=sp.cpu().numpy()[:P],
                pair_pos=pp.cpu().numpy()[:P], miss_ids=miss.cpu().numpy()[:n], n_miss=n,
                status=int(ws[:4].view(torch.int32).item()))


@pytest.mark.parametrize("name,T,E,k,s", ROUTE_CASES + [("chunked", 300, 64, 8, 1.0),
                                                        ("ragged", 103, 96, 10, 1.0)])
@pytest.mark.parametrize("resident", [1.0, 0.6, 0.0])
def test_permute_bit_exact(name, T, E, k, s, resident):
    lg = synth.random_logits(T, E, seed=T + 3 * E, zipf_s=s).numpy()
    ids, _, _ = oracle.route(lg, k)
    if resident == 1.0:
        sm, S = None, E
    else:
        smt, S = synth.random_slot_map(E, resident, seed=E)
        sm = smt.numpy()
        S = max(S, 1)
    ref = oracle.permute(ids, E, sm)
    got = gpu_permute(ids, E, sm, S)
    assert got["status"] == 0
    for key in ("offsets", "sorted_pair", "pair_pos", "miss_ids"):
        assert np.array_equal(got[key], ref[key]), key
    assert got["n_miss"] == ref["n_miss"]


def test_permute_flags_slot_out_of_range():
    ids = np.array([[0, 1], [2, 1]], np.int32)
    got = gpu_permute(ids, 4, np.array([0, 5, 1, -1], np.int32), S=3)
    assert got["status"] & 2
    assert list(got["miss_ids"]) == [1]  # treated as not resident


# ---------------------------------------------------------------- layer
def run_layer(inp, logits=None, x=None, slot_map="default", lay=None):
    dev_inp = inp if inp.gate_q.is_cuda else inp.to(DEV)
    lay = lay or MoeLayer(dev_inp, T_max=(x if x is not None else inp.x).shape[0])
    lg = (inp.logits if logits is None else logits).to(DEV)
    xx = (inp.x if x is None else x).to(DEV)
    sm = slot_map if isinstance(slot_map, str) else (None if slot_map is None else slot_map.to(DEV))
    out = lay.forward(lg, xx, slot_map=sm)
    torch.cuda.synchronize()
    code, bits = lay.status()
    assert code == _lib.MOE_OK, bits
    return {k: v.cpu().numpy() for k, v in out.items()}, lay


def oracle_layer(inp, logits, rows=None, slot_map="default"):
    ids, w, we = oracle.route(np.asarray(logits), inp.cfg.k)
    L = oracle.Layer(inp)
    y = L.rows(ids, w, rows=rows, slot_map=slot_map)
    return ids, w, we, y


def test_tiny_layer_end_to_end():
    """Tiny case: router GEMV on the GPU, then route + FFN, against the oracle."""
    cfg = synth.TINY
    inp = synth.make_layer(cfg, 0)
    lg = oracle.router_logits(inp.x, inp.wg)
    dinp = inp.to(DEV)
    lg_dev = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=DEV)
    _lib.moe_router_logits(dinp.x, _lib.MOE_F32, dinp.wg, cfg.T, cfg.H, cfg.E, lg_dev)
    out, _ = run_layer(dinp, logits=lg_dev)
    ids, w, we, y = oracle_layer(inp, lg)
    assert np.array_equal(out["ids"], ids)
    assert_weights_match(out["w"], w, we)
    check_y(out["y"], y, what="tiny")
    assert out["n_miss"][0] == 0


@pytest.mark.parametrize("cfg", [synth.DECODE_WINDOW, synth.EXPERT_CACHE], ids=lambda c: c.name)
def test_decode_configs_full(cfg):
    inp = synth.make_layer(cfg, 0, device=DEV)
    out, _ = run_layer(inp)
    hinp = inp.to("cpu")
    ids, w, we, y = oracle_layer(hinp, hinp.logits.numpy())
    assert np.array_equal(out["ids"], ids)
    assert_weights_match(out["w"], w, we)
    pm = oracle.permute(ids, cfg.E, None if hinp.slot_map is None else hinp.slot_map.numpy())
    assert out["n_miss"][0] == pm["n_miss"]
    assert np.array_equal(out["miss_ids"][:pm["n_miss"]], pm["miss_ids"])
    check_y(out["y"], y, what=cfg.name)


@pytest.mark.parametrize("T", synth.DECODE48_WINDOWS)
def test_decode48_layers(T):
    """Large-expert-count decode: two of the 48 layers (first and last seed
    streams) at every window size."""
    cfg = synth.DECODE_48
    for layer in (0, 47):
        inp = synth.make_layer(cfg, 0, device=DEV, layer=layer, T=T)
        out, _ = run_layer(inp)
        hinp = inp.to("cpu")
        ids, w, we, y = oracle_layer(hinp, hinp.logits.numpy())
        assert np.array_equal(out["ids"], ids)
        assert_weights_match(out["w"], w, we)
        check_y(out["y"], y, what=f"decode48 T={T} layer {layer}")


@pytest.mark.parametrize("T", [1, 16])
def test_decode48_near_tied_logits_route_bit_exact(T):
    """The one-launch decode kernel routes the window itself (every CTA runs the
    top-k; the softmax weights come from the kernel's own float-float path): at
    512 experts top-10 with logits on a grid of 1/4, so that many are exactly
    equal, its ids and fp32 weights must equal the oracle's bit for bit and ties
    must go to the lower expert id."""
    cfg = synth.DECODE_48
    inp = synth.make_layer(cfg, 0, device=DEV, layer=3, T=T)
    rng = np.random.default_rng(40 + T)
    lg = (np.round(rng.normal(size=(T, cfg.E)) * 2) / 4).astype(np.float32)
    lg[0, :] = np.float32(-1.0)
    lg[0, 100:140] = np.float32(0.5)  # 40 equal maxima: ids 100..109 must be taken
    if T > 1:
        lg[1, :] = np.float32(0.0)     # all equal, with signed zeros
        lg[1, ::3] = np.float32(-0.0)
    out, _ = run_layer(inp, logits=torch.from_numpy(lg))
    hinp = inp.to("cpu")
    ids, w, we, y = oracle_layer(hinp, lg)
    assert list(ids[0]) == list(range(100, 110))
    assert np.array_equal(out["ids"], ids)
    assert_weights_match(out["w"], w, we)
    check_y(out["y"], y, what=f"decode48 near-tied T={T}")


def test_expert_cache_random_slot_map_and_misses():
    cfg = synth.MoeConfig("ec_small", H=1024, I=512, E=64, k=8, T=16, zipf_s=1.2)
    inp = synth.make_layer(cfg, 5)
    smt, S = synth.random_slot_map(cfg.E, 0.6, seed=9)
    # pool with only the resident experts: slot s = the s-th resident expert
    keep = (smt >= 0).nonzero().flatten()
    for kname in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s"):
        setattr(inp, kname, getattr(inp, kname)[keep].contiguous())
    inp.S = S
    inp.slot_map = smt
    out, _ = run_layer(inp)
    ids, w, we, y = oracle_layer(inp, inp.logits.numpy())
    pm = oracle.permute(ids, cfg.E, smt.numpy())
    assert pm["n_miss"] > 0
    assert out["n_miss"][0] == pm["n_miss"]
    assert np.array_equal(out["miss_ids"][:pm["n_miss"]], pm["miss_ids"])
    check_y(out["y"], y, what="random slot map")


def test_prefill_random_slot_map_and_misses():
    """Prefill path (64 tokens: the tcgen05 GEMMs) through a slot map with 60% of the experts
    resident and a shared expert: the miss list equals the oracle's permutation, and y sums the
    resident experts and the shared one."""
    cfg = synth.MoeConfig("pf_ec", H=1024, I=512, E=64, k=8, T=64, shared_I=512, zipf_s=1.2)
    inp = synth.make_layer(cfg, 6)
    smt, S = synth.random_slot_map(cfg.E, 0.6, seed=11)
    keep = (smt >= 0).nonzero().flatten()
    for kname in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s"):
        setattr(inp, kname, getattr(inp, kname)[keep].contiguous())
    inp.S = S
    inp.slot_map = smt
    out, _ = run_layer(inp)
    ids, w, we, y = oracle_layer(inp, inp.logits.numpy())
    pm = oracle.permute(ids, cfg.E, smt.numpy())
    assert pm["n_miss"] > 0
    assert out["n_miss"][0] == pm["n_miss"]
    assert np.array_equal(out["miss_ids"][:pm["n_miss"]], pm["miss_ids"])
    check_y(out["y"], y, what="prefill, random slot map")


def test_prefill_sampled_rows():
    """2,048-token chunk: every output row is finite; the oracle checks sampled
    rows, including rows routed to the hottest expert, the rows with the most
    picks of experts of at most 16 tokens, the first and the last."""
    cfg = synth.PREFILL
    inp = synth.make_layer(cfg, 0, device=DEV)
    out, _ = run_layer(inp)
    hinp = inp.to("cpu")
    ids, w, we = oracle.route(hinp.logits.numpy(), cfg.k)
    assert np.array_equal(out["ids"], ids)
    assert_weights_match(out["w"], w, we)
    assert np.all(np.isfinite(out["y"]))
    counts = np.bincount(ids.ravel(), minlength=cfg.E)
    hot = counts.argmax()
    rows_hot = np.nonzero((ids == hot).any(1))[0]
    # the rows with the most picks of light experts (at most 16 tokens: the jobs
    # that take the smallest token boxes); under this skew a row has 2-3 of them
    n_light = (counts[ids] <= 16).sum(1)
    rows_light = np.argsort(-n_light, kind="stable")[:4]
    assert n_light[rows_light[0]] >= 2
    rng = np.random.default_rng(0)
    rows = sorted(set([0, cfg.T - 1] + list(rng.choice(cfg.T, 10, replace=False)) +
                      list(rows_hot[:3]) + list(rows_hot[-3:]) + list(rows_light)))
    y = oracle.Layer(hinp).rows(ids, w, rows=rows)
    check_y(out["y"][rows], y, what="prefill sampled rows")


def _scale_scales(s_bits, factor, mask=None):
    """fp16 scale bit patterns times `factor` (rounded to fp16), where mask."""
    h = s_bits.view(torch.float16).float()
    scaled = (h * factor).to(torch.float16).float()
    h = scaled if mask is None else torch.where(mask, scaled, h)
    return h.to(torch.float16).view(torch.int16).contiguous()


@pytest.mark.parametrize("case", ["down", "gateup", "subnormal", "mixed"])
def test_prefill_small_scales(case):
    """Prefill with small fp16 block scales: q * s must stay one rounding of the
    exact product for every scale, down to subnormal ones (a form that takes
    16 q times s / 16, say, would lose that below 2^-10). The scales of a whole
    matrix kind are made small (x scaled up where needed, so that h stays a
    normal fp16 number), or subnormal, or small in a random half of the blocks
    of every matrix: y matches the oracle, which uses the same fp16 scales."""
    cfg = synth.MoeConfig("pf_small_" + case, H=512, I=256, E=16, k=4, T=96, shared_I=256, zipf_s=1.0)
    inp = synth.make_layer(cfg, 21)
    g = torch.Generator().manual_seed(5)
    kinds = {"down": ("down_s",), "gateup": ("gate_s", "up_s"), "subnormal": ("down_s",),
             "mixed": ("gate_s", "up_s", "down_s")}[case]
    factor = 2.0 ** -12 if case == "subnormal" else 2.0 ** -6
    for name in kinds:
        m = None
        if case == "mixed":
            m = torch.rand(getattr(inp, name).shape, generator=g) < 0.5
        setattr(inp, name, _scale_scales(getattr(inp, name), factor, m))
        ms = None if m is None else torch.rand(inp.sh[name].shape, generator=g) < 0.5
        inp.sh[name] = _scale_scales(inp.sh[name], factor, ms)
    if case == "gateup":  # x 64 times larger (exact in bf16) keeps g, u and h in range
        xf = torch.from_numpy(synth.bf16_bits_to_f32(inp.x.numpy())) * 64.0
        inp.x = synth.f32_to_bf16_bits(xf).contiguous()
    for name in kinds:  # the three-shift form is exercised
        assert (np.abs(getattr(inp, name).view(torch.float16).float().numpy()) < 2.0 ** -10).any()
    out, _ = run_layer(inp)
    ids, w, we, y = oracle_layer(inp, inp.logits.numpy())
    assert np.array_equal(out["ids"], ids)
    check_y(out["y"], y, what=f"small scales: {case}")


@pytest.mark.parametrize("T", [1, 3, 5, 13, 16, 17, 33, 100])
def test_ragged_windows(T):
    cfg = synth.MoeConfig("rag", H=512, I=256, E=32, k=4, T=T, shared_I=256, zipf_s=1.0)
    inp = synth.make_layer(cfg, T)
    out, _ = run_layer(inp)
    ids, w, we, y = oracle_layer(inp, inp.logits.numpy())
    assert np.array_equal(out["ids"], ids)
    assert_weights_match(out["w"], w, we)
    check_y(out["y"], y, what=f"T={T}")


def test_prefill_k_not_a_multiple_of_slot_steps():
    """Prefill GEMMs with K = 768 in both (12 steps of 64 columns, where a token slot holds 8
    steps for jobs of up to 16 tokens) and two or three jobs per CTA: each job's last, partly
    used token slot must be released before the next job of the CTA reads the ring."""
    cfg = synth.MoeConfig("k768", H=768, I=768, E=64, k=4, T=384, shared_I=768, zipf_s=1.0)
    inp = synth.make_layer(cfg, 5)
    out, _ = run_layer(inp)
    ids, w, we, y = oracle_layer(inp, inp.logits.numpy())
    assert np.array_equal(out["ids"], ids)
    check_y(out["y"], y, what="K = 768 prefill")


def test_min_shapes_and_max_k():
    cfg = synth.MoeConfig("min", H=128, I=128, E=40, k=32, T=3, shared_I=128, zipf_s=0.0)
    inp = synth.make_layer(cfg, 2)
    out, _ = run_layer(inp)
    ids, w, we, y = oracle_layer(inp, inp.logits.numpy())
    assert np.array_equal(out["ids"], ids)
    check_y(out["y"], y, what="min shapes")


def test_no_resident_expert_gives_shared_only():
    cfg = synth.MoeConfig("none", H=256, I=128, E=16, k=4, T=6, shared_I=256, zipf_s=1.0)
    inp = synth.make_layer(cfg, 3)
    sm = torch.full((cfg.E,), -1, dtype=torch.int32)
    out, _ = run_layer(inp, slot_map=sm)
    ids, w, we, y = oracle_layer(inp, inp.logits.numpy(), slot_map=sm.numpy())
    assert out["n_miss"][0] == len(set(ids.ravel().tolist()))
    assert np.array_equal(out["miss_ids"][:out["n_miss"][0]], np.unique(ids))
    check_y(out["y"], y, what="shared only")


def test_empty_window_is_a_noop():
    cfg = synth.MoeConfig("empty", H=256, I=128, E=8, k=2, T=4)
    inp = synth.make_layer(cfg, 0).to(DEV)
    lay = MoeLayer(inp, T_max=4)
    out = lay.alloc_outputs(0)
    out["n_miss"].fill_(5)
    _lib.moe_layer_forward(lay.desc, None, None, lay.x_dtype, 0, None, out["y"], out["ids"],
                           out["w"], out["miss_ids"], out["n_miss"], lay.ws_ptr, lay.ws_bytes)
    torch.cuda.synchronize()
    assert int(out["n_miss"].item()) == 0


@pytest.mark.parametrize("I", [768, 256])
def test_deterministic_and_window_composition_invariant(I):
    """Same inputs, same bits (run to run); and on the decode path a row's output
    does not depend on the other rows of its window, bit for bit, in windows of
    1, 2, 4, 8, 12 and 16 rows: alone, a row's groups of I are split into half
    units, in the 16-row window they are not."""
    cfg = synth.DECODE_WINDOW.with_T(16)
    if I != cfg.I:
        cfg = synth.MoeConfig("inv", H=cfg.H, I=I, E=cfg.E, k=cfg.k, T=16, shared_I=I, zipf_s=cfg.zipf_s)
    inp = synth.make_layer(cfg, 11, device=DEV)
    out1, lay = run_layer(inp)
    out2, _ = run_layer(inp, lay=lay)
    assert hashlib.sha256(out1["y"].tobytes()).hexdigest() == hashlib.sha256(out2["y"].tobytes()).hexdigest()
    rng = np.random.default_rng(3)
    for t, n in ((0, 8), (5, 4), (15, 12), (3, 1), (9, 1), (7, 2)):
        others = rng.permutation([r for r in range(cfg.T) if r != t])[:n - 1]
        rows = torch.tensor([t, *others.tolist()], dtype=torch.long, device=inp.x.device)
        sub, _ = run_layer(inp, logits=inp.logits[rows], x=inp.x[rows], lay=lay)
        assert sub["y"][0].tobytes() == out1["y"][t].tobytes(), (t, n)


@pytest.mark.parametrize("D", [25, 35])
def test_split_tail_groups_match_whole_units(D):
    """A window touching 25 (35) experts has 156 (216) groups of I for 152 SMs:
    the groups past the first round are split into half units. Its rows are
    bitwise equal to the same rows computed alone (every group split) and match
    the oracle."""
    cfg = synth.DECODE_WINDOW.with_T(8)
    inp = synth.make_layer(cfg, 21)
    pool = np.arange(D) * 3
    stride = (D + cfg.T - 1) // cfg.T
    ids = np.array([[pool[(stride * t + j) % D] for j in range(cfg.k)] for t in range(cfg.T)], np.int32)
    assert len(np.unique(ids)) == D
    rng = np.random.default_rng(5)
    w = rng.random((cfg.T, cfg.k)).astype(np.float32) + 0.1
    w = (w / w.sum(1, keepdims=True)).astype(np.float32)
    dinp = inp.to(DEV)
    lay = MoeLayer(dinp, T_max=cfg.T)
    ids_d, w_d = torch.from_numpy(ids).to(DEV), torch.from_numpy(w).to(DEV)
    y = lay.expert_ffn(dinp.x, ids_d, w_d)["y"].cpu().numpy()
    torch.cuda.synchronize()
    code, bits = lay.status()
    assert code == _lib.MOE_OK, bits
    for t in range(cfg.T):
        yt = lay.expert_ffn(dinp.x[t:t + 1], ids_d[t:t + 1], w_d[t:t + 1])["y"].cpu().numpy()
        assert yt[0].tobytes() == y[t].tobytes(), t
    L = oracle.Layer(inp)
    check_y(y, L.rows(ids, w), what="split tail")


def test_launch_count_reported():
    cfg = synth.MoeConfig("lc", H=256, I=128, E=8, k=2, T=4)
    inp = synth.make_layer(cfg, 0)
    run_layer(inp)
    assert _lib.moe_last_launch_count() >= 3


# ---------------------------------------------------------------- one-launch decode path
def test_fused_all_missing_without_shared_gives_zero():
    cfg = synth.MoeConfig("f0", H=512, I=256, E=16, k=4, T=6, zipf_s=1.0)
    inp = synth.make_layer(cfg, 3)
    sm = torch.full((cfg.E,), -1, dtype=torch.int32)
    out, _ = run_layer(inp, slot_map=sm)
    assert np.all(out["y"] == 0)
    ids, _, _ = oracle.route(inp.logits.numpy(), cfg.k)
    assert out["n_miss"][0] == len(np.unique(ids))


def test_fused_no_resident_expert_gives_shared_only():
    cfg = synth.MoeConfig("f1", H=512, I=256, E=16, k=4, T=6, shared_I=512, zipf_s=1.0)
    inp = synth.make_layer(cfg, 4)
    sm = torch.full((cfg.E,), -1, dtype=torch.int32)
    out, _ = run_layer(inp, slot_map=sm)
    ids, w, we, y = oracle_layer(inp, inp.logits.numpy(), slot_map=sm.numpy())
    check_y(out["y"], y, what="fused shared only")


def test_fused_ffn_mode_matches_layer_mode_and_repeats():
    """moe_expert_ffn (routing given) and moe_layer_forward agree bit for bit, and
    repeated calls on one workspace give the same bits (counters reset)."""
    cfg = synth.MoeConfig("f2", H=2048, I=768, E=128, k=8, T=12, shared_I=768, zipf_s=1.1)
    inp = synth.make_layer(cfg, 8, device=DEV)
    out1, lay = run_layer(inp)
    ids = torch.from_numpy(out1["ids"]).to(DEV)
    w = torch.from_numpy(out1["w"]).to(DEV)
    for _ in range(3):
        o2 = lay.expert_ffn(inp.x, ids, w)
        torch.cuda.synchronize()
        assert np.array_equal(o2["y"].cpu().numpy(), out1["y"])
        out3, _ = run_layer(inp, lay=lay)
        assert np.array_equal(out3["y"], out1["y"])
    code, bits = lay.status()
    assert code == _lib.MOE_OK, bits


def test_fused_window_sizes_share_one_workspace():
    cfg = synth.MoeConfig("f3", H=1024, I=512, E=64, k=6, T=16, shared_I=256, zipf_s=1.0)
    inp = synth.make_layer(cfg, 12, device=DEV)
    lay = MoeLayer(inp, T_max=16)
    hinp = inp.to("cpu")
    for T in (16, 1, 7, 16, 3):
        out, _ = run_layer(inp, logits=inp.logits[:T], x=inp.x[:T], lay=lay)
        ids, w, _ = oracle.route(hinp.logits[:T].numpy(), cfg.k)
        y = oracle.Layer(hinp).rows(ids, w)
        check_y(out["y"], y, what=f"T={T}")


def test_fused_flags_non_finite_logit():
    cfg = synth.MoeConfig("f4", H=512, I=256, E=16, k=4, T=4, zipf_s=1.0)
    inp = synth.make_layer(cfg, 1).to(DEV)
    lay = MoeLayer(inp, T_max=4)
    lg = inp.logits.clone()
    lg[1, 3] = float("nan")
    lay.forward(lg, inp.x)
    code, bits = lay.status()
    assert code == _lib.MOE_ERR_DEVICE and bits & 1
    lay.clear_status()
    lay.forward(inp.logits, inp.x)
    assert lay.status()[0] == _lib.MOE_OK


def test_negative_control_one_corrupted_byte_fails_the_gate():
    """Negative control on the GPU path: one flipped bit (the exponent's top bit)
    in one byte of an fp16 scale of a routed expert's down matrix. Against the
    intact layer's oracle, the rows routed to that expert must then fail the
    2e-3 gate, so the gate compares bytes and is not vacuous. The corrupted pool
    must still match its own oracle, and the rows not routed to that expert must
    be bitwise unchanged."""
    cfg = synth.DECODE_WINDOW
    inp = synth.make_layer(cfg, 0, device=DEV)
    out, _ = run_layer(inp)
    hinp = inp.to("cpu")
    ids, w, we, y = oracle_layer(hinp, hinp.logits.numpy())
    check_y(out["y"], y, what="intact")
    e = int(ids[0][0])
    bad = synth.clone_pool(inp)
    b = bad.down_s.view(torch.uint8).view(cfg.E, cfg.H, cfg.I // 32, 2)
    b[e, 0, 0, 1] ^= 0x40
    out_bad, _ = run_layer(bad)
    assert np.array_equal(out_bad["ids"], ids)
    hit = [t for t in range(cfg.T) if e in ids[t]]
    miss = [t for t in range(cfg.T) if e not in ids[t]]
    dy = np.abs(out_bad["y"][hit].astype(np.float64) - y[hit]).max()
    assert dy > TOL * np.abs(y).max(), dy
    y_bad = oracle.Layer(bad.to("cpu")).rows(ids, w, rows=hit)
    check_y(out_bad["y"][hit], y_bad, what="corrupted pool")
    assert np.array_equal(out_bad["y"][miss], out["y"][miss])


# ---------------------------------------------------------------- more shapes and flags
def test_prefill_without_shared_expert():
    cfg = synth.MoeConfig("pf_noshared", H=1024, I=512, E=64, k=6, T=200, zipf_s=1.0)
    inp = synth.make_layer(cfg, 11)
    out, _ = run_layer(inp)
    ids, w, we, y = oracle_layer(inp, inp.logits.numpy())
    assert np.array_equal(out["ids"], ids)
    assert_weights_match(out["w"], w, we)
    check_y(out["y"], y, what="prefill without shared expert")


def test_fp32_chunk_takes_the_separate_path_with_chunked_permutation():
    cfg = synth.MoeConfig("f32_chunk", H=384, I=256, E=48, k=8, T=160, shared_I=128, zipf_s=1.0,
                          x_dtype="f32")
    assert cfg.T * cfg.k > 1024
    inp = synth.make_layer(cfg, 12)
    out, _ = run_layer(inp)
    ids, w, we, y = oracle_layer(inp, inp.logits.numpy())
    assert np.array_equal(out["ids"], ids)
    check_y(out["y"], y, what="fp32 chunk")


def test_fused_slot_beyond_pool_is_flagged_and_treated_as_miss():
    cfg = synth.MoeConfig("badslot", H=1024, I=256, E=32, k=4, T=8, shared_I=256, zipf_s=1.0)
    inp = synth.make_layer(cfg, 13)
    ids, _, _ = oracle.route(inp.logits.numpy(), cfg.k)
    e_bad = int(ids[0][0])
    sm = torch.arange(cfg.E, dtype=torch.int32)
    sm[e_bad] = cfg.E + 5  # beyond the pool's S = E slots
    dinp = inp.to(DEV)
    lay = MoeLayer(dinp, T_max=cfg.T)
    out = lay.forward(dinp.logits, dinp.x, slot_map=sm.to(DEV))
    torch.cuda.synchronize()
    code, bits = lay.status()
    assert bits & 2 and code == _lib.MOE_ERR_DEVICE
    sm_ref = sm.clone()
    sm_ref[e_bad] = -1
    y = oracle.Layer(inp).rows(ids, oracle.route(inp.logits.numpy(), cfg.k)[1], slot_map=sm_ref.numpy())
    check_y(out["y"].cpu().numpy(), y, what="bad slot as miss")
    assert int(out["n_miss"].item()) >= 1
    assert e_bad in out["miss_ids"].cpu().numpy()[:int(out["n_miss"].item())]


@pytest.mark.parametrize("E,k", [(40, 1), (100, 3)])
def test_fused_odd_expert_counts(E, k):
    cfg = synth.MoeConfig("odd", H=1024, I=256, E=E, k=k, T=8, shared_I=256, zipf_s=1.0)
    inp = synth.make_layer(cfg, 14)
    out, _ = run_layer(inp)
    ids, w, we, y = oracle_layer(inp, inp.logits.numpy())
    assert np.array_equal(out["ids"], ids)
    assert_weights_match(out["w"], w, we)
    check_y(out["y"], y, what=f"E={E} k={k}")
