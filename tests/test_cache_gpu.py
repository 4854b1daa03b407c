"""The adaptive cache planner driving the decode path on the GPU: windows read a
pool of a few slots through the planner's slot map, the planner's moves are
copied from a host store of every expert into the pool between windows, and
each window's output equals the oracle's for the experts held at that window."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from routed_expert_ffn_router_gb300 import synth  # noqa: E402
from routed_expert_ffn_router_gb300.cache import ExpertCache  # noqa: E402
from routed_expert_ffn_router_gb300.layer import MoeLayer  # noqa: E402

POOL = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")
TOL = 2e-3


@pytest.mark.gpu
def test_adaptive_cache_drives_the_decode_path():
    dev = torch.device("cuda", 0)
    cfg = synth.MoeConfig("ac", H=512, I=256, E=32, k=4, T=8, shared_I=256, zipf_s=1.2)
    store = synth.make_layer(cfg, 7)                 # host: every expert
    S = 10
    dinp = store.to(dev)
    for name in POOL:                                # the device pool: S empty slots
        t = getattr(store, name)
        setattr(dinp, name, torch.zeros((S,) + tuple(t.shape[1:]), dtype=t.dtype, device=dev))
    dinp.S = S
    lay = MoeLayer(dinp, T_max=cfg.T)
    cache = ExpertCache(1, cfg.E, [S])
    logits, xs = synth.draw_windows(store, 40, seed=3, device="cpu")
    sm_dev = torch.full((cfg.E,), -1, dtype=torch.int32, device=dev)
    ref = oracle.Layer(store)
    misses = []
    for w in range(40):
        out = lay.forward(logits[w].to(dev), xs[w].to(dev), slot_map=sm_dev)
        torch.cuda.synchronize()
        ids, wts = out["ids"].cpu().numpy(), out["w"].cpu().numpy()
        o_ids, _, _ = oracle.route(logits[w].numpy(), cfg.k)
        assert np.array_equal(ids, o_ids)
        sm = cache.slot_map(0)
        held = np.where(sm >= 0, np.arange(cfg.E), -1).astype(np.int32)  # the store, masked
        y = ref.rows(ids, wts, slot_map=held, x=xs[w].numpy())
        yg = out["y"].cpu().double().numpy()
        assert np.abs(yg - y).max() <= TOL * np.abs(y).max(), f"window {w}"
        misses.append(int(out["n_miss"].item()))
        cache.observe(0, ids)
        for _, s, e_in, _ in cache.advance(4):        # 4 batch slots of token + draft
            for name in POOL:
                getattr(dinp, name)[s].copy_(getattr(store, name)[e_in])
        sm_dev.copy_(torch.from_numpy(cache.slot_map(0)))
    assert cache.swapped_total() >= S
    assert misses[0] > 0 and sum(misses[-10:]) < sum(misses[:10])


@pytest.mark.gpu
@pytest.mark.parametrize("path", ["fused_bf16", "separate_f32", "prefill"])
def test_device_pick_counters(path):
    """moe_layer_desc.pick_counts: each call of T <= pick_max_rows rows adds one
    pick per distinct expert its window routes to (resident or not), on every
    path; larger calls add nothing; moe_cache_observe_device reads and clears
    the counters and the planner's heats equal per-window host observation."""
    from routed_expert_ffn_router_gb300 import _lib
    dev = torch.device("cuda", 0)
    T = {"fused_bf16": 8, "separate_f32": 6, "prefill": 40}[path]
    cfg = synth.MoeConfig("pc", H=512, I=256, E=48, k=4, T=T, shared_I=256, zipf_s=1.0,
                          x_dtype="f32" if path == "separate_f32" else "bf16")
    inp = synth.make_layer(cfg, 5)
    smt, S = synth.random_slot_map(cfg.E, 0.5, seed=4)
    keep = (smt >= 0).nonzero().flatten()
    for name in POOL:
        setattr(inp, name, getattr(inp, name)[keep].contiguous())
    inp.S = S
    inp.slot_map = smt
    dinp = inp.to(dev)
    lay = MoeLayer(dinp, T_max=cfg.T)
    counts = torch.zeros(1, cfg.E, dtype=torch.int32, device=dev)
    lay.desc.pick_counts = counts.data_ptr()
    lay.desc.pick_max_rows = 32
    logits, xs = synth.draw_windows(inp, 5, seed=8, device="cpu")
    host = ExpertCache(1, cfg.E, [S])
    expect = np.zeros(cfg.E, np.int64)
    for w in range(5):
        out = lay.forward(logits[w].to(dev), xs[w].to(dev))
        torch.cuda.synchronize()
        assert lay.status()[0] == _lib.MOE_OK
        ids = out["ids"].cpu().numpy()
        if T <= 32:
            expect[np.unique(ids)] += 1
            host.observe(0, ids)
    assert np.array_equal(counts.cpu().numpy()[0], expect)
    cache = ExpertCache(1, cfg.E, [S])
    cache.observe_device(counts)
    torch.cuda.synchronize()
    assert int(counts.abs().sum().item()) == 0
    np.testing.assert_allclose(cache.heat(0), host.heat(0), rtol=1e-12, atol=0)
    if T > 32:  # the same chunk counts once the limit allows it
        lay.desc.pick_max_rows = T
        out = lay.forward(logits[0].to(dev), xs[0].to(dev))
        torch.cuda.synchronize()
        got = counts.cpu().numpy()[0]
        exp1 = np.zeros(cfg.E, np.int32)
        exp1[np.unique(out["ids"].cpu().numpy())] = 1
        assert np.array_equal(got, exp1)
