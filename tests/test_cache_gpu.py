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
