"""The mailbox: experts the slot map does not hold, computed by the library's
host threads ("extended-strata-moe reference", "The mailbox").

CPU tests: the pair list, the host experts against the oracle (the sum of a
row's partials equals the oracle's layer restricted to the missed experts),
determinism across thread counts, and peers that stall or are lost (failure
injected on the host: the call reports a timeout and the mailbox serves the
next call). GPU test: the whole window (held experts on the GPU, missed ones on
the host, added on the GPU) equals the oracle with every expert held."""
import numpy as np
import pytest
import torch

import oracle
from routed_expert_ffn_router_gb300 import _lib, synth
from routed_expert_ffn_router_gb300 import build as libbuild
from routed_expert_ffn_router_gb300.mailbox import Mailbox

TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    libbuild.build()
    _lib.load()


def _case(seed=3, T=6, x_dtype="bf16"):
    cfg = synth.MoeConfig("mb", H=256, I=128, E=24, k=4, T=T, zipf_s=1.0, x_dtype=x_dtype)
    inp = synth.make_layer(cfg, seed)
    sm, _ = synth.random_slot_map(cfg.E, 0.5, seed=seed + 1)
    ids, w, _ = oracle.route(inp.logits.numpy(), cfg.k)
    return cfg, inp, sm.numpy(), ids, w


def test_pairs_lists_the_missed_pairs_in_order():
    mb = Mailbox(_case()[1], n_threads=1)
    ids = np.array([[3, 1], [0, 2], [1, 3]], np.int32)
    sm = np.array([0, -1, 1, -1], np.int32)
    assert list(mb.pairs(ids, sm)) == [0, 1, 4, 5]
    with pytest.raises(_lib.MoeError):
        mb.pairs(np.array([[0, 9]], np.int32), sm)
    cfg, inp, sm, ids, w = _case()
    ref = [p for p in range(ids.size) if sm[ids.ravel()[p]] < 0]
    assert list(mb.pairs(ids, sm)) == ref
    mb.close()


@pytest.mark.parametrize("x_dtype", ["bf16", "f32"])
def test_host_experts_match_the_oracle(x_dtype):
    cfg, inp, sm, ids, w = _case(x_dtype=x_dtype)
    mb = Mailbox(inp, n_threads=3)
    pairs = mb.pairs(ids, sm)
    assert len(pairs) > 0
    part = mb.compute(inp.x, ids, w, pairs)
    y = np.zeros((cfg.T, cfg.H))
    for i, p in enumerate(pairs):
        y[p // cfg.k] += part[i]
    # the oracle restricted to the missed experts (held in their own slots)
    only_missed = np.where(sm < 0, np.arange(cfg.E), -1).astype(np.int32)
    y_ref = oracle.Layer(inp).rows(ids, w, slot_map=only_missed)
    assert np.abs(y - y_ref).max() <= TOL * np.abs(y_ref).max()
    mb.close()


def test_results_do_not_depend_on_the_thread_count():
    cfg, inp, sm, ids, w = _case(seed=7, T=12)
    outs = []
    for n in (1, 4, 7):
        mb = Mailbox(inp, n_threads=n)
        pairs = mb.pairs(ids, sm)
        outs.append(mb.compute(inp.x, ids, w, pairs).tobytes())
        mb.close()
    assert outs[0] == outs[1] == outs[2]


@pytest.mark.parametrize("mode", [1, 2])
def test_a_stalled_or_lost_peer_times_out_and_the_mailbox_recovers(mode):
    cfg, inp, sm, ids, w = _case(seed=9)
    mb = Mailbox(inp, n_threads=2, timeout_ms=300)
    pairs = mb.pairs(ids, sm)
    good = mb.compute(inp.x, ids, w, pairs)
    mb.inject(mode)
    with pytest.raises(_lib.MoeError) as ei:
        mb.compute(inp.x, ids, w, pairs)
    assert ei.value.code == _lib.MOE_ERR_TIMEOUT
    again = mb.compute(inp.x, ids, w, pairs)
    assert again.tobytes() == good.tobytes()
    mb.close()


def test_argument_errors():
    cfg, inp, sm, ids, w = _case()
    mb = Mailbox(inp, n_threads=1)
    pairs = mb.pairs(ids, sm)
    with pytest.raises(_lib.MoeError):
        mb.compute(inp.x, ids, w, pairs[::-1].copy())  # not ascending
    bad = pairs.copy()
    bad[-1] = ids.size
    with pytest.raises(_lib.MoeError):
        mb.compute(inp.x, ids, w, bad)
    assert _lib.load().moe_mailbox_create(0, 10) is None
    with pytest.raises(_lib.MoeError):
        mb.inject(3)
    mb.close()


@pytest.mark.gpu
def test_window_with_missed_experts_equals_every_expert_held():
    from routed_expert_ffn_router_gb300.layer import MoeLayer
    dev = torch.device("cuda", 0)
    cfg = synth.MoeConfig("mbgpu", H=1024, I=512, E=64, k=8, T=16, shared_I=512, zipf_s=1.2)
    store = synth.make_layer(cfg, 5)
    smt, S = synth.random_slot_map(cfg.E, 0.6, seed=2)
    pool = synth.make_layer(cfg, 5)
    keep = (smt >= 0).nonzero().flatten()
    for name in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s"):
        setattr(pool, name, getattr(pool, name)[keep].contiguous())
    pool.S = S
    pool.slot_map = smt
    dpool = pool.to(dev)
    lay = MoeLayer(dpool, T_max=cfg.T)
    mb = Mailbox(store, n_threads=4)
    outs = []
    for _ in range(2):
        out = mb.forward(lay, dpool.logits, dpool.x, dpool.slot_map)
        torch.cuda.synchronize()
        assert lay.status()[0] == _lib.MOE_OK
        assert len(out["mailbox_pairs"]) > 0
        outs.append(out["y"].cpu().numpy())
    assert outs[0].tobytes() == outs[1].tobytes()
    ids, w, _ = oracle.route(store.logits.numpy(), cfg.k)
    y_ref = oracle.Layer(store).rows(ids, w)  # every expert held
    assert np.abs(outs[0] - y_ref).max() <= TOL * np.abs(y_ref).max()
    mb.close()
