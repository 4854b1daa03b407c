"""The seeded synthetic inputs follow the stated recipe: Zipf-biased logits
N(0,1) - s ln r(e) over a seeded popularity permutation, the expert-cache slot
map holding the hottest experts in rank order, weights N(0, 0.02) encoded as
symmetric int4 blocks of 32 with an fp16 scale amax/7, bf16 activations
N(0,1), reproducible per seed, and the routing skew the workloads are sized
for. Logits and ranks are drawn before anything whose size depends on H or I,
so small-H copies of the real configurations carry their exact logits."""
import dataclasses

import numpy as np
import pytest
import torch

from routed_expert_ffn_router_gb300 import synth


def small(cfg, **kw):
    shared = 128 if cfg.shared_I else 0
    return dataclasses.replace(cfg, H=128, I=128, shared_I=shared, **kw)


def decode_weights(q, s):
    """Stored weights of a [rows][K/2] code / [rows][K/32] scale pair (numpy)."""
    q = q.numpy().astype(np.int32)
    lo, hi = q & 0xF, q >> 4
    n = np.stack([lo, hi], axis=-1).reshape(q.shape[0], -1)
    code = n - 16 * (n >> 3)
    scale = s.numpy().view(np.float16).astype(np.float64)
    return code, code * np.repeat(scale, 32, axis=1)


@pytest.mark.parametrize("name", ["decode_window", "expert_cache", "prefill", "decode48"])
def test_logits_are_unit_noise_plus_the_zipf_log_bias(name):
    base = synth.CONFIGS[name]
    cfg = small(base)
    inp = synth.make_layer(cfg, 0, T=2048)
    rank = inp.rank.numpy()
    assert sorted(rank.tolist()) == list(range(1, cfg.E + 1))
    noise = inp.logits.numpy().astype(np.float64) + cfg.zipf_s * np.log(rank)[None, :]
    assert abs(noise.mean()) < 0.01 and abs(noise.std() - 1.0) < 0.01
    # the popularity shows in the column means: they follow -s ln r(e)
    col = inp.logits.numpy().mean(axis=0)
    assert np.corrcoef(col, -np.log(rank))[0, 1] > 0.95


def test_expert_cache_slot_map_holds_the_hottest_in_rank_order():
    cfg = small(synth.EXPERT_CACHE)
    inp = synth.make_layer(cfg, 0)
    assert inp.S == 154 == cfg.n_resident            # floor(0.6 * 256 + 0.5)
    rank = inp.rank.numpy()
    want = np.where(rank <= 154, rank - 1, -1)
    assert np.array_equal(inp.slot_map.numpy(), want)
    assert inp.gate_q.shape[0] == inp.down_s.shape[0] == 154


def test_weights_are_symmetric_int4_blocks_of_the_stated_spread():
    cfg = synth.MoeConfig("w", H=256, I=128, E=3, k=2, T=2, shared_I=128, zipf_s=1.0)
    inp = synth.make_layer(cfg, 4)
    vals = []
    for qn, sn, rows, K in (("gate_q", "gate_s", cfg.I, cfg.H), ("up_q", "up_s", cfg.I, cfg.H),
                            ("down_q", "down_s", cfg.H, cfg.I)):
        for e in range(cfg.E):
            code, w = decode_weights(getattr(inp, qn)[e], getattr(inp, sn)[e])
            assert code.shape == (rows, K)
            assert code.min() >= -7 and code.max() <= 7   # -8 needs |w| > 7.5 scales
            blk = np.abs(code).reshape(rows, K // 32, 32).max(axis=2)
            assert np.all(blk == 7)                       # each block's amax maps to +-7
            vals.append(w.ravel())
    v = np.concatenate(vals)
    assert abs(v.mean()) < 5e-4 and abs(v.std() / 0.02 - 1.0) < 0.03


def test_activations_are_bf16_unit_normal():
    cfg = small(synth.DECODE_WINDOW)
    inp = synth.make_layer(cfg, 0, T=512)
    x = synth.bf16_bits_to_f32(inp.x.numpy()).astype(np.float64)
    assert x.shape == (512, 128)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01


def test_inputs_are_reproducible_per_seed():
    cfg = synth.MoeConfig("r", H=256, I=128, E=4, k=2, T=3, shared_I=128, zipf_s=1.0)
    a, b, c = synth.make_layer(cfg, 7), synth.make_layer(cfg, 7), synth.make_layer(cfg, 8)
    for f in ("logits", "x", "gate_q", "gate_s", "up_q", "down_s"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f
    assert not torch.equal(a.logits, c.logits) and not torch.equal(a.gate_q, c.gate_q)
    assert torch.equal(a.sh["down_q"], b.sh["down_q"])


def _distinct_and_counts(logits, k):
    ids = torch.topk(torch.as_tensor(logits), k, dim=-1).indices.numpy().reshape(-1)
    counts = np.bincount(ids)
    return int((counts > 0).sum()), counts


def test_decode_window_touches_about_two_dozen_experts():
    cfg = small(synth.DECODE_WINDOW)
    inp = synth.make_layer(cfg, 0)
    logits, _ = synth.draw_windows(inp, 64, seed=1)
    d = [_distinct_and_counts(logits[w].numpy(), cfg.k)[0] for w in range(64)]
    assert 20 <= np.mean(d) <= 28


def test_prefill_chunk_routing_is_heavily_skewed():
    cfg = small(synth.PREFILL)
    inp = synth.make_layer(cfg, 0)
    D, counts = _distinct_and_counts(inp.logits.numpy(), cfg.k)
    assert 180 <= D <= 260                 # about 209 of 512 experts touched
    assert 1200 <= counts.max() <= 2800    # the hottest expert takes most of the 2,048 rows
    assert 10 <= int((counts >= 128).sum()) <= 45
    assert counts.sum() == cfg.T * cfg.k
