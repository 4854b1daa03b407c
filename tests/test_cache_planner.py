"""Adaptive expert cache planner (host code of libmoe_gb300.so) and the STRP
profile: pinned by hand-worked cases of the rules in "extended-strata-moe
reference", "The adaptive cache" / "Profile format (STRP)", and compared with
the plain-Python oracle on random routing traces, decision for decision and
heat for heat (no GPU needed)."""
import struct

import numpy as np
import pytest

from oracle.cache_oracle import CacheOracle
from routed_expert_ffn_router_gb300 import _lib
from routed_expert_ffn_router_gb300 import build as libbuild
from routed_expert_ffn_router_gb300.cache import ExpertCache


@pytest.fixture(scope="module", autouse=True)
def lib():
    libbuild.build()
    return _lib.load()


def window(c, layer, rows):
    c.observe(layer, np.asarray(rows, np.int32))


class OracleCache:
    """The oracle behind the library planner's Python interface, so that the
    hand-worked pins below hold for both."""

    def __init__(self, n_layers, n_experts, slots, **params):
        self.o = CacheOracle(n_layers, n_experts, list(np.broadcast_to(slots, (n_layers,))), **params)
        self.max_swaps = self.o.max_swaps

    def set_resident(self, layer, experts):
        self.o.set_resident(layer, list(experts))

    def observe(self, layer, ids):
        self.o.observe(layer, np.asarray(ids).tolist())

    def advance(self, n):
        return self.o.advance(n)

    def rebalance(self, max_swaps=None):
        return self.o.rebalance(self.max_swaps if max_swaps is None else max_swaps)

    def slot_map(self, layer):
        return np.asarray(self.o.slot_map(layer))

    def heat(self, layer):
        return np.asarray(self.o.heat[layer])

    def profile_bytes(self):
        return self.o.profile_bytes()

    def load_profile(self, b):
        self.o.load_profile(b)


@pytest.fixture(params=["library", "oracle"])
def Cache(request):
    return ExpertCache if request.param == "library" else OracleCache


# ----------------------------------------------------------------- pins
def test_half_life(Cache):
    c = Cache(1, 4, [1])
    window(c, 0, [[2]])
    c.advance(350)                       # one half-life
    assert c.heat(0)[2] == 0.5
    c.advance(700)                       # two more
    assert c.heat(0)[2] == 0.125


def test_one_pick_per_expert_and_window_and_large_windows_do_not_count(Cache):
    c = Cache(1, 8, [2])
    window(c, 0, [[1, 2], [2, 1], [1, 3]])
    assert list(c.heat(0)[:4]) == [0.0, 1.0, 1.0, 1.0]
    window(c, 0, [[5, 6]] * 33)          # 33 rows: a large batch
    assert c.heat(0)[5] == 0.0
    window(c, 0, [[5, 6]] * 32)          # 32 rows still count
    assert c.heat(0)[5] == 1.0


def test_free_slots_filled_hottest_first_every_8_tokens(Cache):
    c = Cache(1, 8, [2])
    for _ in range(2):
        window(c, 0, [[5]])
    window(c, 0, [[3]])
    window(c, 0, [[7]])
    assert c.advance(7) == []            # no fill round before 8 tokens
    moves = c.advance(1)
    assert moves == [(0, 0, 5, -1), (0, 1, 3, -1)]   # hotter first; 3 before 7 on equal heat
    assert list(c.slot_map(0)) == [-1, -1, -1, 1, -1, 0, -1, -1]


def test_hysteresis_ratio_plus_picks(Cache):
    """An expert comes in only when heat_in - 2 > 1.5 * heat_out."""
    c = Cache(1, 4, [1])
    c.set_resident(0, [0])
    for _ in range(2):
        window(c, 0, [[0]])              # held: heat 2
    for _ in range(5):
        window(c, 0, [[1]])              # outside: heat 5, 5 - 2 = 3 is not > 3
    assert c.rebalance() == []
    window(c, 0, [[1]])                  # heat 6: 4 > 3
    assert c.rebalance() == [(0, 0, 1, 0)]
    assert list(c.slot_map(0)) == [-1, 0, -1, -1]


def test_swap_round_every_32_tokens_and_cap(Cache):
    c = Cache(1, 200, [100], max_swaps=64, half_life_tokens=1e9)
    c.set_resident(0, range(100))        # held experts 0..99, heat 0
    for _ in range(3):
        window(c, 0, [[e] for e in range(100, 200)][:32])  # 32-row windows: experts 100..131
    for e0 in range(132, 200, 32):
        for _ in range(3):
            window(c, 0, [[e] for e in range(e0, min(e0 + 32, 200))])
    for t in (8, 16, 24):
        moves = c.advance(8)
        assert moves == [], t            # fill rounds: no free slot; no swap round yet
    moves = c.advance(8)                 # clock 32: the swap round
    assert len(moves) == 64              # at most 64 per round
    assert [m[2] for m in moves] == list(range(100, 164))   # equal heat: lower id first
    assert [m[3] for m in moves] == list(range(64))          # coldest held, lower id first


def test_layers_held_whole_are_left_alone(Cache):
    c = Cache(2, 4, [4, 2])
    c.set_resident(0, [0, 1, 2, 3])
    c.set_resident(1, [0, 1])
    for _ in range(10):
        window(c, 0, [[0]])
        window(c, 1, [[3]])
    # layer 1: expert 3 (heat 10) replaces the coldest held expert, 0 (heat 0, the
    # lower id of two); layer 0 holds every expert and is not touched
    assert c.rebalance() == [(1, 0, 3, 0)]
    assert list(c.slot_map(0)) == [0, 1, 2, 3]


def test_argument_errors():
    c = ExpertCache(2, 8, [2, 2])
    with pytest.raises(_lib.MoeError):
        c.observe(2, np.zeros((1, 2), np.int32))        # no such layer
    with pytest.raises(_lib.MoeError):
        c.observe(0, np.full((1, 2), 8, np.int32))      # expert out of range
    with pytest.raises(_lib.MoeError):
        c.set_resident(0, [1, 1])                       # repeated expert
    with pytest.raises(_lib.MoeError):
        c.set_resident(0, [1, 2, 3])                    # more than the slots
    with pytest.raises(ValueError):
        ExpertCache(2, 8, [2, -1])
    L = _lib.load()
    assert L.moe_cache_advance(c.state.ctypes.data, 8, c._moves, c.n_max - 1) == -1  # array too small
    assert L.moe_cache_advance(None, 8, c._moves, c.n_max) == -1


# ----------------------------------------------------------------- STRP
def parse_strp(b):
    """An independent reader of the page's layout."""
    assert b[:4] == b"STRP"
    version, L, E, slots, n = struct.unpack_from("<5I", b, 4)
    pairs = [struct.unpack_from("<2H", b, 24 + 4 * i) for i in range(n)]
    ranks = struct.unpack_from(f"<{L * E}i", b, 24 + 4 * n)
    assert len(b) == 24 + 4 * n + 4 * L * E
    return version, L, E, slots, pairs, ranks


def test_profile_write_layout_and_load(Cache):
    c = Cache(2, 6, [2, 3])
    for _ in range(3):
        window(c, 1, [[4]])
    for _ in range(2):
        window(c, 0, [[5]])
        window(c, 1, [[0]])
    window(c, 0, [[1]])
    version, L, E, slots, pairs, ranks = parse_strp(c.profile_bytes())
    assert (version, L, E, slots) == (1, 2, 6, 5)
    assert pairs == [(1, 4), (0, 5), (1, 0), (0, 1)]   # heat 3, 2, 2, 1; ties: lower layer
    assert ranks[1 * 6 + 4] == 0 and ranks[0 * 6 + 1] == 3 and ranks[0] == -1
    d = Cache(2, 6, [1, 3])
    d.load_profile(c.profile_bytes())
    assert list(d.slot_map(0)) == [-1, -1, -1, -1, -1, 0]      # one slot: the hottest of layer 0
    assert list(d.slot_map(1)) == [1, -1, -1, -1, 0, -1]


@pytest.mark.parametrize("mutate", ["magic", "version", "layers", "experts", "n_ranked", "pair", "short"])
def test_profile_validation(mutate):
    c = ExpertCache(2, 6, [2, 2])
    window(c, 0, [[1]])
    b = bytearray(c.profile_bytes())
    if mutate == "magic":
        b[0:4] = b"STRQ"
    elif mutate == "version":
        struct.pack_into("<I", b, 4, 2)
    elif mutate == "layers":
        struct.pack_into("<I", b, 8, 3)
    elif mutate == "experts":
        struct.pack_into("<I", b, 12, 7)
    elif mutate == "n_ranked":
        struct.pack_into("<I", b, 20, 13)
    elif mutate == "pair":
        struct.pack_into("<2H", b, 24, 0, 6)
    else:
        b = b[:27]
    with pytest.raises(_lib.MoeError):
        c.load_profile(bytes(b))
    with pytest.raises(ValueError):
        CacheOracle(2, 6, [2, 2]).load_profile(bytes(b))


# ----------------------------------------------------------------- oracle parity
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_oracle_on_random_traces(seed):
    rng = np.random.default_rng(seed)
    L, E, k = 4, 40, 4
    slots = [8, 40, 0, 13]                     # a partial, a whole, an empty and a partial layer
    params = dict(half_life_tokens=50.0, round_every_tokens=16, max_swaps=5, fill_every_tokens=4,
                  max_fills=6, in_ratio=1.5, in_picks=2.0, max_window_tokens=32)
    c = ExpertCache(L, E, slots, **params)
    o = CacheOracle(L, E, slots, **params)
    c.set_resident(1, range(40))
    o.set_resident(1, range(40))
    pop = [rng.permutation(E) for _ in range(L)]
    n_fill = n_swap = 0
    for step in range(160):
        if step == 80:                          # the popular experts change
            pop = [rng.permutation(E) for _ in range(L)]
        for l in range(L):
            T = int(rng.choice([1, 2, 4, 8, 16, 33]))
            p = 1.0 / np.arange(1, E + 1) ** 1.1
            p = p[np.argsort(pop[l])]
            p /= p.sum()
            rows = [list(rng.choice(E, size=k, replace=False, p=p)) for _ in range(T)]
            c.observe(l, np.asarray(rows, np.int32))
            o.observe(l, rows)
        n = int(rng.choice([1, 2, 4, 8]))
        moves = c.advance(n)
        assert moves == o.advance(n), step
        n_fill += sum(m[3] < 0 for m in moves)
        n_swap += sum(m[3] >= 0 for m in moves)
        if step % 37 == 36:
            assert c.rebalance(3) == o.rebalance(3), step
        for l in range(L):
            assert list(c.slot_map(l)) == o.slot_map(l), (step, l)
            assert list(c.heat(l)) == o.heat[l], (step, l)
    assert c.swapped_total() == o.swapped
    assert n_fill > 10 and n_swap > 10          # both kinds of round did work
    assert c.profile_bytes() == o.profile_bytes()


def test_observe_layers_equals_per_layer_calls():
    rng = np.random.default_rng(5)
    L, E, T, k = 3, 16, 6, 2
    a, b = ExpertCache(L, E, [4, 4, 4]), ExpertCache(L, E, [4, 4, 4])
    for _ in range(5):
        ids = np.stack([np.stack([rng.choice(E, k, replace=False) for _ in range(T)]) for _ in range(L)])
        a.observe_layers(ids)
        for l in range(L):
            b.observe(l, ids[l])
        assert a.advance(4) == b.advance(4)
    for l in range(L):
        assert list(a.heat(l)) == list(b.heat(l))
    bad = np.zeros((L, T, k), np.int32)
    bad[2, 0, 0] = E                         # out of range in the last layer
    before = [a.heat(l).copy() for l in range(L)]
    with pytest.raises(_lib.MoeError):
        a.observe_layers(bad)
    assert all(np.array_equal(a.heat(l), before[l]) for l in range(L))   # nothing counted


def test_copy_moves_fills_the_pool_slots():
    import torch
    from routed_expert_ffn_router_gb300 import synth
    from routed_expert_ffn_router_gb300.cache import POOL_TENSORS, copy_moves
    cfg = synth.MoeConfig("cm", H=128, I=128, E=8, k=2, T=4, zipf_s=1.0)
    store = synth.make_layer(cfg, 2)
    S = 3

    class Pool:
        pass
    pool = Pool()
    for name in POOL_TENSORS:
        t = getattr(store, name)
        setattr(pool, name, torch.zeros((S,) + tuple(t.shape[1:]), dtype=t.dtype))
    c = ExpertCache(1, cfg.E, [S])
    for e in (6, 6, 1, 4, 4, 4):
        window(c, 0, [[e]])
    moves = c.advance(8)
    assert [m[2] for m in moves] == [4, 6, 1]
    copy_moves(pool, store, moves)
    for _, slot, e_in, _ in moves:
        for name in POOL_TENSORS:
            assert torch.equal(getattr(pool, name)[slot], getattr(store, name)[e_in])


def test_observe_counts_matches_the_oracle_and_per_window_picks():
    """Picks counted outside the planner (the device counters) enter the heat
    as the oracle adds them, bit for bit; with no advance between the windows
    they equal the per-window picks to the last bits of the double sum."""
    rng = np.random.default_rng(12)
    L, E, k = 3, 40, 4
    lib_c = ExpertCache(L, E, [8, 40, 0])
    orc = CacheOracle(L, E, [8, 40, 0])
    per_win = ExpertCache(L, E, [8, 40, 0])
    for step in range(6):
        counts = np.zeros((L, E), np.int32)
        for _ in range(5):  # five windows between planner steps
            ids = rng.integers(0, E, size=(L, 4, k)).astype(np.int32)
            for l in range(L):
                counts[l, np.unique(ids[l])] += 1
                per_win.observe(l, ids[l])
        lib_c.observe_counts(counts)
        orc.observe_counts(counts.tolist())
        for l in range(L):
            assert lib_c.heat(l).tobytes() == np.asarray(orc.heat[l], np.float64).tobytes()
            np.testing.assert_allclose(lib_c.heat(l), per_win.heat(l), rtol=1e-12, atol=0)
        assert lib_c.advance(3) == [tuple(m) for m in orc.advance(3)]
        per_win.advance(3)


def test_observe_counts_rejects_negative_counts():
    c = ExpertCache(2, 8, [2, 2])
    bad = np.zeros((2, 8), np.int32)
    bad[1, 3] = -1
    bad[0, 0] = 5
    with pytest.raises(_lib.MoeError):
        c.observe_counts(bad)
    assert c.heat(0)[0] == 0.0  # validated before anything was added
    with pytest.raises(ValueError):
        c.observe_counts(np.zeros((1, 8), np.int32))
