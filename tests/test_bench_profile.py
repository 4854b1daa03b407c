"""bench.py's per-kernel event profile must count exactly the kernels of the
timed sequence of graph replays (K steps x launches per step), with the bytes
of those same steps. The library's profiler keeps one event pair per launch
recorded during a capture and, on collect, adds the latest elapsed time of every
pair it holds; pairs of a graph that was not replayed must not be counted
again. A fake of the library and of torch's graph capture reproduces those
semantics on the CPU."""
import contextlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


class FakeLib:
    """Profiler semantics of the C library: enable resets everything, a launch
    during capture registers a pair, collect adds every registered pair once,
    forget drops the registered pairs."""

    def __init__(self):
        self.on = False
        self.capturing = False
        self.pairs = []
        self.total = {"fused_decode": [0.0, 0]}
        self.replayed = 0

    def moe_profile_enable(self, n):
        self.on = n > 0
        self.pairs = []
        self.total = {"fused_decode": [0.0, 0]}

    def moe_profile_forget(self):
        self.pairs = []

    def moe_profile_collect(self):
        for _ in self.pairs:
            self.total["fused_decode"][0] += 0.04
            self.total["fused_decode"][1] += 1

    def moe_profile_totals(self):
        return {k: tuple(v) for k, v in self.total.items()}

    def launch(self):
        if self.on and self.capturing:
            self.pairs.append("fused_decode")


class FakeGraph:
    def __init__(self, lib):
        self.lib = lib
        self.n = 0

    def replay(self):
        self.lib.replayed += self.n


class FakeTorch:
    def __init__(self, lib):
        self.lib = lib
        outer = self

        class _Cuda:
            @staticmethod
            def CUDAGraph():
                return FakeGraph(lib)

            @staticmethod
            @contextlib.contextmanager
            def graph(g, stream=None):
                lib.capturing = True
                before = len(lib.pairs)
                outer._g = g
                yield
                lib.capturing = False
                g.n = len(lib.pairs) - before

            @staticmethod
            def stream(s):
                return contextlib.nullcontext()

            @staticmethod
            def synchronize():
                pass
        self.cuda = _Cuda


class FakeWorkload:
    def __init__(self, lib):
        self.lib = lib
        self.calls = []

    def step(self, i, stream=None):
        self.calls.append(i)
        self.lib.launch()


@pytest.mark.parametrize("K", [20, 64, 256, 7])
def test_profile_counts_exactly_the_timed_steps(K):
    lib = FakeLib()
    torch = FakeTorch(lib)
    wl = FakeWorkload(lib)
    R = bench.divisor_le(K, 64)
    n_graphs = min(8, max(1, (64 * 8) // R) if R < 64 else 1)
    reps = K // R
    totals, steps = bench.profile_steps(torch, lib, wl, None, R, reps, n_graphs, 1)
    ms, cnt = totals["fused_decode"]
    assert cnt == K == len(steps)
    # the profiled steps are those of the timed region, in its order of graphs
    timed = [((r % n_graphs) * R + i) for r in range(reps) for i in range(R)]
    assert sorted(steps) == sorted(timed)
