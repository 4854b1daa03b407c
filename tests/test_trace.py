"""Routing traces ("extended-strata-moe reference", "Routing trace format"):
the library's records against an independent struct encoder of the page's
layout, round trips, and malformed buffers (no GPU needed)."""
import struct

import numpy as np
import pytest

from routed_expert_ffn_router_gb300 import _lib
from routed_expert_ffn_router_gb300 import build as libbuild
from routed_expert_ffn_router_gb300 import trace


@pytest.fixture(scope="module", autouse=True)
def lib():
    libbuild.build()
    return _lib.load()


def page_records(layer, ids, w):
    """int32 layer, int32 k, k x int32 expert id, k x float32 weight per token."""
    b = b""
    for t in range(ids.shape[0]):
        k = ids.shape[1]
        b += struct.pack(f"<ii{k}i{k}f", layer, k, *ids[t].tolist(), *w[t].tolist())
    return b


def test_layout_matches_the_page():
    rng = np.random.default_rng(0)
    ids = rng.integers(0, 512, size=(5, 10)).astype(np.int32)
    w = rng.random((5, 10)).astype(np.float32)
    assert trace.encode(7, ids, w) == page_records(7, ids, w)
    # the page's dumping tool writes the weights as 0
    assert trace.encode(7, ids) == page_records(7, ids, np.zeros_like(w))


def test_round_trip_mixed_layers_and_k():
    a = np.array([[3, 1], [0, 2]], np.int32)
    b = np.array([[5, 6, 7, 8]], np.int32)
    wa = np.array([[0.75, 0.25], [0.5, 0.5]], np.float32)
    wb = np.array([[0.4, 0.3, 0.2, 0.1]], np.float32)
    data = trace.encode(0, a, wa) + trace.encode(47, b, wb)
    layer, k, ids, w = trace.decode(data, k_max=4)
    assert list(layer) == [0, 0, 47] and list(k) == [2, 2, 4]
    assert ids.tolist() == [[3, 1, -1, -1], [0, 2, -1, -1], [5, 6, 7, 8]]
    assert np.array_equal(w[:2, :2], wa) and np.array_equal(w[2], wb[0]) and not w[:2, 2:].any()
    assert trace.decode(b"")[0].size == 0


@pytest.mark.parametrize("cut", [1, 7, 8, 20])
def test_truncated_and_malformed(cut):
    data = trace.encode(1, np.array([[1, 2]], np.int32), np.array([[0.5, 0.5]], np.float32))
    with pytest.raises(ValueError):
        trace.decode(data[:len(data) - cut])
    bad = bytearray(data)
    struct.pack_into("<i", bad, 4, 0)          # k = 0
    with pytest.raises(ValueError):
        trace.decode(bytes(bad))
    with pytest.raises(ValueError):
        trace.decode(data, k_max=1)             # k above k_max


def test_write_argument_errors():
    L = _lib.load()
    ids = np.zeros((2, 2), np.int32)
    assert L.moe_trace_write(0, ids.ctypes.data, None, 2, 0, None, 0) == -1       # k < 1
    assert L.moe_trace_write(0, None, None, 2, 2, None, 0) == -1                  # no ids
    buf = (np.zeros(10, np.uint8))
    assert L.moe_trace_write(0, ids.ctypes.data, None, 2, 2, buf.ctypes.data, 10) == -1  # too small


def test_bench_routing_dump(tmp_path):
    """bench.py's MOE_TRACE dump: the windows' routing as consecutive records."""
    import torch
    import bench
    outs = [dict(ids=torch.tensor([[3, 1], [0, 2]], dtype=torch.int32),
                 w=torch.tensor([[0.75, 0.25], [0.5, 0.5]])),
            dict(ids=torch.tensor([[7, 6]], dtype=torch.int32), w=torch.tensor([[0.6, 0.4]]))]
    assert bench.dump_routing(None, outs) == 0
    path = tmp_path / "routing.bin"
    n = bench.dump_routing(str(path), outs)
    data = path.read_bytes()
    assert n == len(data) == 3 * (8 + 16)
    layer, k, ids, w = trace.decode(data, k_max=2)
    assert ids.tolist() == [[3, 1], [0, 2], [7, 6]] and list(layer) == [0, 0, 0]
    assert np.allclose(w, [[0.75, 0.25], [0.5, 0.5], [0.6, 0.4]])
