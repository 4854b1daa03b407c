"""bench.py's end-to-end step stages a window's inputs in one device buffer and
its results in another, so that each step makes one host-to-device and one
device-to-host copy. The views handed to the layer call must tile those
buffers exactly, without overlap, with the alignment the C ABI asks for (x and
y 16-byte aligned), and the read-back prefix must hold y, ids, w and n_miss."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from routed_expert_ffn_router_gb300 import synth  # noqa: E402


def _off(view, base):
    return view.data_ptr() - base.data_ptr()


@pytest.mark.parametrize("name", sorted(synth.CONFIGS))
def test_staged_views_tile_the_buffers(name):
    cfg = synth.CONFIGS[name]
    T = min(cfg.T, 16)
    cfg = cfg.with_T(T)
    x_dtype = torch.int16 if cfg.x_dtype == "bf16" else torch.float32
    xe = 2 if x_dtype == torch.int16 else 4
    din, vin, dout, vout, n_in, n_back = bench.staged_io(torch, cfg, x_dtype, "cpu")

    # inputs: [logits | pad | x], x 256-byte aligned, nothing past x
    assert din.numel() == n_in
    assert _off(vin["logits"], din) == 0 and vin["logits"].shape == (T, cfg.E)
    assert vin["logits"].dtype == torch.float32
    ox = _off(vin["x"], din)
    assert ox % 256 == 0 and ox >= T * cfg.E * 4 and ox - T * cfg.E * 4 < 256
    assert vin["x"].shape == (T, cfg.H) and vin["x"].dtype == x_dtype
    assert ox + T * cfg.H * xe == n_in

    # outputs: y, ids, w, n_miss back to back (the read-back prefix), then miss_ids
    spans = []
    for key, shape, dt in (("y", (T, cfg.H), torch.float32), ("ids", (T, cfg.k), torch.int32),
                           ("w", (T, cfg.k), torch.float32), ("n_miss", (1,), torch.int32)):
        v = vout[key]
        assert v.shape == shape and v.dtype == dt and v.is_contiguous()
        spans.append((_off(v, dout), v.numel() * 4))
    assert spans[0][0] == 0
    for (a, na), (b, _) in zip(spans, spans[1:]):
        assert a + na == b
    assert spans[-1][0] + spans[-1][1] == n_back
    om = _off(vout["miss_ids"], dout)
    assert om % 256 == 0 and om >= n_back and vout["miss_ids"].shape == (cfg.E,)
    assert om + cfg.E * 4 == dout.numel()

    # writes through the views land in the bytes a single copy reads back
    g = torch.Generator().manual_seed(3)
    vout["y"].copy_(torch.randn(T, cfg.H, generator=g))
    vout["ids"].copy_(torch.randint(0, cfg.E, (T, cfg.k), generator=g, dtype=torch.int32))
    vout["w"].copy_(torch.rand(T, cfg.k, generator=g))
    vout["n_miss"].fill_(7)
    vout["miss_ids"].fill_(-1)
    back = dout[:n_back].clone()
    assert torch.equal(bench.carve(torch, back, 0, (T, cfg.H), torch.float32), vout["y"])
    assert torch.equal(bench.carve(torch, back, spans[1][0], (T, cfg.k), torch.int32), vout["ids"])
    assert torch.equal(bench.carve(torch, back, spans[2][0], (T, cfg.k), torch.float32), vout["w"])
    assert int(bench.carve(torch, back, spans[3][0], (1,), torch.int32).item()) == 7


def test_carve_rejects_misaligned_or_oversized_views():
    buf = torch.zeros(64, dtype=torch.uint8)
    with pytest.raises(AssertionError):
        bench.carve(torch, buf, 2, (2,), torch.float32)
    with pytest.raises(AssertionError):
        bench.carve(torch, buf, 0, (17,), torch.float32)
    v = bench.carve(torch, buf, 4, (3,), torch.int32)
    v.fill_(1)
    assert buf[4:16].tolist() == [1, 0, 0, 0] * 3 and buf[:4].sum() == 0 and buf[16:].sum() == 0
