"""moe_expert_ffn_static, the entry point for callers that cannot allocate
device memory (a framework allocator that owns the GPU, plugin code without an
allocator, decode loops that must not call cudaMalloc): it must give the same
layer output as moe_expert_ffn with a caller-owned workspace, call after call,
even though every call reuses the library's one fixed scratch array.

Kept in a file that pytest collects last, so a stop at the first failure has
already run every other test."""
import numpy as np
import pytest
import torch

from routed_expert_ffn_router_gb300 import _lib, synth
from routed_expert_ffn_router_gb300 import build as libbuild
from routed_expert_ffn_router_gb300.layer import MoeLayer

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    libbuild.build()
    _lib.load()


def _route(lg, k):
    T, E = lg.shape
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    _lib.moe_route(lg, T, E, k, ids, w)
    return ids, w


def _cache_layer(cfg, seed):
    """A layer whose pool holds only 60% of the experts (slot map with misses)."""
    inp = synth.make_layer(cfg, seed)
    smt, S = synth.random_slot_map(cfg.E, 0.6, seed=seed + 1)
    keep = (smt >= 0).nonzero().flatten()
    for kname in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s"):
        setattr(inp, kname, getattr(inp, kname)[keep].contiguous())
    inp.S = S
    inp.slot_map = smt
    return inp.to("cuda")


# Three routes through the library, each placing different regions in the
# scratch: the one-launch decode kernel (bf16 rows), the separate permute /
# gate-up / down / combine kernels (fp32 rows), and a slot map with misses.
CASES = {
    "decode_bf16": (synth.MoeConfig("noalloc", H=2048, I=768, E=128, k=8, T=8, shared_I=768,
                                    zipf_s=1.1), False),
    "separate_f32": (synth.MoeConfig("noalloc_f32", H=256, I=128, E=16, k=4, T=6, shared_I=128,
                                     zipf_s=1.0, x_dtype="f32"), False),
    "slot_map_misses": (synth.MoeConfig("noalloc_cache", H=1024, I=512, E=64, k=8, T=16,
                                        zipf_s=1.2), True),
}


@pytest.mark.parametrize("case", list(CASES))
def test_static_scratch_matches_workspace_entry_point_twice(case):
    cfg, cached = CASES[case]
    inp = _cache_layer(cfg, 21) if cached else synth.make_layer(cfg, 21, device="cuda")
    lay = MoeLayer(inp, T_max=cfg.T)
    sm = inp.slot_map if cached else None
    logits, xs = synth.draw_windows(inp, 2, seed=5)
    for call in range(2):  # two calls in a row, different windows
        ids, w = _route(logits[call], cfg.k)
        ref = lay.expert_ffn(xs[call], ids, w, slot_map=sm)
        y = torch.full((cfg.T, cfg.H), float("nan"), device="cuda")
        miss = torch.full((cfg.E,), -5, dtype=torch.int32, device="cuda")
        nm = torch.full((1,), -5, dtype=torch.int32, device="cuda")
        _lib.moe_expert_ffn_static(lay.desc, xs[call], lay.x_dtype, cfg.T, ids, w, sm, y, miss,
                                   nm)
        code, bits = _lib.moe_static_read_status()
        assert code == _lib.MOE_OK, (call, bits)
        y_ref = ref["y"].double().cpu().numpy()
        err = np.abs(y.double().cpu().numpy() - y_ref).max()
        assert err <= TOL * np.abs(y_ref).max(), (call, err)
        n = int(ref["n_miss"].item())
        assert int(nm.item()) == n
        assert (n > 0) == cached
        assert torch.equal(miss[:n], ref["miss_ids"][:n])


def test_static_scratch_rejects_a_chunk_too_large_for_it():
    cfg = synth.MoeConfig("big", H=2048, I=512, E=512, k=10, T=2048, shared_I=512)
    d = _lib.moe_layer_desc()
    d.H, d.I, d.E, d.k, d.S, d.shared_I = cfg.H, cfg.I, cfg.E, cfg.k, cfg.E, cfg.shared_I
    buf = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    for f in ("gate", "up", "down", "shared_gate", "shared_up", "shared_down"):
        setattr(d, f, _lib.moe_qmat(buf.data_ptr(), buf.data_ptr()))
    code = _lib.load().moe_expert_ffn_static(
        d, buf.data_ptr(), _lib.MOE_BF16, cfg.T, buf.data_ptr(), buf.data_ptr(), None,
        buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == _lib.MOE_ERR_UNSUPPORTED
