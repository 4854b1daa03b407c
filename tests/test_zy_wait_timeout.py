"""A bounded device wait that runs out reports MOE_ERR_TIMEOUT and leaves the
context usable (failure detection without a GPU fault).

The failure is made on the host: the workspace's unit-queue counter is left
advanced (as a timed-out or killed call could leave it), so no unit of the
window is handed out, nothing is published, and the reduction's wait for the
window's units gives up after about a second. moe_read_status must then say
MOE_ERR_TIMEOUT; after moe_workspace_init the same window is computed
correctly.

Nothing faults or hangs: the wait is bounded in the kernel, every CTA exits,
and the last one resets the cross-CTA counters."""
import time

import numpy as np
import pytest
import torch

from routed_expert_ffn_router_gb300 import _lib, synth
from routed_expert_ffn_router_gb300 import build as libbuild
from routed_expert_ffn_router_gb300.layer import MoeLayer

pytestmark = pytest.mark.gpu

# byte offset of the decode kernel's unit-queue counter in a workspace: the
# status word (256 B), the counters (256 B), then the cross-CTA counters, of
# which the queue is the third int32
QUEUE_BYTE = 512 + 2 * 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    libbuild.build()
    _lib.load()


def test_expired_wait_reports_timeout_and_the_workspace_recovers():
    cfg = synth.MoeConfig("timeout", H=2048, I=768, E=128, k=8, T=8, shared_I=768, zipf_s=1.1)
    inp = synth.make_layer(cfg, 3, device="cuda")
    lay = MoeLayer(inp, T_max=cfg.T)
    logits, xs = synth.draw_windows(inp, 1, seed=9)
    ref = lay.forward(logits[0], xs[0])
    y_ref = ref["y"].clone()
    torch.cuda.synchronize()
    assert lay.status()[0] == _lib.MOE_OK

    base = lay.ws_ptr - lay.ws.data_ptr()
    q = lay.ws[base + QUEUE_BYTE: base + QUEUE_BYTE + 4].view(torch.int32)
    q.fill_(1 << 24)
    t0 = time.time()
    lay.forward(logits[0], xs[0])
    code, bits = lay.status()  # synchronises
    dt = time.time() - t0
    assert code == _lib.MOE_ERR_TIMEOUT and bits & 4, (code, bits)
    assert dt < 30.0

    lay.clear_status()
    out = lay.forward(logits[0], xs[0])
    torch.cuda.synchronize()
    assert lay.status()[0] == _lib.MOE_OK
    assert torch.equal(out["y"], y_ref)
    assert np.array_equal(out["ids"].cpu().numpy(), ref["ids"].cpu().numpy())
