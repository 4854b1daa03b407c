"""The boundary is a plain C ABI: a C program (compiled by gcc as C11, not C++)
includes include/moe.h, links libmoe_gb300.so and calls its host-side entry
points: status strings, workspace sizing with argument errors, a routing-trace
round trip and the expert-cache planner. Nothing here touches a GPU."""
import os
import shutil
import subprocess
import sys

import pytest

from routed_expert_ffn_router_gb300 import _lib
from routed_expert_ffn_router_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SRC = r"""
#include <stdio.h>
#include <string.h>
#include "moe.h"

int main(void) {
  for (int s = 0; s <= 6; ++s) printf("status %d %s\n", s, moe_status_str((moe_status)s));

  moe_layer_desc d;
  memset(&d, 0, sizeof d);
  d.H = 2048; d.I = 768; d.E = 128; d.k = 8; d.S = 128; d.shared_I = 768;
  const moe_qmat m = {(const uint8_t *)4096, (const uint16_t *)4096};
  d.gate = d.up = d.down = d.shared_gate = d.shared_up = d.shared_down = m;
  printf("ws8 %zu\n", moe_workspace_bytes(&d, 8));
  printf("ws2048 %zu\n", moe_workspace_bytes(&d, 2048));
  d.H = 200;
  printf("wsbad %zu\n", moe_workspace_bytes(&d, 8));
  printf("ffn_bad %d\n", (int)moe_expert_ffn(&d, (void *)4096, MOE_BF16, 8, (int32_t *)4096,
                                             (float *)4096, NULL, (float *)4096, (int32_t *)4096,
                                             (int32_t *)4096, (void *)4096, 1 << 30, NULL));

  int32_t ids[2 * 3] = {5, 1, 7, 2, 0, 3};
  float w[2 * 3] = {0.5f, 0.3f, 0.2f, 0.6f, 0.25f, 0.15f};
  uint8_t buf[256];
  long long n = (long long)moe_trace_write(4, ids, w, 2, 3, buf, (int64_t)sizeof buf);
  int32_t lay[4], kk[4], rid[4 * 3];
  float rw[4 * 3];
  long long r = (long long)moe_trace_read(buf, n, lay, kk, rid, rw, 3, 4);
  int same = r == 2 && memcmp(rid, ids, sizeof ids) == 0 && memcmp(rw, w, sizeof w) == 0 &&
             lay[0] == 4 && lay[1] == 4 && kk[0] == 3 && kk[1] == 3;
  printf("trace %lld %lld %d\n", n, r, same);

  moe_cache_params p;
  memset(&p, 0, sizeof p);
  p.n_layers = 1; p.n_experts = 8; p.half_life_tokens = 350.0; p.round_every_tokens = 32;
  p.max_swaps = 64; p.fill_every_tokens = 8; p.max_fills = 128; p.in_ratio = 1.5;
  p.in_picks = 2.0; p.max_window_tokens = 32;
  int32_t slots[1] = {2};
  size_t nb = moe_cache_state_bytes(&p, slots);
  static double state[1 << 12];
  if (nb == 0 || nb > sizeof state) { printf("cache_bytes %zu\n", nb); return 1; }
  if (moe_cache_init(state, nb, &p, slots) != MOE_OK) return 2;
  int32_t win[1 * 2] = {6, 3};
  if (moe_cache_observe(state, 0, win, 1, 2) != MOE_OK) return 3;
  moe_cache_swap mv[192];
  int32_t nm = moe_cache_advance(state, 8, mv, 192);
  int32_t map[8];
  moe_cache_slot_map(state, 0, map);
  printf("cache %d", nm);
  for (int e = 0; e < 8; ++e) printf(" %d", map[e]);
  printf("\n");
  return 0;
}
"""


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    libbuild.build()
    d = tmp_path_factory.mktemp("cclient")
    src = d / "client.c"
    src.write_text(C_SRC)
    out = d / "client"
    pkg = os.path.dirname(_lib.LIB_PATH)
    cmd = ["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
           "-o", str(out), "-L", pkg, "-l:libmoe_gb300.so", f"-Wl,-rpath,{pkg}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return str(out)


def test_c_program_uses_the_host_entry_points(exe):
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    lines = dict(l.split(" ", 1) for l in r.stdout.strip().splitlines() if not l.startswith("status"))
    status = [l for l in r.stdout.splitlines() if l.startswith("status")]
    assert status[0] == "status 0 ok" and len(status) == 7
    for code in range(7):
        assert status[code] == f"status {code} {_lib.status_str(code)}"
    # the C client and the Python binding size workspaces alike
    import ctypes
    d = _lib.moe_layer_desc()
    d.H, d.I, d.E, d.k, d.S, d.shared_I = 2048, 768, 128, 8, 128, 768
    for f in ("gate", "up", "down", "shared_gate", "shared_up", "shared_down"):
        setattr(d, f, _lib.moe_qmat(4096, 4096))
    L = _lib.load()
    assert int(lines["ws8"]) == L.moe_workspace_bytes(ctypes.byref(d), 8) > 0
    assert int(lines["ws2048"]) == L.moe_workspace_bytes(ctypes.byref(d), 2048)
    assert int(lines["wsbad"]) == 0
    assert int(lines["ffn_bad"]) == _lib.MOE_ERR_UNSUPPORTED  # H = 200: not a multiple of 128
    n, rr, same = lines["trace"].split()
    assert int(n) == 2 * (8 + 8 * 3) and int(rr) == 2 and same == "1"
    # one fill round after 8 tokens: the two experts of the window take the two free slots
    parts = lines["cache"].split()
    assert int(parts[0]) == 2
    m = [int(v) for v in parts[1:]]
    assert sorted(v for v in m if v >= 0) == [0, 1] and m[3] >= 0 and m[6] >= 0
