"""The multi-GPU layout of bench.py is replicas only (each rank runs its own
layer on its own GPU, no collective on the data path): the rank bookkeeping
and the timing reductions (barrier, max over ranks of the elapsed time, sum of
the bytes) are exercised here with two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    try:
        assert d.world == world and d.rank == rank and d.pg is not None
        assert d.pg.get_backend() == "gloo"
        d.barrier()
        ms = 10.0 + 5.0 * rank          # this rank's elapsed time
        byts = 1000.0 * (rank + 1)      # this rank's bytes
        out[rank] = (d.max(ms), d.sum(byts))
        d.barrier()
    finally:
        d.close()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_reduce_like_the_bench():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    # every rank sees the slowest rank's time and the whole job's bytes, so the
    # whole-job value (bytes / max time) is the same on every rank
    assert dict(out) == {0: (15.0, 3000.0), 1: (15.0, 3000.0)}


def test_single_process_has_no_group():
    sys.path.insert(0, ROOT)
    import bench
    saved = {k: os.environ.pop(k, None) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    try:
        d = bench.Dist()
        assert d.world == 1 and d.rank == 0 and d.pg is None
        assert d.max(3.5) == 3.5 and d.sum(7.0) == 7.0
        d.barrier()
        d.close()
    finally:
        for k, v in saved.items():
            if v is not None:
                os.environ[k] = v


@pytest.mark.timeout(300)
def test_reference_arm_under_two_ranks_prints_one_line():
    """`bench.py --impl reference` launched as two ranks: rank 0 alone times the
    CPU oracle and prints the one JSON line; rank 1 exits 0 without work."""
    import json
    import subprocess
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=280, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    # the line carries every key of the bench contract, on the same metric and workload
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e",
                "cpu_baseline"):
        assert key in d, key
    import bench
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["warmup"] >= 3
    assert d["config"]["workload"].startswith("decode_window: 1 layer, T=8 rows")
    assert d["e2e"]["value"] == d["value"] == d["cpu_baseline"]["value"] > 0
    assert d["cpu_baseline"]["cores"] == 1 and d["vs_baseline"] is None
