"""The benchmark's multi-rank plumbing on CPU with the gloo backend (world size 2): the
barrier and the maximum over ranks that the GPU run applies to its timings, and the reference
arm's rule that rank 0 alone runs and prints."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, results):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_env()
    assert (w, r) == (world, rank)
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    # each rank reports its own "time"; every rank must see the largest
    got = bench.max_over_ranks(10.0 + 3.0 * rank, w, "cpu")
    bench.barrier(w)
    results[rank] = got


def test_max_over_ranks_with_gloo():
    world, port = 2, _free_port()
    results = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
    assert dict(results) == {0: 13.0, 1: 13.0}


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        gpus, steps, warmup = 2, 1, 0

    called = []
    monkeypatch.setattr(bench, "oracle_sample", lambda n: called.append(n) or (None, None, None))
    monkeypatch.setattr(bench, "oracle_step", lambda *a: None)
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(Args, 2, 1) == 0
    assert called == [] and buf.getvalue() == ""        # rank 1: no work, no line
    with redirect_stdout(buf):
        assert bench.run_reference(Args, 2, 0) == 0
    assert called == [256] and '"impl": "reference"' in buf.getvalue()


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` end to end on CPU (it times the oracle, no GPU): one JSON
    line with the keys and units of the GPU arm's line, on the same workload."""
    import json
    import subprocess
    sys.path.insert(0, ROOT)
    import bench
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                         timeout=300, cwd=ROOT, check=True).stdout.strip().splitlines()
    line = json.loads(out[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert (line["steps"], line["warmup"], line["n_gpus"]) == (1, 3, 1)
    assert line["config"] == bench.workload_config()
    assert line["value"] > 0 and line["ms_per_step"] > 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
