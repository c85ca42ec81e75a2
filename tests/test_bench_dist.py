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
