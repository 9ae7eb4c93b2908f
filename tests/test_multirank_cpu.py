"""The multi-rank bench path on CPU: two gloo ranks on 127.0.0.1 run the
helpers bench.py uses under torchrun (rank environment, barrier, max and sum
over ranks, the weak-scaling aggregate), and the reference arm runs on rank
0 only."""
import contextlib
import io
import os
import socket
import sys
from datetime import timedelta
from pathlib import Path

import pytest
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", timeout=timedelta(seconds=60))
    try:
        assert bench.dist_env() == (rank, world, rank)
        bench.barrier()
        # per-rank times differ: the aggregate divides all units by the slowest
        secs = 1.0 + rank          # rank 0: 1 s, rank 1: 2 s
        units = 100.0 * (rank + 1)  # rank 0: 100, rank 1: 200
        results[rank] = (bench.reduce_scalar(rank + 1, "max"), bench.reduce_scalar(rank + 1, "sum"),
                         bench.weak_scaling_value(units, secs))
        bench.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_and_aggregate():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        assert codes == [0, 0], codes
        for r in range(world):
            mx, sm, agg = results[r]
            assert mx == 2.0 and sm == 3.0
            assert agg == pytest.approx(300.0 / 2.0)  # (100 + 200) units / max(1 s, 2 s)


def test_single_rank_helpers_are_identities(monkeypatch):
    for key in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(key, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.reduce_scalar(3.5, "max") == 3.5
    assert bench.weak_scaling_value(10.0, 4.0) == 2.5


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"]))
    assert out.getvalue() == ""
