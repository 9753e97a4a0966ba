"""The benchmark's multi-rank host logic on CPU: two gloo ranks (world size 2), no GPU.

bench.py runs one replica of the step per GPU ("replicas only"): each rank times its own work,
the per-kernel times become the maximum over ranks, and the reported value is the work of all
ranks over that time.  The reference arm runs on rank 0 only.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        # rank r measured (1 + r, 10 - r, 5) ms: the slowest rank's value wins element-wise
        out[rank] = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 5.0], ws, "cpu")
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ws = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as manager:
        out = manager.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, ws, port, out)) for r in range(ws)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        assert out[0] == [2.0, 10.0, 5.0]
        assert out[1] == [2.0, 10.0, 5.0]


def test_max_over_ranks_single_rank_is_identity():
    assert bench.max_over_ranks([3.0, 4.5], 1, "cpu") == [3.0, 4.5]


def test_whole_job_rate_counts_every_rank():
    # 2 ranks x 1e12 flop in 2 ms: 1e15 flop/s; one rank alone: half of it
    assert bench.whole_job_rate(2, 1e12, 2.0) == pytest.approx(1e15)
    assert bench.whole_job_rate(1, 1e12, 2.0) == pytest.approx(5e14)


def test_reference_arm_runs_on_rank_zero_only():
    class Args:
        steps, warmup, ref_rows = 1, 3, 1
    assert bench.run_reference(Args(), 2, 1) is None


def test_dist_env(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "4")
    monkeypatch.setenv("RANK", "3")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench._dist() == (4, 3, 1)
