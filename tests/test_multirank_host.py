"""The multi-rank path of bench.py on CPU: two gloo ranks (one process each)
run the same host logic the GPU ranks run (rank discovery, barrier, slowest
rank's time, whole-job rate); the reference arm does its work on rank 0 only.
The data path has no collective: every rank runs its own replica."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": "2", "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        import bench
        ws, r, local = bench._dist()
        slowest = bench._max_over_ranks(10.0 + rank, ws)   # rank 1 is the slow one: 11 ms
        bench._barrier(ws)
        rate = bench.whole_job_rate(1000, 5, ws, slowest)
        q.put((rank, ws, r, local, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_time_and_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r0, ws, r, local, slowest, rate) in enumerate(res):
        assert (r0, ws, r, local) == (rank, 2, rank, rank)
        assert slowest == 11.0
        assert rate == pytest.approx(1000 * 5 * 2 / 0.011)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""


def test_whole_job_rate_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_rate(1000, 5, 1, 10.0)
    assert bench.whole_job_rate(1000, 5, 4, 10.0) == pytest.approx(4 * one)
