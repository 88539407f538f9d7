"""bench.py's multi-rank logic on CPU with two gloo ranks (127.0.0.1): the slowest
rank's time decides, the job's value counts every rank's work (replicas, weak
scaling), and under --impl reference only rank 0 runs and prints."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.rank_env()
        slowest = bench.max_over_ranks(1.0 + rank, dist, "cpu")
        value = bench.whole_job_tflops(2e12, 3, slowest, w)
        q.put((r, w, lr, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for r, (rank, w, lr, slowest, value) in enumerate(got):
        assert (rank, w, lr) == (r, 2, r)
        assert slowest == 2.0                       # max over ranks
        assert abs(value - 2 * 2e12 * 3 / 2.0 / 1e12) < 1e-9


def test_reference_arm_only_rank0_prints(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""
