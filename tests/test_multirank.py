"""The N > 1 path of bench.py on CPU: two gloo ranks (spawned processes,
rendezvous on 127.0.0.1) reduce their step times to the slowest rank's, and
the job's throughput counts every rank's work (weak scaling)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [12.5, 17.25][rank]                     # rank 1 is the slower one
    worst = bench.max_over_ranks(ms, dist)
    dist.barrier()
    q.put((rank, worst, bench.job_tflops(1.0e12, world, worst)))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in out] == [0, 1]
    assert all(w == 17.25 for _, w, _ in out)
    # 2 ranks x 1 TFLOP per step in 17.25 ms
    assert all(abs(v - 2.0 / 17.25e-3) < 1e-9 for _, _, v in out)


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert abs(bench.job_tflops(2.0e12, 1, 4.0) - 500.0) < 1e-9
