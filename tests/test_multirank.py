"""The benchmark's multi-rank host logic on CPU: world size 2 over gloo.

Each rank runs its own copy of the workload (heads are independent, so there
is no data-path collective); the only exchange is the max of the per-rank
timings, and the whole-job value counts every rank's FLOPs over the slowest
rank's time."""
import importlib.util
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        # rank-dependent "timings": rank 0 slower on the first, rank 1 on the second
        got = b.max_over_ranks([10.0 - rank, 1.0 + rank, 3.0])
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == [10.0, 2.0, 3.0]
    assert out[1] == [10.0, 2.0, 3.0]


def test_single_process_is_identity_and_job_value():
    b = _bench()
    assert b.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    # 2 ranks x 1e12 FLOPs each in 1 ms (slowest rank) = 2000 TFLOPS
    assert b.job_tflops(1e12, 2, 1.0) == pytest.approx(2000.0)
