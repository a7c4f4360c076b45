"""The N>1 host logic of bench.py on CPU: two gloo ranks.

Each rank times its own independent batch; the job's time is the slowest
rank's (all ranks agree on it), and the job's value counts every rank's
tokens over that time (weak scaling).  No data-path collective exists.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, times, out_q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], dist, torch.device("cpu"))
        val = bench.weak_scaling_value(world, 4096, 10, ms)
        out_q.put((rank, ms, val, bench.rank_batch_seed(rank)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_weak_scaling_value():
    world, port = 2, _free_port()
    times = [31.0, 37.5]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r[1] for r in res] == [37.5, 37.5]
    assert res[0][2] == res[1][2] == pytest.approx(2 * 4096 * 10 / 0.0375)
    assert res[0][3] != res[1][3]  # each rank its own batch


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, None, None) == 12.5
    assert bench.weak_scaling_value(1, 4096, 100, 300.0) == pytest.approx(4096 * 100 / 0.3)
