"""The multi-GPU (replicas over heads) host logic of bench.py, run as two gloo
ranks on the CPU: the max over ranks and the whole-job throughput."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slower one
        m = bench.max_over_ranks(local_ms)
        dist.barrier()
        v = bench.weak_scaling_value(131072, world, m)
        q.put((rank, m, v, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_and_weak_scaling():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, m, v, env in res:
        assert m == 15.0                                  # max over ranks, seen by every rank
        assert v == pytest.approx(131072 * 2 / 0.015)     # all ranks' tokens over the slowest time
        assert env[0] == 2 and env[1] == rank


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.weak_scaling_value(1000, 1, 1.0) == pytest.approx(1e6)
