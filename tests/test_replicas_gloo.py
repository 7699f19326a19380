"""The multi-replica path of bench.py, on CPU with two gloo ranks.

Every box here has one GPU, so N > 1 only ever runs independent replicas
(the path has no exchange step).  What the ranks share is host logic: a
barrier, the maximum step time over ranks, and the whole-job throughput
computed from it.  Two processes on 127.0.0.1 check that logic."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [0.25, 0.40][rank]                       # the second replica is slower
    dist.barrier()
    step_ms = bench.reduce_max(local_ms, world, "cpu")
    value = bench.job_throughput(1 << 30, world, step_ms)
    q.put((rank, step_ms, value, bench.dist_env()))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_step():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, step_ms, value, env in res:
        assert step_ms == pytest.approx(0.40)
        assert value == pytest.approx(2 * (1 << 30) / 0.40e-3 / 1e9)
        assert env[0] == rank and env[1] == 2


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(1.5, 1, "cpu") == 1.5
    assert bench.job_throughput(10 ** 9, 1, 1000.0) == pytest.approx(1.0)
