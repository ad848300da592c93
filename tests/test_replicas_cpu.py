"""The multi-GPU path of bench.py on CPU: two gloo ranks.

bench.py --gpus N runs N independent replicas (the SGMV path has no exchange
step): the only collective is the reduction of each rank's timed interval to
the slowest one, from which the whole job's rows/s follows.  Here two
processes on the gloo backend report different intervals; both must see the
maximum, and the throughput must count both replicas' rows.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        dist.barrier()
        elapsed, kernel_s = bench.max_over_ranks([1.0 + rank, 0.5 - 0.25 * rank], world)
        value = bench.replica_throughput(world, K=100, T=32, elapsed=elapsed)
        dist.barrier()
        q.put((rank, elapsed, kernel_s, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_interval():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, elapsed, kernel_s, value in out:
        assert elapsed == 2.0 and kernel_s == 0.5
        assert value == pytest.approx(2 * 100 * 32 / 2.0)


def test_one_rank_needs_no_collective():
    import bench

    assert bench.max_over_ranks([3.0, 1.0], 1) == [3.0, 1.0]
    assert bench.replica_throughput(1, 10, 8, 2.0) == 40.0
