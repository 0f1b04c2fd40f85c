"""The N > 1 path of the benchmark on CPU: two gloo ranks, replicas of the
workload, step times reduced by maximum, whole-job throughput summed over
ranks.  (The forward has no cross-sequence exchange, so replicas are the
whole multi-GPU design: no data-path collective exists to test.)"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, local = bench.dist_env()
    mine = [1.0 + rank, 5.0 - 2 * rank]            # rank 0: [1, 5]; rank 1: [2, 3]
    got = bench.reduce_over_ranks(mine, torch.device("cpu"))
    value = bench.job_throughput(8192, ws, got[0])
    dist.barrier()
    q.put((rank, ws, r, local, got, value))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_by_max_and_sum_tokens():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ws, r, local, got, value in results:
        assert ws == world and r == rank and local == rank
        assert got == [2.0, 5.0]                        # element-wise maximum over ranks
        assert value == pytest.approx(8192 * 2 / 2.0e-3)  # both ranks' tokens over the slowest time


def test_single_process_reduction_is_identity():
    import bench
    assert bench.reduce_over_ranks([1.5, 2.5], torch.device("cpu")) == [1.5, 2.5]
    assert bench.job_throughput(100, 1, 1.0) == pytest.approx(1e5)
