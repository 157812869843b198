"""The N>1 path of the benchmark on CPU: two gloo ranks run the same
aggregation the GPU job uses (max over ranks of the step time; whole-job
throughput = units of all ranks / that time).  Each rank is an independent
replica on its own batch, so no other collective is involved."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.0][rank]                       # rank 1 is the slow one
    agg = bench.max_over_ranks(ms, dist, "cpu")
    thr = bench.job_throughput(128 * 64, world, agg)
    q.put((rank, agg, thr))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, agg, thr in res:
        assert agg == 5.0
        assert thr == pytest.approx(2 * 128 * 64 / 5e-3)


def test_single_rank_aggregation_is_identity():
    import bench
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.job_throughput(100, 1, 1.0) == pytest.approx(1e5)
