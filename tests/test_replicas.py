"""The multi-GPU bench path runs independent replicas (the hot path has no
exchange step): ranks meet at barriers, time their own steps, and rank 0
reports the slowest rank's time and the bytes of all ranks.  This checks
that logic over two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), QMOE_BENCH_BACKEND="gloo")
    import torch.distributed as dist
    import bench
    r, w = bench.dist_init(world)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    # each rank "took" a different time; the job's step time is the slowest
    ms = bench.max_over_ranks(1.0 + 0.5 * rank, w)
    out[rank] = (ms, bench.job_throughput(1e9, ms, w))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    # every rank agrees on the max (1.5 ms) and on the whole-job figure:
    # 2 ranks x 1 GB per step / 1.5 ms = 1333.3 GB/s
    for rank in range(world):
        ms, gbs = res[rank]
        assert ms == pytest.approx(1.5)
        assert gbs == pytest.approx(2 * 1e9 / 1.5e-3 / 1e9)


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.job_throughput(2e9, 2.0, 1) == pytest.approx(1000.0)
