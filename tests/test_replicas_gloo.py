"""The multi-GPU mode of bench.py runs independent replicas (the decode step has
no exchange); the only cross-rank step is the max over ranks of the timings and
the whole-job aggregate. Covered here with two gloo ranks on CPU."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mx = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)], "cpu")
        q.put((rank, mx))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got[0] == got[1] == [2.0, 5.0, 0.5]


def test_whole_job_aggregate_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    # two replicas each moving 1 GB in 1 ms: 2000 GB/s for the job
    assert bench.whole_job_gbs(1e9, 2, 1.0) == pytest.approx(2000.0)
    assert bench.whole_job_gbs(1e9, 1, 0.5) == pytest.approx(2000.0)
