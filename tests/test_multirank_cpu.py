"""Host logic of the multi-GPU path on CPU ranks (gloo, world size 2).

Every rank runs the whole per-GPU workload (replicas; the path needs no
collective on its data). The benchmark reports all ranks' work over the
slowest rank's time, which these ranks check with the same helpers."""
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


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = 2.0 + rank          # rank 1 is the slow one
    ms = bench.reduce_max_over_ranks(ms_local, dist, "cpu")
    thr = bench.job_throughput(1.0e9, ms, world)
    q.put((rank, ms, thr))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_reduce_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, thr in res:
        assert ms == 3.0                            # slowest rank's time, on every rank
        assert thr == pytest.approx(2 * 1.0e9 / 3.0e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max_over_ranks(1.5) == 1.5
    assert bench.job_throughput(10.0, 2.0, 1) == pytest.approx(5000.0)
