"""bench.py's multi-GPU path is N independent replicas (the attention path has
no exchange step): each rank times its own step, the job's step time is the
maximum over ranks, and the reported rate sums every rank's work. This runs
that host logic as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, ms_by_rank, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup(None)
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    rate, ms = bench.replica_rate(1000.0, ms_by_rank[rank], w)
    out[rank] = (rate, ms)
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_sum_the_work():
    ms_by_rank = [10.0, 25.0]
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, ms_by_rank, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        res = dict(out)
    for r in range(2):
        rate, ms = res[r]
        assert ms == pytest.approx(25.0)
        assert rate == pytest.approx(2 * 1000.0 / 25e-3)


def test_single_process_needs_no_process_group():
    import bench
    rate, ms = bench.replica_rate(500.0, 4.0, 1)
    assert ms == 4.0 and rate == pytest.approx(500.0 / 4e-3)
