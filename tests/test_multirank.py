"""The N>1 benchmark path on CPU: two gloo ranks on 127.0.0.1.  Each rank
runs its own independent problem (no collective on the data path); only the
timing and flop totals are combined: max over ranks for the time, sum for the
work.  This checks that aggregation, and the rank/env plumbing."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    dist = bench.dist_init(w, "gloo")
    ms = 10.0 + 5.0 * rank          # this rank's elapsed time
    flops = 1e12 * (rank + 1)       # this rank's work
    out[rank] = (bench.reduce_max(ms, dist), bench.reduce_sum(flops, dist))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == (15.0, 3e12)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.5, None) == 3.5 and bench.reduce_sum(2.0, None) == 2.0
