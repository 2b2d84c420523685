"""The N>1 benchmark path on CPU: two gloo ranks on 127.0.0.1 run the code
bench.py runs under torchrun, with a CPU stand-in for the timed GPU step.

Each rank reads its rank and world size from the environment, picks its own
seeded copy of the workload (independent replicas: attention heads share
nothing, so no collective touches the data), times its stand-in step, and
the ranks combine their figures with bench.aggregate (max over ranks for the
time, sum for the work).  Rank 0 then builds the JSON line with
bench.result_line, the function bench.py's own arm prints; the test checks
its n_gpus, value and scaling."""
import json
import os
import socket
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _stand_in_step(q, k, v, rank):
    """CPU work in place of the GPU step: one score block per head
    (q k^T of the first 64 rows), plus a rank-dependent pause so the ranks'
    times differ and the max over ranks is the slower one."""
    acc = 0.0
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            acc += float(np.abs(q[b, h, :64] @ k[b, h, :64].T).sum())
    time.sleep(0.02 * (rank + 1))
    return acc


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from exact_tiled_attention_04_gb300 import inputs as I
    w_env, r_env, local = bench.dist_env()
    assert (w_env, r_env, local) == (world, rank, rank)
    dist = bench.dist_init(w_env, "gloo")
    w = I.WORKLOADS["tail_n1000"]
    wr = bench.rank_workload(w, rank)
    q, k, v = I.make(wr)
    steps = 3
    t0 = time.perf_counter()
    for _ in range(steps):
        _stand_in_step(q, k, v, rank)
    ms_local = (time.perf_counter() - t0) * 1e3
    ms_total, flops_all, value = bench.aggregate(ms_local, w.flops() * steps, dist)
    line = None
    if rank == 0:
        line = bench.result_line(
            w, w_env, steps, 3, ms_total, value, splits=0, launch="cpu stand-in", frac_of_peak=None,
            roofline={}, e2e={}, gpu_launches=0, clocks={}, entry="stand-in")
        line = json.loads(json.dumps(line))  # what rank 0 prints
    out[rank] = {"ms_local": ms_local, "ms_total": ms_total, "flops_all": flops_all, "value": value,
                 "checksum": float(np.asarray(q, np.float64).sum()), "seed": wr.seed, "line": line}
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_bench_line():
    import bench
    from exact_tiled_attention_04_gb300 import inputs as I
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    r0, r1 = out[0], out[1]
    w = I.WORKLOADS["tail_n1000"]
    # independent replicas: every rank its own seed and inputs
    assert r0["seed"] != r1["seed"] and r0["checksum"] != r1["checksum"]
    # aggregation: the slower rank's time, both ranks' work
    assert r0["ms_total"] == r1["ms_total"] == max(r0["ms_local"], r1["ms_local"])
    assert r0["flops_all"] == r1["flops_all"] == 2 * 3 * w.flops()
    expect = 2 * 3 * w.flops() / (max(r0["ms_local"], r1["ms_local"]) * 1e-3) / 1e12
    line = r0["line"]
    assert r1["line"] is None
    assert line["n_gpus"] == 2 and line["scaling"] == "weak"
    assert line["value"] == pytest.approx(expect, rel=1e-12)
    assert line["ms_per_step"] == pytest.approx(max(r0["ms_local"], r1["ms_local"]) / 3, rel=1e-12)
    assert line["metric"] == bench.METRIC and line["unit"] == "TFLOP/s"
    assert line["config"]["workload"] == "tail_n1000"
    assert line["config"]["parallelism"] == "independent replica per GPU x2"


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.5, None) == 3.5 and bench.reduce_sum(2.0, None) == 2.0
    assert bench.aggregate(2.0, 4e12, None) == (2.0, 4e12, 2000.0)
