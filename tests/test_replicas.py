"""The N>1 path of bench.py: independent replicas, one process per GPU, no collective on
the data path. Each rank times its own replica; the job time is the slowest rank's
(max over ranks) and the job's throughput is all ranks' units over that time. These
checks run the same helpers as two gloo ranks on the CPU (no GPU involved).
"""

import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank), "PMOE_BENCH_BACKEND": "gloo"})
    import bench
    import torch.distributed as dist
    try:
        ws, r, local = bench.dist_init()
        # rank-dependent replica times (ms) for the same number of steps
        steps = 50
        my_ms = 10.0 + 7.5 * r
        bench.barrier(ws)
        job_ms = bench.reduce_max(my_ms, ws, torch.device("cpu"))
        value = ws * 1 * steps / (job_ms / 1e3)
        agg = bench.aggregate([steps] * ws, [(10.0 + 7.5 * i) / 1e3 for i in range(ws)])
        out_q.put((r, ws, local, job_ms, value, agg))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(2))
    for r, (rank, ws, local, job_ms, value, agg) in enumerate(res):
        assert (rank, ws, local) == (r, 2, r)
        assert job_ms == pytest.approx(17.5)           # the slower replica's time
        assert value == pytest.approx(2 * 50 / 0.0175)  # both replicas' tokens over it
        assert agg == pytest.approx(value)


def test_single_rank_needs_no_process_group(monkeypatch):
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_init() == (1, 0, 0)
    assert bench.reduce_max(3.25, 1, torch.device("cpu")) == 3.25
    assert bench.aggregate([7], [0.5]) == 14.0
