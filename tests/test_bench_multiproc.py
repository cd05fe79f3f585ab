"""The bench's multi-process (N > 1) host logic with two gloo ranks on the CPU: the barrier,
the slowest-rank time and the whole-job rate (weak scaling: every rank runs the same workload
and the units of all ranks count), and the reference arm's rank policy (rank 0 alone works)."""
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import sys

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.dist_env()
        bench.barrier(w)
        dev = torch.device("cpu")
        # rank r took (r + 1) ms for 1000 units: the job is paced by the slowest rank
        ms, per_gpu, job = bench.whole_job_rate(1000.0, float(r + 1), w, dev)
        worst = bench.max_over_ranks(float(10 * r), w, dev)

        class A:  # the reference arm on a rank other than 0 does no work and prints nothing
            steps, warmup, gpus = 1, 0, w
        skipped = bench.run_reference(A) is None if r != 0 else True
        q.put((r, w, lr, ms, per_gpu, job, worst, skipped))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_and_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, lr, ms, per_gpu, job, worst, skipped in res:
        assert w == 2 and lr == r
        assert ms == pytest.approx(2.0)                 # slowest rank
        assert per_gpu == pytest.approx(1000.0 / 2e-3)  # units per second per GPU
        assert job == pytest.approx(2 * per_gpu)        # all ranks' units
        assert worst == pytest.approx(10.0)
        assert skipped
