"""The N > 1 host path of bench.py on CPU: two gloo ranks (no GPU).

The layer shards by (b, h) with no exchange, so the multi-rank run is
replicas: every rank draws its own batch, the ranks meet only at the timing
barrier, the job time is the slowest rank's, and only rank 0 reports (also
for the oracle arm).
"""

import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    import sys

    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import numpy as np
    import torch
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import gen

        cfg = dict(gen.CONFIGS["tiny"])
        cfg["seed"] = bench.rank_seed(cfg["seed"], rank)
        inp = gen.make_inputs(name="tiny", **cfg)
        fp = torch.tensor([float(np.abs(inp.q).sum()), float(inp.v[0, 0, 0, 0])], dtype=torch.float64)
        got = [torch.zeros_like(fp) for _ in range(world)]
        dist.all_gather(got, fp)
        slowest = bench.max_over_ranks(10.0 + 3.0 * rank, dist, "cpu")
        args = type("A", (), {"steps": 1, "warmup": 0, "gpus": world})()
        ref = bench.run_reference(args, rank) if rank != 0 else "skipped"
        queue.put((rank, [g.tolist() for g in got], slowest, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_are_independent_replicas():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        rank, got, slowest, ref = queue.get(timeout=120)
        res[rank] = (got, slowest, ref)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got0, got1 = res[0][0], res[1][0]
    assert got0 == got1  # both ranks see the same gathered fingerprints
    assert got0[0] != got0[1]  # ... and the two batches differ
    assert res[0][1] == res[1][1] == 13.0  # max over ranks
    assert res[1][2] is None  # the oracle arm runs on rank 0 only


def test_job_throughput_counts_every_rank():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    one = bench.job_throughput(4 * 8192, 1, 1.0)
    assert one == pytest.approx(4 * 8192 / 1e-3)
    assert bench.job_throughput(4 * 8192, 8, 1.0) == pytest.approx(8 * one)
    assert bench.rank_seed(2, 0) == 2 and bench.rank_seed(2, 3) != bench.rank_seed(2, 1)
