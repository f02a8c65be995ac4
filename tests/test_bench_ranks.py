"""Multi-rank timing reduction of bench.py, run as two gloo ranks on the CPU.

Each rank times its own shard; the whole-job figure takes the slowest rank's time and the
sum of all ranks' work."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r ran for 10 + 5 r ms and processed 1e9 * (r + 1) flops
        t, work = bench.whole_job(10.0 + 5.0 * rank, 1e9 * (rank + 1), world, torch.device("cpu"))
        q.put((rank, t, work))
    finally:
        dist.destroy_process_group()


def test_whole_job_max_time_and_summed_work():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, t, work in got:
        assert t == pytest.approx(15.0)
        assert work == pytest.approx(3e9)


def test_whole_job_single_rank_is_identity():
    import bench
    assert bench.whole_job(7.5, 123.0, 1, None) == (7.5, 123.0)


def _shard_worker(rank, world, port, q):
    import torch
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        w = bench.workload_by_name("base_encoder").replace(B=4, H=2)
        x = bench.draw(w, seed=0 + rank)  # what each rank of bench.py draws: seed + rank
        flops = bench.algorithmic_flops(w, x["kv_len"])
        # the shard's fingerprint, and the whole-job reduction of equal per-rank work
        fp = float(x["q"].float().sum() + x["k"].float().sum() + x["v"].float().sum())
        t, work = bench.whole_job(1.0, flops, world, torch.device("cpu"))
        q.put((rank, fp, flops, work, tuple(x["q"].shape)))
    finally:
        dist.destroy_process_group()


def test_each_rank_draws_its_own_shard_of_the_same_shape():
    """Weak scaling: every rank of bench.py draws its own seeded batch (seed + rank) of the
    per-GPU workload, so the shards differ in content but not in shape or work, and the job's
    work is the ranks' sum; no data moves between ranks."""
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    (_, fp0, f0, w0, s0), (_, fp1, f1, w1, s1) = got
    assert s0 == s1
    assert fp0 != fp1
    # the key padding differs per shard, so the per-rank work may differ; the job sums it
    assert w0 == pytest.approx(f0 + f1) and w1 == pytest.approx(f0 + f1)
