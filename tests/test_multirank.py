"""The N > 1 launch of the benchmark on CPU: two gloo ranks, each with its own synthetic
batch (seeded by rank) and its own timing; the job's time is the slowest rank's and its
throughput counts every rank's sequences (weak scaling, no collective in the data path)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench._dist()
        fls, _ = bench.load_workload(1, seed=r, batch=1, ctx=256)
        fl = fls[0]
        # a different per-rank step time; every rank must see the slowest
        ms = [3.0, 5.0][r]
        dist.barrier()
        worst = bench.max_over_ranks(ms, w)
        value = bench.job_throughput(w, 1, worst * 1e-3)
        q.put((r, w, local, worst, value, fl.q[0, 0, :8].tolist(), int(fl.targets.sum())))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, l0, worst0, v0, q0, t0), (r1, w1, l1, worst1, v1, q1, t1) = res
    assert (r0, r1, w0, w1, l0, l1) == (0, 1, 2, 2, 0, 1)
    assert worst0 == worst1 == 5.0
    assert v0 == v1 == pytest.approx(2 * 1 / 5e-3)
    # each rank decodes its own synthetic batch
    assert q0 != q1


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.job_throughput(1, 8, 0.5) == 16.0
