"""The replicas path of bench.py under two ranks, on the CPU with the gloo backend.

Streams are independent, so N GPUs run N replicas with no collective on the data path; the only
collectives are the barrier and the max-over-ranks reduction of the timed region.  These tests
run that host logic in two processes: each rank gets its own streams' inputs, both ranks see the
slowest rank's time, and the rate counts every rank's streams.  A rank that fails before the
reduction makes the others' reduction end with an error instead of hanging.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import workloads as wl

STEPS = 50


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q, fail_rank):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    from datetime import timedelta

    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=timedelta(seconds=20))
    try:
        cfg = bench.rank_workload(wl.TINY, rank)
        logits = wl.logits(cfg)
        if rank == fail_rank:
            raise SystemExit(3)  # leaves before the reduction
        ms = 10.0 * (rank + 1)  # this rank's timed region
        job = bench.max_over_ranks(ms, world)
        q.put(("ok", rank, job, bench.whole_job_rate(world, cfg.N, STEPS, job), cfg.base_seed,
               float(np.asarray(logits, dtype=np.float64).sum())))
    except RuntimeError as e:  # the collective failed because a peer is gone
        q.put(("error", rank, str(e)[:200]))
    finally:
        if rank != fail_rank:
            dist.destroy_process_group()


def _run(world, fail_rank=-1):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q, fail_rank)) for r in range(world)]
    for p in procs:
        p.start()
    n_reports = world - (1 if fail_rank >= 0 else 0)
    res = [q.get(timeout=180) for _ in range(n_reports)]
    for p in procs:
        p.join(timeout=60)
        if p.is_alive():
            p.kill()
    return res, [p.exitcode for p in procs]


def test_two_rank_replicas_share_the_slowest_time():
    res, codes = _run(2)
    assert codes == [0, 0]
    res = sorted(res, key=lambda r: r[1])
    assert all(r[0] == "ok" for r in res)
    (_, _, job0, v0, seed0, sum0), (_, _, job1, v1, seed1, sum1) = res
    assert job0 == job1 == 20.0                       # the slower rank's 20 ms
    assert v0 == v1 == 2 * wl.TINY.N * STEPS / 0.020  # whole job: both ranks' streams
    assert seed1 == seed0 + wl.TINY.N                 # rank 1 owns the next N streams' seeds
    assert sum0 != sum1                               # so its inputs differ


def test_one_rank_is_the_identity():
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.rank_workload(wl.HEADLINE, 0) is wl.HEADLINE
    assert bench.whole_job_rate(1, 32, 50, 5.8) == pytest.approx(32 * 50 / 0.0058)


def test_a_rank_that_leaves_ends_the_others_reduction():
    res, codes = _run(2, fail_rank=1)
    assert codes[1] == 3
    assert len(res) == 1 and res[0][0] == "error" and res[0][1] == 0
