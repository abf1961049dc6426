"""bench.py's multi-rank bookkeeping on CPU: two gloo ranks (127.0.0.1),
the job time is the slowest rank's, the whole-job rate counts every rank's
units, and --gpus must match the launched world size."""
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


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.0 + rank, dist)  # rank 1 is the slow one
        q.put((rank, ms, bench.whole_job_rate(240, ms, world)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [ms for _, ms, _ in res] == [2.0, 2.0]
    # 240 units per rank per step, 2 ranks, 2 ms per step: 240 000 units/s
    assert all(rate == pytest.approx(240_000.0) for _, _, rate in res)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.whole_job_rate(15, 0.5, 1) == pytest.approx(30_000.0)


def test_gpus_must_match_the_launched_ranks():
    bench.check_world(1, 1)
    bench.check_world(4, 4)
    with pytest.raises(SystemExit) as e:
        bench.check_world(2, 1)
    assert "torch.distributed.run" in str(e.value)
