"""The N > 1 host path of bench.py on CPU ranks (gloo, world size 2).

On N GPUs every rank runs an independent replica of the forward pass on its
own inputs (the heads are independent problems: no data-path collective);
the only cross-rank steps are the barriers around the timed region and the
max over ranks of the step time. These tests run those steps as two gloo
processes and check the whole-job numbers rank 0 reports."""
import os
import socket

import numpy as np
import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, ms_by_rank, queue):
    import torch.distributed as dist

    import bench
    import synth

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_barrier(world)
        ms = bench.max_over_ranks(ms_by_rank[rank], world)
        value = bench.job_throughput(1000, world, ms)
        # replicas draw their own inputs (seed = rank)
        q, _, _ = synth.make_inputs(synth.CONFIGS["tiny"], seed=rank)
        bench.rank_barrier(world)
        queue.put((rank, ms, value, int(q.view(np.uint16).astype(np.int64).sum())))
    finally:
        dist.destroy_process_group()


def _run_ranks(world, ms_by_rank):
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, ms_by_rank, queue)) for r in range(world)]
    for p in procs:
        p.start()
    out = [queue.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out)


def test_two_ranks_take_the_slowest_time():
    res = _run_ranks(2, [3.0, 5.0])
    assert [r[1] for r in res] == [5.0, 5.0]  # every rank sees the max
    # whole-job rate: both ranks' queries over the slowest rank's time
    assert res[0][2] == pytest.approx(2 * 1000 / 5e-3)
    # the replicas' inputs differ
    assert res[0][3] != res[1][3]


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(4.0, 1) == 4.0
    assert bench.job_throughput(1000, 1, 4.0) == pytest.approx(1000 / 4e-3)
    bench.rank_barrier(1)


def test_reference_arm_other_ranks_do_no_work():
    import argparse

    import bench

    args = argparse.Namespace(config="tiny", steps=1, warmup=0)
    assert bench.run_reference(args, 1, 2) is None
