"""Host-side logic of the multi-rank benchmark on CPU: two gloo ranks, each
decoding its own batch (replicas, no data-path collective). The job's time is
the slowest rank's; its throughput counts every rank's tokens; only rank 0
prints the reference arm's line."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as tdist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.max_over_ranks(1.0 + rank * 0.5)       # rank 1 is the slow one
    out[rank] = (t, bench.weak_scaling_value(16, world, t))
    tdist.barrier()
    tdist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_tokens():
    world = 2
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 1.5
    assert out[0][1] == pytest.approx(16 * 2 / 1.5e-3)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.weak_scaling_value(16, 1, 0.3) == pytest.approx(16 / 0.3e-3)


def test_reference_arm_prints_on_rank_zero_only(capsys):
    import argparse
    import bench
    args = argparse.Namespace(steps=1, warmup=0)
    bench.run_reference(args, rank=1, world=2)
    assert capsys.readouterr().out == ""
