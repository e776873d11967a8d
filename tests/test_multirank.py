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


def _seq_split_worker(rank, world, port, out):
    """One rank of a sequence split: attention over its contiguous share of the
    positions, in the library's partial-state format (each row normalised over
    the share, with its log-sum-exp), then an all-gather of (out, lse) and the
    merge. The device path cannot run on these CPU ranks, so each rank's share
    goes through the oracle."""
    import numpy as np
    import torch
    import torch.distributed as tdist

    import kvp_synth as syn
    import oracle as orc
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    B, T, H, G, d = 1, 640, 4, 2, 32
    k, v = syn.kv_inputs(21, B, T, H, d)
    q = syn.q_inputs(21, B, H * G, d)
    s = syn.normal_f32(21, 5, (B, T, H))
    now = T - 1
    exp = orc.mask_kvzap(s, orc.threshold_at_quantile(s, 0.7), now)[0]
    lo, hi = rank * T // world, (rank + 1) * T // world
    mp = (hi - lo + 15) // 16
    part = orc.compact_dense(k[:, lo:hi], v[:, lo:hi], exp[:, :, lo:hi], now, 0, n_pages_cap=B * H * mp,
                             max_pages=mp)
    o_r, l_r = orc.decode_attention_lse(q, part, now)
    o_all = [torch.empty(o_r.shape, dtype=torch.float64) for _ in range(world)]
    l_all = [torch.empty(l_r.shape, dtype=torch.float64) for _ in range(world)]
    tdist.all_gather(o_all, torch.from_numpy(o_r.astype(np.float64)))
    tdist.all_gather(l_all, torch.from_numpy(l_r))
    o_m, l_m = orc.merge_attention(torch.stack(o_all).numpy(), torch.stack(l_all).numpy())
    mpw = (T + 15) // 16
    whole = orc.compact_dense(k, v, exp, now, 0, n_pages_cap=B * H * mpw, max_pages=mpw)
    o_w, l_w = orc.decode_attention_lse(q, whole, now)
    out[rank] = (float(np.abs(o_m - o_w).max()), float(np.abs(l_m - l_w).max()))
    tdist.barrier()
    tdist.destroy_process_group()


def test_sequence_split_over_two_gloo_ranks_merges_to_the_whole():
    world = 2
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_seq_split_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    for r in range(world):
        d_out, d_lse = out[r]
        assert d_out <= 2e-6 and d_lse <= 1e-12, (r, d_out, d_lse)
