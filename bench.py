#!/usr/bin/env python
"""Benchmark of the pruned-KV decode path on GB300.

One step = the whole path over one batch: KVzap-Linear scores of every cached
token (tcgen05), keep/evict mask, compaction of the survivors into 16-token
pages, split-KV decode attention of the batch's query tokens. Workload: a
Llama-3-8B-shaped layer (d_model 4096, 32 query / 8 KV heads, head_dim 128,
batch 16, 8192 cached tokens, threshold at each head's 75th-percentile score,
last 128 tokens always kept). Metric: decode tokens/s (batch / step time).

Arms:
  default            the CUDA path through the C ABI (device-resident inputs),
                     plus an end-to-end leg with pinned host inputs copied in
                     and the output copied back inside the timed region, plus
                     the oracle timed on a bounded sample (cpu_baseline)
  --impl reference   the oracle (float64 CPU reference) on host cores, on a
                     bounded sample per step
Multi-GPU (torchrun): every rank runs its own batch (weak scaling, no data-path
collective); rank 0 prints the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

if "--impl" in sys.argv and "reference" in sys.argv or "--cpu-baseline-only" in sys.argv:
    # the oracle is timed single-threaded: every library below runs on one core
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_v] = "1"

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "pruned-KV decode tokens/s at 1 GB300; effective HBM GB/s vs ~8 TB/s peak"
UNIT = "tokens/s"
WORKLOAD = dict(name="llama3_8b_layer", d_model=4096, n_q_heads=32, n_kv_heads=8, head_dim=128, batch=16,
                n_pos=8192, prune_q=0.75, window=128)


# DRAM read + write bytes per row of hidden states of the tcgen05 scorer
# (KVzap-Linear, d_model 4096, 8 heads), from an ncu capture of that kernel on
# 32,768 rows: (268.592 + 3.492) MB / 32,768 rows. Valid while the scorer kernel
# is unchanged.
SCORE_DRAM_BYTES_PER_ROW = 272.084e6 / 32768

# Kernels of this library launched per step at this workload's size (B*H <= 1024):
# scorer (on the weight split once at set-up), segment count + copy pass of the
# compaction with the mask fused in, decode attention; one more (the mask
# kernel) with --mask separate. The compaction and attention calls also issue
# one memset each.
KERNELS_PER_STEP = {"fused": 4, "separate": 5}


def scorer_overhead(w=WORKLOAD, ffn_hidden=14336, mlp_hidden=1024):
    """The KVzap summary's overhead figures ("메모리 및 계산 효율": about 0.02 % of the linear-projection FLOPs
    for KVzap-Linear, about 1.1 % for KVzap-MLP) as closed forms for this layer's shape: scorer multiply-adds
    per token over the layer's Q, K, V, O and gated feed-forward projections."""
    D, Hq, H, d = w["d_model"], w["n_q_heads"], w["n_kv_heads"], w["head_dim"]
    proj = 2 * D * Hq * d + 2 * D * H * d + 3 * D * ffn_hidden
    lin = D * H
    mlp = D * mlp_hidden + mlp_hidden * H
    return {"projection_macs_per_token": proj, "linear_macs_per_token": lin, "linear_fraction": lin / proj,
            "mlp_macs_per_token": mlp, "mlp_fraction": mlp / proj, "ffn_hidden": ffn_hidden, "mlp_hidden": mlp_hidden}


def config_desc(w=WORKLOAD, mask_mode=None):
    return {
        "workload": (f"{w['name']}: one layer, d_model {w['d_model']}, {w['n_q_heads']} q / {w['n_kv_heads']} kv "
                     f"heads, head_dim {w['head_dim']}, batch {w['batch']}, context {w['n_pos']}, KVzap-Linear "
                     f"scorer, threshold at each head's {int(w['prune_q'] * 100)}th-percentile score, last "
                     f"{w['window']} tokens kept; step = score + mask + compact + decode attention"
                     f"{ {'fused': ' (mask fused into the compaction)', 'separate': ' (mask as its own kernel)'}.get(mask_mode, '')}"),
        "global_batch": w["batch"],
        "seq_len": w["n_pos"],
        "parallelism": "replicas: each rank decodes its own batch",
        "l2": "inputs larger than L2 (hidden states 1.07 GB, dense K/V 1.07 GB per step); no flush",
    }


# --------------------------------------------------------------------------- oracle sample (CPU)

class OracleSample:
    """One sequence of the workload drawn once on the host; run(rows) times the
    oracle over the last `rows` cached positions of it (score, mask,
    compaction, attention of the sequence's query heads) and returns (seconds,
    sequences-equivalent = rows / n_pos)."""

    def __init__(self, seed: int = 0, w=WORKLOAD):
        import kvp_synth as syn
        self.w = w
        D, H, d, T = w["d_model"], w["n_kv_heads"], w["head_dim"], w["n_pos"]
        G = w["n_q_heads"] // H
        self.x, self.W = syn.linear_inputs(seed, T, D, H)
        self.k, self.v = syn.kv_inputs(seed, 1, T, H, d)
        self.q = syn.q_inputs(seed, 1, H * G, d)
        self.tau = np.zeros((1, H), np.float32)  # the oracle's work does not depend on tau's value
        self.phases = {"score": 0.0, "mask": 0.0, "compact": 0.0, "attention": 0.0}

    def run(self, rows: int):
        import oracle as orc
        w = self.w
        H, T = w["n_kv_heads"], w["n_pos"]
        now, pos0 = T - 1, T - rows
        t0 = time.perf_counter()
        s = orc.score_linear(self.x[pos0:], self.W).reshape(1, rows, H)
        t1 = time.perf_counter()
        exp = orc.mask_kvzap(s, self.tau, now, window=w["window"], pos0=pos0)[0]
        t2 = time.perf_counter()
        mp = (rows + 15) // 16
        c = orc.compact_dense(self.k[:, pos0:], self.v[:, pos0:], exp, now, 0, H * mp, mp)
        t3 = time.perf_counter()
        orc.decode_attention(self.q, c, now)
        t4 = time.perf_counter()
        for k, dt in zip(("score", "mask", "compact", "attention"), (t1 - t0, t2 - t1, t3 - t2, t4 - t3)):
            self.phases[k] += dt
        return t4 - t0, rows / T


def run_cpu_baseline(budget_s: float):
    """About `budget_s` seconds of oracle work, single-threaded."""
    T = WORKLOAD["n_pos"]
    sample = OracleSample()
    t1, _ = sample.run(T)
    total_t, total_seq, runs = t1, 1.0, 1
    while total_t < budget_s and runs < 1000:
        t, sq = sample.run(T)
        total_t += t
        total_seq += sq
        runs += 1
    return {"value": total_seq / total_t, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{runs} full sequences of the workload (one sequence's 8192 cached positions, drawn once "
                      f"and re-run): float64 score, mask, compaction and attention of its query heads, one thread",
            "seconds": total_t, "phase_seconds": {k: round(v, 3) for k, v in sample.phases.items()}}


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    T = WORKLOAD["n_pos"]
    budget = 120.0
    sample = OracleSample()
    t1, _ = sample.run(T)
    rows = int(max(64, min(T, budget / max(1, args.steps + args.warmup) / (t1 / T))))
    for _ in range(args.warmup):
        sample.run(rows)
    total_t, total_seq = 0.0, 0.0
    for _ in range(args.steps):
        t, sq = sample.run(rows)
        total_t += t
        total_seq += sq
    value = total_seq / total_t
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": config_desc(), "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"per step the last {rows} cached positions of one sequence ({rows / T:.4f} of "
                                   f"a sequence's decode step): score, mask, compaction, attention in float64"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while timing."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"kvp_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9 and p[0].isdigit() and int(p[0]) == self.index:
                    rows.append(p)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


def max_over_ranks(x: float, device=None) -> float:
    """The largest of every rank's x (the job is as slow as its slowest rank);
    x itself when no process group is running."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(batch_per_rank: int, world: int, ms_per_step: float) -> float:
    """Decode tokens/s of the whole job: every rank decodes its own batch of
    one token per sequence per step."""
    return batch_per_rank * world / (ms_per_step * 1e-3)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def run_gpu(args, rank: int, world: int):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import kv_cache_pruning_gb300 as kvp

    w = dict(WORKLOAD)
    if args.batch:
        w["batch"] = args.batch
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    B, T, H, Hq, d, D = w["batch"], w["n_pos"], w["n_kv_heads"], w["n_q_heads"], w["head_dim"], w["d_model"]
    n_tok = B * T
    now = T - 1

    # ---- seeded synthetic inputs, resident in HBM
    g = torch.Generator(device=dev)
    g.manual_seed(1000 * args.seed + rank)
    x = torch.randn(n_tok, D, generator=g, device=dev).to(torch.bfloat16)
    W = torch.randn(H, D, generator=g, device=dev) / math.sqrt(D)
    K = torch.randn(B, T, H, d, generator=g, device=dev).to(torch.bfloat16)
    V = torch.randn(B, T, H, d, generator=g, device=dev).to(torch.bfloat16)
    q = torch.randn(B, Hq, d, generator=g, device=dev).to(torch.bfloat16)

    # ---- buffers, sized once (keep-all capacity), reused by every step
    max_pages = (T + 15) // 16
    n_pages_cap = B * H * max_pages
    cache = kvp.PagedKV.allocate(B, H, d, n_pages_cap, max_pages, device=dev)
    scores = torch.empty(n_tok, H, dtype=torch.float32, device=dev)
    separate = args.mask == "separate"  # the mask's own outputs exist only when it runs as its own kernel
    expire = torch.empty(B, H, T, dtype=torch.int32, device=dev) if separate else None
    bits = torch.empty(B, H, (T + 31) // 32, dtype=torch.int32, device=dev) if separate else None
    count = torch.empty(B, H, dtype=torch.int32, device=dev) if separate else None
    out = torch.empty(B, Hq, d, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_s = torch.empty(kvp.kvp_score_workspace_bytes(0, n_tok, D, H), dtype=torch.uint8, device=dev)
    ws_c = torch.empty(kvp.kvp_compact_workspace_bytes(B, H, T), dtype=torch.uint8, device=dev)
    ws_a = torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, Hq, H, d), dtype=torch.uint8, device=dev)

    # ---- the layer's scorer weight in tensor-core form, made once per layer
    # like the weight itself (set-up, untimed)
    Ws = kvp.kvp_score_split_weight(W)

    # ---- threshold per (b, h): the 75th-percentile score, chosen on the device
    # (harness set-up, untimed)
    kvp.kvp_score(x, W, out=scores, workspace=ws_s, status=status)
    tau = kvp.kvp_threshold(scores.view(B, T, H), w["prune_q"])
    fused = args.mask == "fused"

    stream = torch.cuda.current_stream(dev)
    # event slots per step: before score, [mask,] compact, attention, after
    names = ["score", "mask+compact", "decode_attn"] if fused else ["score", "mask", "compact", "decode_attn"]
    N_EV = len(names) + 1

    def step(evs=None):
        e = iter(evs) if evs is not None else None
        if e is not None:
            next(e).record(stream)
        kvp.kvp_score(x, Ws, scorer=kvp.KVP_SCORER_LINEAR_SPLIT, n_kv_heads=H, out=scores, status=status)
        if e is not None:
            next(e).record(stream)
        if fused:
            kvp.kvp_compact_masked(K, V, now, 0, cache, mode=kvp.KVP_MASK_KVZAP, scores=scores, tau=tau,
                                   window=w["window"], status=status, workspace=ws_c)
        else:
            kvp.kvp_mask(mode=kvp.KVP_MASK_KVZAP, batch=B, n_kv_heads=H, n_pos=T, now=now, scores=scores, tau=tau,
                         window=w["window"], expire=expire, keep_bits=bits, count=count)
            if e is not None:
                next(e).record(stream)
            kvp.kvp_compact(K, V, expire, now, 0, cache, status=status, workspace=ws_c)
        if e is not None:
            next(e).record(stream)
        kvp.kvp_decode_attn(q, cache, now, out=out, workspace=ws_a, status=status)
        if e is not None:
            next(e).record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert status.item() == 0, kvp.status_string(status.item())
    count = cache.count
    kept = int(count.sum().item())
    surv_pages = int(((count + 15) // 16).sum().item())

    dist = world > 1
    if dist:
        import torch.distributed as tdist
    # The step is captured once as a CUDA graph (its kernels and memsets as
    # nodes) and replayed: no host launch work inside the timed region.
    graph = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        assert status.item() == 0, kvp.status_string(status.item())
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        if dist:
            tdist.barrier()
        torch.cuda.synchronize()
        t_start.record(stream)
        for i in range(args.steps):
            if graph is not None:
                graph.replay()
            else:
                step()
        t_end.record(stream)
        torch.cuda.synchronize()
        if dist:
            tdist.barrier()
    clocks = clk.summary()
    assert status.item() == 0, kvp.status_string(status.item())
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), dev)
    ms_step = total_ms / args.steps

    # ---- per-phase times: eager steps with an event between phases (a
    # separate loop, so these events are not inside the timed region above)
    n_break = max(3, min(args.steps, 50))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(N_EV)] for _ in range(n_break)]
    for i in range(n_break):
        step(evs[i])
    torch.cuda.synchronize()
    per = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(N_EV - 1)] for i in range(n_break)])
    k_ms = per.mean(axis=0)  # per phase of `names` (per launch, ms)

    # ---- algorithmic bytes (what the method must move)
    x_b = n_tok * D * 2
    score_b = x_b + Ws.numel() * 2 + n_tok * H * 4
    mask_b = n_tok * H * 4 + B * H * 4 + B * H * T * 4 + B * H * ((T + 31) // 32) * 4 + B * H * 4
    row_b = d * 2
    compact_b = 2 * B * H * T * 4 + 2 * kept * 2 * row_b + kept * 4 + B * H * max_pages * 16 * 4 \
        + B * H * max_pages * 4
    attn_b = surv_pages * 16 * (2 * row_b + 4) + B * Hq * d * 2 + B * Hq * d * 4
    # fused: the mask reads the scores and thresholds and writes nothing of its own
    fused_b = n_tok * H * 4 + B * H * 4 + (compact_b - 2 * B * H * T * 4)
    kb = [score_b, fused_b, attn_b] if fused else [score_b, mask_b, compact_b, attn_b]
    step_b = sum(kb)
    hbm, _, peak_kind = measured_peaks()
    kernels = {n: {"ms": float(k_ms[i]), "bytes": int(kb[i]), "GB_s": kb[i] / (k_ms[i] * 1e-3) / 1e9,
                   "frac_of_hbm": kb[i] / (k_ms[i] * 1e-3) / 1e9 / hbm} for i, n in enumerate(names)}
    dom = int(np.argmax(k_ms))
    traffic = args.traffic
    if traffic is None and names[dom] == "score":
        traffic = SCORE_DRAM_BYTES_PER_ROW * n_tok
    roofline = {"bound": "hbm", "kernel": names[dom], "achieved": kb[dom] / (k_ms[dom] * 1e-3) / 1e9,
                "peak": hbm, "unit": "GB/s", "frac": kb[dom] / (k_ms[dom] * 1e-3) / 1e9 / hbm,
                "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else peak_kind,
                "traffic": traffic}
    value = weak_scaling_value(B, world, ms_step)

    # ---- end to end: pinned host inputs in, result out, inside the timed region
    e2e = None
    if not args.no_e2e:
        xh = x.cpu().pin_memory()
        Kh, Vh, qh = K.cpu().pin_memory(), V.cpu().pin_memory(), q.cpu().pin_memory()
        Wh, tauh = Ws.cpu().pin_memory(), tau.cpu().pin_memory()
        outh = torch.empty_like(out, device="cpu").pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (xh, Kh, Vh, qh, Wh, tauh))
        d2h = outh.numel() * outh.element_size()

        def e2e_step():
            for dst, src in ((x, xh), (K, Kh), (V, Vh), (q, qh), (Ws, Wh), (tau, tauh)):
                dst.copy_(src, non_blocking=True)
            step()
            outh.copy_(out, non_blocking=True)

        n_e2e = max(3, min(args.steps, args.e2e_steps))
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        if dist:
            tdist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, dev)
        e2e = {"value": weak_scaling_value(B, world, e_ms), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e_ms, "steps": n_e2e,
               "h2d_GB_s": h2d / (e_ms * 1e-3) / 1e9}

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-only",
                            "--cpu-budget", str(args.cpu_budget)], capture_output=True, text=True, cwd=ROOT)
        try:
            cpu = json.loads(r.stdout.strip().splitlines()[-1])
        except Exception:
            cpu = {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": "failed: " + r.stderr[-300:]}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded torch RNG, N(0,1) hidden states and K/V)",
        "config": dict(config_desc(w, args.mask), cuda_graph=graph is not None), "e2e": e2e,
        "gpu_launches": KERNELS_PER_STEP[args.mask] * args.steps, "roofline": roofline,
        "kernels": kernels, "effective_step_GB_s": step_b / (ms_step * 1e-3) / 1e9,
        "scored_tokens_per_s": n_tok / (k_ms[0] * 1e-3),
        "scorer_overhead": scorer_overhead(w),
        "kept_fraction": kept / (B * H * T), "clocks": clocks, "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvp", choices=["kvp", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0, help="override the batch (profiling runs only)")
    ap.add_argument("--workload", default="llama3_8b_layer",
                    choices=["llama3_8b_layer", "mlp_prefill", "dms_decode", "llama65b_mha", "prune_sweep",
                             "threshold", "quant_tier", "quant_decode", "gqa_sweep", "mla_sweep", "mla_dms_decode"],
                    help="llama3_8b_layer = the bench line; the others print measurement lines "
                         "(see bench_workloads.py)")
    ap.add_argument("--eager", action="store_true", help="launch every step from the host (no CUDA graph)")
    ap.add_argument("--mask", default="fused", choices=["fused", "separate"],
                    help="fused: the mask is computed inside the compaction's passes (kvp_compact_masked); "
                         "separate: kvp_mask writes expire, then kvp_compact reads it")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--cpu-baseline-only", action="store_true")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the dominant kernel from an ncu capture of this kernel "
                         "(default: the scorer's measured bytes per row times the rows of one launch)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.cpu_baseline_only:
        print(json.dumps(run_cpu_baseline(args.cpu_budget)), flush=True)
        return
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if world > 1 and args.impl != "reference":
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.workload != "llama3_8b_layer":
        import torch
        import __graft_entry__
        import bench_workloads
        __graft_entry__.build()
        import kv_cache_pruning_gb300 as kvp
        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
        torch.cuda.set_device(dev)
        bench_workloads.run(args.workload, kvp, dev, measured_peaks())
        return
    run_gpu(args, rank, world)
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
