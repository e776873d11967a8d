"""Measurement runs of the other synthetic workloads (bench.py --workload NAME).

The default bench line is the 8-layer Llama-65B-shaped MHA decode step; these
runs measure the rest of the path on the shapes it is quoted for:

  mlp_prefill    KVzap-MLP scoring of 4 x 32,768 prompt tokens (d_model 4096 ->
                 1024 GELU -> 8 heads; tensor-bound), 80% pruned, compaction into
                 16-token pages, then 64 decode steps (new token scored, appended,
                 GQA attention over the survivors)
  dms_decode     DMS delayed eviction, Qwen-3-8B-shaped attention: batch 64,
                 4,096-token prompt, 1,024 decode steps, evict flag
                 ~Bernoulli(7/8), eviction 256 steps after the flag, 128-token
                 window, re-compaction every 64 steps into a second pool
  llama65b_mha   8 MHA layers (64 heads, d_model 8192), batch 1, 131,072 cached
                 tokens, KVzap-Linear with per-(layer, head) keep rates ~Beta(2,5),
                 then 32 decode steps over all 8 layers
  prune_sweep    decode attention on the Llama-3-8B-shaped cache at pruning
                 levels 0 / 50 / 75 / 87.5 / 93.75 / 96.9 %: tokens/s against the
                 inverse of the kept fraction
  prune_sweep_long  the same sweep on one layer of the 65B-shaped MHA stack
                 (64 heads, 131,072 cached tokens, batch 1)

Decode loops are captured once in a CUDA graph (the C-ABI calls only enqueue
work on the current stream) and replayed for timing, so host launch overhead
is not measured. Inputs are seeded torch draws on the device.
"""
from __future__ import annotations

import json
import math

import torch


def _ev():
    return torch.cuda.Event(enable_timing=True)


def _time(fn, reps=1):
    torch.cuda.synchronize()
    a, b = _ev(), _ev()
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def _graph(fn):
    """Capture fn (after one eager warm-up) and return a replay callable."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g.replay


def _randn_bf16(shape, gen, dev, std=1.0):
    return (torch.randn(shape, generator=gen, device=dev, dtype=torch.bfloat16) * std).contiguous()


def _tau_quantile(kvp, scores_bth, q):
    """Per-(b, h) lower order statistic at index floor(q (T-1)), chosen on the device."""
    return kvp.kvp_threshold(scores_bth.contiguous(), q)


def mlp_prefill(kvp, dev, peaks, seed=0):
    B, T, D, HID, H, Hq, d, steps, reserve = 4, 32768, 4096, 1024, 8, 32, 128, 64, 64
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    x = _randn_bf16((B * T, D), g, dev)
    w1 = _randn_bf16((HID, D), g, dev, 1 / math.sqrt(D))
    w2 = _randn_bf16((H, HID), g, dev, 1 / math.sqrt(HID))
    K = _randn_bf16((B, T, H, d), g, dev)
    V = _randn_bf16((B, T, H, d), g, dev)
    xs = _randn_bf16((steps, B, D), g, dev)
    ks = _randn_bf16((steps, B, H, d), g, dev)
    vs = _randn_bf16((steps, B, H, d), g, dev)
    qs = _randn_bf16((steps, B, Hq, d), g, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    MLP = kvp.KVP_SCORER_MLP
    scores = torch.empty(B * T, H, dtype=torch.float32, device=dev)
    ws = torch.empty(kvp.kvp_score_workspace_bytes(MLP, B * T, D, H, HID), dtype=torch.uint8, device=dev)

    def score():
        kvp.kvp_score(x, w1, None, w2, None, scorer=MLP, out=scores, workspace=ws, status=st)

    for _ in range(3):
        score()
    ms_score = _time(score, reps=10)
    flops = 2.0 * B * T * D * HID + 2.0 * B * T * HID * H
    tau = _tau_quantile(kvp, scores.view(B, T, H), 0.8)
    now = T - 1
    expire, _, count = kvp.kvp_mask(mode=kvp.KVP_MASK_KVZAP, batch=B, n_kv_heads=H, n_pos=T, now=now,
                                    scores=scores, tau=tau)
    mp = (T + reserve + 15) // 16
    cache = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp, device=dev)

    def prefill_rest():
        kvp.kvp_mask(mode=kvp.KVP_MASK_KVZAP, batch=B, n_kv_heads=H, n_pos=T, now=now, scores=scores, tau=tau,
                     expire=expire, count=count, want_bits=False)
        kvp.kvp_compact(K, V, expire, now, reserve, cache, status=st)

    prefill_rest()
    ms_mask_compact = _time(prefill_rest, reps=10)
    kept = int(count.sum().item())
    snapshot = [t.clone() for t in (cache.k_pool, cache.v_pool, cache.expire_pool, cache.page_table, cache.remap,
                                    cache.count)]
    s_new = torch.empty(B, H, dtype=torch.float32, device=dev)
    ws_new = torch.empty(kvp.kvp_score_workspace_bytes(MLP, B, D, H, HID), dtype=torch.uint8, device=dev)
    out = torch.empty(steps, B, Hq, d, dtype=torch.float32, device=dev)
    ws_a = torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, Hq, H, d), dtype=torch.uint8, device=dev)

    def restore():
        for dst, src in zip((cache.k_pool, cache.v_pool, cache.expire_pool, cache.page_table, cache.remap,
                             cache.count), snapshot):
            dst.copy_(src)

    def decode():
        for i in range(steps):
            t = T + i
            kvp.kvp_score(xs[i], w1, None, w2, None, scorer=MLP, out=s_new, workspace=ws_new, status=st)
            kvp.kvp_append(cache, ks[i], vs[i], t, mode=kvp.KVP_MASK_KVZAP, score=s_new, tau=tau, status=st)
            kvp.kvp_decode_attn(qs[i], cache, t, out=out[i], workspace=ws_a, status=st)

    replay = _graph(lambda: (restore(), decode()))
    ms_restore = _time(lambda: restore(), reps=3)
    ms_decode = _time(replay, reps=3) - ms_restore
    torch.cuda.synchronize()
    assert st.item() == 0, kvp.status_string(st.item())

    # the same steps with L2 flushed before each one (the survivors, about 109 MB, fit in the 129 MB L2):
    # one CUDA graph per step, events around the step only
    def one_step(i):
        t = T + i
        kvp.kvp_score(xs[i], w1, None, w2, None, scorer=MLP, out=s_new, workspace=ws_new, status=st)
        kvp.kvp_append(cache, ks[i], vs[i], t, mode=kvp.KVP_MASK_KVZAP, score=s_new, tau=tau, status=st)
        kvp.kvp_decode_attn(qs[i], cache, t, out=out[i], workspace=ws_a, status=st)

    restore()
    step_graphs = []
    for i in range(steps):
        one_step(i)  # warm-up of step i; restore() below resets the cache
    for i in range(steps):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            one_step(i)
        step_graphs.append(gr)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    restore()
    torch.cuda.synchronize()
    ms_flushed = 0.0
    for i in range(steps):
        flush.zero_()
        a, b_ = _ev(), _ev()
        a.record()
        step_graphs[i].replay()
        b_.record()
        torch.cuda.synchronize()
        ms_flushed += a.elapsed_time(b_)
    assert st.item() == 0, kvp.status_string(st.item())
    kv_pages = int(((cache.count + 15) // 16).sum().item())
    attn_bytes = kv_pages * 16 * (2 * d * 2 + 4)
    return {
        "workload": "mlp_prefill: KVzap-MLP d_model 4096 -> 1024 (GELU) -> 8, batch 4 x 32768 prompt tokens, "
                    "80% pruned, 128-token window, 64 decode steps (GQA 32/8, head_dim 128)",
        "scorer_ms": ms_score, "scorer_tflops": flops / (ms_score * 1e-3) / 1e12,
        "scorer_frac_of_bf16_peak": flops / (ms_score * 1e-3) / 1e12 / peaks[1],
        "scored_tokens_per_s": B * T / (ms_score * 1e-3),
        "mask_compact_ms": ms_mask_compact, "kept_fraction": kept / (B * H * T),
        "decode_ms_per_step": ms_decode / steps, "decode_tokens_per_s": B * steps / (ms_decode * 1e-3),
        "decode_ms_per_step_l2_flushed": ms_flushed / steps,
        "decode_tokens_per_s_l2_flushed": B * steps / (ms_flushed * 1e-3),
        "attn_bytes_last_step": attn_bytes, "peaks": {"hbm_gbs": peaks[0], "bf16_tflops": peaks[1]},
    }


def dms_decode(kvp, dev, peaks, seed=0, steps=1024):
    B, T0, H, Hq, d, delay, W, every, reserve = 64, 4096, 8, 32, 128, 256, 128, 64, 64
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    K = _randn_bf16((B, T0, H, d), g, dev)
    V = _randn_bf16((B, T0, H, d), g, dev)
    pos = torch.arange(T0, device=dev, dtype=torch.int32)
    f0 = torch.where(torch.rand((B, H, T0), generator=g, device=dev) < 7 / 8, pos, -1).to(torch.int32)
    ks = _randn_bf16((steps, B, H, d), g, dev)
    vs = _randn_bf16((steps, B, H, d), g, dev)
    qs = _randn_bf16((steps, B, Hq, d), g, dev)
    tpos = (T0 + torch.arange(steps, device=dev, dtype=torch.int32)).view(steps, 1, 1)
    fs = torch.where(torch.rand((steps, B, H), generator=g, device=dev) < 7 / 8, tpos, -1).to(torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    now0 = T0 - 1
    expire, _, _ = kvp.kvp_mask(mode=kvp.KVP_MASK_DMS, batch=B, n_kv_heads=H, n_pos=T0, now=now0, flag_step=f0,
                                delay=delay, window=W, want_bits=False)
    mp = (T0 + steps + reserve + 15) // 16
    cap = B * H * mp
    pools = [kvp.PagedKV.allocate(B, H, d, cap, mp, device=dev) for _ in range(2)]
    out = torch.empty(steps, B, Hq, d, dtype=torch.float32, device=dev)
    ws_a = torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, Hq, H, d), dtype=torch.uint8, device=dev)
    ws_c = torch.empty(kvp.kvp_compact_workspace_bytes(B, H, T0), dtype=torch.uint8, device=dev)
    ws_p = torch.empty(kvp.kvp_compact_paged_workspace_bytes(B, H, mp), dtype=torch.uint8, device=dev)
    pages_read = torch.zeros((), dtype=torch.int64, device=dev)

    def prefill():
        kvp.kvp_compact(K, V, expire, now0, reserve, pools[0], status=st, workspace=ws_c)

    def decode(count_pages=False):
        cur = 0
        for i in range(steps):
            t = T0 + i
            if i > 0 and i % every == 0:
                kvp.kvp_compact_paged(pools[cur], t, reserve, pools[1 - cur], status=st, workspace=ws_p)
                cur = 1 - cur
            c = pools[cur]
            kvp.kvp_append(c, ks[i], vs[i], t, mode=kvp.KVP_MASK_DMS, flag_step=fs[i], delay=delay, window=W,
                           status=st)
            kvp.kvp_decode_attn(qs[i], c, t, out=out[i], workspace=ws_a, status=st)
            if count_pages:
                pages_read.add_(((c.count + 15) // 16).sum())

    prefill()
    decode(count_pages=True)  # eager pass: algorithmic bytes of the attention steps
    torch.cuda.synchronize()
    assert st.item() == 0, kvp.status_string(st.item())
    total_pages = int(pages_read.item())
    prefill()
    replay = _graph(decode)
    ms_pref = _time(prefill, reps=3)
    ms = _time(lambda: (prefill(), replay()), reps=3) - ms_pref
    torch.cuda.synchronize()
    assert st.item() == 0, kvp.status_string(st.item())
    attn_bytes = total_pages * 16 * (2 * d * 2 + 4)
    return {
        "workload": "dms_decode: batch 64, 32 q / 8 kv heads, head_dim 128, 4096-token prompt + 1024 steps, "
                    "evict ~Bernoulli(7/8), delay 256, window 128, re-compaction every 64 steps",
        "decode_ms_total": ms, "decode_ms_per_step": ms / steps, "decode_tokens_per_s": B * steps / (ms * 1e-3),
        "attn_pages_read_total": total_pages, "attn_bytes_total": attn_bytes,
        "effective_GB_s_attention_bytes_over_loop_time": attn_bytes / (ms * 1e-3) / 1e9,
        "frac_of_hbm": attn_bytes / (ms * 1e-3) / 1e9 / peaks[0],
        "dense_kv_bytes_last_step": B * H * (T0 + steps) * 2 * d * 2,
    }


def llama65b_mha(kvp, dev, peaks, seed=0, steps=32, n_layers=8):
    B, T, D, H, d, reserve = 1, 131072, 8192, 64, 128, 32
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    layers = []
    ms_score = ms_mc = 0.0
    score_bytes = 0
    scores = torch.empty(B * T, H, dtype=torch.float32, device=dev)
    ws_s = torch.empty(kvp.kvp_score_workspace_bytes(0, B * T, D, H), dtype=torch.uint8, device=dev)
    ws_c = torch.empty(kvp.kvp_compact_workspace_bytes(B, H, T), dtype=torch.uint8, device=dev)
    for layer in range(n_layers):
        x = _randn_bf16((B * T, D), g, dev)
        w = torch.randn((H, D), generator=g, device=dev) / math.sqrt(D)
        K = _randn_bf16((B, T, H, d), g, dev)
        V = _randn_bf16((B, T, H, d), g, dev)
        kvp.kvp_score(x, w, out=scores, workspace=ws_s, status=st)
        ms_score += _time(lambda: kvp.kvp_score(x, w, out=scores, workspace=ws_s, status=st), reps=3)
        score_bytes += x.numel() * 2
        # per-head keep rate r ~ Beta(2,5) (2nd smallest of 6 uniforms); tau at quantile 1 - r
        r = torch.rand((H, 6), generator=g, device=dev).sort(dim=1).values[:, 1]
        srt = scores.view(T, H).sort(dim=0).values
        idx = torch.floor((1 - r) * (T - 1)).long()
        tau = srt.gather(0, idx.view(1, H)).view(B, H).contiguous()
        expire, _, count = kvp.kvp_mask(mode=kvp.KVP_MASK_KVZAP, batch=B, n_kv_heads=H, n_pos=T, now=T - 1,
                                        scores=scores, tau=tau, want_bits=False)
        torch.cuda.synchronize()
        pages = int(((count + reserve + 15) // 16).sum().item())
        mp = (T + reserve + 15) // 16
        cache = kvp.PagedKV.allocate(B, H, d, pages, mp, device=dev)

        def mc():
            kvp.kvp_mask(mode=kvp.KVP_MASK_KVZAP, batch=B, n_kv_heads=H, n_pos=T, now=T - 1, scores=scores, tau=tau,
                         expire=expire, count=count, want_bits=False)
            kvp.kvp_compact(K, V, expire, T - 1, reserve, cache, status=st, workspace=ws_c)

        mc()
        ms_mc += _time(mc, reps=1)
        layers.append(dict(w=w, tau=tau, cache=cache,
                           snap=[t.clone() for t in (cache.expire_pool, cache.page_table, cache.remap, cache.count)]))
        del x, K, V
        torch.cuda.empty_cache()
    xs = _randn_bf16((steps, n_layers, B, D), g, dev)
    ks = _randn_bf16((steps, n_layers, B, H, d), g, dev)
    vs = _randn_bf16((steps, n_layers, B, H, d), g, dev)
    qs = _randn_bf16((steps, n_layers, B, H, d), g, dev)
    out = torch.empty(B, H, d, dtype=torch.float32, device=dev)
    s_new = torch.empty(B, H, dtype=torch.float32, device=dev)
    ws_a = torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, H, H, d), dtype=torch.uint8, device=dev)

    def restore():
        for L in layers:
            c = L["cache"]
            for dst, src in zip((c.expire_pool, c.page_table, c.remap, c.count), L["snap"]):
                dst.copy_(src)

    for L in layers:  # each layer's scorer weight in tensor-core form, once, like the weight itself
        L["w_split"] = kvp.kvp_score_split_weight(L["w"])

    def decode():
        for i in range(steps):
            t = T + i
            for li, L in enumerate(layers):
                kvp.kvp_score(xs[i, li], L["w_split"], scorer=kvp.KVP_SCORER_LINEAR_SPLIT, n_kv_heads=H,
                              out=s_new, status=st)
                kvp.kvp_append(L["cache"], ks[i, li], vs[i, li], t, mode=kvp.KVP_MASK_KVZAP, score=s_new,
                               tau=L["tau"], status=st)
                kvp.kvp_decode_attn(qs[i, li], L["cache"], t, out=out, workspace=ws_a, status=st)

    replay = _graph(lambda: (restore(), decode()))
    ms_restore = _time(restore, reps=3)
    ms = _time(replay, reps=3) - ms_restore
    torch.cuda.synchronize()
    assert st.item() == 0, kvp.status_string(st.item())
    pages = sum(int(((L["cache"].count + 15) // 16).sum().item()) for L in layers)
    kept = sum(int(L["cache"].count.sum().item()) for L in layers)
    step_bytes = pages * 16 * (2 * d * 2 + 4)
    return {
        "workload": "llama65b_mha: 8 layers x (64 heads MHA, head_dim 128, d_model 8192), batch 1, 131072 cached "
                    "tokens, KVzap-Linear, keep rate per (layer, head) ~Beta(2,5), 128-token window, 32 decode steps",
        "prefill_score_ms_8_layers": ms_score, "prefill_score_GB_s": score_bytes / (ms_score * 1e-3) / 1e9,
        "prefill_mask_compact_ms_8_layers": ms_mc,
        "kept_fraction": kept / (n_layers * H * (T + steps)),
        "decode_ms_per_step": ms / steps, "decode_tokens_per_s": B * steps / (ms * 1e-3),
        "attn_bytes_last_step_8_layers": step_bytes,
        "effective_GB_s_last_step_bytes": step_bytes / (ms / steps * 1e-3) / 1e9,
        "frac_of_hbm": step_bytes / (ms / steps * 1e-3) / 1e9 / peaks[0],
    }


def prune_sweep(kvp, dev, peaks, seed=0, calls=10, reps=5):
    """Decode attention over the Llama-3-8B-shaped cache (batch 16, 8,192 cached
    tokens, 32 q / 8 kv heads, head_dim 128) at several pruning levels: the
    threshold at each head's q-quantile score, 128-token window, q = 0 keeps
    everything. The kernel reads only surviving pages, so decode tokens/s should
    rise as the inverse of the kept fraction while the kernel stays HBM-bound;
    fixed per-call costs bend the curve at high pruning."""
    B, T, H, Hq, d, W = 16, 8192, 8, 32, 128, 128
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    K = _randn_bf16((B, T, H, d), g, dev)
    V = _randn_bf16((B, T, H, d), g, dev)
    q = _randn_bf16((B, Hq, d), g, dev)
    s = torch.randn((B, T, H), generator=g, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    mp = (T + 15) // 16
    cache = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp, device=dev)
    out = torch.empty(B, Hq, d, dtype=torch.float32, device=dev)
    ws_a = torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, Hq, H, d), dtype=torch.uint8, device=dev)
    ws_c = torch.empty(kvp.kvp_compact_workspace_bytes(B, H, T), dtype=torch.uint8, device=dev)
    points = []
    for prune_q in (0.0, 0.5, 0.75, 0.875, 0.9375, 0.96875):
        tau = (torch.full((B, H), -math.inf, device=dev) if prune_q == 0.0 else _tau_quantile(kvp, s, prune_q))
        expire, _, _ = kvp.kvp_mask(mode=kvp.KVP_MASK_KVZAP, batch=B, n_kv_heads=H, n_pos=T, now=T - 1,
                                    scores=s.view(B * T, H), tau=tau, window=W, want_bits=False)
        kvp.kvp_compact(K, V, expire, T - 1, 0, cache, status=st, workspace=ws_c)
        torch.cuda.synchronize()
        assert st.item() == 0, kvp.status_string(st.item())
        kept = int(cache.count.sum().item())
        pages = int(((cache.count + 15) // 16).sum().item())

        def calls_fn():
            for _ in range(calls):
                kvp.kvp_decode_attn(q, cache, T - 1, out=out, workspace=ws_a, status=st)

        replay = _graph(calls_fn)
        ms = _time(replay, reps=reps) / calls
        nbytes = pages * 16 * (2 * d * 2 + 4) + B * Hq * d * (2 + 4)
        points.append({"prune_q": prune_q, "kept_fraction": kept / (B * H * T), "surviving_pages": pages,
                       "decode_attn_us": ms * 1e3, "decode_tokens_per_s": B / (ms * 1e-3),
                       "GB_s": nbytes / (ms * 1e-3) / 1e9, "frac_of_hbm": nbytes / (ms * 1e-3) / 1e9 / peaks[0]})
    assert st.item() == 0, kvp.status_string(st.item())
    base = points[0]
    for p in points:
        p["speedup_vs_keep_all"] = p["decode_tokens_per_s"] / base["decode_tokens_per_s"]
        p["inverse_kept_ratio"] = base["kept_fraction"] / p["kept_fraction"]
    return {"workload": "prune_sweep: decode attention, batch 16, 8192 cached tokens, 32 q / 8 kv heads, "
                        "head_dim 128, threshold at each head's q-quantile score, 128-token window; "
                        "each point = a CUDA graph of 10 calls",
            "points": points}


def prune_sweep_long(kvp, dev, peaks, seed=0, calls=5, reps=3):
    """Decode attention over one layer of the 65B-shaped MHA stack (batch 1,
    131,072 cached tokens, 64 heads, head_dim 128: 4.3 GB of dense K/V) at
    pruning levels from 0 to 96.9 %, the threshold at each head's q-quantile
    score, 128-token window: with gigabytes of survivors the call's fixed
    cost is small, so decode tokens/s follow the inverse of the kept
    fraction much further than on the 16 x 8,192-token cache."""
    B, T, H, d, W = 1, 131072, 64, 128, 128
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    K = _randn_bf16((B, T, H, d), g, dev)
    V = _randn_bf16((B, T, H, d), g, dev)
    q = _randn_bf16((B, H, d), g, dev)
    s = torch.randn((B, T, H), generator=g, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    mp = (T + 15) // 16
    cache = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp, device=dev)
    out = torch.empty(B, H, d, dtype=torch.float32, device=dev)
    ws_a = torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, H, H, d), dtype=torch.uint8, device=dev)
    ws_c = torch.empty(kvp.kvp_compact_workspace_bytes(B, H, T), dtype=torch.uint8, device=dev)
    points = []
    for prune_q in (0.0, 0.5, 0.75, 0.875, 0.9375, 0.96875):
        tau = torch.full((B, H), -math.inf, device=dev) if prune_q == 0.0 else _tau_quantile(kvp, s, prune_q)
        kvp.kvp_compact_masked(K, V, T - 1, 0, cache, mode=kvp.KVP_MASK_KVZAP, scores=s.view(B * T, H), tau=tau,
                               window=W, status=st, workspace=ws_c)
        torch.cuda.synchronize()
        assert st.item() == 0, kvp.status_string(st.item())
        kept = int(cache.count.sum().item())
        pages = int(((cache.count + 15) // 16).sum().item())

        def calls_fn():
            for _ in range(calls):
                kvp.kvp_decode_attn(q, cache, T - 1, out=out, workspace=ws_a, status=st)

        ms = _time(_graph(calls_fn), reps=reps) / calls
        nbytes = pages * 16 * (2 * d * 2 + 4) + B * H * d * (2 + 4)
        points.append({"prune_q": prune_q, "kept_fraction": kept / (B * H * T), "surviving_pages": pages,
                       "decode_attn_us": ms * 1e3, "decode_tokens_per_s": B / (ms * 1e-3),
                       "GB_s": nbytes / (ms * 1e-3) / 1e9, "frac_of_hbm": nbytes / (ms * 1e-3) / 1e9 / peaks[0]})
    assert st.item() == 0, kvp.status_string(st.item())
    base = points[0]
    for p in points:
        p["speedup_vs_keep_all"] = p["decode_tokens_per_s"] / base["decode_tokens_per_s"]
        p["inverse_kept_ratio"] = base["kept_fraction"] / p["kept_fraction"]
    return {"workload": "prune_sweep_long: decode attention, one 65B-shaped MHA layer, batch 1, 131072 cached "
                        "tokens, 64 heads, head_dim 128, threshold at each head's q-quantile score, 128-token window; "
                        "each point = a CUDA graph of 5 calls",
            "points": points}


def threshold(kvp, dev, peaks, seed=0, calls=10, reps=5):
    """Per-(b, h) threshold selection on the device (kvp_threshold, four radix
    passes) at the score shapes of three layers: the tiny case, the Llama-3-8B
    layer (batch 16, 8,192 tokens, 8 kv heads, 75th percentile) and one
    Llama-65B MHA layer (1 x 131,072 tokens, 64 heads). Each result is checked
    against torch.kthvalue; torch's time is printed beside ours for context."""
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    points = []
    for name, B, T, H, q in (("tiny", 1, 512, 2, 0.5), ("llama3_8b_layer", 16, 8192, 8, 0.75),
                             ("llama65b_mha_layer", 1, 131072, 64, 0.6)):
        s = torch.randn((B, T, H), generator=g, device=dev)
        tau = torch.empty(B, H, dtype=torch.float32, device=dev)
        ws = torch.empty(kvp.kvp_threshold_workspace_bytes(B, H), dtype=torch.uint8, device=dev)
        kvp.kvp_threshold(s, q, out=tau, workspace=ws)
        kth = int(math.floor(q * (T - 1))) + 1
        ref = torch.kthvalue(s, kth, dim=1).values
        torch.cuda.synchronize()
        assert torch.equal(tau, ref), name

        def calls_fn():
            for _ in range(calls):
                kvp.kvp_threshold(s, q, out=tau, workspace=ws)

        replay = _graph(calls_fn)
        ms = _time(replay, reps=reps) / calls
        ms_torch = _time(lambda: torch.kthvalue(s, kth, dim=1), reps=reps)
        nbytes = B * T * H * 4
        points.append({"shape": name, "batch": B, "n_pos": T, "n_kv_heads": H, "q": q, "threshold_us": ms * 1e3,
                       "torch_kthvalue_us_eager": ms_torch * 1e3, "score_bytes": nbytes,
                       "GB_s_one_read": nbytes / (ms * 1e-3) / 1e9,
                       "frac_of_hbm_one_read": nbytes / (ms * 1e-3) / 1e9 / peaks[0]})
    return {"workload": "threshold: per-(b, h) rank-floor(q(T-1)) score chosen on the device; "
                        "each point = a CUDA graph of 10 calls (memset + 4 radix passes each)",
            "points": points}


def quant_tier(kvp, dev, peaks, seed=0, calls=10, reps=5):
    """Quantize instead of drop on the Llama-3-8B-shaped layer (batch 16,
    8,192 cached tokens, 32 q / 8 kv heads, head_dim 128): tau at each head's
    75th-percentile score (bf16 tier: those entries plus the 128-token window),
    and the entries below tau but at or above tau_q in the fp8 tier, for
    tau_q at the 50th and 25th percentiles and at -inf (every entry kept in
    some form). Times the fp8-tier compaction and the two-tier attention (CUDA
    graphs of 10 calls) next to the one-tier attention over the bf16 tier
    alone; bytes are the pages each call reads."""
    pts = _quant_tier(kvp, dev, peaks, 16, 8192, 8, 32, 128, seed, calls, reps)
    return {"workload": "quant_tier: Llama-3-8B layer (batch 16 x 8192 tokens, 32 q / 8 kv heads, head_dim 128), "
                        "tau at the 75th percentile, fp8 tier for tau_q <= s < tau; CUDA graphs of 10 calls",
            "points": pts}


def quant_tier_mha(kvp, dev, peaks, seed=0, calls=5, reps=3):
    """The same tiers on one layer of the 65B-shaped MHA stack (batch 1,
    131,072 cached tokens, 64 heads, one query head per kv head, head_dim
    128): tau at the 75th percentile, tau_q at the 50th / 25th / -inf."""
    pts = _quant_tier(kvp, dev, peaks, 1, 131072, 64, 64, 128, seed, calls, reps)
    return {"workload": "quant_tier_mha: one 65B-shaped MHA layer (batch 1 x 131072 tokens, 64 heads, head_dim 128), "
                        "tau at the 75th percentile, fp8 tier for tau_q <= s < tau; CUDA graphs of 5 calls",
            "points": pts}


def _quant_tier(kvp, dev, peaks, B, T, H, Hq, d, seed, calls, reps):
    W = 128
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    K = _randn_bf16((B, T, H, d), g, dev)
    V = _randn_bf16((B, T, H, d), g, dev)
    q = _randn_bf16((B, Hq, d), g, dev)
    s = torch.randn((B, T, H), generator=g, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    mp = (T + 15) // 16
    ca = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp, device=dev)
    cq = kvp.QuantPagedKV.allocate(B, H, d, B * H * mp, mp, device=dev)
    out = torch.empty(B, Hq, d, dtype=torch.float32, device=dev)
    ws_a = torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, Hq, H, d), dtype=torch.uint8, device=dev)
    ws_c = torch.empty(kvp.kvp_compact_workspace_bytes(B, H, T), dtype=torch.uint8, device=dev)
    tau = _tau_quantile(kvp, s, 0.75)
    kvp.kvp_compact_masked(K, V, T - 1, 0, ca, mode=kvp.KVP_MASK_KVZAP, scores=s.view(B * T, H), tau=tau, window=W,
                           status=st, workspace=ws_c)
    torch.cuda.synchronize()
    pages_a = int(((ca.count + 15) // 16).sum().item())
    bytes_a = pages_a * 16 * (2 * d * 2 + 4) + B * Hq * d * (2 + 4)

    def one_tier():
        for _ in range(calls):
            kvp.kvp_decode_attn(q, ca, T - 1, out=out, workspace=ws_a, status=st)

    ms_one = _time(_graph(one_tier), reps=reps) / calls
    points = [{"tau_q": "tau (no fp8 tier)", "bf16_kept_fraction": int(ca.count.sum()) / (B * H * T),
               "fp8_fraction": 0.0, "attention_us": ms_one * 1e3, "attention_bytes": bytes_a,
               "frac_of_hbm": bytes_a / (ms_one * 1e-3) / 1e9 / peaks[0]}]
    for name, tq in (("50th percentile", _tau_quantile(kvp, s, 0.5)), ("25th percentile", _tau_quantile(kvp, s, 0.25)),
                     ("-inf", torch.full((B, H), -math.inf, device=dev))):
        def comp():
            kvp.kvp_compact_quant(K, V, s, tau, tq, cq, window=W, status=st, workspace=ws_c)

        ms_comp = _time(_graph(comp), reps=reps)
        torch.cuda.synchronize()
        assert st.item() == 0, kvp.status_string(st.item())
        nq = int(cq.count.sum().item())
        pages_q = int(((cq.count + 15) // 16).sum().item())
        bytes_q = pages_q * (2 * 16 * d + 3 * 16 * 4)

        def two_tier():
            for _ in range(calls):
                kvp.kvp_decode_attn_two_tier(q, ca, cq, T - 1, out=out, workspace=ws_a, status=st)

        ms_two = _time(_graph(two_tier), reps=reps) / calls
        assert st.item() == 0, kvp.status_string(st.item())
        nbytes = bytes_a + bytes_q
        comp_bytes = nq * 2 * d * 2 + nq * 2 * d + pages_q * 3 * 16 * 4 + B * T * H * 4
        points.append({"tau_q": name, "bf16_kept_fraction": int(ca.count.sum()) / (B * H * T),
                       "fp8_fraction": nq / (B * H * T), "fp8_pages": pages_q,
                       "compact_quant_us": ms_comp * 1e3,
                       "compact_quant_frac_of_hbm": comp_bytes / (ms_comp * 1e-3) / 1e9 / peaks[0],
                       "attention_us": ms_two * 1e3, "attention_bytes": nbytes,
                       "frac_of_hbm": nbytes / (ms_two * 1e-3) / 1e9 / peaks[0],
                       "decode_tokens_per_s": B / (ms_two * 1e-3)})
    return points


def quant_decode(kvp, dev, peaks, seed=0, steps=64, reps=3):
    """A decode loop over both tiers on the Llama-3-8B-shaped layer (batch
    16, 8,192-token prompt, 32 q / 8 kv heads, head_dim 128): tau at each
    head's 75th-percentile prompt score, tau_q at the 25th, 128-token window.
    Each step appends the new token to the bf16 tier (kvp_append) and, when
    its score is in [tau_q, tau), to the fp8 tier (kvp_append_quant), then runs
    the two-tier attention; the 64 steps are one CUDA graph. The one-tier loop
    (the same steps without the fp8 tier) is timed beside it."""
    B, T, H, Hq, d, W = 16, 8192, 8, 32, 128, 128
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    K = _randn_bf16((B, T + steps, H, d), g, dev)
    V = _randn_bf16((B, T + steps, H, d), g, dev)
    q = _randn_bf16((steps, B, Hq, d), g, dev)
    s = torch.randn((B, T + steps, H), generator=g, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    reserve = steps
    mp = (T + reserve + 15) // 16
    ws_c = torch.empty(kvp.kvp_compact_workspace_bytes(B, H, T), dtype=torch.uint8, device=dev)
    ws_a = torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, Hq, H, d), dtype=torch.uint8, device=dev)
    out = torch.empty(B, Hq, d, dtype=torch.float32, device=dev)
    sp = s[:, :T].contiguous()
    tau = _tau_quantile(kvp, sp, 0.75)
    tau_q = _tau_quantile(kvp, sp, 0.25)
    Kp, Vp = K[:, :T], V[:, :T]
    k_new = [K[:, T + i].contiguous() for i in range(steps)]
    v_new = [V[:, T + i].contiguous() for i in range(steps)]
    s_new = [s[:, T + i].contiguous() for i in range(steps)]
    res = {}
    for tiers in (1, 2):
        ca = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp, device=dev)
        cq = kvp.QuantPagedKV.allocate(B, H, d, B * H * mp, mp, device=dev)

        def prefill():
            kvp.kvp_compact_masked(Kp, Vp, T - 1, reserve, ca, mode=kvp.KVP_MASK_KVZAP, scores=sp, tau=tau, window=W,
                                   status=st, workspace=ws_c)
            if tiers == 2:
                kvp.kvp_compact_quant(Kp, Vp, sp, tau, tau_q, cq, reserve=reserve, window=W, status=st,
                                      workspace=ws_c)

        def loop():
            for i in range(steps):
                t = T + i
                kvp.kvp_append(ca, k_new[i], v_new[i], t, mode=kvp.KVP_MASK_KVZAP, score=s_new[i], tau=tau,
                               window=W, status=st)
                if tiers == 2:
                    kvp.kvp_append_quant(cq, k_new[i], v_new[i], t, score=s_new[i], tau=tau, tau_q=tau_q, window=W,
                                         status=st)
                    kvp.kvp_decode_attn_two_tier(q[i], ca, cq, t, out=out, workspace=ws_a, status=st)
                else:
                    kvp.kvp_decode_attn(q[i], ca, t, out=out, workspace=ws_a, status=st)

        prefill()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            loop()
        best = 1e30
        for _ in range(reps):
            prefill()               # the loop appends: start every replay from the prompt's caches
            torch.cuda.synchronize()
            best = min(best, _time(gr.replay))
        assert st.item() == 0, kvp.status_string(st.item())
        res[tiers] = {"ms_per_step": best / steps, "decode_tokens_per_s": B / (best / steps * 1e-3),
                      "bf16_slots": int(ca.count.sum().item()), "fp8_slots": int(cq.count.sum().item())}
    return {"workload": "quant_decode: Llama-3-8B layer, batch 16, 8192-token prompt + 64 decode steps, "
                        "tau 75th / tau_q 25th percentile, window 128; each step = append (both tiers) + attention; "
                        "the 64 steps are one CUDA graph",
            "one_tier": res[1], "two_tier": res[2]}


def gqa_sweep(kvp, dev, peaks, seed=0, calls=10, reps=5):
    """Decode attention on the Llama-3-8B-shaped cache (batch 16, 8,192 cached
    tokens, 8 kv heads, head_dim 128) with 1, 2, 4 and 8 query heads per kv
    head, kept whole and 75 % pruned: the call time of the kernel each group
    size is dispatched to (CUDA graphs of 10 calls)."""
    B, T, H, d = 16, 8192, 8, 128
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    K = _randn_bf16((B, T, H, d), g, dev)
    V = _randn_bf16((B, T, H, d), g, dev)
    s = torch.randn((B, T, H), generator=g, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    mp = (T + 15) // 16
    cache = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp, device=dev)
    points = []
    for prune_q in (0.0, 0.75):
        tau = torch.full((B, H), -math.inf, device=dev) if prune_q == 0.0 else _tau_quantile(kvp, s, prune_q)
        kvp.kvp_compact_masked(K, V, T - 1, 0, cache, mode=kvp.KVP_MASK_KVZAP, scores=s.view(B * T, H), tau=tau,
                               status=st)
        torch.cuda.synchronize()
        pages = int(((cache.count + 15) // 16).sum().item())
        for G in (1, 2, 4, 8):
            Hq = H * G
            q = _randn_bf16((B, Hq, d), g, dev)
            out = torch.empty(B, Hq, d, dtype=torch.float32, device=dev)
            ws = torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, Hq, H, d), dtype=torch.uint8, device=dev)

            def calls_fn():
                for _ in range(calls):
                    kvp.kvp_decode_attn(q, cache, T - 1, out=out, workspace=ws, status=st)

            ms = _time(_graph(calls_fn), reps=reps) / calls
            nbytes = pages * 16 * (2 * d * 2 + 4) + B * Hq * d * (2 + 4)
            points.append({"prune_q": prune_q, "group": G, "surviving_pages": pages, "decode_attn_us": ms * 1e3,
                           "GB_s": nbytes / (ms * 1e-3) / 1e9, "frac_of_hbm": nbytes / (ms * 1e-3) / 1e9 / peaks[0]})
    assert st.item() == 0, kvp.status_string(st.item())
    return {"workload": "gqa_sweep: decode attention, batch 16, 8192 cached tokens, 8 kv heads, head_dim 128, "
                        "1/2/4/8 query heads per kv head, keep-all and 75 % pruned; CUDA graphs of 10 calls",
            "points": points}


def mla_sweep(kvp, dev, peaks, seed=0, calls=10, reps=5):
    """MLA latent cache (DeepSeek-V3-shaped attention: latent rows of 512 + 64
    values, batch 16, 8,192 cached tokens): latent compaction with the mask
    fused in, then absorbed decode attention with 16, 32, 64 and 128 query
    heads, kept whole and 75 % pruned (CUDA graphs of 10 calls). Bytes count
    the surviving pages (16 rows of 1,152 bytes + 64 bytes of expire values)
    and the query and output rows; flops count 2 x 16 x (576 + 512) per page
    and head."""
    B, T, row, dc = 16, 8192, kvp.LATENT_ROW, kvp.KVP_MLA_LATENT_DIM
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    lat = _randn_bf16((B, T, row), g, dev)
    s = torch.randn((B, T, 1), generator=g, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    mp = (T + 15) // 16
    cache = kvp.LatentPagedKV.allocate(B, B * mp, mp, device=dev)
    ws_c = torch.empty(kvp.kvp_compact_workspace_bytes(B, 1, T), dtype=torch.uint8, device=dev)
    points = []
    for prune_q in (0.0, 0.75):
        tau = torch.full((B, 1), -math.inf, device=dev) if prune_q == 0.0 else _tau_quantile(kvp, s, prune_q)

        def compact_fn():
            for _ in range(calls):
                kvp.kvp_compact_latent(lat, T - 1, 0, cache, mode=kvp.KVP_MASK_KVZAP, scores=s.view(B, T),
                                       tau=tau.view(B), workspace=ws_c, status=st)

        ms_c = _time(_graph(compact_fn), reps=reps) / calls
        torch.cuda.synchronize()
        pages = int(((cache.count + 15) // 16).sum().item())
        kept = int(cache.count.sum().item())
        c_bytes = B * T * 4 + 2 * kept * row * 2 + pages * 16 * 4
        for Hq in (16, 32, 64, 128):
            q = _randn_bf16((B, Hq, row), g, dev)
            out = torch.empty(B, Hq, dc, dtype=torch.float32, device=dev)
            ws = torch.zeros(kvp.kvp_decode_attn_mla_workspace_bytes(B, Hq, 0), dtype=torch.uint8, device=dev)

            def calls_fn():
                for _ in range(calls):
                    kvp.kvp_decode_attn_mla(q, cache, T - 1, out=out, workspace=ws, status=st)

            ms = _time(_graph(calls_fn), reps=reps) / calls
            nbytes = pages * (16 * row * 2 + 64) + B * Hq * (row * 2 + dc * 4)
            flops = 2.0 * 16 * pages * Hq * (row + dc)
            points.append({"prune_q": prune_q, "q_heads": Hq, "surviving_pages": pages,
                           "compact_latent_us": ms_c * 1e3,
                           "compact_frac_of_hbm": c_bytes / (ms_c * 1e-3) / 1e9 / peaks[0],
                           "decode_attn_mla_us": ms * 1e3, "GB_s": nbytes / (ms * 1e-3) / 1e9,
                           "frac_of_hbm": nbytes / (ms * 1e-3) / 1e9 / peaks[0],
                           "TFLOP_s": flops / (ms * 1e-3) / 1e12,
                           "frac_of_bf16_peak": flops / (ms * 1e-3) / 1e12 / peaks[1]})
    assert st.item() == 0, kvp.status_string(st.item())
    return {"workload": "mla_sweep: MLA latent cache, batch 16, 8192 cached tokens, rows of 512 + 64, latent "
                        "compaction and absorbed decode attention at 16/32/64/128 query heads, keep-all and 75 % "
                        "pruned; CUDA graphs of 10 calls",
            "points": points}


def mla_dms_decode(kvp, dev, peaks, seed=0, steps=256):
    """The DMS decode loop on an MLA latent cache (rows of 512 + 64 values):
    batch 64, 4,096-token prompt, then per step the new latent row is
    appended and absorbed attention runs over the present rows; every 64
    steps the cache is re-compacted. Run with 16 and with 128 query heads.
    Bytes count the surviving pages read by the attention steps."""
    B, T0, delay, W, every, reserve = 64, 4096, 256, 128, 64, 64
    row, dc = kvp.LATENT_ROW, kvp.KVP_MLA_LATENT_DIM
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    lat = _randn_bf16((B, T0, row), g, dev)
    pos = torch.arange(T0, device=dev, dtype=torch.int32)
    f0 = torch.where(torch.rand((B, T0), generator=g, device=dev) < 7 / 8, pos, -1).to(torch.int32)
    ls = _randn_bf16((steps, B, row), g, dev)
    tpos = (T0 + torch.arange(steps, device=dev, dtype=torch.int32)).view(steps, 1)
    fs = torch.where(torch.rand((steps, B), generator=g, device=dev) < 7 / 8, tpos, -1).to(torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    now0 = T0 - 1
    mp = (T0 + steps + reserve + 15) // 16
    pools = [kvp.LatentPagedKV.allocate(B, B * mp, mp, device=dev) for _ in range(2)]
    ws_c = torch.empty(kvp.kvp_compact_workspace_bytes(B, 1, T0), dtype=torch.uint8, device=dev)
    ws_p = torch.empty(kvp.kvp_compact_paged_workspace_bytes(B, 1, mp), dtype=torch.uint8, device=dev)
    points = []
    for Hq in (16, 128):
        qs = _randn_bf16((steps, B, Hq, row), g, dev)
        out = torch.empty(steps, B, Hq, dc, dtype=torch.float32, device=dev)
        ws_a = torch.zeros(kvp.kvp_decode_attn_mla_workspace_bytes(B, Hq, 0), dtype=torch.uint8, device=dev)
        pages_read = torch.zeros((), dtype=torch.int64, device=dev)

        def prefill():
            kvp.kvp_compact_latent(lat, now0, reserve, pools[0], mode=kvp.KVP_MASK_DMS, flag_step=f0, delay=delay,
                                   window=W, workspace=ws_c, status=st)

        def decode(count_pages=False):
            cur = 0
            for i in range(steps):
                t = T0 + i
                if i > 0 and i % every == 0:
                    kvp.kvp_compact_latent_paged(pools[cur], t, reserve, pools[1 - cur], workspace=ws_p, status=st)
                    cur = 1 - cur
                c = pools[cur]
                kvp.kvp_append_latent(c, ls[i], t, mode=kvp.KVP_MASK_DMS, flag_step=fs[i], delay=delay, window=W,
                                      status=st)
                kvp.kvp_decode_attn_mla(qs[i], c, t, out=out[i], workspace=ws_a, status=st)
                if count_pages:
                    pages_read.add_(((c.count + 15) // 16).sum())

        prefill()
        decode(count_pages=True)  # eager pass: algorithmic bytes of the attention steps
        torch.cuda.synchronize()
        assert st.item() == 0, kvp.status_string(st.item())
        total_pages = int(pages_read.item())
        prefill()
        replay = _graph(decode)
        ms_pref = _time(prefill, reps=3)
        ms = _time(lambda: (prefill(), replay()), reps=3) - ms_pref
        torch.cuda.synchronize()
        assert st.item() == 0, kvp.status_string(st.item())
        attn_bytes = total_pages * (16 * row * 2 + 64)
        points.append({"q_heads": Hq, "decode_ms_per_step": ms / steps, "decode_tokens_per_s": B * steps / (ms * 1e-3),
                       "attn_pages_read_total": total_pages, "attn_bytes_total": attn_bytes,
                       "frac_of_hbm": attn_bytes / (ms * 1e-3) / 1e9 / peaks[0],
                       "dense_latent_bytes_last_step": B * (T0 + steps) * row * 2})
    return {"workload": f"mla_dms_decode: MLA latent cache, batch 64, 4096-token prompt + {steps} steps, rows of "
                        "512 + 64, evict ~Bernoulli(7/8), delay 256, window 128, re-compaction every 64 steps; 16 and "
                        "128 query heads",
            "points": points}


def seq_split(kvp, dev, peaks, seed=0, calls=5, reps=3):
    """A long sequence attended in two parts and merged on the device (the
    building blocks of a sequence split): one 65B-shaped MHA layer (batch 1,
    131,072 cached tokens, 64 heads, head_dim 128), tau at each head's 75th
    percentile; the cache of the whole sequence against two caches of its
    halves, each attended with its log-sum-exp (kvp_decode_attn_lse) and the
    rows merged (kvp_attn_merge); CUDA graphs of 5 calls."""
    B, T, H, d, W = 1, 131072, 64, 128, 128
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    K = _randn_bf16((B, T, H, d), g, dev)
    V = _randn_bf16((B, T, H, d), g, dev)
    q = _randn_bf16((B, H, d), g, dev)
    s = torch.randn((B, T, H), generator=g, device=dev)
    tau = _tau_quantile(kvp, s, 0.75)
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    # a part's positions count from its first token: the second half is compacted and attended at its own
    # step T / 2 - 1, so that its last 128 tokens are the recent window the whole sequence keeps
    def cache_of(lo, hi, now):
        n = hi - lo
        mp = (n + 15) // 16
        c = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp, device=dev)
        ws = torch.empty(kvp.kvp_compact_workspace_bytes(B, H, n), dtype=torch.uint8, device=dev)
        kvp.kvp_compact_masked(K[:, lo:hi], V[:, lo:hi], now, 0, c, mode=kvp.KVP_MASK_KVZAP,
                               scores=s[:, lo:hi].contiguous().view(B * n, H), tau=tau, window=W, status=st,
                               workspace=ws)
        return c

    nows = [T - 1, T // 2 - 1]
    whole = cache_of(0, T, T - 1)
    parts = [cache_of(0, T // 2, nows[0]), cache_of(T // 2, T, nows[1])]
    torch.cuda.synchronize()
    assert st.item() == 0, kvp.status_string(st.item())
    ws_a = [torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, H, H, d), dtype=torch.uint8, device=dev)
            for _ in range(3)]
    out = torch.empty(B, H, d, dtype=torch.float32, device=dev)
    outs = torch.empty(2, B, H, d, dtype=torch.float32, device=dev)
    lses = torch.empty(2, B, H, dtype=torch.float32, device=dev)
    lse = torch.empty(B, H, dtype=torch.float32, device=dev)

    def one():
        for _ in range(calls):
            kvp.kvp_decode_attn(q, whole, T - 1, out=out, workspace=ws_a[0], status=st)

    def split():
        for _ in range(calls):
            for i in range(2):
                kvp.kvp_decode_attn_lse(q, parts[i], nows[i], out=outs[i], lse=lses[i], workspace=ws_a[1 + i],
                                        status=st)
            kvp.kvp_attn_merge(outs, lses, out=out, lse=lse)

    ms_one = _time(_graph(one), reps=reps) / calls
    ms_split = _time(_graph(split), reps=reps) / calls
    torch.cuda.synchronize()
    assert st.item() == 0, kvp.status_string(st.item())
    pages = [int(((c.count + 15) // 16).sum().item()) for c in (whole, *parts)]
    page_bytes = 16 * (2 * d * 2 + 4)
    return {"workload": "seq_split: one 65B-shaped MHA layer (batch 1 x 131072 tokens, 64 heads, head_dim 128), tau at "
                        "the 75th percentile; whole cache against two half caches attended with their log-sum-exps "
                        "and merged; CUDA graphs of 5 calls",
            "points": [{"form": "whole", "pages": pages[0], "attention_us": ms_one * 1e3,
                        "frac_of_hbm": pages[0] * page_bytes / (ms_one * 1e-3) / 1e9 / peaks[0]},
                       {"form": "two halves + merge", "pages": pages[1] + pages[2], "attention_us": ms_split * 1e3,
                        "frac_of_hbm": (pages[1] + pages[2]) * page_bytes / (ms_split * 1e-3) / 1e9 / peaks[0]}]}


RUNNERS = {"mlp_prefill": mlp_prefill, "dms_decode": dms_decode, "llama65b_mha": llama65b_mha,
           "prune_sweep": prune_sweep, "prune_sweep_long": prune_sweep_long, "threshold": threshold,
           "quant_tier": quant_tier, "quant_tier_mha": quant_tier_mha, "quant_decode": quant_decode, "gqa_sweep": gqa_sweep, "mla_sweep": mla_sweep,
           "mla_dms_decode": mla_dms_decode, "seq_split": seq_split}


def run(name, kvp, dev, peaks):
    res = RUNNERS[name](kvp, dev, peaks)
    res["name"] = name
    print(json.dumps(res), flush=True)
    return res
