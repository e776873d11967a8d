"""The three large configurations at their stated sizes, through the library
as the measurement workloads run them, against the oracle on the same seeded
inputs (drawn with the fast Philox generator of kvp_synth: each holds
hundreds of millions of values).

* KVzap-MLP prefill scoring (KVzap summary, "KVzap의 구조"): d_model 4096 ->
  1024 (GELU) -> 8 over 4 x 32,768 tokens, every score compared; the
  persistent scorer then runs about 27 tiles per CTA, through its
  accumulator double buffer and the 64-k-block ring. A 40,000-row case with
  and without biases is compared as well.
* Llama-65B-shaped MHA layer (KVzap summary, "실제 적용"): 1 x 131,072 tokens,
  64 heads, d_model 8192, per-head keep rates ~ Beta(2, 5); scores, mask
  (near-threshold entries excluded and counted), fused mask + compaction and
  compaction bit-exact, attention at the prompt's last token and through 32
  decode steps (append, attention).
* DMS delayed eviction, Qwen-3-8B-shaped (DMS article, "지연 삭제 (Delayed
  Eviction)"): batch 64, 32 / 8 heads, 4,096-token prompt, evict bit ~
  Bernoulli(7/8), delay 256, recompaction every 64 steps; 192 decode steps
  with the caches bit-exact after every recompaction and at the end, and
  the attention compared at every step.

* MLA latent cache, DeepSeek-V3-shaped attention (DMS article, "주요 요점"
  and "앞으로의 전망"): batch 16 x 8,192 tokens of 512 + 64-value rows, 128
  query heads (the tensor-core kernel), kept whole and at each element's
  75th-percentile score; four batch elements compared with the oracle in full.

Bars: scores within 1e-3 relative, masks / pools / tables bit-exact,
attention within max-abs 2e-2, mean-abs 2e-3 and 1e-2 relative per head."""
import math

import numpy as np
import pytest
import torch

import kvp_synth as syn
import oracle as orc
from helpers import (check_attention, check_scores, compare_paged, dev_bf16, dev_f32, dev_i32,
                     oracle_linear_scores, oracle_mlp_scores, status_word)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


# --------------------------------------------------------------------------- KVzap-MLP scorer

@pytest.mark.parametrize("n_tok,bias", [(4 * 32768, False), (40000, True), (40000, False)])
def test_mlp_scorer_prefill_size(kvp, n_tok, bias):
    D, HID, H = 4096, 1024, 8
    x = syn.fast_normal_bf16(3, syn.S_X, (n_tok, D))
    w1 = syn.fast_normal_bf16(3, syn.S_W1, (HID, D), std=1.0 / math.sqrt(D))
    w2 = syn.fast_normal_bf16(3, syn.S_W2, (H, HID), std=1.0 / math.sqrt(HID))
    b1 = syn.normal_f32(3, 78, (HID,), std=0.1) if bias else None
    b2 = syn.normal_f32(3, 79, (H,)) if bias else None
    st = status_word()
    xd = dev_bf16(x)
    s = kvp.kvp_score(xd, dev_bf16(w1), dev_f32(b1) if bias else None, dev_bf16(w2),
                      dev_f32(b2) if bias else None, scorer=kvp.KVP_SCORER_MLP, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    del xd
    # every CTA of the persistent grid runs several 128-row x 256-column tiles
    tiles = ((n_tok + 127) // 128) * (HID // 256)
    assert tiles >= 8 * torch.cuda.get_device_properties(0).multi_processor_count
    ref, scale = oracle_mlp_scores(x, w1, w2, b1, b2)
    worst = check_scores(s.cpu().numpy(), ref, scale)
    print(f"MLP scorer, {n_tok} rows: worst error / bound = {worst:.3g}")


# --------------------------------------------------------------------------- Llama-65B-shaped MHA layer

def test_llama65b_mha_layer_full_size(kvp):
    cfg = syn.WORKLOADS["llama65b_mha"]
    B, T, D, H, d = cfg["batch"], cfg["n_pos"], cfg["d_model"], cfg["n_kv_heads"], cfg["head_dim"]
    Hq, steps, reserve = cfg["n_q_heads"], cfg["steps"], cfg["reserve"]
    now = T - 1
    x = syn.fast_normal_bf16(0, syn.S_X, (B * T, D))
    w = syn.normal_f32(0, syn.S_W, (H, D), std=1.0 / math.sqrt(D))
    st = status_word()

    # ---- scores: the layer's weight split once, the prompt scored with it (as the workload does)
    ws = kvp.kvp_score_split_weight(dev_f32(w))
    xd = dev_bf16(x)
    s_gpu = kvp.kvp_score(xd, ws, scorer=kvp.KVP_SCORER_LINEAR_SPLIT, n_kv_heads=H, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    del xd
    s_ref, scale = oracle_linear_scores(x, w)
    del x
    check_scores(s_gpu.cpu().numpy(), s_ref, scale)
    del scale

    # ---- per-head keep rates r ~ Beta(2, 5), the threshold at quantile 1 - r of the head's scores
    r = syn.beta_2_5(0, syn.S_KEEPRATE, (H,))
    s3 = s_ref.reshape(B, T, H)
    tau = orc.threshold_at_quantile(s3, 1.0 - r)
    exp_g, _, cnt_g = kvp.kvp_mask(mode=kvp.KVP_MASK_KVZAP, batch=B, n_kv_heads=H, n_pos=T, now=now,
                                   scores=s_gpu, tau=dev_f32(tau), want_bits=False)
    torch.cuda.synchronize()
    exp_r, keep_r, _, cnt_r = orc.mask_kvzap(s3, tau, now)
    near = (np.abs(s3 - tau[:, None, :]) <= 1e-3).transpose(0, 2, 1)
    print(f"near-threshold entries excluded from the mask comparison: {int(near.sum())} of {near.size}")
    np.testing.assert_array_equal(exp_g.cpu().numpy()[~near], exp_r[~near])
    kept = keep_r.mean(axis=(0, 2))
    # heterogeneous survivor lengths: each head keeps about its own rate (plus the window)
    assert np.all(np.abs(kept - (r + 128.0 / T)) < 2e-3), (kept, r)
    del exp_g, s_gpu

    # ---- compaction of the oracle's keep set, and the fused mask + compaction on fp32 scores
    k = syn.fast_normal_bf16(0, syn.S_K, (B, T, H, d))
    v = syn.fast_normal_bf16(0, syn.S_V, (B, T, H, d))
    mp = (T + steps + reserve + 15) // 16
    need = int(((cnt_r + reserve + 15) // 16).sum())
    ref_c = orc.compact_dense(k, v, exp_r, now, reserve, need, mp)
    kd, vd = dev_bf16(k), dev_bf16(v)
    c = kvp.PagedKV.allocate(B, H, d, need, mp)
    kvp.kvp_compact(kd, vd, dev_i32(exp_r), now, reserve, c, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    compare_paged(c, ref_c, what="compact")
    s32 = s3.astype(np.float32)
    exp32 = orc.mask_kvzap(s32, tau, now)[0]
    ref_f = orc.compact_dense(k, v, exp32, now, reserve, int(((orc.mask(exp32, now)[2] + reserve + 15) // 16).sum()),
                              mp)
    cf = kvp.PagedKV.allocate(B, H, d, ref_f.k_pool.shape[0], mp)
    kvp.kvp_compact_masked(kd, vd, now, reserve, cf, mode=kvp.KVP_MASK_KVZAP, scores=dev_f32(s32.reshape(B * T, H)),
                           tau=dev_f32(tau), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    compare_paged(cf, ref_f, what="fused mask + compaction")
    del kd, vd, cf, ref_f, k, v, s3, s32, s_ref

    # ---- attention at the prompt's last token, then 32 decode steps: the new token scored, appended
    # under the same threshold, attention over the survivors. Both sides take the keep decision of a new
    # token on the same fp32 score (the oracle's); the device scorer's output for it is compared separately.
    q0 = syn.normal_bf16(0, syn.S_Q, (B, Hq, d))
    o = kvp.kvp_decode_attn(dev_bf16(q0), c, now, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    check_attention(o.cpu().numpy(), orc.decode_attention(q0, ref_c, now))
    ws_a = torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, Hq, H, d), dtype=torch.uint8, device="cuda")
    for i in range(steps):
        t = T + i
        xn = syn.normal_bf16(0, syn.step_stream(i, 1), (B, D))
        kn = syn.normal_bf16(0, syn.step_stream(i, 2), (B, H, d))
        vn = syn.normal_bf16(0, syn.step_stream(i, 3), (B, H, d))
        qn = syn.normal_bf16(0, syn.step_stream(i, 4), (B, Hq, d))
        sn_gpu = kvp.kvp_score(dev_bf16(xn), ws, scorer=kvp.KVP_SCORER_LINEAR_SPLIT, n_kv_heads=H, status=st)
        sn_ref, sn_scale = oracle_linear_scores(xn, w)
        sn32 = sn_ref.astype(np.float32)
        kvp.kvp_append(c, dev_bf16(kn), dev_bf16(vn), t, mode=kvp.KVP_MASK_KVZAP, score=dev_f32(sn32),
                       tau=dev_f32(tau), status=st)
        orc.append(ref_c, kn, vn, t, orc.expire_kvzap(sn32, tau, t))
        o = kvp.kvp_decode_attn(dev_bf16(qn), c, t, workspace=ws_a, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        check_scores(sn_gpu.cpu().numpy(), sn_ref, sn_scale)
        if i in (0, 1, steps // 2, steps - 1):   # the oracle's attention over 64 long heads takes seconds
            check_attention(o.cpu().numpy(), orc.decode_attention(qn, ref_c, t))
    compare_paged(c, ref_c, what="after 32 decode steps")


# --------------------------------------------------------------------------- DMS delayed-eviction loop

def test_dms_decode_loop_qwen3_8b_shape(kvp):
    cfg = syn.WORKLOADS["dms_decode"]
    B, T0, H, Hq, d = cfg["batch"], cfg["n_pos"], cfg["n_kv_heads"], cfg["n_q_heads"], cfg["head_dim"]
    delay, every, reserve, W = cfg["delay"], cfg["recompact_every"], cfg["reserve"], 128
    steps = 3 * every
    p_evict = cfg["evict_p"]
    now0 = T0 - 1
    k = syn.fast_normal_bf16(1, syn.S_K, (B, T0, H, d))
    v = syn.fast_normal_bf16(1, syn.S_V, (B, T0, H, d))
    f0 = np.where(syn.fast_uniform(1, syn.S_FLAG, (B, H, T0)) < p_evict, np.arange(T0)[None, None, :], -1)
    st = status_word()

    # ---- the prompt: DMS expire values, compaction
    exp_g, _, _ = kvp.kvp_mask(mode=kvp.KVP_MASK_DMS, batch=B, n_kv_heads=H, n_pos=T0, now=now0,
                               flag_step=dev_i32(f0), delay=delay, window=W, want_bits=False)
    exp_r = orc.mask_dms(f0, now0, delay, W)[0]
    torch.cuda.synchronize()
    np.testing.assert_array_equal(exp_g.cpu().numpy(), exp_r)
    mp = (T0 + steps + reserve + 15) // 16
    cap = B * H * mp
    ref = orc.compact_dense(k, v, exp_r, now0, reserve, cap, mp)
    pools = [kvp.PagedKV.allocate(B, H, d, cap, mp) for _ in range(2)]
    kvp.kvp_compact(dev_bf16(k), dev_bf16(v), exp_g, now0, reserve, pools[0], status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    compare_paged(pools[0], ref, what="prompt")
    del k, v, exp_g

    ws_a = torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, Hq, H, d), dtype=torch.uint8, device="cuda")
    ws_p = torch.empty(kvp.kvp_compact_paged_workspace_bytes(B, H, mp), dtype=torch.uint8, device="cuda")
    cur = 0
    recompactions = 0
    for i in range(steps):
        t = T0 + i
        if i > 0 and i % every == 0:
            kvp.kvp_compact_paged(pools[cur], t, reserve, pools[1 - cur], status=st, workspace=ws_p)
            cur = 1 - cur
            ref = orc.compact_paged(ref, t, reserve, cap, mp)
            torch.cuda.synchronize()
            assert st.item() == 0
            compare_paged(pools[cur], ref, what=f"recompaction at step {t}")
            recompactions += 1
        kn = syn.fast_normal_bf16(1, syn.step_stream(i, 2), (B, H, d))
        vn = syn.fast_normal_bf16(1, syn.step_stream(i, 3), (B, H, d))
        qn = syn.fast_normal_bf16(1, syn.step_stream(i, 4), (B, Hq, d))
        fn = np.where(syn.fast_uniform(1, syn.step_stream(i, 5), (B, H)) < p_evict, t, -1)
        kvp.kvp_append(pools[cur], dev_bf16(kn), dev_bf16(vn), t, mode=kvp.KVP_MASK_DMS, flag_step=dev_i32(fn),
                       delay=delay, window=W, status=st)
        orc.append(ref, kn, vn, t, orc.expire_dms(fn, t, delay, W))
        o = kvp.kvp_decode_attn(dev_bf16(qn), pools[cur], t, workspace=ws_a, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        check_attention(o.cpu().numpy(), orc.decode_attention(qn, ref, t))
    assert recompactions == 2
    compare_paged(pools[cur], ref, what="end of the loop")
    # delayed eviction at work: entries flagged in the last `delay` steps of the prompt are still cached
    assert int(ref.count.sum()) > B * H * (T0 // 8)


# --------------------------------------------------------------------------- MLA latent cache

@pytest.mark.parametrize("prune_q", [0.0, 0.75])
def test_mla_latent_cache_128_heads_full_size(kvp, prune_q):
    B, T, Hq, row, dc = 16, 8192, 128, kvp.LATENT_ROW, kvp.KVP_MLA_LATENT_DIM
    now = T - 1
    lat = syn.fast_normal_bf16(5, syn.S_LAT, (B, T, row))
    s = syn.normal_f32(5, 61, (B, T, 1))
    tau = (np.full((B, 1), -np.inf, np.float32) if prune_q == 0.0 else orc.threshold_at_quantile(s, prune_q))
    q = syn.fast_normal_bf16(5, syn.S_Q, (B, Hq, row))
    mp = T // 16
    st = status_word()
    c = kvp.LatentPagedKV.allocate(B, B * mp, mp)
    kvp.kvp_compact_latent(dev_bf16(lat), now, 0, c, mode=kvp.KVP_MASK_KVZAP, scores=dev_f32(s[:, :, 0].copy()),
                           tau=dev_f32(tau[:, 0].copy()), status=st)
    out = kvp.kvp_decode_attn_mla(dev_bf16(q), c, now, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    o = out.cpu().numpy()
    sel = [0, 5, 10, 15]
    exp = orc.mask_kvzap(s[sel], tau[sel], now)[0][:, 0]
    ref_c = orc.compact_latent_dense(lat[sel], exp, now, 0, len(sel) * mp, mp)
    np.testing.assert_array_equal(c.count.cpu().numpy()[sel], ref_c.count[:, 0])
    ref = orc.decode_attention_mla(q[sel], ref_c, dc, now)
    check_attention(o[sel], ref)
    # each softmax weight rounded to bf16 once: |error| <= (2^-9 + margin) * max |row value| of the element
    u = 2.0 ** -9 + 2.0 ** -20
    vmax = np.abs(orc.widen_bf16(lat[sel])[:, :, :dc]).max(axis=1)
    assert (np.abs(o[sel] - ref) <= u * vmax[:, None, :] + 1e-5).all()
    kept = int(ref_c.count.sum())
    print(f"MLA 128 heads, pruned at q = {prune_q}: {kept} of {len(sel) * T} slots kept in the compared elements")
