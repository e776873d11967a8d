"""The Llama-3-8B-shaped layer at its full size (batch 16, 8192 cached
tokens, d_model 4096, 32 query / 8 kv heads, threshold at each head's
75th-percentile score), run through the library exactly as bench.py launches
it, against the oracle on the same seeded inputs.

Scores: all 131,072 x 8 within 1e-3 relative. Mask: bit-exact except entries
whose oracle score lies within 1e-3 of the threshold (counted). Compaction
and attention take the oracle's keep set so that one near-threshold flip
cannot move every later page: pools, page table, remap and counts bit-exact,
attention within the attention tolerances."""
import numpy as np
import pytest
import torch

import kvp_synth as syn
import oracle as orc
from helpers import (check_attention, check_scores, dev_bf16, dev_f32, dev_i32, host_bits,
                     oracle_linear_scores, status_word)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_llama3_8b_layer_full_size(kvp):
    cfg = syn.WORKLOADS["llama3_8b_layer"]
    B, T, H, Hq, d, D = cfg["batch"], cfg["n_pos"], cfg["n_kv_heads"], cfg["n_q_heads"], cfg["head_dim"], cfg["d_model"]
    now = T - 1
    x, w = syn.linear_inputs(0, B * T, D, H)
    k, v = syn.kv_inputs(0, B, T, H, d)
    q = syn.q_inputs(0, B, Hq, d)

    # ---- score (all rows)
    st = status_word()
    xd = dev_bf16(x)
    s_gpu = kvp.kvp_score(xd, dev_f32(w), status=st)
    torch.cuda.synchronize()
    del xd
    assert st.item() == 0
    s_ref, scale = oracle_linear_scores(x, w)
    check_scores(s_gpu.cpu().numpy(), s_ref, scale)

    # ---- mask with the GPU's scores vs the oracle's, near-threshold entries excluded
    s_ref3 = s_ref.reshape(B, T, H)
    tau = orc.threshold_at_quantile(s_ref3, cfg["prune_q"])
    exp_g, bits_g, cnt_g = kvp.kvp_mask(mode=kvp.KVP_MASK_KVZAP, batch=B, n_kv_heads=H, n_pos=T, now=now,
                                        scores=s_gpu, tau=dev_f32(tau))
    torch.cuda.synchronize()
    exp_r, keep_r, bits_r, cnt_r = orc.mask_kvzap(s_ref3, tau, now)
    near = (np.abs(s_ref3 - tau[:, None, :]) <= 1e-3).transpose(0, 2, 1)
    n_near = int(near.sum())
    print(f"near-threshold entries excluded from the mask comparison: {n_near} of {near.size}")
    np.testing.assert_array_equal(exp_g.cpu().numpy()[~near], exp_r[~near])
    assert abs(keep_r.mean() - 0.262) < 0.01   # 75th percentile plus the window's share

    # ---- compaction and attention on the oracle's keep set
    mp = (T + 15) // 16
    cap = B * H * mp
    ref_c = orc.compact_dense(k, v, exp_r.astype(np.int32), now, 0, cap, mp)
    c = kvp.PagedKV.allocate(B, H, d, cap, mp)
    kvp.kvp_compact(dev_bf16(k), dev_bf16(v), dev_i32(exp_r), now, 0, c, status=st)
    o = kvp.kvp_decode_attn(dev_bf16(q), c, now, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    np.testing.assert_array_equal(c.count.cpu().numpy(), ref_c.count)
    np.testing.assert_array_equal(c.page_table.cpu().numpy(), ref_c.page_table)
    np.testing.assert_array_equal(c.remap.cpu().numpy(), ref_c.remap)
    used = ref_c.pages_used
    np.testing.assert_array_equal(c.expire_pool.cpu().numpy()[:used], ref_c.expire_pool[:used])
    np.testing.assert_array_equal(host_bits(c.k_pool)[:used], ref_c.k_pool[:used])
    np.testing.assert_array_equal(host_bits(c.v_pool)[:used], ref_c.v_pool[:used])
    check_attention(o.cpu().numpy(), orc.decode_attention(q, ref_c, now))


def test_llama3_8b_layer_full_size_fused_and_fp8_tier(kvp):
    """The same layer through the entry points the benchmark step and the fp8
    tier use, on fp32 scores that both sides share (so every threshold
    decision is taken in the same precision): the device threshold equals the
    oracle's order statistic, the fused mask + compaction equals the oracle's
    mask then compaction, the fp8-tier compaction (tau_q at the 50th
    percentile) is bit-exact, and the two-tier attention is within the
    attention tolerances."""
    cfg = syn.WORKLOADS["llama3_8b_layer"]
    B, T, H, Hq, d = cfg["batch"], cfg["n_pos"], cfg["n_kv_heads"], cfg["n_q_heads"], cfg["head_dim"]
    now = T - 1
    k, v = syn.kv_inputs(0, B, T, H, d)
    q = syn.q_inputs(0, B, Hq, d)
    s32 = syn.normal_f32(0, 61, (B, T, H))
    st = status_word()
    sd = dev_f32(s32)

    # ---- threshold on the device, bit for bit
    tau = orc.threshold_at_quantile(s32, cfg["prune_q"])
    tau_q = orc.threshold_at_quantile(s32, 0.5)
    tau_d = kvp.kvp_threshold(sd, cfg["prune_q"])
    tq_d = kvp.kvp_threshold(sd, 0.5)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tau_d.cpu().numpy(), tau)
    np.testing.assert_array_equal(tq_d.cpu().numpy(), tau_q)

    # ---- fused mask + compaction
    mp = (T + 15) // 16
    cap = B * H * mp
    exp_r = orc.mask_kvzap(s32, tau, now)[0].astype(np.int32)
    ref_c = orc.compact_dense(k, v, exp_r, now, 0, cap, mp)
    kd, vd = dev_bf16(k), dev_bf16(v)
    c = kvp.PagedKV.allocate(B, H, d, cap, mp)
    kvp.kvp_compact_masked(kd, vd, now, 0, c, mode=kvp.KVP_MASK_KVZAP, scores=sd.view(B * T, H), tau=tau_d, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    np.testing.assert_array_equal(c.count.cpu().numpy(), ref_c.count)
    np.testing.assert_array_equal(c.page_table.cpu().numpy(), ref_c.page_table)
    np.testing.assert_array_equal(c.remap.cpu().numpy(), ref_c.remap)
    used = ref_c.pages_used
    np.testing.assert_array_equal(c.expire_pool.cpu().numpy()[:used], ref_c.expire_pool[:used])
    np.testing.assert_array_equal(host_bits(c.k_pool)[:used], ref_c.k_pool[:used])
    np.testing.assert_array_equal(host_bits(c.v_pool)[:used], ref_c.v_pool[:used])

    # ---- fp8 tier and the two-tier attention
    ref_q = orc.compact_quant_dense(k, v, s32, tau, tau_q, 0, cap, mp)
    cq = kvp.QuantPagedKV.allocate(B, H, d, cap, mp)
    kvp.kvp_compact_quant(kd, vd, sd, tau_d, tq_d, cq, status=st)
    o = kvp.kvp_decode_attn_two_tier(dev_bf16(q), c, cq, now, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    usedq = ref_q.pages_used
    np.testing.assert_array_equal(cq.count.cpu().numpy(), ref_q.count)
    np.testing.assert_array_equal(cq.page_table.cpu().numpy(), ref_q.page_table)
    np.testing.assert_array_equal(cq.kq_pool.cpu().numpy()[:usedq], ref_q.kq_pool[:usedq])
    np.testing.assert_array_equal(cq.vq_pool.cpu().numpy()[:usedq], ref_q.vq_pool[:usedq])
    np.testing.assert_array_equal(cq.kscale.cpu().numpy()[:usedq].view(np.uint32), ref_q.kscale[:usedq].view(np.uint32))
    np.testing.assert_array_equal(cq.vscale.cpu().numpy()[:usedq].view(np.uint32), ref_q.vscale[:usedq].view(np.uint32))
    np.testing.assert_array_equal(cq.start_pool.cpu().numpy()[:usedq], ref_q.start_pool[:usedq])
    check_attention(o.cpu().numpy(), orc.decode_attention_two_tier(q, ref_c, ref_q, now))
