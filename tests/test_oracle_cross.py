"""The two oracles (C++ and numpy, written independently) against each other
on the same seeded inputs, function by function: integer and byte results
bit-exact, float64 results within a few ulps of each other's summation
order. CPU only."""
import numpy as np
import pytest

import kvp_synth as syn
import oracle

C, N = oracle.cpp_impl, oracle.numpy_impl


def _same_cache(a, b):
    for name in ("k_pool", "v_pool", "expire_pool", "page_table", "remap", "count"):
        np.testing.assert_array_equal(getattr(a, name), getattr(b, name), err_msg=name)
    assert a.pages_used == b.pages_used


def _same_qcache(a, b):
    for name in ("kq_pool", "vq_pool", "start_pool", "page_table", "remap", "count"):
        np.testing.assert_array_equal(getattr(a, name), getattr(b, name), err_msg=name)
    np.testing.assert_array_equal(a.kscale.view(np.uint32), b.kscale.view(np.uint32))
    np.testing.assert_array_equal(a.vscale.view(np.uint32), b.vscale.view(np.uint32))
    assert a.pages_used == b.pages_used


def test_scores_agree():
    x, w = syn.linear_inputs(11, 400, 320, 6)
    b = syn.normal_f32(11, 40, (6,))
    np.testing.assert_allclose(C.score_linear(x, w, b), N.score_linear(x, w, b), rtol=1e-12, atol=1e-12)
    x, w1, w2 = syn.mlp_inputs(11, 64, 256, 512, 5)
    b1, b2 = syn.normal_f32(11, 41, (512,), std=0.1), syn.normal_f32(11, 42, (5,))
    np.testing.assert_allclose(C.score_mlp(x, w1, w2, b1, b2), N.score_mlp(x, w1, w2, b1, b2), rtol=1e-12,
                               atol=1e-12)
    u = np.linspace(-9, 9, 1001)
    np.testing.assert_allclose(C.gelu(u), N.gelu(u), rtol=1e-12, atol=1e-15)  # two erf implementations


@pytest.mark.parametrize("window", [128, 7, 0])
def test_masks_and_thresholds_agree(window):
    B, T, H = 3, 900, 5
    s = syn.normal_f32(12, 1, (B, T, H)).astype(np.float64)
    s[0, 3, 1] = np.nan
    s[1, :10, 2] = -np.inf
    tau = N.threshold_at_quantile(s, 0.6)
    np.testing.assert_array_equal(C.threshold_at_quantile(s, 0.6), tau)
    qh = np.array([0.0, 0.2, 0.5, 0.9, 1.0])
    np.testing.assert_array_equal(C.threshold_at_quantile(s, qh), N.threshold_at_quantile(s, qh))
    for a, b in zip(C.mask_kvzap(s, tau, T - 1, window), N.mask_kvzap(s, tau, T - 1, window)):
        np.testing.assert_array_equal(a, b)
    f = np.where(syn.bernoulli(12, 2, (B, H, T), 0.875), np.arange(T)[None, None, :], -1)
    for now in (T - 1, T + 300):
        for a, b in zip(C.mask_dms(f, now, 256, window), N.mask_dms(f, now, 256, window)):
            np.testing.assert_array_equal(a, b)


def test_compaction_append_and_attention_agree():
    B, T, H, G, d, reserve = 2, 1200, 3, 4, 64, 20
    k, v = syn.kv_inputs(13, B, T, H, d)
    q = syn.q_inputs(13, B, H * G, d)
    s = syn.normal_f32(13, 3, (B, T, H))
    tau = N.threshold_at_quantile(s, 0.7)
    exp = N.mask_kvzap(s, tau, T - 1)[0]
    mp = (T + reserve + 15) // 16
    cap = B * H * mp
    a, b = C.compact_dense(k, v, exp, T - 1, reserve, cap, mp), N.compact_dense(k, v, exp, T - 1, reserve, cap, mp)
    _same_cache(a, b)
    np.testing.assert_allclose(C.decode_attention(q, a, T - 1), N.decode_attention(q, b, T - 1), rtol=1e-6,
                               atol=1e-7)
    for i in range(10):
        t = T + i
        kn, vn = syn.normal_bf16(13, 100 + i, (B, H, d)), syn.normal_bf16(13, 200 + i, (B, H, d))
        en = N.expire_kvzap(syn.normal_f32(13, 300 + i, (B, H)), tau, t)
        C.append(a, kn, vn, t, en)
        N.append(b, kn, vn, t, en)
    _same_cache(a, b)
    a2, b2 = C.compact_paged(a, T + 140, 4, cap, mp), N.compact_paged(b, T + 140, 4, cap, mp)
    _same_cache(a2, b2)
    np.testing.assert_allclose(C.decode_attention(q, a2, T + 140, 0.1), N.decode_attention(q, b2, T + 140, 0.1),
                               rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(C.dense_attention(q, k, v, T - 1), N.dense_attention(q, k, v, T - 1), rtol=1e-6,
                               atol=1e-7)
    np.testing.assert_allclose(C.window_attention(q, k, v, T - 1), N.window_attention(q, k, v, T - 1), rtol=1e-6,
                               atol=1e-7)
    with pytest.raises(oracle.CapacityError):
        C.compact_dense(k, v, exp, T - 1, reserve, 3, mp)


def test_fp8_tier_agrees():
    B, T, H, G, d, reserve = 2, 700, 2, 2, 128, 8
    k, v = syn.kv_inputs(14, B, T, H, d)
    q = syn.q_inputs(14, B, H * G, d)
    s = syn.normal_f32(14, 4, (B, T, H))
    tau, tau_q = N.threshold_at_quantile(s, 0.7), N.threshold_at_quantile(s, 0.3)
    vals = np.concatenate([np.linspace(-500, 500, 20001), [0.0, -0.0, np.nan, 1e-9, -1e-9]])
    np.testing.assert_array_equal(C.e4m3_encode(vals), N.e4m3_encode(vals))
    codes = np.arange(256, dtype=np.uint8)
    np.testing.assert_array_equal(C.e4m3_decode(codes), N.e4m3_decode(codes))
    ca, sa = C.quantize_rows(k.reshape(-1, d))
    cb, sb = N.quantize_rows(k.reshape(-1, d))
    np.testing.assert_array_equal(ca, cb)
    np.testing.assert_array_equal(sa.view(np.uint32), sb.view(np.uint32))
    mp = (T + reserve + 15) // 16
    cap = B * H * mp
    qa = C.compact_quant_dense(k, v, s, tau, tau_q, reserve, cap, mp)
    qb = N.compact_quant_dense(k, v, s, tau, tau_q, reserve, cap, mp)
    _same_qcache(qa, qb)
    f = np.where(syn.bernoulli(14, 5, (B, H, T), 0.5), np.arange(T)[None, None, :], -1)
    _same_qcache(C.compact_quant_dense(k, v, None, None, None, reserve, cap, mp, flag_step_bht=f, delay=64),
                 N.compact_quant_dense(k, v, None, None, None, reserve, cap, mp, flag_step_bht=f, delay=64))
    sn = syn.normal_f32(14, 6, (B, H))
    kn, vn = syn.normal_bf16(14, 7, (B, H, d)), syn.normal_bf16(14, 8, (B, H, d))
    C.append_quant(qa, kn, vn, T, sn, tau, tau_q)
    N.append_quant(qb, kn, vn, T, sn, tau, tau_q)
    _same_qcache(qa, qb)
    exp = N.mask_kvzap(s, tau, T - 1)[0]
    a = N.compact_dense(k, v, exp, T - 1, reserve, cap, mp)
    for now in (T - 1, T + 200):
        np.testing.assert_allclose(C.decode_attention_two_tier(q, a, qa, now),
                                   N.decode_attention_two_tier(q, a, qb, now), rtol=1e-6, atol=1e-7)


def test_latent_cache_agrees():
    B, T, Hq, R, dc = 2, 600, 6, 576, 512
    lat = syn.latent_inputs(15, B, T, R)
    s = syn.normal_f32(15, 9, (B, T, 1))
    tau = N.threshold_at_quantile(s, 0.5)
    exp = N.mask_kvzap(s, tau, T - 1)[0][:, 0]
    mp = (T + 15) // 16
    a, b = C.compact_latent_dense(lat, exp, T - 1, 0, B * mp, mp), N.compact_latent_dense(lat, exp, T - 1, 0, B * mp, mp)
    _same_cache(a, b)
    q = syn.q_inputs(15, B, Hq, R)
    np.testing.assert_allclose(C.decode_attention_mla(q, a, dc, T - 1), N.decode_attention_mla(q, b, dc, T - 1),
                               rtol=1e-6, atol=1e-7)


def test_closed_forms_agree():
    assert C.kv_cache_bytes(80, 8192, 128000) == N.kv_cache_bytes(80, 8192, 128000)
    assert C.linear_projection_macs(4096, 32, 8, 128, 14336) == N.linear_projection_macs(4096, 32, 8, 128, 14336)
    assert C.scorer_macs(4096, 8) == N.scorer_macs(4096, 8)
    assert C.scorer_macs(4096, 8, 512) == N.scorer_macs(4096, 8, 512)


def test_thread_count_does_not_change_results():
    x, w = syn.linear_inputs(16, 257, 128, 4)
    k, v = syn.kv_inputs(16, 3, 300, 2, 64)
    s = syn.normal_f32(16, 1, (3, 300, 2))
    tau = N.threshold_at_quantile(s, 0.5)
    q = syn.q_inputs(16, 3, 4, 64)
    exp = N.mask_kvzap(s, tau, 299)[0]
    res = []
    for n in (1, 3, 0):
        C.set_threads(n)
        c = C.compact_dense(k, v, exp, 299, 0, 3 * 2 * 19, 19)
        res.append((C.score_linear(x, w), C.decode_attention(q, c, 299), c.k_pool.copy()))
    C.set_threads(0)
    for r in res[1:]:
        for a, b in zip(r, res[0]):
            np.testing.assert_array_equal(a, b)
