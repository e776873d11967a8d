"""GPU path vs the oracle, element by element, on the same seeded inputs.

Bars: masks, expire values, page tables, remap lists and pools bit-exact;
scores within 1e-3 relative (to max(|s|, ||x_t * w_h||_2)); attention within
max-abs 2e-2, mean-abs 2e-3 and 1e-2 relative per head."""
import math

import numpy as np
import pytest
import torch

import kvp_synth as syn
import oracle as orc
from helpers import check_attention, check_scores, dev_bf16, dev_f32, dev_i32, host_bits, status_word

pytestmark = pytest.mark.gpu


def _linear_scale(x_bits, w):
    """||x_t * w_h||_2 per (t, h): the size of the dot product's terms."""
    x = orc.widen_bf16(x_bits)
    return np.sqrt((x * x) @ (np.asarray(w, np.float64) ** 2).T)


# --------------------------------------------------------------------------- score

@pytest.mark.parametrize("n_tok,D,H,bias", [
    (512, 256, 2, False),     # tiny workload shape, one layer
    (1000, 4096, 8, True),    # Llama-3-8B width, 8 tiles with a ragged tail
    (300, 512, 64, False),    # 64 heads (widest weight tile), ragged
    (129, 1032, 5, True),     # d_model not a multiple of 64, odd head count
    (1, 64, 1, False),        # single token, single head
    # decode-step sizes: up to 64 rows go to the CUDA-core dot products
    (1, 8192, 64, True),      # one new token of the 65B-shaped MHA layer
    (16, 4096, 8, True),      # the Llama-3-8B layer's batch of new tokens
    (61, 1032, 5, False),     # ragged last group of 8 rows, d_model not a multiple of 64
    (64, 4096, 8, False),     # the largest count on that path
    (65, 4096, 8, True),      # the smallest on the tensor-core path
])
def test_score_linear(kvp, n_tok, D, H, bias):
    x, w = syn.linear_inputs(0, n_tok, D, H)
    b = syn.normal_f32(0, 77, (H,)) if bias else None
    ref = orc.score_linear(x, w, b)
    st = status_word()
    s = kvp.kvp_score(dev_bf16(x), dev_f32(w), dev_f32(b) if bias else None, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    check_scores(s.cpu().numpy(), ref, _linear_scale(x, w))


def test_score_linear_strided_rows(kvp):
    n_tok, D, H = 200, 512, 8
    x, w = syn.linear_inputs(1, n_tok, D + 64, H)
    xs = dev_bf16(x)[:, :D]  # row stride D + 64
    s = kvp.kvp_score(xs, dev_f32(w[:, :D].copy()))
    torch.cuda.synchronize()
    check_scores(s.cpu().numpy(), orc.score_linear(x[:, :D], w[:, :D]), _linear_scale(x[:, :D], w[:, :D]))


@pytest.mark.parametrize("n_tok", [1, 9, 64])
def test_score_linear_split_weight_few_rows(kvp, n_tok):
    """The few-row path on the pre-split weight gives the LINEAR call's scores
    bit for bit, and both are within the oracle tolerance."""
    D, H = 8192, 64
    x, w = syn.linear_inputs(9, n_tok, D, H)
    b = syn.normal_f32(9, 30, (H,))
    wd = dev_f32(w)
    xd = dev_bf16(x)
    s_lin = kvp.kvp_score(xd, wd, dev_f32(b))
    s_split = kvp.kvp_score(xd, kvp.kvp_score_split_weight(wd), dev_f32(b), scorer=kvp.KVP_SCORER_LINEAR_SPLIT,
                            n_kv_heads=H)
    torch.cuda.synchronize()
    assert torch.equal(s_lin, s_split)
    check_scores(s_split.cpu().numpy(), orc.score_linear(x, w, b), _linear_scale(x, w))


def test_score_linear_split_weight(kvp):
    # the pre-split operand: row 2h = bf16(w[h]) (round to nearest even), row
    # 2h+1 = bf16(w[h] - bf16(w[h])), rows past 2H zero; scores from it are
    # bit-identical to the LINEAR call and within the oracle tolerance
    n_tok, D, H = 3000, 4096, 8
    x, w = syn.linear_inputs(4, n_tok, D, H)
    b = syn.normal_f32(4, 30, (H,))
    wd = dev_f32(w)
    ws = kvp.kvp_score_split_weight(wd)
    torch.cuda.synchronize()
    assert ws.shape == (16, D) and ws.dtype == torch.bfloat16
    wt = torch.from_numpy(np.asarray(w, np.float32))
    hi = wt.to(torch.bfloat16)
    lo = (wt - hi.float()).to(torch.bfloat16)
    got = ws.cpu()
    assert torch.equal(got[0:2 * H:2].view(torch.int16), hi.view(torch.int16))
    assert torch.equal(got[1:2 * H:2].view(torch.int16), lo.view(torch.int16))
    assert not got[2 * H:].float().any()
    xd = dev_bf16(x)
    s_lin = kvp.kvp_score(xd, wd, dev_f32(b))
    s_split = kvp.kvp_score(xd, ws, dev_f32(b), scorer=kvp.KVP_SCORER_LINEAR_SPLIT, n_kv_heads=H)
    torch.cuda.synchronize()
    assert torch.equal(s_lin, s_split)
    ref = orc.score_linear(x, w, b)
    scale = np.sqrt(orc.widen_bf16(x) ** 2 @ (np.asarray(w, np.float64) ** 2).T)
    check_scores(s_split.cpu().numpy(), ref, scale)


@pytest.mark.parametrize("n_tok,D,hidden,H,bias", [
    (300, 512, 512, 8, True),
    (128, 256, 1024, 8, False),
    (77, 320, 256, 3, True),
])
def test_score_mlp(kvp, n_tok, D, hidden, H, bias):
    x, w1, w2 = syn.mlp_inputs(0, n_tok, D, hidden, H)
    b1 = syn.normal_f32(0, 78, (hidden,), std=0.1) if bias else None
    b2 = syn.normal_f32(0, 79, (H,)) if bias else None
    ref = orc.score_mlp(x, w1, w2, b1, b2)
    st = status_word()
    s = kvp.kvp_score(dev_bf16(x), dev_bf16(w1), dev_f32(b1) if bias else None, dev_bf16(w2),
                      dev_f32(b2) if bias else None, scorer=kvp.KVP_SCORER_MLP, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    # natural error scale: the 2-norm of the hidden terms z_j * w2[h, j]
    u = orc.widen_bf16(x) @ orc.widen_bf16(w1).T + (0 if b1 is None else b1[None, :])
    z = orc.gelu(u)
    scale = np.sqrt((z * z) @ (orc.widen_bf16(w2) ** 2).T)
    check_scores(s.cpu().numpy(), ref, scale)


@pytest.mark.parametrize("n_tok,bias", [(1, True), (4, False), (13, True), (64, False), (65, True)])
def test_score_mlp_decode_rows(kvp, n_tok, bias):
    """A decode step's few rows at the MLP prefill config's width (d_model
    4096 -> 1024 -> 8): up to 64 rows on the CUDA-core path, 65 on the tensor
    cores; both within the score tolerance."""
    D, hidden, H = 4096, 1024, 8
    x, w1, w2 = syn.mlp_inputs(6, n_tok, D, hidden, H)
    b1 = syn.normal_f32(6, 78, (hidden,), std=0.1) if bias else None
    b2 = syn.normal_f32(6, 79, (H,)) if bias else None
    st = status_word()
    s = kvp.kvp_score(dev_bf16(x), dev_bf16(w1), dev_f32(b1) if bias else None, dev_bf16(w2),
                      dev_f32(b2) if bias else None, scorer=kvp.KVP_SCORER_MLP, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    u = orc.widen_bf16(x) @ orc.widen_bf16(w1).T + (0 if b1 is None else b1[None, :])
    z = orc.gelu(u)
    check_scores(s.cpu().numpy(), orc.score_mlp(x, w1, w2, b1, b2), np.sqrt((z * z) @ (orc.widen_bf16(w2) ** 2).T))


# --------------------------------------------------------------------------- mask

@pytest.mark.parametrize("B,T,H,window", [(1, 512, 2, 128), (3, 1000, 5, 128), (2, 33, 3, 7), (1, 4096, 8, 0),
                                          (2, 700, 12, 128),   # two batches of heads per thread
                                          (1, 300, 70, 128)])  # heads past the shared-memory counts
def test_mask_kvzap_bit_exact(kvp, B, T, H, window):
    s = syn.normal_f32(2, 11, (B, T, H))
    s[0, 5, 0] = np.nan
    tau = syn.normal_f32(2, 12, (B, H), std=0.5)
    tau[0, 0] = -np.inf
    now = T - 1
    exp_r, keep_r, bits_r, cnt_r = orc.mask_kvzap(s, tau, now, window=window)
    exp, bits, cnt = kvp.kvp_mask(mode=kvp.KVP_MASK_KVZAP, batch=B, n_kv_heads=H, n_pos=T, now=now,
                                  scores=dev_f32(s), tau=dev_f32(tau), window=window)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(exp.cpu().numpy(), exp_r)
    np.testing.assert_array_equal(bits.cpu().numpy().view(np.uint32), bits_r)
    np.testing.assert_array_equal(cnt.cpu().numpy(), cnt_r)


@pytest.mark.parametrize("delay,now", [(256, 4095), (40, 3000), (0, 4095)])
def test_mask_dms_bit_exact(kvp, delay, now):
    B, H, T = 4, 8, 4096
    ev = syn.bernoulli(0, syn.S_FLAG, (B, H, T), 7 / 8)
    f = np.where(ev, np.arange(T)[None, None, :], -1).astype(np.int32)
    exp_r, keep_r, bits_r, cnt_r = orc.mask_dms(f, now, delay)
    exp, bits, cnt = kvp.kvp_mask(mode=kvp.KVP_MASK_DMS, batch=B, n_kv_heads=H, n_pos=T, now=now,
                                  flag_step=dev_i32(f), delay=delay)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(exp.cpu().numpy(), exp_r)
    np.testing.assert_array_equal(bits.cpu().numpy().view(np.uint32), bits_r)
    np.testing.assert_array_equal(cnt.cpu().numpy(), cnt_r)


# --------------------------------------------------------------------------- threshold

def _check_tau(t_gpu, t_ref):
    # bit-identical values (NaN == NaN; -0.0 and +0.0 are one value)
    np.testing.assert_array_equal(t_gpu, t_ref)


@pytest.mark.parametrize("B,T,H,q", [
    (1, 512, 2, 0.5),
    (16, 8192, 8, 0.75),       # a Llama-3-8B layer's scores
    (3, 1000, 40, 0.3),        # two head groups, the second partial
    (2, 1, 5, 0.9),            # one position
    (4, 777, 3, 0.0),
    (4, 777, 3, 1.0),
    (1, 131072, 64, 0.6),      # the 65B-MHA layer: one b, 64 heads, long rows
    (2, 700, 12, 0.4),         # 16-byte loads whose row of 3 does not divide the block
    (2, 900, 44, 0.7),         # second head group of 12
])
def test_threshold_matches_oracle(kvp, B, T, H, q):
    s = syn.normal_f32(4, 40, (B, T, H))
    tau = kvp.kvp_threshold(dev_f32(s), q)
    torch.cuda.synchronize()
    _check_tau(tau.cpu().numpy(), orc.threshold_at_quantile(s, q))


@pytest.mark.parametrize("H", [6, 8])   # one score per load; four heads per 16-byte load
def test_threshold_ties_and_special_values(kvp, H):
    B, T = 3, 2000
    s = (np.round(syn.normal_f32(5, 41, (B, T, H)) * 2) / 2).astype(np.float32)   # heavy ties
    s[0, :300, 0] = np.nan                  # NaN ranks last
    s[0, 300:310, 0] = np.inf
    s[1, :500, 1] = -np.inf
    s[1, 500:900, 1] = -0.0
    s[2, :, 2] = np.nan                     # all NaN
    s[2, :, 3] = 1.5                        # all equal
    s[2, ::2, 4] = -0.0                     # signed zeros mixed with +0.0 below
    s[2, 1::2, 4] = 0.0
    for q in [0.0, 0.05, 0.25, 0.5, 0.8, 0.86, 0.999, 1.0]:
        tau = kvp.kvp_threshold(dev_f32(s), q)
        torch.cuda.synchronize()
        _check_tau(tau.cpu().numpy(), orc.threshold_at_quantile(s, q))


def test_threshold_then_mask_prunes_the_quantile(kvp):
    """Device threshold feeding the mask: per head, exactly T - k entries score
    at or above it when the scores are distinct (k = floor(q (T - 1)))."""
    B, T, H, q = 4, 4096, 8, 0.75
    s = syn.normal_f32(6, 42, (B, T, H))
    sd = dev_f32(s)
    tau = kvp.kvp_threshold(sd, q)
    exp, bits, cnt = kvp.kvp_mask(mode=kvp.KVP_MASK_KVZAP, batch=B, n_kv_heads=H, n_pos=T, now=T - 1,
                                  scores=sd.view(B * T, H), tau=tau, window=0)
    torch.cuda.synchronize()
    k = math.floor(q * (T - 1))
    np.testing.assert_array_equal(cnt.cpu().numpy(), np.full((B, H), T - k))


# --------------------------------------------------------------------------- compact

def _compare_cache(gpu, ref: orc.PagedCache):
    np.testing.assert_array_equal(gpu.count.cpu().numpy(), ref.count, err_msg="count")
    np.testing.assert_array_equal(gpu.page_table.cpu().numpy(), ref.page_table, err_msg="page_table")
    np.testing.assert_array_equal(gpu.remap.cpu().numpy(), ref.remap, err_msg="remap")
    used = ref.pages_used
    np.testing.assert_array_equal(gpu.expire_pool.cpu().numpy()[:used], ref.expire_pool[:used], err_msg="expire")
    np.testing.assert_array_equal(host_bits(gpu.k_pool)[:used], ref.k_pool[:used], err_msg="k_pool")
    np.testing.assert_array_equal(host_bits(gpu.v_pool)[:used], ref.v_pool[:used], err_msg="v_pool")


def _kvzap_case(B, T, H, d, seed=3, tau_std=0.7):
    k, v = syn.kv_inputs(seed, B, T, H, d)
    s = syn.normal_f32(seed, 21, (B, T, H))
    tau = syn.normal_f32(seed, 22, (B, H), std=tau_std)
    exp, keep, bits, cnt = orc.mask_kvzap(s, tau, T - 1)
    return k, v, exp.astype(np.int32), cnt


@pytest.mark.parametrize("B,T,H,d,reserve", [
    (1, 512, 2, 64, 0),
    (2, 3000, 3, 128, 5),      # 3 chunks, ragged
    (4, 1030, 8, 128, 64),
    (2, 17, 2, 64, 16),        # tiny ragged, reserve a full page
    (131, 40, 8, 64, 3),       # more than 1024 (b, h): page bases from the separate base pass
])
def test_compact_dense_bit_exact(kvp, B, T, H, d, reserve):
    k, v, exp, cnt = _kvzap_case(B, T, H, d)
    max_pages = (T + reserve + 15) // 16
    cap = B * H * max_pages
    ref = orc.compact_dense(k, v, exp, T - 1, reserve, cap, max_pages)
    st = status_word()
    dst = kvp.PagedKV.allocate(B, H, d, cap, max_pages)
    kvp.kvp_compact(dev_bf16(k), dev_bf16(v), dev_i32(exp), T - 1, reserve, dst, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_cache(dst, ref)
    # rows past count in a (b, h)'s last page are zero, expire 0
    ep = dst.expire_pool.cpu().numpy()
    assert (ep[ref.pages_used:] == 0).all()


def test_compact_strided_source(kvp):
    # K/V as a [B, H, T, d] tensor viewed as [B, T, H, d]
    B, T, H, d = 2, 700, 4, 128
    k, v, exp, cnt = _kvzap_case(B, T, H, d, seed=5)
    kt = dev_bf16(np.ascontiguousarray(k.transpose(0, 2, 1, 3))).permute(0, 2, 1, 3)
    vt = dev_bf16(np.ascontiguousarray(v.transpose(0, 2, 1, 3))).permute(0, 2, 1, 3)
    max_pages = (T + 15) // 16
    ref = orc.compact_dense(k, v, exp, T - 1, 0, B * H * max_pages, max_pages)
    st = status_word()
    dst = kvp.PagedKV.allocate(B, H, d, B * H * max_pages, max_pages)
    kvp.kvp_compact(kt, vt, dev_i32(exp), T - 1, 0, dst, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_cache(dst, ref)


def test_compact_keep_all_and_keep_none(kvp):
    B, T, H, d = 1, 300, 2, 64
    k, v = syn.kv_inputs(6, B, T, H, d)
    for exp in [np.full((B, H, T), orc.NEVER, np.int32), np.zeros((B, H, T), np.int32)]:
        ref = orc.compact_dense(k, v, exp, T - 1, 3, 64, 32)
        st = status_word()
        dst = kvp.PagedKV.allocate(B, H, d, 64, 32)
        kvp.kvp_compact(dev_bf16(k), dev_bf16(v), dev_i32(exp), T - 1, 3, dst, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        _compare_cache(dst, ref)


def test_compact_capacity_status(kvp):
    B, T, H, d = 1, 256, 2, 64
    k, v = syn.kv_inputs(6, B, T, H, d)
    exp = dev_i32(np.full((B, H, T), orc.NEVER, np.int32))
    st = status_word()
    dst = kvp.PagedKV.allocate(B, H, d, 20, 32)  # needs 32 pages in all
    kvp.kvp_compact(dev_bf16(k), dev_bf16(v), exp, T - 1, 0, dst, status=st)
    torch.cuda.synchronize()
    assert st.item() == kvp.KVP_ERR_CAPACITY
    st.zero_()
    dst = kvp.PagedKV.allocate(B, H, d, 64, 15)  # a (b, h) needs 16 > max_pages
    kvp.kvp_compact(dev_bf16(k), dev_bf16(v), exp, T - 1, 0, dst, status=st)
    torch.cuda.synchronize()
    assert st.item() == kvp.KVP_ERR_CAPACITY
    # the same check when more than 1024 (b, h) take the separate base pass
    B, T, H = 130, 32, 8
    k, v = syn.kv_inputs(6, B, T, H, d)
    exp = dev_i32(np.full((B, H, T), orc.NEVER, np.int32))
    st.zero_()
    dst = kvp.PagedKV.allocate(B, H, d, 2000, 2)  # needs 2 * 1040 pages
    kvp.kvp_compact(dev_bf16(k), dev_bf16(v), exp, T - 1, 0, dst, status=st)
    torch.cuda.synchronize()
    assert st.item() == kvp.KVP_ERR_CAPACITY


# --------------------------------------------------------------------------- fused mask + compact

@pytest.mark.parametrize("B,T,H,d,reserve,window,strided", [
    (1, 512, 2, 64, 0, 128, False),
    (2, 3000, 3, 128, 5, 128, True),    # ragged segments, [B, H, T, d] storage viewed as [B, T, H, d]
    (4, 1030, 8, 128, 64, 7, False),
    (2, 17, 2, 64, 16, 0, False),       # tiny ragged, no window
    (131, 40, 8, 64, 3, 16, False),     # more than 1024 (b, h): page bases from the separate base pass
])
def test_compact_masked_kvzap_bit_exact(kvp, B, T, H, d, reserve, window, strided):
    """Mask fused into the compaction == the oracle's mask followed by its
    compaction, and == the two GPU calls in sequence."""
    k, v = syn.kv_inputs(7, B, T, H, d)
    s = syn.normal_f32(7, 21, (B, T, H))
    s[0, min(5, T - 1), 0] = np.nan
    tau = syn.normal_f32(7, 22, (B, H), std=0.7)
    tau[0, 0] = -np.inf                 # keeps every entry of that head
    tau[-1, -1] = np.inf                # keeps only the window of that head
    now = T - 1
    exp_r = orc.mask_kvzap(s, tau, now, window=window)[0]
    max_pages = (T + reserve + 15) // 16
    cap = B * H * max_pages
    ref = orc.compact_dense(k, v, exp_r, now, reserve, cap, max_pages)
    if strided:
        kd = dev_bf16(np.ascontiguousarray(k.transpose(0, 2, 1, 3))).permute(0, 2, 1, 3)
        vd = dev_bf16(np.ascontiguousarray(v.transpose(0, 2, 1, 3))).permute(0, 2, 1, 3)
    else:
        kd, vd = dev_bf16(k), dev_bf16(v)
    sd, td = dev_f32(s), dev_f32(tau)
    st = status_word()
    dst = kvp.PagedKV.allocate(B, H, d, cap, max_pages)
    kvp.kvp_compact_masked(kd, vd, now, reserve, dst, mode=kvp.KVP_MASK_KVZAP, scores=sd, tau=td, window=window,
                           status=st)
    two = kvp.PagedKV.allocate(B, H, d, cap, max_pages)
    exp, _, _ = kvp.kvp_mask(mode=kvp.KVP_MASK_KVZAP, batch=B, n_kv_heads=H, n_pos=T, now=now, scores=sd, tau=td,
                             window=window)
    kvp.kvp_compact(kd, vd, exp, now, reserve, two, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_cache(dst, ref)
    for name in ("k_pool", "v_pool", "expire_pool", "page_table", "remap", "count"):
        assert torch.equal(getattr(dst, name), getattr(two, name)), name


@pytest.mark.parametrize("delay,window,now_back", [(256, 128, 0), (40, 32, 0), (0, 128, 300)])
def test_compact_masked_dms_bit_exact(kvp, delay, window, now_back):
    B, T, H, d = 3, 2100, 4, 128
    k, v, f, _ = _dms_stream(B, T, H, d, delay, window, seed=12)
    now = T - 1 - now_back              # entries past `now` are in the source too: expire decides
    exp_r = orc.mask_dms(f, now, delay, window=window)[0]
    max_pages = (T + 15) // 16
    cap = B * H * max_pages
    ref = orc.compact_dense(k, v, exp_r, now, 0, cap, max_pages)
    st = status_word()
    dst = kvp.PagedKV.allocate(B, H, d, cap, max_pages)
    kvp.kvp_compact_masked(dev_bf16(k), dev_bf16(v), now, 0, dst, mode=kvp.KVP_MASK_DMS, flag_step=dev_i32(f),
                           delay=delay, window=window, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_cache(dst, ref)


def test_compact_masked_and_quant_empty_source(kvp):
    """No positions at all: every (b, h) gets its reserve's pages (zeroed),
    count 0, remap -1; the fp8 tier likewise."""
    B, T, H, d, reserve = 2, 0, 3, 64, 20
    k = np.zeros((B, T, H, d), np.uint16)
    s = np.zeros((B, T, H), np.float32)
    tau = np.zeros((B, H), np.float32)
    mp = 4
    ref = orc.compact_dense(k, k, np.zeros((B, H, T), np.int32), 0, reserve, B * H * mp, mp)
    refq = orc.compact_quant_dense(k, k, s, tau, tau - 1, reserve, B * H * mp, mp)
    st = status_word()
    kd = torch.zeros((B, T, H, d), dtype=torch.bfloat16, device="cuda")
    sd = torch.zeros((B * T, H), dtype=torch.float32, device="cuda")
    c = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp)
    c.k_pool.fill_(1.0)      # the reserved rows must come back zeroed
    kvp.kvp_compact_masked(kd, kd, 0, reserve, c, mode=kvp.KVP_MASK_KVZAP, scores=sd, tau=dev_f32(tau), status=st)
    cq = kvp.QuantPagedKV.allocate(B, H, d, B * H * mp, mp)
    cq.kq_pool.fill_(7)
    kvp.kvp_compact_quant(kd, kd, sd, dev_f32(tau), dev_f32(tau - 1), cq, reserve=reserve, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_cache(c, ref)
    _compare_qcache(cq, refq)
    assert ref.pages_used == B * H * 2


def test_compact_masked_capacity_status(kvp):
    B, T, H, d = 1, 256, 2, 64
    k, v = syn.kv_inputs(6, B, T, H, d)
    s = dev_f32(np.zeros((B, T, H), np.float32))
    tau = dev_f32(np.full((B, H), -np.inf, np.float32))   # keeps all 512 entries: 32 pages
    st = status_word()
    dst = kvp.PagedKV.allocate(B, H, d, 20, 32)
    kvp.kvp_compact_masked(dev_bf16(k), dev_bf16(v), T - 1, 0, dst, mode=kvp.KVP_MASK_KVZAP, scores=s, tau=tau,
                           status=st)
    torch.cuda.synchronize()
    assert st.item() == kvp.KVP_ERR_CAPACITY


# --------------------------------------------------------------------------- fp8 tier

def _compare_qcache(gpu, ref: orc.QuantPagedCache):
    np.testing.assert_array_equal(gpu.count.cpu().numpy(), ref.count, err_msg="count")
    np.testing.assert_array_equal(gpu.page_table.cpu().numpy(), ref.page_table, err_msg="page_table")
    np.testing.assert_array_equal(gpu.remap.cpu().numpy(), ref.remap, err_msg="remap")
    used = ref.pages_used
    np.testing.assert_array_equal(gpu.kq_pool.cpu().numpy()[:used], ref.kq_pool[:used], err_msg="K codes")
    np.testing.assert_array_equal(gpu.vq_pool.cpu().numpy()[:used], ref.vq_pool[:used], err_msg="V codes")
    np.testing.assert_array_equal(gpu.kscale.cpu().numpy()[:used].view(np.uint32),
                                  ref.kscale[:used].view(np.uint32), err_msg="K scales")
    np.testing.assert_array_equal(gpu.vscale.cpu().numpy()[:used].view(np.uint32),
                                  ref.vscale[:used].view(np.uint32), err_msg="V scales")
    np.testing.assert_array_equal(gpu.start_pool.cpu().numpy()[:used], ref.start_pool[:used], err_msg="start")


def _quant_case(B, T, H, d, seed, kv_std=1.0):
    k, v = syn.kv_inputs(seed, B, T, H, d)
    if kv_std != 1.0:
        k = syn.f32_to_bf16_bits((orc.widen_bf16(k) * kv_std).astype(np.float32))
    s = syn.normal_f32(seed, 31, (B, T, H))
    s[0, min(3, T - 1), 0] = np.nan
    tau = syn.normal_f32(seed, 32, (B, H), std=0.3) + np.float32(0.7)
    tau_q = syn.normal_f32(seed, 33, (B, H), std=0.3) - np.float32(0.7)
    tau_q[-1, -1] = -np.inf                # every entry below tau goes to the fp8 tier
    tau_q[0, -1] = tau[0, -1]              # empty fp8 tier for this head
    return k, v, s, tau.astype(np.float32), tau_q.astype(np.float32)


@pytest.mark.parametrize("B,T,H,d,reserve,window,strided", [
    (1, 512, 2, 64, 0, 128, False),
    (2, 3000, 3, 128, 5, 128, True),
    (4, 1030, 8, 128, 64, 7, False),
    (2, 17, 2, 64, 16, 0, False),
    (131, 40, 8, 64, 3, 16, False),     # more than 1024 (b, h): page bases from the separate base pass
])
def test_compact_quant_bit_exact(kvp, B, T, H, d, reserve, window, strided):
    """fp8-tier compaction: codes, scales, start steps, page tables and remap
    lists bit-identical to the oracle."""
    k, v, s, tau, tau_q = _quant_case(B, T, H, d, seed=13, kv_std=3.0)
    max_pages = (T + reserve + 15) // 16
    cap = B * H * max_pages
    ref = orc.compact_quant_dense(k, v, s, tau, tau_q, reserve, cap, max_pages, window=window)
    if strided:
        kd = dev_bf16(np.ascontiguousarray(k.transpose(0, 2, 1, 3))).permute(0, 2, 1, 3)
        vd = dev_bf16(np.ascontiguousarray(v.transpose(0, 2, 1, 3))).permute(0, 2, 1, 3)
    else:
        kd, vd = dev_bf16(k), dev_bf16(v)
    st = status_word()
    dst = kvp.QuantPagedKV.allocate(B, H, d, cap, max_pages)
    kvp.kvp_compact_quant(kd, vd, dev_f32(s), dev_f32(tau), dev_f32(tau_q), dst, reserve=reserve, window=window,
                          status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_qcache(dst, ref)


def test_compact_quant_special_rows(kvp):
    """All-zero rows (scale 0, codes 0), rows with one huge element (everything
    else in the subnormal range), exact ties on the E4M3 grid, and rows at
    scale exactly 1 that hold every finite E4M3 value (codes 0..126 and
    129..254), so that each code's encoding is compared once."""
    B, T, H, d = 1, 64, 2, 128
    rng = np.random.default_rng(5)
    kf = rng.standard_normal((B, T, H, d)).astype(np.float32)
    kf[0, 0] = 0.0                                    # zero rows
    kf[0, 1, :, :] *= 1e-3
    kf[0, 1, :, 0] = 300.0                            # one large element, the rest tiny
    grid = orc.e4m3_positive_values()[:127]
    mids = np.resize(((grid[:-1] + grid[1:]) / 2)[20:], d - 1)
    kf[0, 2, :, 0] = 448.0                            # scale exactly 1: the others are exact ties
    kf[0, 2, :, 1:] = mids
    full = orc.e4m3_positive_values()[:127]           # codes 0..126 (0 .. 448)
    kf[0, 3, :, :127] = full                          # scale 1 (amax 448): every code is its own value
    kf[0, 3, :, 127] = 448.0
    kf[0, 4, :, :126] = -full[1:]                     # codes 129..254
    kf[0, 4, :, 126] = 448.0
    kf[0, 4, :, 127] = 1.0
    k = syn.f32_to_bf16_bits(kf)
    v = syn.f32_to_bf16_bits(kf[:, ::-1].copy())
    s = np.zeros((B, T, H), np.float32)
    tau = np.ones((B, H), np.float32)
    tau_q = np.full((B, H), -1.0, np.float32)
    ref = orc.compact_quant_dense(k, v, s, tau, tau_q, 0, 16, 8)
    st = status_word()
    dst = kvp.QuantPagedKV.allocate(B, H, d, 16, 8)
    kvp.kvp_compact_quant(dev_bf16(k), dev_bf16(v), dev_f32(s), dev_f32(tau), dev_f32(tau_q), dst, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_qcache(dst, ref)


@pytest.mark.parametrize("d", [64, 128])
def test_append_quant_bit_exact(kvp, d):
    """fp8-tier compaction of [0, T0), then appends of T0..T-1: bit-identical
    to the oracle at every slot; an exhausted reserve records
    KVP_ERR_CAPACITY and leaves that (b, h) unchanged."""
    B, T0, T, H = 3, 700, 780, 4
    k, v = syn.kv_inputs(19, B, T, H, d)
    s = syn.normal_f32(19, 51, (B, T, H))
    tau = np.full((B, H), 0.6, np.float32)
    tau_q = np.full((B, H), -0.4, np.float32)
    tau_q[0, 0] = -np.inf                 # every token below tau: this (b, h)'s reserve runs out first
    reserve, mp = 48, (T + 48 + 15) // 16
    cap = B * H * mp
    ref = orc.compact_quant_dense(k[:, :T0], v[:, :T0], s[:, :T0], tau, tau_q, reserve, cap, mp)
    st = status_word()
    cq = kvp.QuantPagedKV.allocate(B, H, d, cap, mp)
    kvp.kvp_compact_quant(dev_bf16(k[:, :T0].copy()), dev_bf16(v[:, :T0].copy()), dev_f32(s[:, :T0].copy()),
                          dev_f32(tau), dev_f32(tau_q), cq, reserve=reserve, status=st)
    kd, vd, sd = dev_bf16(k), dev_bf16(v), dev_f32(s)
    tq_d, tau_d = dev_f32(tau_q), dev_f32(tau)
    t_fail = None
    for t in range(T0, T):
        try:
            orc.append_quant(ref, k[:, t], v[:, t], t, s[:, t], tau, tau_q)
        except orc.CapacityError:
            t_fail = t
            break
        kvp.kvp_append_quant(cq, kd[:, t].contiguous(), vd[:, t].contiguous(), t, score=sd[:, t].contiguous(),
                             tau=tau_d, tau_q=tq_d, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_qcache(cq, ref)
    assert t_fail is not None, "the test expects the reserve of (0, 0) to run out"
    before = cq.count.clone()
    kvp.kvp_append_quant(cq, kd[:, t_fail].contiguous(), vd[:, t_fail].contiguous(), t_fail,
                         score=sd[:, t_fail].contiguous(), tau=tau_d, tau_q=tq_d, status=st)
    torch.cuda.synchronize()
    assert st.item() == kvp.KVP_ERR_CAPACITY
    assert int(cq.count[0, 0]) == int(before[0, 0])


def test_step_in_cuda_graph_matches_eager(kvp):
    """Score, fused mask + compaction and attention captured as one CUDA graph
    (the copy pass and the attention launched as programmatic dependents)
    replay to the same bits as the eager calls."""
    B, T, H, G, d, D = 2, 3000, 4, 4, 128, 256
    x, w = syn.linear_inputs(23, B * T, D, H)
    k, v = syn.kv_inputs(23, B, T, H, d)
    q = syn.q_inputs(23, B, H * G, d)
    xd, wd, kd, vd, qd = dev_bf16(x), torch.from_numpy(w).cuda(), dev_bf16(k), dev_bf16(v), dev_bf16(q)
    ws_split = kvp.kvp_score_split_weight(wd)
    scores = torch.empty(B * T, H, dtype=torch.float32, device="cuda")
    st = status_word()
    kvp.kvp_score(xd, ws_split, scorer=kvp.KVP_SCORER_LINEAR_SPLIT, n_kv_heads=H, out=scores, status=st)
    tau = kvp.kvp_threshold(scores.view(B, T, H), 0.75)
    mp = (T + 15) // 16
    outs = []
    for use_graph in (False, True):
        cache = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp)
        out = torch.empty(B, H * G, d, dtype=torch.float32, device="cuda")
        ws_c = torch.empty(kvp.kvp_compact_workspace_bytes(B, H, T), dtype=torch.uint8, device="cuda")
        ws_a = torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, H * G, H, d), dtype=torch.uint8, device="cuda")

        def step():
            kvp.kvp_score(xd, ws_split, scorer=kvp.KVP_SCORER_LINEAR_SPLIT, n_kv_heads=H, out=scores, status=st)
            kvp.kvp_compact_masked(kd, vd, T - 1, 0, cache, mode=kvp.KVP_MASK_KVZAP, scores=scores, tau=tau,
                                   status=st, workspace=ws_c)
            kvp.kvp_decode_attn(qd, cache, T - 1, out=out, workspace=ws_a, status=st)

        if use_graph:
            step()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step()
            cache.count.zero_()
            out.zero_()
            for _ in range(3):
                g.replay()
        else:
            step()
        torch.cuda.synchronize()
        assert st.item() == 0
        outs.append((out.clone(), cache.count.clone(), cache.page_table.clone()))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)


def _dms_stream(B, T, H, d, delay, window, seed):
    k, v = syn.kv_inputs(seed, B, T, H, d)
    pos = np.arange(T)[None, None, :]
    f = np.where(syn.bernoulli(seed, 8, (B, H, T), 0.875), pos, -1).astype(np.int32)
    exp = orc.expire_dms(f, pos, delay, window).astype(np.int32)
    return k, v, f, exp


def test_append_then_paged_recompaction(kvp):
    """Prefill compaction, appends of the next tokens, then a paged re-compaction:
    bit-exact against the oracle at every stage."""
    B, T0, steps, H, d = 3, 700, 90, 4, 128
    delay, window, reserve = 60, 32, 96
    T = T0 + steps
    k, v, f, exp = _dms_stream(B, T, H, d, delay, window, seed=9)
    max_pages = (T + reserve + 15) // 16
    cap = B * H * max_pages
    now0 = T0 - 1
    ref = orc.compact_dense(k[:, :T0], v[:, :T0], exp[:, :, :T0], now0, reserve, cap, max_pages)
    st = status_word()
    c = kvp.PagedKV.allocate(B, H, d, cap, max_pages)
    kvp.kvp_compact(dev_bf16(k[:, :T0].copy()), dev_bf16(v[:, :T0].copy()), dev_i32(exp[:, :, :T0].copy()), now0,
                    reserve, c, status=st)
    kd, vd, fd = dev_bf16(k), dev_bf16(v), dev_i32(f)
    for t in range(T0, T):
        orc.append(ref, k[:, t], v[:, t], t, exp[:, :, t])
        kvp.kvp_append(c, kd[:, t].contiguous(), vd[:, t].contiguous(), t, mode=kvp.KVP_MASK_DMS,
                       flag_step=fd[:, :, t].contiguous(), delay=delay, window=window, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_cache(c, ref)
    now = T - 1
    ref2 = orc.compact_paged(ref, now, 16, cap, max_pages)
    c2 = kvp.PagedKV.allocate(B, H, d, cap, max_pages)
    kvp.kvp_compact_paged(c, now, 16, c2, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_cache(c2, ref2)


def test_append_kvzap_and_reserve_exhausted(kvp):
    B, T, H, d = 2, 100, 2, 64
    k, v = syn.kv_inputs(4, B, T + 40, H, d)
    exp = np.full((B, H, T), orc.NEVER, np.int32)
    reserve = 12  # 100 + 12 = 112 slots = 7 pages exactly
    max_pages = 8
    ref = orc.compact_dense(k[:, :T], v[:, :T], exp, T - 1, reserve, 64, max_pages)
    st = status_word()
    c = kvp.PagedKV.allocate(B, H, d, 64, max_pages)
    kvp.kvp_compact(dev_bf16(k[:, :T].copy()), dev_bf16(v[:, :T].copy()), dev_i32(exp), T - 1, reserve, c, status=st)
    score = syn.normal_f32(4, 30, (12, B, H))
    tau = np.zeros((B, H), np.float32)
    for i in range(12):
        t = T + i
        orc.append(ref, k[:, t], v[:, t], t, orc.expire_kvzap(score[i], tau, t, 128))
        kvp.kvp_append(c, dev_bf16(k[:, t].copy()), dev_bf16(v[:, t].copy()), t, mode=kvp.KVP_MASK_KVZAP,
                       score=dev_f32(score[i]), tau=dev_f32(tau), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_cache(c, ref)
    kvp.kvp_append(c, dev_bf16(k[:, T].copy()), dev_bf16(v[:, T].copy()), T + 12, mode=kvp.KVP_MASK_KVZAP,
                   score=dev_f32(score[0]), tau=dev_f32(tau), status=st)
    torch.cuda.synchronize()
    assert st.item() == kvp.KVP_ERR_CAPACITY
    np.testing.assert_array_equal(c.count.cpu().numpy(), ref.count)  # unchanged


# --------------------------------------------------------------------------- attention

def _attn_case(kvp, B, T, H, G, d, tau_std=0.7, seed=3, reserve=0, pps=0, peaked=False):
    k, v, exp, cnt = _kvzap_case(B, T, H, d, seed=seed, tau_std=tau_std)
    q = syn.q_inputs(seed, B, H * G, d)
    if peaked:  # q x 8 and 16 planted keys equal to q: a sharp softmax
        qf = orc.widen_bf16(q) * 8.0
        q = syn.f32_to_bf16_bits(qf.astype(np.float32))
        k = k.copy()
        for i in range(16):
            t = (i * 97 + 11) % T
            exp[:, :, t] = orc.NEVER
            k[:, t, :, :] = syn.f32_to_bf16_bits((qf[:, ::G, :] / 8.0).astype(np.float32))
    max_pages = (T + reserve + 15) // 16
    cap = B * H * max_pages
    now = T - 1
    ref_c = orc.compact_dense(k, v, exp, now, reserve, cap, max_pages)
    ref = orc.decode_attention(q, ref_c, now)
    st = status_word()
    c = kvp.PagedKV.allocate(B, H, d, cap, max_pages)
    kvp.kvp_compact(dev_bf16(k), dev_bf16(v), dev_i32(exp), now, reserve, c, status=st)
    out = kvp.kvp_decode_attn(dev_bf16(q), c, now, grid_limit=pps, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return out.cpu().numpy(), ref


@pytest.mark.parametrize("B,T,H,G,d,pps", [
    (1, 512, 2, 2, 64, 0),       # tiny workload shape
    (2, 2000, 8, 4, 128, 0),     # Llama-3-8B GQA 4: more warps than pages, one piece per slice
    (2, 2000, 8, 4, 128, 3),     # 3 CTAs: slices span several (b, h)
    (1, 3000, 4, 1, 128, 5),     # MHA
    (2, 1500, 2, 8, 128, 0),     # GQA 8
    (3, 777, 3, 2, 64, 1),       # one CTA: 8 slices
    (1, 900, 2, 8, 64, 7),
    (1, 1200, 4, 4, 64, 2),
    (7, 3333, 5, 4, 128, 2),     # ragged everything, slices cross (b, h) boundaries
    (1, 3000, 3, 1, 64, 0),      # odd B*H with G = 1: every workspace region stays 16-byte aligned
    (3, 2200, 3, 1, 128, 0),
    (1, 32768, 1, 4, 128, 0),    # one (b, h) over more than 32 slices: the merge goes in chunks of 32
])
def test_decode_attn(kvp, B, T, H, G, d, pps):
    o, ref = _attn_case(kvp, B, T, H, G, d, pps=pps)
    check_attention(o, ref)


@pytest.mark.parametrize("G,d", [(4, 128), (1, 128), (8, 64)])
def test_decode_attn_peaked(kvp, G, d):
    o, ref = _attn_case(kvp, 2, 1500, 2, G, d, peaked=True)
    check_attention(o, ref)


def test_decode_attn_split_independent(kvp):
    outs = [_attn_case(kvp, 1, 2500, 2, 4, 128, pps=p)[0] for p in (1, 2, 5, 0)]
    for o in outs[1:]:
        np.testing.assert_allclose(o, outs[0], rtol=0, atol=1e-5)


@pytest.mark.parametrize("d,grid", [(128, 4), (128, 5), (128, 6), (64, 5), (128, 0)])
def test_decode_attn_one_head_per_kv_head_many_pieces(kvp, d, grid):
    """One query head per kv head (MHA), one long head among short ones: with
    a capped grid the long head's pages span about 32 to 48 slices, the range
    where the merge at a slice end can stage every piece in the warp's idle
    ring; every piece must count (a per-head relative check catches one that
    is dropped)."""
    B, T, H, G = 1, 12000, 3, 1
    k, v = syn.kv_inputs(31, B, T, H, d)
    s = syn.normal_f32(31, 21, (B, T, H))
    tau = np.array([[-np.inf, 2.5, 1.5]], np.float32)   # head 0 keeps everything, the others few entries
    exp = orc.mask_kvzap(s, tau, T - 1)[0].astype(np.int32)
    q = syn.q_inputs(31, B, H * G, d)
    mp = (T + 15) // 16
    ref_c = orc.compact_dense(k, v, exp, T - 1, 0, B * H * mp, mp)
    c = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp)
    st = status_word()
    kvp.kvp_compact(dev_bf16(k), dev_bf16(v), dev_i32(exp), T - 1, 0, c, status=st)
    o = kvp.kvp_decode_attn(dev_bf16(q), c, T - 1, grid_limit=grid, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    check_attention(o.cpu().numpy(), orc.decode_attention(q, ref_c, T - 1))


def test_decode_attn_workspace_reused_across_calls(kvp):
    """One zero-filled workspace serves consecutive calls on different caches
    and grids: every result equals the one from a fresh zeroed workspace, and
    the workspace's counters are zero again after each call."""
    B, T, H, G, d = 3, 2100, 4, 4, 128
    q = dev_bf16(syn.q_inputs(11, B, H * G, d))
    st = status_word()
    caches = []
    for seed, tau_std in ((21, 0.7), (22, 0.2), (23, 1.5)):
        k, v, exp, _ = _kvzap_case(B, T, H, d, seed=seed, tau_std=tau_std)
        c = kvp.PagedKV.allocate(B, H, d, B * H * (T // 16 + 1), T // 16 + 1)
        kvp.kvp_compact(dev_bf16(k), dev_bf16(v), dev_i32(exp), T - 1, 0, c, status=st)
        caches.append(c)
    ws = torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, H * G, H, d), dtype=torch.uint8, device="cuda")
    for c in caches:
        for grid in (0, 3, 1):
            o = kvp.kvp_decode_attn(q, c, T - 1, grid_limit=grid, workspace=ws, status=st)
            fresh = kvp.kvp_decode_attn(q, c, T - 1, grid_limit=grid, status=st)
            torch.cuda.synchronize()
            assert st.item() == 0
            assert torch.equal(o, fresh)
            assert int(ws[: B * H * 4].view(torch.int32).abs().sum()) == 0   # counters back to zero


def _two_tier_case(kvp, B, T, H, G, d, pps=0, now=None, seed=17, empty_q=False):
    k, v = syn.kv_inputs(seed, B, T, H, d)
    q = syn.q_inputs(seed, B, H * G, d)
    s = syn.normal_f32(seed, 41, (B, T, H))
    tau = (syn.normal_f32(seed, 42, (B, H), std=0.3) + np.float32(0.7)).astype(np.float32)
    tau_q = tau.copy() if empty_q else (syn.normal_f32(seed, 43, (B, H), std=0.3) - np.float32(0.5)).astype(np.float32)
    if not empty_q:
        tau_q[-1, -1] = -np.inf
    now = T - 1 if now is None else now
    exp = orc.mask_kvzap(s, tau, now)[0].astype(np.int32)
    mp = (T + 15) // 16
    cap = B * H * mp
    ref_a = orc.compact_dense(k, v, exp, now, 0, cap, mp)
    ref_q = orc.compact_quant_dense(k, v, s, tau, tau_q, 0, cap, mp)
    ref = orc.decode_attention_two_tier(q, ref_a, ref_q, now)
    st = status_word()
    kd, vd = dev_bf16(k), dev_bf16(v)
    ca = kvp.PagedKV.allocate(B, H, d, cap, mp)
    kvp.kvp_compact(kd, vd, dev_i32(exp), now, 0, ca, status=st)
    cq = kvp.QuantPagedKV.allocate(B, H, d, cap, mp)
    kvp.kvp_compact_quant(kd, vd, dev_f32(s), dev_f32(tau), dev_f32(tau_q), cq, status=st)
    qd = dev_bf16(q)
    out = kvp.kvp_decode_attn_two_tier(qd, ca, cq, now, grid_limit=pps, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return out, ref, (qd, ca, cq, now, st)


@pytest.mark.parametrize("B,T,H,G,d,pps", [
    (1, 512, 2, 2, 64, 0),
    (2, 2000, 8, 4, 128, 0),     # Llama-3-8B GQA 4
    (2, 2000, 8, 4, 128, 3),     # 3 CTAs: slices cross tiers and (b, h)
    (1, 3000, 4, 1, 128, 5),
    (2, 1500, 2, 8, 128, 0),
    (3, 777, 3, 2, 64, 1),
    (7, 3333, 5, 4, 128, 2),
    (2, 1500, 4, 4, 64, 0),      # G = 4 at head_dim 64 (the tensor-core kernel with one 64-column box per row)
])
def test_decode_attn_two_tier(kvp, B, T, H, G, d, pps):
    out, ref, _ = _two_tier_case(kvp, B, T, H, G, d, pps=pps)
    check_attention(out.cpu().numpy(), ref)


def test_decode_attn_two_tier_visibility_and_empty_tier(kvp):
    """Before any fp8 entry's start step the result is the bf16 tier's alone;
    with an empty fp8 tier the two-tier kernel (CUDA-core page math) agrees
    with kvp_decode_attn (tensor-core page math) to fp32 rounding."""
    B, T, H, G, d = 2, 1200, 4, 4, 128
    out, ref, _ = _two_tier_case(kvp, B, T, H, G, d, now=100)   # now < 0 + window: no fp8 slot visible
    check_attention(out.cpu().numpy(), ref)
    out, ref, (qd, ca, cq, now, st) = _two_tier_case(kvp, B, T, H, G, d, empty_q=True)
    assert int(cq.count.sum()) == 0
    one = kvp.kvp_decode_attn(qd, ca, now, status=st)
    torch.cuda.synchronize()
    np.testing.assert_allclose(out.cpu().numpy(), one.cpu().numpy(), rtol=0, atol=2e-5)
    check_attention(out.cpu().numpy(), ref)


def test_two_tier_decode_loop(kvp):
    """Prefill both tiers at step T0 - 1, then decode steps T0..T-1: each new
    token is appended to the bf16 tier (kvp_append, KVzap rule) and, when its
    score falls in [tau_q, tau), to the fp8 tier (kvp_append_quant); every
    step's two-tier attention is checked against the oracle's. Window 32, so
    that entries cross from the bf16 tier to the fp8 tier during the loop."""
    B, T0, T, H, G, d, W = 2, 600, 680, 4, 4, 128, 32
    k, v = syn.kv_inputs(29, B, T, H, d)
    q_all = syn.normal_f32(29, 71, (T - T0, B, H * G, d))
    s = syn.normal_f32(29, 72, (B, T, H))
    tau = np.full((B, H), 0.5, np.float32)
    tau_q = np.full((B, H), -0.5, np.float32)
    now0 = T0 - 1
    reserve, mp = 96, (T + 96 + 15) // 16
    cap = B * H * mp
    exp0 = orc.mask_kvzap(s[:, :T0], tau, now0, window=W)[0].astype(np.int32)
    ref_a = orc.compact_dense(k[:, :T0], v[:, :T0], exp0, now0, reserve, cap, mp)
    ref_q = orc.compact_quant_dense(k[:, :T0], v[:, :T0], s[:, :T0], tau, tau_q, reserve, cap, mp, window=W)
    st = status_word()
    ca = kvp.PagedKV.allocate(B, H, d, cap, mp)
    cq = kvp.QuantPagedKV.allocate(B, H, d, cap, mp)
    kvp.kvp_compact(dev_bf16(k[:, :T0].copy()), dev_bf16(v[:, :T0].copy()), dev_i32(exp0), now0, reserve, ca,
                    status=st)
    kvp.kvp_compact_quant(dev_bf16(k[:, :T0].copy()), dev_bf16(v[:, :T0].copy()), dev_f32(s[:, :T0].copy()),
                          dev_f32(tau), dev_f32(tau_q), cq, reserve=reserve, window=W, status=st)
    kd, vd, sd, tau_d, tq_d = dev_bf16(k), dev_bf16(v), dev_f32(s), dev_f32(tau), dev_f32(tau_q)
    ws = torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, H * G, H, d), dtype=torch.uint8, device="cuda")
    for i, t in enumerate(range(T0, T)):
        orc.append(ref_a, k[:, t], v[:, t], t, orc.expire_kvzap(s[:, t], tau, t, W))
        orc.append_quant(ref_q, k[:, t], v[:, t], t, s[:, t], tau, tau_q, window=W)
        kvp.kvp_append(ca, kd[:, t].contiguous(), vd[:, t].contiguous(), t, mode=kvp.KVP_MASK_KVZAP,
                       score=sd[:, t].contiguous(), tau=tau_d, window=W, status=st)
        kvp.kvp_append_quant(cq, kd[:, t].contiguous(), vd[:, t].contiguous(), t, score=sd[:, t].contiguous(),
                             tau=tau_d, tau_q=tq_d, window=W, status=st)
        qb = syn.f32_to_bf16_bits(q_all[i])
        o = kvp.kvp_decode_attn_two_tier(dev_bf16(qb), ca, cq, t, workspace=ws, status=st)
        if i % 8 == 0 or t == T - 1:
            torch.cuda.synchronize()
            assert st.item() == 0
            check_attention(o.cpu().numpy(), orc.decode_attention_two_tier(qb, ref_a, ref_q, t))
    _compare_cache(ca, ref_a)
    _compare_qcache(cq, ref_q)


def test_decode_attn_largest_pair_count(kvp):
    """4096 (b, h) pairs, the most the kernel's shared page prefix holds, with
    short and empty heads mixed in; one more pair is refused on the host."""
    B, T, H, G, d = 512, 70, 8, 1, 64
    k, v = syn.kv_inputs(31, B, T, H, d)
    q = syn.q_inputs(31, B, H * G, d)
    s = syn.normal_f32(31, 81, (B, T, H))
    tau = syn.normal_f32(31, 82, (B, H), std=1.0)
    tau[::7, :] = np.inf                  # window only
    now = T - 1
    exp = orc.mask_kvzap(s, tau, now, window=3)[0].astype(np.int32)
    exp[::5, ::3, :] = 0                  # some heads keep nothing
    mp = (T + 15) // 16
    ref_c = orc.compact_dense(k, v, exp, now, 0, B * H * mp, mp)
    st = status_word()
    c = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp)
    kvp.kvp_compact(dev_bf16(k), dev_bf16(v), dev_i32(exp), now, 0, c, status=st)
    o = kvp.kvp_decode_attn(dev_bf16(q), c, now, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_cache(c, ref_c)
    check_attention(o.cpu().numpy(), orc.decode_attention(q, ref_c, now))
    big = kvp.PagedKV.allocate(B + 1, H, d, 8, 1)
    with pytest.raises(kvp.KvpError):
        kvp.kvp_decode_attn(dev_bf16(syn.q_inputs(31, B + 1, H * G, d)), big, now, status=st)


@pytest.mark.parametrize("B,T,H,d,delay,window,reserve", [
    (2, 1000, 4, 128, 256, 128, 0),
    (3, 777, 3, 64, 40, 16, 20),
    (131, 40, 8, 64, 8, 4, 3),          # more than 1024 (b, h)
])
def test_compact_quant_dms_bit_exact(kvp, B, T, H, d, delay, window, reserve):
    """DMS flags: the fp8 tier holds the flagged entries with start =
    max(flag + delay, pos + window), bit-exact against the oracle."""
    k, v, f, _ = _dms_stream(B, T, H, d, delay, window, seed=33)
    mp = (T + reserve + 15) // 16
    cap = B * H * mp
    ref = orc.compact_quant_dense(k, v, None, None, None, reserve, cap, mp, window=window, flag_step_bht=f,
                                  delay=delay)
    st = status_word()
    cq = kvp.QuantPagedKV.allocate(B, H, d, cap, mp)
    kvp.kvp_compact_quant(dev_bf16(k), dev_bf16(v), None, None, None, cq, mode=kvp.KVP_MASK_DMS,
                          flag_step=dev_i32(f), delay=delay, reserve=reserve, window=window, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_qcache(cq, ref)


def test_two_tier_dms_decode_loop(kvp):
    """DMS decode with quantize-instead-of-evict: prefill both tiers, then
    each step appends the token to the bf16 tier (kvp_append, DMS rule) and,
    if flagged, to the fp8 tier (kvp_append_quant, DMS); the two-tier
    attention at every step matches the oracle's, and the flagged entries
    cross into the fp8 tier as their delay runs out."""
    B, T0, T, H, G, d, delay, W = 2, 500, 580, 4, 4, 128, 24, 16
    k, v, f, exp = _dms_stream(B, T, H, d, delay, W, seed=37)
    q_all = syn.normal_f32(37, 91, (T - T0, B, H * G, d))
    now0 = T0 - 1
    reserve, mp = 96, (T + 96 + 15) // 16
    cap = B * H * mp
    ref_a = orc.compact_dense(k[:, :T0], v[:, :T0], exp[:, :, :T0], now0, reserve, cap, mp)
    ref_q = orc.compact_quant_dense(k[:, :T0], v[:, :T0], None, None, None, reserve, cap, mp, window=W,
                                    flag_step_bht=f[:, :, :T0], delay=delay)
    st = status_word()
    ca = kvp.PagedKV.allocate(B, H, d, cap, mp)
    cq = kvp.QuantPagedKV.allocate(B, H, d, cap, mp)
    kvp.kvp_compact(dev_bf16(k[:, :T0].copy()), dev_bf16(v[:, :T0].copy()), dev_i32(exp[:, :, :T0].copy()), now0,
                    reserve, ca, status=st)
    kvp.kvp_compact_quant(dev_bf16(k[:, :T0].copy()), dev_bf16(v[:, :T0].copy()), None, None, None, cq,
                          mode=kvp.KVP_MASK_DMS, flag_step=dev_i32(f[:, :, :T0].copy()), delay=delay,
                          reserve=reserve, window=W, status=st)
    kd, vd, fd = dev_bf16(k), dev_bf16(v), dev_i32(f)
    ws = torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, H * G, H, d), dtype=torch.uint8, device="cuda")
    for i, t in enumerate(range(T0, T)):
        orc.append(ref_a, k[:, t], v[:, t], t, exp[:, :, t])
        orc.append_quant(ref_q, k[:, t], v[:, t], t, None, None, None, window=W, flag_bh=f[:, :, t], delay=delay)
        ft = fd[:, :, t].contiguous()
        kvp.kvp_append(ca, kd[:, t].contiguous(), vd[:, t].contiguous(), t, mode=kvp.KVP_MASK_DMS, flag_step=ft,
                       delay=delay, window=W, status=st)
        kvp.kvp_append_quant(cq, kd[:, t].contiguous(), vd[:, t].contiguous(), t, mode=kvp.KVP_MASK_DMS,
                             flag_step=ft, delay=delay, window=W, status=st)
        qb = syn.f32_to_bf16_bits(q_all[i])
        o = kvp.kvp_decode_attn_two_tier(dev_bf16(qb), ca, cq, t, workspace=ws, status=st)
        if i % 10 == 0 or t == T - 1:
            torch.cuda.synchronize()
            assert st.item() == 0
            check_attention(o.cpu().numpy(), orc.decode_attention_two_tier(qb, ref_a, ref_q, t))
    _compare_cache(ca, ref_a)
    _compare_qcache(cq, ref_q)


def test_decode_attn_keep_all_is_dense_and_window(kvp):
    B, T, H, G, d = 1, 1100, 2, 4, 128
    k, v = syn.kv_inputs(8, B, T, H, d)
    q = syn.q_inputs(8, B, H * G, d)
    now = T - 1
    mp = (T + 15) // 16
    for exp, ref in [(np.full((B, H, T), orc.NEVER, np.int32), orc.dense_attention(q, k, v, now)),
                     (orc.mask_kvzap(np.full((B, T, H), -np.inf, np.float32), np.zeros((B, H), np.float32),
                                     now)[0].astype(np.int32), orc.window_attention(q, k, v, now))]:
        c = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp)
        st = status_word()
        kvp.kvp_compact(dev_bf16(k), dev_bf16(v), dev_i32(exp), now, 0, c, status=st)
        o = kvp.kvp_decode_attn(dev_bf16(q), c, now, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        check_attention(o.cpu().numpy(), ref)


def test_decode_attn_empty_heads_and_expired_slots(kvp):
    # window 0 and tau +inf for head 0: nothing kept -> zero rows; later `now`
    # turns slots of head 1 absent without re-compaction (masked in attention)
    B, T, H, G, d = 1, 400, 2, 2, 64
    k, v = syn.kv_inputs(10, B, T, H, d)
    q = syn.q_inputs(10, B, H * G, d)
    s = syn.normal_f32(10, 21, (B, T, H))
    tau = np.array([[np.inf, 0.5]], np.float32)
    exp = orc.mask_kvzap(s, tau, T - 1, window=0)[0].astype(np.int32)
    exp[0, 1, ::3] = T + 5   # these leave the cache at step T+5
    mp = (T + 15) // 16
    for now in (T - 1, T + 5):
        ref = orc.decode_attention(q, orc.compact_dense(k, v, exp, T - 1, 0, B * H * mp, mp), now)
        c = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp)
        st = status_word()
        kvp.kvp_compact(dev_bf16(k), dev_bf16(v), dev_i32(exp), T - 1, 0, c, status=st)
        o = kvp.kvp_decode_attn(dev_bf16(q), c, now, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        on = o.cpu().numpy()
        assert (on[0, :G] == 0).all()
        check_attention(on, ref)


# --------------------------------------------------------------------------- chained path

def test_chain_score_mask_compact_attend_tiny(kvp):
    """The tiny workload end to end on the GPU: scores from the scorer, the
    per-head median threshold from the oracle's scores, then mask, compaction and
    attention; near-threshold entries (|s - tau| <= 1e-3) are excluded from the
    mask comparison and the downstream steps take the oracle's keep set."""
    cfg = syn.WORKLOADS["tiny"]
    B, T, H, G, d, D = 1, cfg["n_pos"], cfg["n_kv_heads"], 2, cfg["head_dim"], cfg["d_model"]
    x, w = syn.linear_inputs(0, B * T, D, H)
    k, v = syn.kv_inputs(0, B, T, H, d)
    q = syn.q_inputs(0, B, H * G, d)
    s_ref = orc.score_linear(x, w).reshape(B, T, H)
    tau = orc.threshold_at_quantile(s_ref, 0.5)
    s_gpu = kvp.kvp_score(dev_bf16(x), dev_f32(w))
    exp_g, _, cnt_g = kvp.kvp_mask(mode=kvp.KVP_MASK_KVZAP, batch=B, n_kv_heads=H, n_pos=T, now=T - 1,
                                   scores=s_gpu, tau=dev_f32(tau))
    torch.cuda.synchronize()
    exp_r = orc.mask_kvzap(s_ref, tau, T - 1)[0]
    near = np.abs(s_ref - tau[:, None, :]).transpose(0, 2, 1) <= 1e-3
    assert near.sum() <= 4
    np.testing.assert_array_equal(exp_g.cpu().numpy()[~near], exp_r[~near])
    kept = (T - 1 < exp_r).sum(axis=2)
    assert np.all(np.abs(kept / T - 0.627) < 0.05)  # ~37% pruned: median minus the window's share
    mp = (T + 15) // 16
    ref_c = orc.compact_dense(k, v, exp_r.astype(np.int32), T - 1, 0, B * H * mp, mp)
    c = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp)
    st = status_word()
    kvp.kvp_compact(dev_bf16(k), dev_bf16(v), dev_i32(exp_r), T - 1, 0, c, status=st)
    o = kvp.kvp_decode_attn(dev_bf16(q), c, T - 1, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_cache(c, ref_c)
    check_attention(o.cpu().numpy(), orc.decode_attention(q, ref_c, T - 1))


@pytest.mark.parametrize("G,grid", [(4, 0), (4, 3), (8, 0), (8, 3)])
def test_decode_attn_bad_page_ids(kvp, G, grid):
    """A page id outside [0, n_pages_cap) in the page table records
    KVP_ERR_BOUNDS; that page is read as no slots and everything else as
    usual: the output equals the oracle's with that page's slots expired
    (G = 4: the CUDA-core kernel; G = 8: the tensor-core page math)."""
    B, T, H, d = 2, 1500, 4, 128
    k, v, exp, cnt = _kvzap_case(B, T, H, d, seed=5)
    q = syn.q_inputs(5, B, H * G, d)
    max_pages = (T + 15) // 16
    cap = B * H * max_pages
    now = T - 1
    ref_c = orc.compact_dense(k, v, exp, now, 0, cap, max_pages)
    st = status_word()
    c = kvp.PagedKV.allocate(B, H, d, cap, max_pages)
    kvp.kvp_compact(dev_bf16(k), dev_bf16(v), dev_i32(exp), now, 0, c, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    pt = c.page_table.clone()
    for b, h, j, val in [(0, 1, 3, -9), (1, 0, 0, cap + 7), (1, 3, 5, cap)]:
        assert j * 16 < int(c.count[b, h])
        ref_c.expire_pool[ref_c.page_table[b, h, j]] = 0  # the oracle: every slot of the page gone
        pt[b, h, j] = val
    c_bad = kvp.PagedKV(c.k_pool, c.v_pool, c.expire_pool, pt, c.remap, c.count)
    out = kvp.kvp_decode_attn(dev_bf16(q), c_bad, now, grid_limit=grid, status=st)
    torch.cuda.synchronize()
    assert st.item() == kvp.KVP_ERR_BOUNDS
    check_attention(out.cpu().numpy(), orc.decode_attention(q, ref_c, now))
