"""GPU parity of the MLA latent-cache path (DMS article, "주요 요점" and "앞으로의
전망": the method over Multi-Head Latent Attention's single latent cache)
against the oracle's section 6: latent compaction, append and re-compaction
bit-exact, absorbed decode attention within the attention tolerances.

Every test here has passed on a GB300."""

import numpy as np
import pytest
import torch

import kvp_synth as syn
import oracle as orc
from helpers import check_attention, dev_bf16, dev_f32, dev_i32, host_bits, status_word

pytestmark = pytest.mark.gpu

DC, DR = 512, 64
ROW = DC + DR


def _compare_latent(gpu, ref: orc.PagedCache):
    np.testing.assert_array_equal(gpu.count.cpu().numpy(), ref.count[:, 0], err_msg="count")
    np.testing.assert_array_equal(gpu.page_table.cpu().numpy(), ref.page_table[:, 0], err_msg="page_table")
    np.testing.assert_array_equal(gpu.remap.cpu().numpy(), ref.remap[:, 0], err_msg="remap")
    used = ref.pages_used
    np.testing.assert_array_equal(gpu.expire_pool.cpu().numpy()[:used], ref.expire_pool[:used], err_msg="expire")
    np.testing.assert_array_equal(host_bits(gpu.pool)[:used], ref.k_pool[:used], err_msg="pool")


def _kvzap_latent(B, T, seed, tau_std=0.7, window=128):
    lat = syn.latent_inputs(seed, B, T, ROW)
    s = syn.normal_f32(seed, 51, (B, T, 1))
    tau = syn.normal_f32(seed, 52, (B, 1), std=tau_std)
    exp = orc.mask_kvzap(s, tau, T - 1, window=window)[0][:, 0].astype(np.int32)   # [B, T]
    return lat, s, tau, exp


@pytest.mark.parametrize("B,T,reserve,window,strided", [
    (1, 512, 0, 128, False),
    (2, 3000, 5, 128, True),     # ragged, several segments, rows 640 values apart
    (3, 17, 16, 8, False),       # tiny ragged, a reserved full page
    (5, 1030, 64, 32, False),
])
def test_compact_latent_kvzap_bit_exact(kvp, B, T, reserve, window, strided):
    lat, s, tau, exp = _kvzap_latent(B, T, seed=31, window=window)
    mp = (T + reserve + 15) // 16
    cap = B * mp
    now = T - 1
    ref = orc.compact_latent_dense(lat, exp, now, reserve, cap, mp)
    src = dev_bf16(lat)
    if strided:
        wide = torch.zeros((B, T, ROW + 64), dtype=torch.bfloat16, device="cuda")
        wide[:, :, :ROW] = src
        src = wide[:, :, :ROW]
    st = status_word()
    dst = kvp.LatentPagedKV.allocate(B, cap, mp)
    kvp.kvp_compact_latent(src, now, reserve, dst, mode=kvp.KVP_MASK_KVZAP, scores=dev_f32(s[:, :, 0]),
                           tau=dev_f32(tau[:, 0]), window=window, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_latent(dst, ref)


@pytest.mark.parametrize("delay,window", [(256, 128), (40, 100)])
def test_compact_latent_dms_bit_exact(kvp, delay, window):
    B, T = 3, 2100
    lat = syn.latent_inputs(33, B, T, ROW)
    pos = np.arange(T)[None, :]
    f = np.where(syn.bernoulli(33, 8, (B, T), 0.875), pos, -1).astype(np.int32)
    exp = orc.expire_dms(f, pos, delay, window).astype(np.int32)
    now = T - 1
    mp = (T + 15) // 16
    ref = orc.compact_latent_dense(lat, exp, now, 0, B * mp, mp)
    st = status_word()
    dst = kvp.LatentPagedKV.allocate(B, B * mp, mp)
    kvp.kvp_compact_latent(dev_bf16(lat), now, 0, dst, mode=kvp.KVP_MASK_DMS, flag_step=dev_i32(f), delay=delay,
                           window=window, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_latent(dst, ref)


def test_latent_append_then_paged_recompaction(kvp):
    """Prefill compaction, appends of the next tokens (DMS flags), then a paged
    re-compaction: bit-exact against the oracle at every stage."""
    B, T0, steps = 3, 700, 90
    delay, window, reserve = 60, 32, 96
    T = T0 + steps
    lat = syn.latent_inputs(35, B, T, ROW)
    pos = np.arange(T)[None, :]
    f = np.where(syn.bernoulli(35, 8, (B, T), 0.875), pos, -1).astype(np.int32)
    exp = orc.expire_dms(f, pos, delay, window).astype(np.int32)
    mp = (T + reserve + 15) // 16
    cap = B * mp
    now0 = T0 - 1
    ref = orc.compact_latent_dense(lat[:, :T0], exp[:, :T0], now0, reserve, cap, mp)
    st = status_word()
    c = kvp.LatentPagedKV.allocate(B, cap, mp)
    kvp.kvp_compact_latent(dev_bf16(lat[:, :T0].copy()), now0, reserve, c, mode=kvp.KVP_MASK_DMS,
                           flag_step=dev_i32(f[:, :T0].copy()), delay=delay, window=window, status=st)
    ld, fd = dev_bf16(lat), dev_i32(f)
    for t in range(T0, T):
        orc.append(ref, lat[:, t][:, None, :], lat[:, t][:, None, :], t, exp[:, t][:, None])
        kvp.kvp_append_latent(c, ld[:, t].contiguous(), t, mode=kvp.KVP_MASK_DMS, flag_step=fd[:, t].contiguous(),
                              delay=delay, window=window, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_latent(c, ref)
    now = T - 1
    ref2 = orc.compact_paged(ref, now, 16, cap, mp)
    c2 = kvp.LatentPagedKV.allocate(B, cap, mp)
    kvp.kvp_compact_latent_paged(c, now, 16, c2, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_latent(c2, ref2)


def test_latent_append_kvzap_and_reserve_exhausted(kvp):
    B, T = 2, 100
    lat = syn.latent_inputs(36, B, T + 20, ROW)
    exp = np.full((B, T), orc.NEVER, np.int32)
    reserve, mp = 12, 8   # 100 + 12 = 112 slots = 7 pages exactly
    ref = orc.compact_latent_dense(lat[:, :T], exp, T - 1, reserve, 64, mp)
    st = status_word()
    c = kvp.LatentPagedKV.allocate(B, 64, mp)
    kvp.kvp_compact_latent(dev_bf16(lat[:, :T].copy()), T - 1, reserve, c, mode=kvp.KVP_MASK_KVZAP,
                           scores=dev_f32(np.zeros((B, T), np.float32)), tau=dev_f32(np.zeros(B, np.float32)),
                           status=st)
    score = syn.normal_f32(36, 30, (12, B))
    tau = np.zeros(B, np.float32)
    for i in range(12):
        t = T + i
        orc.append(ref, lat[:, t][:, None, :], lat[:, t][:, None, :], t,
                   orc.expire_kvzap(score[i], tau, t, 128)[:, None])
        kvp.kvp_append_latent(c, dev_bf16(lat[:, t].copy()), t, mode=kvp.KVP_MASK_KVZAP, score=dev_f32(score[i]),
                              tau=dev_f32(tau), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _compare_latent(c, ref)
    kvp.kvp_append_latent(c, dev_bf16(lat[:, T].copy()), T + 12, mode=kvp.KVP_MASK_KVZAP, score=dev_f32(score[0]),
                          tau=dev_f32(tau), status=st)
    torch.cuda.synchronize()
    assert st.item() == kvp.KVP_ERR_CAPACITY
    np.testing.assert_array_equal(c.count.cpu().numpy(), ref.count[:, 0])  # unchanged


# --------------------------------------------------------------------------- attention

def _mla_case(kvp, B, T, Hq, n_splits=0, seed=37, tau_std=0.7, peaked=False, q_zero=False, workspace=None):
    lat, s, tau, exp = _kvzap_latent(B, T, seed, tau_std=tau_std)
    q = syn.q_inputs(seed, B, Hq, ROW)
    if q_zero:
        q = np.zeros_like(q)
    if peaked:  # query x 8 and 16 planted rows equal to head 0's query: a sharp softmax
        qf = orc.widen_bf16(q) * 8.0
        q = syn.f32_to_bf16_bits(qf.astype(np.float32))
        lat, s = lat.copy(), s.copy()
        for i in range(16):
            t = (i * 97 + 11) % T
            s[:, t, 0] = np.float32(1e30)   # kept for good, on both sides
            lat[:, t, :] = syn.f32_to_bf16_bits((qf[:, 0, :] / 8.0).astype(np.float32))
        exp = orc.mask_kvzap(s, tau, T - 1)[0][:, 0].astype(np.int32)
    mp = (T + 15) // 16
    now = T - 1
    ref_c = orc.compact_latent_dense(lat, exp, now, 0, B * mp, mp)
    ref = orc.decode_attention_mla(q, ref_c, DC, now)
    st = status_word()
    c = kvp.LatentPagedKV.allocate(B, B * mp, mp)
    kvp.kvp_compact_latent(dev_bf16(lat), now, 0, c, mode=kvp.KVP_MASK_KVZAP, scores=dev_f32(s[:, :, 0]),
                           tau=dev_f32(tau[:, 0]), status=st)
    out = kvp.kvp_decode_attn_mla(dev_bf16(q), c, now, n_splits=n_splits, workspace=workspace, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return out.cpu().numpy(), ref, c, q, now


@pytest.mark.parametrize("B,T,Hq,n_splits", [
    (1, 512, 16, 0),
    (2, 2000, 16, 3),
    (3, 1500, 20, 0),      # a ragged head tile (heads 16..19 of a second tile)
    (1, 3000, 128, 2),     # DeepSeek-V3's 128 heads: one 128-head tile, four CTAs (output quarters) per slice
    (2, 700, 1, 1),        # one head, one slice: the output is written without a merge
    (4, 300, 16, 64),      # more slices than pages: empty slices are skipped by the merge
    (2, 4100, 32, 0),
    (1, 2000, 40, 3),      # 64-head tiles from 33 heads: five of the eight warps have heads
    (2, 1100, 72, 0),      # tensor-core kernel with rows 72..127 of its tile empty; many slices of 1-2 pages
    (1, 5000, 100, 1),     # one slice: the output written without a merge, 105 blocks through the ring
    (2, 900, 136, 0),      # two 128-head tiles, the second with 8 heads
])
def test_decode_attn_mla(kvp, B, T, Hq, n_splits):
    o, ref, *_ = _mla_case(kvp, B, T, Hq, n_splits)
    check_attention(o, ref)
    if Hq < TC_FROM:
        # mma.sync paths: bf16 products are exact in fp32 and p enters as a
        # hi + lo pair (about 2^-16 relative): the outputs, weighted means of
        # N(0,1) values, stay well inside 1e-4
        np.testing.assert_allclose(o, ref, rtol=0, atol=1e-4)
    else:
        check_bf16_p_bound(o, ref, syn.latent_inputs(37, B, T, ROW))


# From this many query heads on, the tcgen05 kernel runs; it rounds each
# softmax weight p to bf16 once (no lo part) and sums the rounded values.
TC_FROM = 65


def check_bf16_p_bound(o, ref, lat):
    """The product takes p_j (1 + d_j), |d_j| <= u = 2^-9 (one bf16 rounding,
    plus a margin for the fp32 logits and exponential), and the normaliser the
    unrounded sum of p: o_hat - o = sum_j w_j d_j v_j, so |o_hat - o| <=
    u * max_j |v_j| over the batch element's rows (all of them: a superset
    of the kept ones)."""
    u = 2.0 ** -9 + 2.0 ** -20
    vmax = np.abs(orc.widen_bf16(lat)[:, :, :DC]).max(axis=1)          # [B, DC]
    bound = u * vmax[:, None, :] + 1e-5
    err = np.abs(o - ref)
    assert (err <= bound).all(), (err.max(), float((err / bound).max()))


@pytest.mark.parametrize("Hq", [16, 48])
def test_decode_attn_mla_peaked(kvp, Hq):
    o, ref, *_ = _mla_case(kvp, 2, 1500, Hq, peaked=True)
    check_attention(o, ref)


def test_decode_attn_mla_zero_query_is_the_mean(kvp):
    """q = 0: every present row weighs the same, so each head's output is the
    mean of the kept rows' compressed values (closed form)."""
    o, _, c, _, now = _mla_case(kvp, 2, 900, 16, q_zero=True)
    pool = orc.widen_bf16(host_bits(c.pool))
    ep = c.expire_pool.cpu().numpy()
    pt = c.page_table.cpu().numpy()
    cnt = c.count.cpu().numpy()
    for b in range(2):
        j = np.arange(cnt[b])
        pg, r = pt[b, j // 16], j % 16
        keep = ep[pg, r] > now
        mean = pool[pg[keep], r[keep], :DC].mean(axis=0)
        np.testing.assert_allclose(o[b], np.broadcast_to(mean, (16, DC)), rtol=0, atol=2e-5)


def test_decode_attn_mla_split_independent(kvp):
    outs = [_mla_case(kvp, 2, 2500, 16, n_splits=n)[0] for n in (1, 2, 7, 0)]
    for o in outs[1:]:
        np.testing.assert_allclose(o, outs[0], rtol=0, atol=1e-5)


@pytest.mark.parametrize("Hq", [32, 72])
def test_decode_attn_mla_workspace_reused(kvp, Hq):
    """One workspace serves consecutive calls on different caches without any
    clearing (it starts full of garbage here): each result equals a fresh
    workspace's."""
    B, T, ns = 2, 1800, 5
    ws = torch.full((kvp.kvp_decode_attn_mla_workspace_bytes(B, Hq, ns),), 0x7F, dtype=torch.uint8, device="cuda")
    for seed in (41, 42, 43):
        o, _, c, q, now = _mla_case(kvp, B, T, Hq, n_splits=ns, seed=seed, workspace=ws)
        fresh = kvp.kvp_decode_attn_mla(dev_bf16(q), c, now, n_splits=ns)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(o, fresh.cpu().numpy())


@pytest.mark.parametrize("Hq", [16, 128])
def test_decode_attn_mla_empty_batch_element(kvp, Hq):
    """A batch element with no slots gives zero rows; the others are unchanged."""
    B, T = 3, 600
    lat, s, tau, exp = _kvzap_latent(B, T, seed=45, window=0)
    exp[1, :] = 0          # nothing of batch element 1 is present (score -inf, no window)
    q = syn.q_inputs(45, B, Hq, ROW)
    mp = (T + 15) // 16
    now = T - 1
    ref = orc.decode_attention_mla(q, orc.compact_latent_dense(lat, exp, now, 0, B * mp, mp), DC, now)
    st = status_word()
    c = kvp.LatentPagedKV.allocate(B, B * mp, mp)
    kvp.kvp_compact_latent(dev_bf16(lat), now, 0, c, mode=kvp.KVP_MASK_KVZAP,
                           scores=dev_f32(np.where(np.arange(B)[:, None] == 1, -np.inf, s[:, :, 0])
                                          .astype(np.float32)),
                           tau=dev_f32(tau[:, 0]), window=0, status=st)
    torch.cuda.synchronize()
    assert int(c.count[1]) == 0
    for ns in (1, 4):
        out = kvp.kvp_decode_attn_mla(dev_bf16(q), c, now, n_splits=ns, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        o = out.cpu().numpy()
        assert (o[1] == 0).all()
        check_attention(o[[0, 2]], ref[[0, 2]])


@pytest.mark.parametrize("Hq", [16, 128])
def test_mla_decode_loop(kvp, Hq):
    """DMS decode loop on a latent cache: per step the new row is appended and
    attention runs; every 24 steps the cache is re-compacted. Each step's
    output matches the oracle's (16 heads: the mma.sync kernel; 128: the
    tensor-core kernel, also within its bf16-weight bound)."""
    B, T0, steps = 2, 400, 60
    delay, window, reserve = 48, 32, 64
    T = T0 + steps
    lat = syn.latent_inputs(47, B, T, ROW)
    pos = np.arange(T)[None, :]
    f = np.where(syn.bernoulli(47, 8, (B, T), 0.875), pos, -1).astype(np.int32)
    exp = orc.expire_dms(f, pos, delay, window).astype(np.int32)
    mp = (T + reserve + 15) // 16
    cap = B * mp
    ref = orc.compact_latent_dense(lat[:, :T0], exp[:, :T0], T0 - 1, reserve, cap, mp)
    st = status_word()
    c = kvp.LatentPagedKV.allocate(B, cap, mp)
    kvp.kvp_compact_latent(dev_bf16(lat[:, :T0].copy()), T0 - 1, reserve, c, mode=kvp.KVP_MASK_DMS,
                           flag_step=dev_i32(f[:, :T0].copy()), delay=delay, window=window, status=st)
    ld, fd = dev_bf16(lat), dev_i32(f)
    ws = torch.zeros(kvp.kvp_decode_attn_mla_workspace_bytes(B, Hq, 0), dtype=torch.uint8, device="cuda")
    for i, t in enumerate(range(T0, T)):
        if i and i % 24 == 0:
            ref = orc.compact_paged(ref, t - 1, reserve, cap, mp)
            c2 = kvp.LatentPagedKV.allocate(B, cap, mp)
            kvp.kvp_compact_latent_paged(c, t - 1, reserve, c2, status=st)
            c = c2
        orc.append(ref, lat[:, t][:, None, :], lat[:, t][:, None, :], t, exp[:, t][:, None])
        kvp.kvp_append_latent(c, ld[:, t].contiguous(), t, mode=kvp.KVP_MASK_DMS, flag_step=fd[:, t].contiguous(),
                              delay=delay, window=window, status=st)
        q = syn.q_inputs(47, B, Hq, ROW, stream=syn.step_stream(i, 3))
        o = kvp.kvp_decode_attn_mla(dev_bf16(q), c, t, workspace=ws, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        ref_o = orc.decode_attention_mla(q, ref, DC, t)
        check_attention(o.cpu().numpy(), ref_o)
        if Hq >= TC_FROM:
            check_bf16_p_bound(o.cpu().numpy(), ref_o, lat)

@pytest.mark.parametrize("Hq,n_splits", [(16, 0), (16, 3), (40, 3), (128, 0), (128, 3)])
def test_decode_attn_mla_bad_page_ids(kvp, Hq, n_splits):
    """A page id outside [0, n_pages_cap) in the page table records
    KVP_ERR_BOUNDS; that page is read as no slots, the rest as usual (the
    oracle with the page's slots expired)."""
    B, T = 2, 1500
    _, _, c, q, now = _mla_case(kvp, B, T, Hq, n_splits)
    lat, s, tau, exp = _kvzap_latent(B, T, 37)
    mp = (T + 15) // 16
    ref_c = orc.compact_latent_dense(lat, exp, now, 0, B * mp, mp)
    pt = c.page_table.clone()
    cap = c.pool.shape[0]
    for b, j, val in [(0, 2, -7), (1, 0, cap + 100), (1, 40, cap)]:
        assert j * 16 < int(c.count[b])
        ref_c.expire_pool[ref_c.page_table[b, 0, j]] = 0  # the oracle: every slot of the page gone
        pt[b, j] = val
    c_bad = kvp.LatentPagedKV(c.pool, c.expire_pool, pt, c.remap, c.count)
    st = status_word()
    out = kvp.kvp_decode_attn_mla(dev_bf16(q), c_bad, now, n_splits=n_splits, status=st)
    torch.cuda.synchronize()
    assert st.item() == kvp.KVP_ERR_BOUNDS
    ref = orc.decode_attention_mla(q, ref_c, DC, now)
    o = out.cpu().numpy()
    check_attention(o, ref)
    if Hq >= TC_FROM:
        check_bf16_p_bound(o, ref, lat)
    else:
        np.testing.assert_allclose(o, ref, rtol=0, atol=1e-4)
