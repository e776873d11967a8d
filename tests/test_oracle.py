"""Pins for the oracle: each check ties an oracle function to something other
than itself (the pages' printed figures, hand-worked rule timelines, textbook
values, closed forms, invariants, library routines, brute force). CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.stats import norm

import kvp_synth as syn
import oracle

# every pin runs against both implementations of the oracle: the C++ one and the numpy one
IMPLS = {"cpp": oracle.cpp_impl, "numpy": oracle.numpy_impl}


@pytest.fixture(params=sorted(IMPLS))
def orc(request):
    return IMPLS[request.param]

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _exp_list(v):
    return [oracle.NEVER if e == "never" else e for e in v]


def _widen(bits):
    """bf16 bits -> float64 through torch's own bfloat16 type (a library routine)."""
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def _bits(a):
    return syn.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


# --------------------------------------------------------------------------- score

def test_widen_bf16_exact(orc):
    vals = np.array([0.0, 1.0, -2.5, 0.1015625, 3.0e38, -1.0e-38], dtype=np.float32)
    b = _bits(vals)
    back = orc.widen_bf16(b)
    # bf16 keeps the top 16 bits of float32: exact for these, rounded otherwise
    np.testing.assert_array_equal(back[:4], [0.0, 1.0, -2.5, 0.1015625])
    assert orc.widen_bf16(np.array([0x3F80], np.uint16))[0] == 1.0
    assert orc.widen_bf16(np.array([0xC000], np.uint16))[0] == -2.0


def test_score_linear_unit_columns_pick_inputs(orc):
    # W[h] = e_{k_h}: head h must read exactly column k_h of x (catches a transposed W)
    rng = np.random.default_rng(1)
    n, D, H = 37, 48, 5
    x = _bits(rng.standard_normal((n, D)))
    ks = [3, 0, 47, 11, 11]
    W = np.zeros((H, D), np.float32)
    for h, k in enumerate(ks):
        W[h, k] = 1.0
    s = orc.score_linear(x, W)
    xf = orc.widen_bf16(x)
    for h, k in enumerate(ks):
        np.testing.assert_array_equal(s[:, h], xf[:, k])


def test_score_linear_bias_and_full_sum(orc):
    D, H = 64, 3
    x = _bits(np.ones((4, D)))
    W = np.tile(np.arange(D, dtype=np.float32), (H, 1)) * np.array([[1], [2], [-1]], np.float32)
    s = orc.score_linear(x, W, bias=np.array([0.5, 0.0, -3.0]))
    closed = D * (D - 1) / 2  # sum of 0..D-1: every term of the dot product counts
    np.testing.assert_array_equal(s, np.tile([closed + 0.5, 2 * closed, -closed - 3.0], (4, 1)))
    s0 = orc.score_linear(x, np.zeros((H, D), np.float32), bias=np.array([1.0, 2.0, 3.0]))
    np.testing.assert_array_equal(s0, np.tile([1.0, 2.0, 3.0], (4, 1)))


def test_gelu_matches_textbook_phi(orc):
    g = _gold("gelu_phi.json")
    for p in g["points"]:
        assert orc.gelu(np.array(p["u"])) == pytest.approx(p["u"] * p["phi"], abs=1e-15)
    u = np.linspace(-8, 8, 1001)
    np.testing.assert_allclose(orc.gelu(u), u * norm.cdf(u), rtol=0, atol=1e-14)
    big = np.array([30.0, -30.0])
    np.testing.assert_allclose(orc.gelu(big), [30.0, 0.0], atol=1e-12)


def test_score_mlp_selection_weights(orc):
    # W1 row j reads x[:, k_j] scaled by c_j; W2 row h picks hidden unit j_h.
    # Then s[:, h] = GELU(c_{j_h} x[:, k_{j_h}] + b1) + b2 exactly, checked with Phi.
    rng = np.random.default_rng(2)
    n, D, hid, H = 19, 32, 24, 3
    x = _bits(rng.standard_normal((n, D)))
    W1 = np.zeros((hid, D), np.float32)
    ks = rng.integers(0, D, hid)
    cs = np.array([0.5, 1.0, 2.0, -1.0] * (hid // 4), np.float32)
    W1[np.arange(hid), ks] = cs
    W2 = np.zeros((H, hid), np.float32)
    js = [5, 0, 23]
    for h, j in enumerate(js):
        W2[h, j] = 1.0
    b1 = np.linspace(-0.5, 0.5, hid)
    b2 = np.array([0.25, 0.0, -1.0])
    s = orc.score_mlp(x, _bits(W1), _bits(W2), b1=b1, b2=b2)
    xf = orc.widen_bf16(x)
    for h, j in enumerate(js):
        u = cs[j] * xf[:, ks[j]] + b1[j]
        np.testing.assert_allclose(s[:, h], u * norm.cdf(u) + b2[h], rtol=0, atol=1e-13)


def test_score_mlp_sums_hidden_units(orc):
    # all hidden units equal: s = hidden * GELU(u) (catches a dropped hidden term)
    D, hid = 16, 40
    x = _bits(np.full((2, D), 0.25))
    W1 = _bits(np.full((hid, D), 0.125))
    W2 = _bits(np.ones((1, hid)))
    s = orc.score_mlp(x, W1, W2)
    u = D * 0.25 * 0.125
    assert s[0, 0] == pytest.approx(hid * u * norm.cdf(u), abs=1e-13)


# --------------------------------------------------------------------------- mask

def test_kvzap_rule_worked_example(orc):
    g = _gold("mask_rules.json")["kvzap"]
    s = np.array([np.nan if v == "nan" else v for v in g["scores"]], dtype=np.float32)
    T = len(s)
    exp, keep, bits, count = orc.mask_kvzap(s[None, :, None], np.array([[g["tau"]]], np.float32),
                                            g["now"], window=g["window"])
    assert list(exp[0, 0]) == _exp_list(g["expire"])
    assert list(np.nonzero(keep[0, 0])[0]) == g["present"]
    assert count[0, 0] == g["count"]
    assert T == 10
    e = _gold("mask_rules.json")["kvzap_early"]
    _, keep, _, count = orc.mask_kvzap(np.array(e["scores"], np.float32)[None, :, None],
                                       np.array([[e["tau"]]], np.float32), e["now"], window=e["window"])
    assert list(np.nonzero(keep[0, 0])[0]) == e["present"] and count[0, 0] == e["count"]


def test_dms_rule_worked_timeline(orc):
    g = _gold("mask_rules.json")["dms"]
    f = np.array(g["flag_step"])[None, None, :]
    T = f.shape[2]
    for now_s, want in g["timeline"].items():
        now = int(now_s)
        exp, keep, _, _ = orc.mask_dms(f, now, delay=g["delay"], window=g["window"])
        assert list(exp[0, 0]) == _exp_list(g["expire"])
        have = [p for p in range(T) if p <= now and keep[0, 0, p]]
        assert have == want, (now, have, want)


@pytest.mark.parametrize("delay", [1, 129, 256, 300])
def test_dms_delay_present_until_f_plus_d_minus_1(orc, delay):
    # flagged at its own step f (= position): present at f+d-1, gone at f+d when the
    # delay outlasts the window; otherwise the window decides (gone at f+window)
    W = 128
    f = np.array([7, 500, 1000])
    exp = orc.expire_dms(f, f, delay, W)
    for fi, e in zip(f, exp):
        gone = fi + max(delay, W)
        assert e == gone
        assert orc.present(e, gone - 1) and not orc.present(e, gone)
    assert orc.expire_dms(np.array([-1]), np.array([3]), delay, W)[0] == orc.NEVER


def test_mask_keep_all_and_window_only(orc):
    rng = np.random.default_rng(3)
    B, T, H = 2, 700, 3
    s = rng.standard_normal((B, T, H)).astype(np.float32)
    now = T - 1
    _, keep, bits, count = orc.mask_kvzap(s, np.full((B, H), -np.inf, np.float32), now)
    assert (count == T).all() and keep.all()
    _, keep, bits, count = orc.mask_kvzap(np.full((B, T, H), -np.inf, np.float32),
                                          np.zeros((B, H), np.float32), now)
    assert (count == 128).all()
    assert keep[:, :, T - 128:].all() and not keep[:, :, : T - 128].any()
    # fewer than 128 cached tokens: everything is in the window
    _, _, _, count = orc.mask_kvzap(np.full((1, 50, 1), -np.inf, np.float32), np.zeros((1, 1), np.float32), 49)
    assert count[0, 0] == 50


def test_mask_monotone_in_tau_and_popcount(orc):
    rng = np.random.default_rng(4)
    B, T, H = 2, 333, 4
    s = rng.standard_normal((B, T, H)).astype(np.float32)
    prev = None
    for tau in [-3.0, -1.0, 0.0, 0.5, 2.0, 9.0]:
        _, keep, bits, count = orc.mask_kvzap(s, np.full((B, H), tau, np.float32), T - 1)
        pop = np.vectorize(lambda w: bin(int(w)).count("1"))(bits).sum(axis=2)
        np.testing.assert_array_equal(pop, count)
        # bit i of word w is position 32w+i
        for p in [0, 31, 32, 100, T - 1]:
            np.testing.assert_array_equal((bits[:, :, p // 32] >> (p % 32)) & 1, keep[:, :, p])
        if prev is not None:
            assert (count <= prev).all()
        prev = count


def test_threshold_quantile_prunes_expected_share(orc):
    rng = np.random.default_rng(5)
    B, T, H = 1, 512, 2
    s = rng.standard_normal((B, T, H))
    for q in [0.5, 0.75]:
        tau = orc.threshold_at_quantile(s, q)
        above = (s.astype(np.float32) >= tau[:, None, :]).sum(axis=1)
        # distinct scores: exactly T - floor(q (T-1)) are at or above the order statistic
        assert (above == T - math.floor(q * (T - 1))).all()


def test_threshold_quantile_rank_by_brute_force(orc):
    """The threshold is the rank-k element, k = floor(q (T - 1)), with ties and
    special values: brute force over a tiny column counts the scores strictly
    below it (at most k) and at or below it (more than k); NaN ranks last."""
    rng = np.random.default_rng(8)
    B, T, H = 2, 23, 3
    s = rng.integers(-3, 4, size=(B, T, H)).astype(np.float32) * 0.5   # many ties
    s[0, :4, 0] = [np.inf, -np.inf, -0.0, 0.0]
    s[1, :6, 1] = np.nan                                                 # 6 NaN of 23
    for q in [0.0, 0.1, 0.5, 0.77, 0.9, 1.0]:
        k = math.floor(q * (T - 1))
        tau = orc.threshold_at_quantile(s, q)
        for b in range(B):
            for h in range(H):
                col = [float(x) for x in s[b, :, h]]
                num = [x for x in col if x == x]
                t = float(tau[b, h])
                if k >= len(num):
                    assert t != t                    # rank among the NaN: the answer is NaN
                    continue
                assert t in num
                assert sum(1 for x in num if x < t) <= k < sum(1 for x in num if x <= t)


def test_threshold_quantile_special_cases(orc):
    """q = 0 and q = 1 give the column's minimum and maximum, q = 0.5 at odd T
    the median (library routines), with no NaN present."""
    rng = np.random.default_rng(9)
    s = rng.standard_normal((3, 101, 4)).astype(np.float32)
    np.testing.assert_array_equal(orc.threshold_at_quantile(s, 0.0), s.min(axis=1))
    np.testing.assert_array_equal(orc.threshold_at_quantile(s, 1.0), s.max(axis=1))
    np.testing.assert_array_equal(orc.threshold_at_quantile(s, 0.5), np.median(s, axis=1))


def test_threshold_per_head_quantiles_rank_by_brute_force(orc):
    """One quantile per kv head (heads with their own keep rates): each head's
    threshold is that head's rank-floor(q_h (T - 1)) element, counted by brute
    force over the column; heads kept whole (q = 0) and pruned to their last
    element (q = 1) included."""
    rng = np.random.default_rng(10)
    B, T, H = 2, 37, 5
    s = rng.integers(-4, 5, size=(B, T, H)).astype(np.float32) * 0.25
    q = np.array([0.0, 0.3, 0.55, 0.9, 1.0])
    tau = orc.threshold_at_quantile(s, q)
    assert tau.shape == (B, H)
    for b in range(B):
        for h in range(H):
            k = math.floor(q[h] * (T - 1))
            col = sorted(float(x) for x in s[b, :, h])
            t = float(tau[b, h])
            assert sum(1 for x in col if x < t) <= k < sum(1 for x in col if x <= t)


def test_dms_bernoulli_keep_rate(orc):
    # 8x compression: evict bit ~ Bernoulli(7/8) -> outside the delay band ~1/8 kept
    B, H, T = 4, 8, 4096
    ev = syn.bernoulli(0, syn.S_FLAG, (B, H, T), 7 / 8)
    f = np.where(ev, np.arange(T)[None, None, :], -1)
    now = T - 1
    _, keep, _, count = orc.mask_dms(f, now, delay=256)
    old = keep[:, :, : T - 256]
    n = old.size
    rate = old.mean()
    assert abs(rate - 1 / 8) < 5 * math.sqrt(n * (1 / 8) * (7 / 8)) / n
    assert keep[:, :, T - 256:].all()  # within the delay: everything still present


# --------------------------------------------------------------------------- compact

def _toy(B=2, T=300, H=3, d=16, seed=0):
    k = syn.normal_bf16(seed, 5, (B, T, H, d))
    v = syn.normal_bf16(seed, 6, (B, T, H, d))
    return k, v


def test_compact_rows_remap_pages(orc):
    B, T, H, d = 2, 300, 3, 16
    k, v = _toy(B, T, H, d)
    rng = np.random.default_rng(6)
    s = rng.standard_normal((B, T, H)).astype(np.float32)
    tau = np.full((B, H), 0.3, np.float32)
    now = T - 1
    exp, keep, _, count = orc.mask_kvzap(s, tau, now)
    reserve = 5
    maxp = (T + reserve + 15) // 16
    c = orc.compact_dense(k, v, exp, now, reserve, n_pages_cap=B * H * maxp, max_pages=maxp)
    base = 0
    for b in range(B):
        for h in range(H):
            n = int(count[b, h])
            assert c.count[b, h] == n
            r = c.remap[b, h, :n]
            assert (np.diff(r) > 0).all() and (c.remap[b, h, n:] == -1).all()
            np.testing.assert_array_equal(r, np.nonzero(keep[b, h])[0])
            npg = (n + reserve + 15) // 16
            np.testing.assert_array_equal(c.page_table[b, h, :npg], base + np.arange(npg))
            assert (c.page_table[b, h, npg:] == -1).all()
            for j in [0, n // 2, n - 1]:
                pg, row = c.page_table[b, h, j // 16], j % 16
                np.testing.assert_array_equal(c.k_pool[pg, row], k[b, r[j], h])
                np.testing.assert_array_equal(c.v_pool[pg, row], v[b, r[j], h])
                assert c.expire_pool[pg, row] == exp[b, h, r[j]]
            # unused rows of the last pages are zero, expire 0 (never present)
            for j in range(n, npg * 16):
                pg, row = c.page_table[b, h, j // 16], j % 16
                assert c.expire_pool[pg, row] == 0 and not c.k_pool[pg, row].any()
            base += npg
    assert c.pages_used == base


def test_compact_keep_all_is_identity(orc):
    B, T, H, d = 1, 64, 2, 8
    k, v = _toy(B, T, H, d)
    exp = np.full((B, H, T), orc.NEVER)
    c = orc.compact_dense(k, v, exp, T - 1, 0, n_pages_cap=8, max_pages=4)
    for h in range(H):
        np.testing.assert_array_equal(c.remap[h * 0, h, :T], np.arange(T))
        rows = c.k_pool[c.page_table[0, h, :4]].reshape(T, d)
        np.testing.assert_array_equal(rows, k[0, :, h])


def test_compact_capacity_error(orc):
    k, v = _toy(1, 64, 1, 8)
    exp = np.full((1, 1, 64), orc.NEVER)
    with pytest.raises(orc.CapacityError):
        orc.compact_dense(k, v, exp, 63, 0, n_pages_cap=3, max_pages=8)
    with pytest.raises(orc.CapacityError):
        orc.compact_dense(k, v, exp, 63, 1, n_pages_cap=10, max_pages=4)


def test_paged_recompaction_equals_dense_on_same_set(orc):
    # prefill compaction at step 60, then appends of positions 61..120, then a
    # paged re-compaction at 120 == one dense compaction of positions 0..120 at 120
    B, T, H, d = 2, 121, 2, 16
    k, v = _toy(B, T, H, d)
    pos = np.arange(T)[None, None, :]
    f = np.where(syn.bernoulli(1, 8, (B, H, T), 0.875), pos, -1)
    exp = orc.expire_dms(f, pos, delay=40, window=16)
    c1 = orc.compact_dense(k[:, :61], v[:, :61], exp[:, :, :61], 60, reserve=64, n_pages_cap=200, max_pages=20)
    for t in range(61, T):
        orc.append(c1, k[:, t], v[:, t], t, exp[:, :, t])
    c2 = orc.compact_paged(c1, T - 1, reserve=3, n_pages_cap=200, max_pages=20)
    ref = orc.compact_dense(k, v, exp, T - 1, reserve=3, n_pages_cap=200, max_pages=20)
    for name in ["k_pool", "v_pool", "expire_pool", "page_table", "remap", "count", "pages_used"]:
        np.testing.assert_array_equal(getattr(c2, name), getattr(ref, name), err_msg=name)


def test_append_fills_reserved_slots(orc):
    B, T, H, d = 1, 40, 2, 8
    k, v = _toy(B, T, H, d)
    exp = np.full((B, H, T), orc.NEVER)
    exp[0, 1, :10] = 5
    c = orc.compact_dense(k, v, exp, T - 1, reserve=2, n_pages_cap=20, max_pages=4)
    kn = syn.normal_bf16(3, 1, (B, H, d))
    vn = syn.normal_bf16(3, 2, (B, H, d))
    orc.append(c, kn, vn, T, np.array([[orc.NEVER, 77]]))
    assert list(c.count[0]) == [41, 31]
    pg, row = c.slot_rows(0, 1, [30])
    np.testing.assert_array_equal(c.k_pool[pg[0], row[0]], kn[0, 1])
    assert c.expire_pool[pg[0], row[0]] == 77 and c.remap[0, 1, 30] == T
    orc.append(c, kn, vn, T + 1, np.full((1, 2), orc.NEVER))
    with pytest.raises(orc.CapacityError):  # head 0: 40 + 2 reserve = 42 = 3 pages -> 48 slots
        for i in range(10):
            orc.append(c, kn, vn, T + 2 + i, np.full((1, 2), orc.NEVER))


# --------------------------------------------------------------------------- attention

def _sdpa_ref(q_bits, k_bits, v_bits, allowed, scale=None):
    """torch's scaled_dot_product_attention in float64 with a boolean mask over
    the dense cache [B, T, H, d]; an independent library routine."""
    q = torch.from_numpy(_widen(q_bits))          # [B, Hq, d]
    K = torch.from_numpy(_widen(k_bits))          # [B, T, H, d]
    V = torch.from_numpy(_widen(v_bits))
    B, Hq, d = q.shape
    H = K.shape[2]
    g = Hq // H
    K = K.permute(0, 2, 1, 3).repeat_interleave(g, dim=1)  # [B, Hq, T, d]
    V = V.permute(0, 2, 1, 3).repeat_interleave(g, dim=1)
    m = torch.from_numpy(np.asarray(allowed)).repeat_interleave(g, dim=1)[:, :, None, :]  # [B,Hq,1,T]
    o = torch.nn.functional.scaled_dot_product_attention(q[:, :, None, :], K, V, attn_mask=m, scale=scale)
    return o[:, :, 0, :].numpy()


def test_dense_attention_matches_library_sdpa(orc):
    B, T, H, Hq, d = 2, 90, 2, 6, 32
    k, v = _toy(B, T, H, d)
    q = syn.normal_bf16(0, 7, (B, Hq, d))
    now = T - 1
    o = orc.dense_attention(q, k, v, now)
    ref = _sdpa_ref(q, k, v, np.ones((B, H, T), bool))
    np.testing.assert_allclose(o, ref, rtol=1e-6, atol=1e-7)
    ow = orc.window_attention(q, k, v, now, window=20)
    allowed = np.zeros((B, H, T), bool)
    allowed[:, :, T - 20:] = True
    np.testing.assert_allclose(ow, _sdpa_ref(q, k, v, allowed), rtol=1e-6, atol=1e-7)


def test_decode_attention_equals_masked_sdpa(orc):
    # paged pruned attention == library attention over the dense cache with the
    # rule's presence mask (catches any page/slot/remap/GQA indexing slip)
    B, T, H, Hq, d = 2, 333, 2, 8, 64
    k, v = _toy(B, T, H, d)
    q = syn.normal_bf16(0, 7, (B, Hq, d))
    rng = np.random.default_rng(8)
    s = rng.standard_normal((B, T, H)).astype(np.float32)
    now = T - 1
    exp, keep, _, _ = orc.mask_kvzap(s, np.full((B, H), 0.6, np.float32), now)
    c = orc.compact_dense(k, v, exp, now, 7, n_pages_cap=100, max_pages=30)
    o = orc.decode_attention(q, c, now)
    np.testing.assert_allclose(o, _sdpa_ref(q, k, v, keep), rtol=1e-6, atol=1e-7)


def test_decode_attention_special_cases(orc):
    B, T, H, Hq, d = 1, 400, 2, 4, 64
    k, v = _toy(B, T, H, d)
    q = syn.normal_bf16(0, 7, (B, Hq, d))
    now = T - 1
    cap = dict(n_pages_cap=100, max_pages=30)
    # keep-all threshold -> dense attention
    exp, *_ = orc.mask_kvzap(np.zeros((B, T, H), np.float32), np.full((B, H), -np.inf, np.float32), now)
    c = orc.compact_dense(k, v, exp, now, 0, **cap)
    np.testing.assert_allclose(orc.decode_attention(q, c, now), orc.dense_attention(q, k, v, now), rtol=1e-6, atol=1e-7)
    # score -inf everywhere -> last-128 sliding window attention
    exp, *_ = orc.mask_kvzap(np.full((B, T, H), -np.inf, np.float32), np.zeros((B, H), np.float32), now)
    c = orc.compact_dense(k, v, exp, now, 0, **cap)
    np.testing.assert_allclose(orc.decode_attention(q, c, now), orc.window_attention(q, k, v, now), rtol=1e-6, atol=1e-7)
    # q = 0 -> mean of the kept V rows (closed form)
    q0 = np.zeros_like(q)
    o = orc.decode_attention(q0, c, now)
    vm = orc.widen_bf16(v[0, T - 128:, :, :]).mean(axis=0)  # [H, d]
    np.testing.assert_allclose(o[0], np.repeat(vm, Hq // H, axis=0), rtol=1e-6, atol=1e-7)


def test_decode_attention_dominant_key_and_empty(orc):
    d = 16
    k = np.zeros((1, 8, 1, d), np.uint16)
    v = syn.normal_bf16(0, 6, (1, 8, 1, d))
    kf = np.zeros((1, 8, 1, d), np.float32)
    kf[0, 5, 0, 0] = 256.0  # logit 256*q0*scale = 60 above the others
    k = _bits(kf)
    q = _bits(np.concatenate([[60 * 4.0 / 256.0], np.zeros(d - 1)]).reshape(1, 1, d))
    exp = np.full((1, 1, 8), orc.NEVER)
    c = orc.compact_dense(k, v, exp, 7, 0, n_pages_cap=2, max_pages=2)
    o = orc.decode_attention(q, c, 7)
    np.testing.assert_allclose(o[0, 0], orc.widen_bf16(v[0, 5, 0]), rtol=0, atol=1e-20 + 1e-24)
    # nothing present -> zero output
    exp0 = np.zeros((1, 1, 8), np.int64)
    c0 = orc.compact_dense(k, v, exp0, 7, 0, n_pages_cap=2, max_pages=2)
    assert c0.count[0, 0] == 0 and (orc.decode_attention(q, c0, 7) == 0).all()


# --------------------------------------------------------------------------- closed forms

def test_kv_cache_size_matches_page(orc):
    g = _gold("kv_cache_size.json")
    nb = orc.kv_cache_bytes(g["n_layers"], g["d_model"], g["n_tokens"], g["elem_bytes"])
    # 335.54e9 bytes: the page prints the integer part of the decimal-GB figure
    assert 0 <= nb / 1e9 - g["printed_total_gb"] < g["printed_precision_gb"]


def test_scorer_overhead_matches_page(orc):
    g = _gold("scorer_overhead.json")
    m = g["model"]
    proj = orc.linear_projection_macs(m["d_model"], m["n_q_heads"], m["n_kv_heads"], m["head_dim"], m["ffn_hidden"])
    lin = 100.0 * orc.scorer_macs(m["d_model"], m["n_kv_heads"]) / proj
    mlp = 100.0 * orc.scorer_macs(m["d_model"], m["n_kv_heads"], g["mlp_hidden_reading"]) / proj
    assert round(lin, g["linear_printed_digits"]) == g["linear_percent"]
    assert round(mlp, g["mlp_printed_digits"]) == g["mlp_percent"]


# --------------------------------------------------------------------------- fp8 tier

def test_e4m3_table_matches_closed_form_and_torch(orc):
    """All 256 codes: the closed form (1 + m/8) 2^(e-7), subnormals (m/8) 2^-6,
    NaN at 0x7F / 0xFF, against torch's float8_e4m3fn decoding (a library
    routine) and a few textbook values."""
    codes = np.arange(256, dtype=np.uint8)
    mine = orc.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(mine, lib)   # NaN == NaN here
    assert orc.e4m3_decode([0x38])[0] == 1.0 and orc.e4m3_decode([0x7E])[0] == 448.0
    assert orc.e4m3_decode([0x01])[0] == 2.0 ** -9 and orc.e4m3_decode([0x08])[0] == 2.0 ** -6
    assert orc.e4m3_decode([0xB8])[0] == -1.0


def test_e4m3_encode_matches_torch_cast(orc):
    """Round to nearest, ties to even, against torch's float8 cast on values
    up to 464 (above it torch gives NaN, the encoder saturates to 448)."""
    rng = np.random.default_rng(3)
    grid = orc.e4m3_positive_values()[:127]
    mids = (grid[:-1] + grid[1:]) / 2                                   # exact ties
    v = np.concatenate([rng.uniform(-464, 464, 4000), rng.standard_normal(4000) * 0.01,
                        mids, -mids, grid, -grid, [464.0, -464.0, 2.0 ** -10, -2.0 ** -11]]).astype(np.float32)
    mine = orc.e4m3_encode(v)
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(mine, lib)
    np.testing.assert_array_equal(orc.e4m3_encode([500.0, -1e6, np.nan]), [0x7E, 0xFE, 0x7F])


def test_quantize_rows_bounds_and_exact_cases(orc):
    """Per-row scale = amax / 448: the largest element encodes to +-448 exactly;
    every element of the normal range is within half an E4M3 step (2^-4
    relative), the subnormal range within 2^-10 scale; zero rows stay zero;
    rows on the E4M3 grid times a power of two come back exactly."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    bits = syn.f32_to_bf16_bits(x)
    codes, scale = orc.quantize_rows(bits)
    xb = orc.widen_bf16(bits)
    back = orc.dequantize_rows(codes, scale)
    amax_idx = np.abs(xb).argmax(axis=1)
    assert np.all((codes[np.arange(64), amax_idx] & 0x7F) == 0x7E)
    y = np.abs(xb) / scale[:, None]
    normal = y >= 2.0 ** -6
    err = np.abs(back - xb)
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(xb[normal]) * (1 + 1e-6))
    assert np.all(err[~normal] <= 2.0 ** -10 * np.broadcast_to(scale[:, None], err.shape)[~normal] * (1 + 1e-6))
    zc, zs = orc.quantize_rows(np.zeros((2, 64), np.uint16))
    assert (zc == 0).all() and (zs == 0).all()
    grid = orc.e4m3_positive_values()[:127]
    ex = rng.choice(np.concatenate([grid, -grid]), size=(8, 64)) * 2.0 ** 3
    ex[:, 0] = 448.0 * 2.0 ** 3
    eb = syn.f32_to_bf16_bits(ex.astype(np.float32))
    c2, s2 = orc.quantize_rows(eb)
    np.testing.assert_array_equal(s2, np.full(8, 8.0, np.float32))
    np.testing.assert_array_equal(orc.dequantize_rows(c2, s2), ex)


def test_quant_tier_partitions_the_entries(orc):
    """With tau_q <= tau every entry is in exactly one class: kept bf16
    (s >= tau), fp8 tier (tau_q <= s < tau), dropped (s < tau_q or NaN)."""
    rng = np.random.default_rng(6)
    B, T, H = 2, 300, 3
    s = rng.standard_normal((B, T, H))
    s[0, :5, 0] = np.nan
    tau = np.full((B, H), 0.5)
    tq = np.full((B, H), -0.5)
    fp8 = orc.quant_tier_select(s, tau, tq)
    st = s.transpose(0, 2, 1)
    keep = st >= 0.5
    drop = ~(st >= -0.5)
    assert ((keep.astype(int) + fp8.astype(int) + drop.astype(int)) == 1).all()
    assert not fp8[0, 0, :5].any()
    assert not orc.quant_tier_select(s, tau, tau).any()     # tau_q = tau: no fp8 tier


def test_two_tier_attention_reduces_to_known_cases(orc):
    """(1) An empty fp8 tier gives the one-tier attention. (2) tau = +inf and
    tau_q = -inf put every entry in the window (bf16) or, once out of it, in
    the fp8 tier; with rows exactly representable in E4M3 (one element at
    448 x 2^k, the rest on the grid x 2^k) that is dense attention over every
    position, brute force. (3) A step before the window has passed shows no
    fp8 slot at all: the last-128 window attention."""
    rng = np.random.default_rng(7)
    B, T, H, G, d = 1, 300, 2, 2, 64
    grid = orc.e4m3_positive_values()[:127]
    grid = grid[(grid >= 2.0 ** -3) & (grid <= 4.0)]
    def rows():
        r = rng.choice(np.concatenate([grid, -grid]), size=(B, T, H, d)) * 0.25
        r[..., 0] = 448.0 * 0.25 * np.where(rng.random((B, T, H)) < 0.5, 1, -1)
        return syn.f32_to_bf16_bits(r.astype(np.float32))
    k, v = rows(), rows()
    q = syn.f32_to_bf16_bits((rng.standard_normal((B, H * G, d)) * 0.05).astype(np.float32))
    s = rng.standard_normal((B, T, H))
    mp = T // 16 + 2
    now = T - 1
    # (1)
    tau = np.zeros((B, H))
    exp = orc.mask_kvzap(s, tau, now)[0]
    ca = orc.compact_dense(k, v, exp, now, 0, B * H * mp, mp)
    cq = orc.compact_quant_dense(k, v, s, tau, tau, 0, B * H * mp, mp)
    assert cq.count.sum() == 0
    np.testing.assert_array_equal(orc.decode_attention_two_tier(q, ca, cq, now), orc.decode_attention(q, ca, now))
    # (2)
    inf = np.full((B, H), np.inf)
    exp = orc.mask_kvzap(s, inf, now)[0]
    ca = orc.compact_dense(k, v, exp, now, 0, B * H * mp, mp)
    cq = orc.compact_quant_dense(k, v, s, inf, -inf, 0, B * H * mp, mp)
    assert (cq.count == T).all()
    two = orc.decode_attention_two_tier(q, ca, cq, now)
    np.testing.assert_allclose(two, orc.dense_attention(q, k, v, now), rtol=0, atol=1e-6)
    # (3) at a step before any fp8 entry is visible (now < 0 + window)
    early = 100
    exp_e = orc.mask_kvzap(s[:, :early + 1], inf[:, :], early)[0]
    ca_e = orc.compact_dense(k[:, :early + 1], v[:, :early + 1], exp_e, early, 0, B * H * mp, mp)
    cq_e = orc.compact_quant_dense(k[:, :early + 1], v[:, :early + 1], s[:, :early + 1], inf, -inf, 0, B * H * mp, mp)
    np.testing.assert_allclose(orc.decode_attention_two_tier(q, ca_e, cq_e, early),
                               orc.window_attention(q, k, v, early), rtol=0, atol=1e-6)


def test_quant_append_equals_one_compaction(orc):
    """Compacting positions [0, T0) into the fp8 tier and appending T0..T-1
    one at a time gives the same tier (codes, scales, starts, remap, count)
    as one compaction of [0, T) with the same reserve budget."""
    rng = np.random.default_rng(12)
    B, T0, T, H, d = 2, 90, 140, 3, 64
    k = syn.f32_to_bf16_bits(rng.standard_normal((B, T, H, d)).astype(np.float32))
    v = syn.f32_to_bf16_bits(rng.standard_normal((B, T, H, d)).astype(np.float32))
    s = rng.standard_normal((B, T, H))
    tau = np.full((B, H), 0.6)
    tq = np.full((B, H), -0.4)
    mp = 16
    step = orc.compact_quant_dense(k[:, :T0], v[:, :T0], s[:, :T0], tau, tq, 64, B * H * mp, mp)
    for t in range(T0, T):
        orc.append_quant(step, k[:, t], v[:, t], t, s[:, t], tau, tq)
    once = orc.compact_quant_dense(k, v, s, tau, tq, 64, B * H * mp, mp)
    np.testing.assert_array_equal(step.count, once.count)
    for b in range(B):
        for h in range(H):
            n = int(once.count[b, h])
            np.testing.assert_array_equal(step.remap[b, h, :n], once.remap[b, h, :n])
            p1, r1 = step.slot_rows(b, h, np.arange(n))
            p2, r2 = once.slot_rows(b, h, np.arange(n))
            np.testing.assert_array_equal(step.kq_pool[p1, r1], once.kq_pool[p2, r2])
            np.testing.assert_array_equal(step.vq_pool[p1, r1], once.vq_pool[p2, r2])
            np.testing.assert_array_equal(step.kscale[p1, r1], once.kscale[p2, r2])
            np.testing.assert_array_equal(step.start_pool[p1, r1], once.start_pool[p2, r2])
    # the reserve runs out: an error, nothing written
    tight = orc.compact_quant_dense(k[:, :T0], v[:, :T0], s[:, :T0], tau, np.full((B, H), -np.inf), 0, B * H * mp, mp)
    full = tight.count.copy()
    with pytest.raises(orc.CapacityError):
        for t in range(T0, T):
            orc.append_quant(tight, k[:, t], v[:, t], t, s[:, t], tau, np.full((B, H), -np.inf))
    assert (tight.count >= full).all()


def test_dms_fp8_tier_takes_over_where_eviction_was(orc):
    """DMS flags: the fp8 tier holds exactly the flagged entries, each from the
    step its bf16 copy is gone; at every step an entry is in exactly one tier,
    and on rows exactly representable in E4M3 the two-tier attention equals
    dense attention over every position (nothing is dropped any more)."""
    rng = np.random.default_rng(14)
    B, T, H, G, d, delay, W = 1, 260, 2, 2, 64, 40, 16
    grid = orc.e4m3_positive_values()[:127]
    grid = grid[(grid >= 2.0 ** -3) & (grid <= 4.0)]

    def rows():
        r = rng.choice(np.concatenate([grid, -grid]), size=(B, T, H, d)) * 0.25
        r[..., 0] = 448.0 * 0.25
        return syn.f32_to_bf16_bits(r.astype(np.float32))
    k, v = rows(), rows()
    q = syn.f32_to_bf16_bits((rng.standard_normal((B, H * G, d)) * 0.05).astype(np.float32))
    pos = np.arange(T)[None, None, :]
    f = np.where(rng.random((B, H, T)) < 0.875, pos, -1)
    mp = T // 16 + 2
    for now in (120, T - 1):
        exp = orc.mask_dms(f[:, :, :now + 1], now, delay, window=W)[0]
        ca = orc.compact_dense(k[:, :now + 1], v[:, :now + 1], exp, now, 0, B * H * mp, mp)
        cq = orc.compact_quant_dense(k[:, :now + 1], v[:, :now + 1], None, None, None, 0, B * H * mp, mp,
                                     window=W, flag_step_bht=f[:, :, :now + 1], delay=delay)
        assert (cq.count == (f[:, :, :now + 1] >= 0).sum(axis=2)).all()
        in_a = orc.present(exp, now).sum()
        vis_b = sum(int((now >= cq.start_pool[cq.slot_rows(0, h, np.arange(cq.count[0, h]))]).sum()) for h in range(H))
        assert in_a + vis_b == H * (now + 1)
        np.testing.assert_allclose(orc.decode_attention_two_tier(q, ca, cq, now),
                                   orc.dense_attention(q, k, v, now), rtol=0, atol=1e-6)


# --------------------------------------------------------------------------- latent cache (MLA)

def test_mla_absorbed_attention_equals_decompressed_heads(orc):
    """The absorbed form is MLA's decompressed attention. Per head j the keys
    [c_t W_UK_j^T, k_rope_t] and values c_t W_UV_j^T with the query
    [q_nope_j, q_rope_j], by torch's scaled_dot_product_attention in float64
    (a library routine), give the oracle's latent attention of the absorbed
    query [q_nope_j W_UK_j, q_rope_j] followed by W_UV_j, on a pruned latent
    cache. W_UK_j is a random permutation times 1/2, so the absorbed query is
    exactly a bf16 value (the path's input format) and the two sides differ
    only by float64 rounding; W_UV_j is a general matrix."""
    rng = np.random.default_rng(21)
    B, T, Hq, dc, dr, dv = 2, 150, 3, 64, 16, 24
    lat = syn.f32_to_bf16_bits(rng.standard_normal((B, T, dc + dr)).astype(np.float32))
    s = rng.standard_normal((B, T, 1))
    now = T - 1
    exp = orc.mask_kvzap(s, np.full((B, 1), 0.3), now, window=16)[0][:, 0]      # [B, T]
    mp = T // 16 + 2
    cache = orc.compact_latent_dense(lat, exp, now, 0, B * mp, mp)
    w_uk = np.stack([np.eye(dc)[rng.permutation(dc)] * 0.5 for _ in range(Hq)])  # [Hq, dn = dc, dc]
    w_uv = rng.standard_normal((Hq, dv, dc)) / math.sqrt(dc)
    q_nope = orc.widen_bf16(syn.f32_to_bf16_bits(rng.standard_normal((B, Hq, dc)).astype(np.float32)))
    q_rope = orc.widen_bf16(syn.f32_to_bf16_bits(rng.standard_normal((B, Hq, dr)).astype(np.float32)))
    q_abs = np.concatenate([np.einsum("bhn,hnc->bhc", q_nope, w_uk), q_rope], axis=2)
    q_bits = syn.f32_to_bf16_bits(q_abs.astype(np.float32))
    np.testing.assert_array_equal(orc.widen_bf16(q_bits), q_abs)                 # exact in bf16
    scale = 1.0 / math.sqrt(dc + dr)
    got = np.einsum("bhc,hvc->bhv", orc.decode_attention_mla(q_bits, cache, dc, now, scale).astype(np.float64), w_uv)
    L = orc.widen_bf16(lat)
    keep = orc.present(exp, now)
    for b in range(B):
        C = torch.from_numpy(L[b, keep[b]])
        for j in range(Hq):
            kj = torch.cat([C[:, :dc] @ torch.from_numpy(w_uk[j]).T, C[:, dc:]], dim=1)   # decompressed keys
            vj = C[:, :dc] @ torch.from_numpy(w_uv[j]).T                               # decompressed values
            qj = torch.from_numpy(np.concatenate([q_nope[b, j], q_rope[b, j]]))
            ref = torch.nn.functional.scaled_dot_product_attention(qj[None, None, None], kj[None, None],
                                                                   vj[None, None], scale=scale)[0, 0, 0].numpy()
            np.testing.assert_allclose(got[b, j], ref, rtol=2e-6, atol=1e-7)


def test_mla_latent_pruning_special_cases(orc):
    """Keep-all reduces to dense latent attention (brute force over every
    position); a score of -inf keeps exactly the last-window rows; the page
    layout is section 3's with one kv head."""
    rng = np.random.default_rng(22)
    B, T, Hq, dc, dr = 1, 200, 4, 32, 8
    lat = syn.f32_to_bf16_bits(rng.standard_normal((B, T, dc + dr)).astype(np.float32))
    q = syn.f32_to_bf16_bits((rng.standard_normal((B, Hq, dc + dr)) * 0.3).astype(np.float32))
    now = T - 1
    mp = T // 16 + 2
    L = orc.widen_bf16(lat)
    qf = orc.widen_bf16(q)
    scale = 1.0 / math.sqrt(dc + dr)

    def brute(lo):
        out = np.zeros((B, Hq, dc))
        for j in range(Hq):
            C = L[0, lo:now + 1]
            w = np.exp((C @ qf[0, j]) * scale - ((C @ qf[0, j]) * scale).max())
            out[0, j] = (w @ C[:, :dc]) / w.sum()
        return out
    keep_all = np.full((B, T), orc.NEVER)
    c = orc.compact_latent_dense(lat, keep_all, now, 0, B * mp, mp)
    np.testing.assert_allclose(orc.decode_attention_mla(q, c, dc, now), brute(0), rtol=0, atol=1e-6)
    s = np.full((B, T, 1), -np.inf)
    exp = orc.mask_kvzap(s, np.zeros((B, 1)), now, window=40)[0][:, 0]
    c = orc.compact_latent_dense(lat, exp, now, 0, B * mp, mp)
    assert int(c.count[0, 0]) == 40
    np.testing.assert_array_equal(c.remap[0, 0, :40], np.arange(T - 40, T))
    np.testing.assert_allclose(orc.decode_attention_mla(q, c, dc, now), brute(T - 40), rtol=0, atol=1e-6)


def test_mla_attention_closed_forms(orc):
    """Closed forms of the latent attention: q = 0 weighs every present row the
    same (the mean of their compressed parts); a row whose logit is 60 above
    every other one takes all the weight (its compressed part, to e^-60); a
    row that has expired by `now` takes none."""
    rng = np.random.default_rng(23)
    B, T, dc, dr = 1, 120, 32, 8
    lat = syn.f32_to_bf16_bits(rng.standard_normal((B, T, dc + dr)).astype(np.float32))
    now = T - 1
    mp = T // 16 + 2
    exp = np.full((B, T), orc.NEVER)
    exp[0, 10:30] = now          # gone at `now`: never present
    cache = orc.compact_latent_dense(lat, exp, now, 0, B * mp, mp)
    L = orc.widen_bf16(lat)[0]
    keep = np.ones(T, bool)
    keep[10:30] = False
    q0 = np.zeros((B, 1, dc + dr), np.uint16)
    np.testing.assert_allclose(orc.decode_attention_mla(q0, cache, dc, now)[0, 0], L[keep, :dc].mean(axis=0),
                               rtol=0, atol=1e-6)
    # a query along row 50's direction, scaled so its logit leads by more than 60
    j = 50
    u = L[j] / np.linalg.norm(L[j])
    others = np.delete(L[keep], np.flatnonzero(np.flatnonzero(keep) == j), axis=0)
    gap = np.linalg.norm(L[j]) - (others @ u).max()
    assert gap > 0
    q = syn.f32_to_bf16_bits((u * (64.0 / gap) * math.sqrt(dc + dr)).astype(np.float32))[None, None]
    qf = orc.widen_bf16(q)[0, 0]
    logits = (L[keep] @ qf) / math.sqrt(dc + dr)
    assert np.sort(logits)[-1] - np.sort(logits)[-2] > 60
    np.testing.assert_allclose(orc.decode_attention_mla(q, cache, dc, now)[0, 0], L[j, :dc], rtol=1e-6, atol=1e-20)


def test_mla_attention_empty_batch_element(orc):
    """A batch element with no present latent row gives a zero row of the
    compressed width (dc values, not the row's dc + dr); the others are
    unaffected."""
    rng = np.random.default_rng(24)
    B, T, Hq, dc, dr = 2, 40, 3, 16, 8
    lat = syn.f32_to_bf16_bits(rng.standard_normal((B, T, dc + dr)).astype(np.float32))
    q = syn.f32_to_bf16_bits(rng.standard_normal((B, Hq, dc + dr)).astype(np.float32))
    exp = np.full((B, T), orc.NEVER)
    exp[1] = 0
    now = T - 1
    c = orc.compact_latent_dense(lat, exp, now, 0, B * 4, 4)
    o = orc.decode_attention_mla(q, c, dc, now)
    assert o.shape == (B, Hq, dc)
    assert (o[1] == 0).all()
    alone = orc.decode_attention_mla(q[:1], orc.compact_latent_dense(lat[:1], exp[:1], now, 0, 4, 4), dc, now)
    np.testing.assert_array_equal(o[0], alone[0])
