"""Pins of the oracle's attention with its log-sum-exp, and of the merge of
attention over disjoint parts ([DMS] "DMS 작동 방식": standard attention over
the kept entries, whose softmax normaliser the log-sum-exp is). CPU only.

- lse against scipy's logsumexp of the brute-force logits of the present
  positions, and the rows against scipy's softmax, with bf16 widened here
  (not by the oracle);
- the merge of the two halves of a sequence equals the whole (an identity
  of the softmax), including a head with no entries in one half and a head
  with none at all;
- the two oracles (C++ and numpy) against each other."""
import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import kvp_synth as syn
import oracle

IMPLS = [oracle.cpp_impl, oracle.numpy_impl]


def _widen(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _inputs(B=2, T=70, H=2, G=2, d=16, seed=11, q_keep=0.5):
    k, v = syn.kv_inputs(seed, B, T, H, d)
    q = syn.q_inputs(seed, B, H * G, d)
    s = syn.normal_f32(seed, 5, (B, T, H))
    tau = oracle.threshold_at_quantile(s, q_keep)
    now = T - 1
    exp = oracle.mask_kvzap(s, tau, now, window=8)[0]
    return k, v, q, exp, now


def _cache(impl, k, v, exp, now):
    B, T, H, _ = k.shape
    mp = (T + 15) // 16 + 1
    return impl.compact_dense(k, v, exp, now, 0, n_pages_cap=B * H * mp, max_pages=mp)


@pytest.mark.parametrize("impl", IMPLS, ids=["cpp", "numpy"])
def test_lse_is_the_log_of_the_softmax_normaliser(impl):
    k, v, q, exp, now = _inputs()
    B, T, H, d = k.shape
    G = q.shape[1] // H
    scale = 1.0 / math.sqrt(d)
    out, lse = impl.decode_attention_lse(q, _cache(impl, k, v, exp, now), now)
    for b in range(B):
        for h in range(H):
            pos = np.nonzero(now < exp[b, h])[0]
            K, V = _widen(k[b, pos, h]), _widen(v[b, pos, h])
            for j in range(h * G, (h + 1) * G):
                logits = K @ _widen(q[b, j]) * scale
                assert lse[b, j] == pytest.approx(logsumexp(logits), rel=1e-13, abs=1e-13)
                np.testing.assert_allclose(out[b, j], softmax(logits) @ V, rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("impl", IMPLS, ids=["cpp", "numpy"])
def test_merge_of_two_halves_is_the_whole(impl):
    k, v, q, exp, now = _inputs(T=96)
    T = k.shape[1]
    exp = exp.copy()
    exp[0, 0, :48] = np.minimum(exp[0, 0, :48], now)  # (0, 0): nothing in the first half
    exp[1, 1, :] = np.minimum(exp[1, 1, :], now)      # (1, 1): nothing at all
    halves = [slice(0, 48), slice(48, T)]
    parts = [impl.decode_attention_lse(q, _cache(impl, k[:, sl], v[:, sl], exp[:, :, sl], now), now) for sl in halves]
    o_m, l_m = impl.merge_attention(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    o_w, l_w = impl.decode_attention_lse(q, _cache(impl, k, v, exp, now), now)
    G = q.shape[1] // k.shape[2]
    assert np.isneginf(parts[0][1][0, :G]).all() and np.isneginf(l_w[1, G:2 * G]).all()
    np.testing.assert_allclose(o_m, o_w, rtol=0, atol=2e-6)  # the parts' rows are float32
    fin = np.isfinite(l_w)
    np.testing.assert_allclose(l_m[fin], l_w[fin], rtol=1e-13, atol=1e-13)
    assert np.array_equal(np.isneginf(l_m), ~fin)
    assert (o_m[1, G:2 * G] == 0).all()
    # a part alone is itself; an all-empty set of parts is zero with lse -inf
    o1, l1 = impl.merge_attention(parts[1][0][None], parts[1][1][None])
    np.testing.assert_allclose(o1, parts[1][0], rtol=0, atol=1e-7)
    o0, l0 = impl.merge_attention(np.zeros((2, 3, 4)), np.full((2, 3), -np.inf))
    assert (o0 == 0).all() and np.isneginf(l0).all()


def test_the_two_oracles_agree_on_lse_and_merge():
    k, v, q, exp, now = _inputs(B=3, T=100, H=2, G=4, d=32, seed=12)
    oc, lc = oracle.cpp_impl.decode_attention_lse(q, _cache(oracle.cpp_impl, k, v, exp, now), now)
    on, ln = oracle.numpy_impl.decode_attention_lse(q, _cache(oracle.numpy_impl, k, v, exp, now), now)
    np.testing.assert_allclose(oc, on, rtol=0, atol=1e-6)
    np.testing.assert_allclose(lc, ln, rtol=1e-13, atol=1e-13)
    outs = np.stack([oc.astype(np.float64), on.astype(np.float64) * 0.5])
    lses = np.stack([lc, ln - 1.0])
    lses[1, 0, 0] = -np.inf
    mc, mlc = oracle.cpp_impl.merge_attention(outs, lses)
    mn, mln = oracle.numpy_impl.merge_attention(outs, lses)
    np.testing.assert_allclose(mc, mn, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(mlc, mln, rtol=1e-13, atol=1e-13)
