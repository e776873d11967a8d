"""Decode attention with each row's log-sum-exp (kvp_decode_attn_lse) and the
merge of attention over disjoint parts (kvp_attn_merge), against the oracle
([DMS] "DMS 작동 방식": standard attention over the kept entries).

- lse at 1, 2, 4 and 8 query heads per kv head and head_dim 64 / 128 (the
  CUDA-core and the tensor-core kernels; heads that one warp takes whole and
  heads split over warps and merged), an empty head giving -inf; the rows
  bit-identical to kvp_decode_attn's;
- a sequence split into two caches, each attended with its lse, and merged
  on the device: the whole's attention within the attention tolerances;
- the merge kernel alone against the oracle's merge, with empty parts, three
  parts, and the arguments it rejects."""
import numpy as np
import pytest
import torch

import kvp_synth as syn
import oracle as orc
from helpers import check_attention, dev_bf16, dev_f32, status_word

pytestmark = pytest.mark.gpu


def _inputs(B, T, H, G, d, seed, q_keep=0.6):
    k, v = syn.kv_inputs(seed, B, T, H, d)
    q = syn.q_inputs(seed, B, H * G, d)
    s = syn.normal_f32(seed, 5, (B, T, H))
    now = T - 1
    exp = orc.mask_kvzap(s, orc.threshold_at_quantile(s, q_keep), now, window=16)[0].astype(np.int32)
    exp[0, H - 1, :] = np.minimum(exp[0, H - 1, :], now)  # (0, H - 1): no entries
    return k, v, q, exp, now


def _caches(kvp, k, v, exp, now):
    B, T, H, d = k.shape
    mp = (T + 15) // 16
    ref = orc.compact_dense(k, v, exp, now, 0, n_pages_cap=B * H * mp, max_pages=mp)
    c = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp)
    st = status_word()
    kvp.kvp_compact(dev_bf16(k), dev_bf16(v), torch.from_numpy(np.ascontiguousarray(exp)).cuda(), now, 0, c,
                    status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return ref, c


def _check_lse(got, ref):
    got = got.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isneginf(got), ~fin)
    np.testing.assert_allclose(got[fin], ref[fin], rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("B,T,H,G,d", [(2, 3000, 4, 1, 128), (2, 2000, 4, 2, 64), (3, 1777, 3, 4, 128),
                                       (2, 2500, 2, 8, 128), (2, 1500, 4, 8, 64), (1, 40, 2, 4, 128)])
def test_decode_attn_lse_matches_oracle(kvp, B, T, H, G, d):
    k, v, q, exp, now = _inputs(B, T, H, G, d, seed=31 + G + d)
    ref, c = _caches(kvp, k, v, exp, now)
    qd = dev_bf16(q)
    st = status_word()
    out, lse = kvp.kvp_decode_attn_lse(qd, c, now, status=st)
    out_plain = kvp.kvp_decode_attn(qd, c, now, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(out, out_plain)
    o_ref, l_ref = orc.decode_attention_lse(q, ref, now)
    check_attention(out.cpu().numpy(), o_ref)
    _check_lse(lse, l_ref)
    assert np.isneginf(lse[0, (H - 1) * G:].cpu().numpy()).all()


@pytest.mark.parametrize("G,d", [(1, 128), (4, 128), (8, 64)])
def test_sequence_split_into_two_caches_merges_to_the_whole(kvp, G, d):
    B, T, H = 2, 2400, 4
    k, v, q, exp, now = _inputs(B, T, H, G, d, seed=41 + G)
    exp[1, 0, :T // 2] = np.minimum(exp[1, 0, :T // 2], now)  # (1, 0): nothing in the first half
    halves = [slice(0, T // 2), slice(T // 2, T)]
    qd = dev_bf16(q)
    st = status_word()
    outs, lses = [], []
    for sl in halves:
        _, c = _caches(kvp, np.ascontiguousarray(k[:, sl]), np.ascontiguousarray(v[:, sl]),
                       np.ascontiguousarray(exp[:, :, sl]), now)
        o, lse = kvp.kvp_decode_attn_lse(qd, c, now, status=st)
        outs.append(o)
        lses.append(lse)
    out, lse = kvp.kvp_attn_merge(torch.stack(outs), torch.stack(lses))
    torch.cuda.synchronize()
    assert st.item() == 0
    ref, _ = _caches(kvp, k, v, exp, now)
    o_ref, l_ref = orc.decode_attention_lse(q, ref, now)
    check_attention(out.cpu().numpy(), o_ref)
    _check_lse(lse, l_ref)
    assert (out[0, (H - 1) * G:] == 0).all()


def test_attn_merge_matches_the_oracle_merge(kvp):
    P, rows, d = 3, 37, 128
    outs = syn.normal_f32(51, 1, (P, rows, d))
    lses = syn.normal_f32(51, 2, (P, rows)) * 4.0
    lses[0, :5] = -np.inf          # rows 0-4: no slots in part 0
    lses[:, 7] = -np.inf           # row 7: no slots anywhere
    lses[1, 9] = lses[0, 9] + 60   # row 9: part 1 dominates
    out, lse = kvp.kvp_attn_merge(dev_f32(outs), dev_f32(lses))
    o_ref, l_ref = orc.merge_attention(outs, lses)
    torch.cuda.synchronize()
    np.testing.assert_allclose(out.cpu().numpy(), o_ref, rtol=1e-5, atol=1e-6)
    _check_lse(lse, l_ref)
    assert (out[7] == 0).all()
    # one part is itself; d = 4 (one float4 a row); no rows: nothing to do
    o1, l1 = kvp.kvp_attn_merge(dev_f32(outs[:1]), dev_f32(lses[:1]))
    fin = np.isfinite(lses[0])
    np.testing.assert_allclose(o1.cpu().numpy()[fin], outs[0][fin], rtol=1e-6, atol=1e-7)
    o4, _ = kvp.kvp_attn_merge(dev_f32(outs[:, :, :4]), dev_f32(lses))
    np.testing.assert_allclose(o4.cpu().numpy(), orc.merge_attention(outs[:, :, :4], lses)[0], rtol=1e-5, atol=1e-6)
    kvp.kvp_attn_merge(torch.zeros((2, 0, 8), device="cuda"), torch.zeros((2, 0), device="cuda"))
    with pytest.raises(kvp.KvpError):
        kvp.kvp_attn_merge(torch.zeros((2, 3, 6), device="cuda"), torch.zeros((2, 3), device="cuda"))
