"""A decode step captured once as a CUDA graph and replayed for every step
(DeInfer summary, "나. 페이지드 KV 캐시 및 CUDA Graph 통합": fixed-address buffers
so that the step replays as a graph), against the oracle.

The step is: KVzap-Linear score of the new token's hidden state, append of
its K/V under the threshold (kvp_append_devpos), attention of the query rows
over the survivors (kvp_decode_attn_devpos), then the position in device
memory is advanced by one. The per-step inputs are copied into the graph's
fixed input buffers before each replay. Every 32 steps the cache is
recompacted outside the graph into the other pool, and the graph captured on
that pool is replayed from then on. Each step's output is compared with the
oracle's append + attention, and the caches bit-exactly at the end."""
import math

import numpy as np
import pytest
import torch

import kvp_synth as syn
import oracle as orc
from helpers import check_attention, check_scores, compare_paged, dev_bf16, dev_f32, oracle_linear_scores, status_word

pytestmark = pytest.mark.gpu


def test_graph_replayed_decode_step_matches_oracle(kvp):
    B, T0, H, G, d, D, W = 2, 1000, 4, 4, 128, 512, 128
    Hq, steps, every, reserve = H * G, 80, 32, 40
    now0 = T0 - 1
    k, v = syn.kv_inputs(7, B, T0, H, d)
    x0, w = syn.linear_inputs(7, B * T0, D, H)
    xs = syn.normal_bf16(7, 200, (steps, B, D))
    ks = syn.normal_bf16(7, 201, (steps, B, H, d))
    vs = syn.normal_bf16(7, 202, (steps, B, H, d))
    qs = syn.normal_bf16(7, 203, (steps, B, Hq, d))

    # ---- the harness's threshold: each head's 75th-percentile prompt score (oracle), moved by 2e-3 where a
    # new token's oracle score would lie within 1e-3 of it, so that the device scorer's rounding cannot
    # flip a keep decision taken inside the graph
    s_prompt = orc.score_linear(x0, w).reshape(B, T0, H)
    tau = orc.threshold_at_quantile(s_prompt, 0.75)
    s_new, s_new_scale = oracle_linear_scores(xs.reshape(steps * B, D), w)
    s_new = s_new.reshape(steps, B, H)
    for _ in range(100):
        near = np.abs(s_new - tau[None].astype(np.float64)) <= 1e-3
        if not near.any():
            break
        tau = np.where(near.any(axis=0), tau + np.float32(2e-3), tau).astype(np.float32)
    assert not (np.abs(s_new - tau[None].astype(np.float64)) <= 1e-3).any()

    # ---- oracle: prompt compaction (on its fp32 scores), then the steps
    mp = (T0 + steps + reserve + 15) // 16
    cap = B * H * mp
    s32 = s_prompt.astype(np.float32)
    ref = orc.compact_dense(k, v, orc.mask_kvzap(s32, tau, now0)[0], now0, reserve, cap, mp)

    # ---- device: fixed buffers, two pools, the prompt compacted into pool 0
    st = status_word()
    pools = [kvp.PagedKV.allocate(B, H, d, cap, mp) for _ in range(2)]
    wsplit = kvp.kvp_score_split_weight(dev_f32(w))
    tau_d = dev_f32(tau)
    x_buf = torch.zeros((B, D), dtype=torch.bfloat16, device="cuda")
    k_buf = torch.zeros((B, H, d), dtype=torch.bfloat16, device="cuda")
    v_buf = torch.zeros((B, H, d), dtype=torch.bfloat16, device="cuda")
    q_buf = torch.zeros((B, Hq, d), dtype=torch.bfloat16, device="cuda")
    s_buf = torch.zeros((B, H), dtype=torch.float32, device="cuda")
    out = torch.zeros((B, Hq, d), dtype=torch.float32, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws_a = torch.zeros(kvp.kvp_decode_attn_workspace_bytes(B, Hq, H, d), dtype=torch.uint8, device="cuda")
    ws_p = torch.empty(kvp.kvp_compact_paged_workspace_bytes(B, H, mp), dtype=torch.uint8, device="cuda")

    def step(cache, status):
        kvp.kvp_score(x_buf, wsplit, scorer=kvp.KVP_SCORER_LINEAR_SPLIT, n_kv_heads=H, out=s_buf, status=status)
        kvp.kvp_append_devpos(cache, k_buf, v_buf, pos, mode=kvp.KVP_MASK_KVZAP, score=s_buf, tau=tau_d,
                              window=W, status=status)
        kvp.kvp_decode_attn_devpos(q_buf, cache, pos, out=out, workspace=ws_a, status=status)
        pos.add_(1)

    # one eager run of the step on each (still empty) pool sets up the launch paths before any capture; the
    # pools' page tables are -1 then, so the appends record KVP_ERR_CAPACITY in a scratch status word
    scratch = status_word()
    for c in pools:
        pos.fill_(T0)
        step(c, scratch)
    torch.cuda.synchronize()
    assert scratch.item() == kvp.KVP_ERR_CAPACITY
    graphs = []
    for c in pools:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(c, st)
        graphs.append(g)

    kvp.kvp_compact_masked(dev_bf16(k), dev_bf16(v), now0, reserve, pools[0], mode=kvp.KVP_MASK_KVZAP,
                           scores=dev_f32(s32.reshape(B * T0, H)), tau=tau_d, window=W, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    compare_paged(pools[0], ref, what="prompt")

    xs_d, ks_d, vs_d, qs_d = dev_bf16(xs), dev_bf16(ks), dev_bf16(vs), dev_bf16(qs)
    pos.fill_(T0)
    cur = 0
    for i in range(steps):
        t = T0 + i
        if i > 0 and i % every == 0:
            kvp.kvp_compact_paged(pools[cur], t, reserve, pools[1 - cur], status=st, workspace=ws_p)
            cur = 1 - cur
            ref = orc.compact_paged(ref, t, reserve, cap, mp)
        x_buf.copy_(xs_d[i])
        k_buf.copy_(ks_d[i])
        v_buf.copy_(vs_d[i])
        q_buf.copy_(qs_d[i])
        graphs[cur].replay()
        torch.cuda.synchronize()
        assert st.item() == 0, kvp.status_string(st.item())
        check_scores(s_buf.cpu().numpy(), s_new[i], s_new_scale.reshape(steps, B, H)[i])
        orc.append(ref, ks[i], vs[i], t, orc.expire_kvzap(s_new[i], tau, t))
        check_attention(out.cpu().numpy(), orc.decode_attention(qs[i], ref, t))
    assert int(pos.item()) == T0 + steps
    compare_paged(pools[cur], ref, what="after the replays")


def test_devpos_entry_points_read_the_position_and_reject_bad_ones(kvp):
    """The device-position forms equal the host-position forms for the same
    position; a negative position, or one whose expire value would reach
    KVP_EXPIRE_NEVER, records KVP_ERR_INVALID and leaves the cache as it is."""
    B, T, H, G, d = 2, 300, 2, 4, 128
    k, v = syn.kv_inputs(8, B, T, H, d)
    s = syn.normal_f32(8, 21, (B, T, H))
    tau = orc.threshold_at_quantile(s, 0.6)
    exp = orc.mask_kvzap(s, tau, T - 1)[0].astype(np.int32)
    mp = (T + 8 + 15) // 16
    kn, vn = dev_bf16(syn.normal_bf16(8, 30, (B, H, d))), dev_bf16(syn.normal_bf16(8, 31, (B, H, d)))
    sn = dev_f32(syn.normal_f32(8, 32, (B, H)))
    q = dev_bf16(syn.q_inputs(8, B, H * G, d))
    caches = []
    for _ in range(2):
        c = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp)
        st = status_word()
        kvp.kvp_compact(dev_bf16(k), dev_bf16(v), torch.from_numpy(exp).cuda(), T - 1, 8, c, status=st)
        caches.append(c)
    st = status_word()
    kvp.kvp_append(caches[0], kn, vn, T, mode=kvp.KVP_MASK_KVZAP, score=sn, tau=dev_f32(tau), status=st)
    o_host = kvp.kvp_decode_attn(q, caches[0], T, status=st)
    pos = torch.full((1,), T, dtype=torch.int32, device="cuda")
    kvp.kvp_append_devpos(caches[1], kn, vn, pos, mode=kvp.KVP_MASK_KVZAP, score=sn, tau=dev_f32(tau), status=st)
    o_dev = kvp.kvp_decode_attn_devpos(q, caches[1], pos, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(o_host, o_dev)
    for name in ("k_pool", "v_pool", "expire_pool", "page_table", "remap", "count"):
        assert torch.equal(getattr(caches[0], name), getattr(caches[1], name)), name
    before = [getattr(caches[1], n).clone() for n in ("k_pool", "expire_pool", "remap", "count")]
    for bad, delay in ((-1, 0), (2**31 - 1 - 128, 0), (2**31 - 300, 256)):
        st = status_word()
        pos.fill_(bad)
        kvp.kvp_append_devpos(caches[1], kn, vn, pos, mode=kvp.KVP_MASK_DMS,
                              flag_step=torch.zeros(B, H, dtype=torch.int32, device="cuda"), delay=delay, status=st)
        torch.cuda.synchronize()
        assert st.item() == kvp.KVP_ERR_INVALID, (bad, st.item())
    after = [getattr(caches[1], n) for n in ("k_pool", "expire_pool", "remap", "count")]
    for a, b in zip(before, after):
        assert torch.equal(a, b)
