"""Device-side failure handling without a GPU fault: the bounded wait that
every kernel puts on its mbarriers gives up, records KVP_ERR_TIMEOUT in the
caller's status word and returns, and the context stays usable.

kvp_selftest_wait makes one warp wait on an mbarrier that nothing arrives on
(a flag that nothing sets), so the wait must run out; nothing traps, faults or
hangs."""

import numpy as np
import pytest
import torch

import kvp_synth as syn
import oracle as orc
from helpers import check_attention, dev_bf16, dev_i32, status_word

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ns", [0, 1_000_000, 20_000_000])
def test_wait_gives_up_records_timeout_and_context_stays_usable(kvp, limit_ns):
    st = status_word()
    waited = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvp.kvp_selftest_wait(limit_ns, status=st, waited_us=waited)
    torch.cuda.synchronize()
    assert st.item() == kvp.KVP_ERR_TIMEOUT
    w = int(waited.item())
    # the wait lasts at least the limit and stops soon after it (the clock is
    # read every 1024 probes of the barrier)
    assert limit_ns // 1000 <= w < limit_ns // 1000 + 200_000, w

    # the context is usable: a small decode attention matches the oracle
    B, T, H, G, d = 1, 700, 2, 4, 128
    k, v = syn.kv_inputs(5, B, T, H, d)
    s = syn.normal_f32(5, 21, (B, T, H))
    tau = syn.normal_f32(5, 22, (B, H), std=0.7)
    exp = orc.mask_kvzap(s, tau, T - 1)[0].astype(np.int32)
    q = syn.q_inputs(5, B, H * G, d)
    mp = (T + 15) // 16
    ref = orc.decode_attention(q, orc.compact_dense(k, v, exp, T - 1, 0, B * H * mp, mp), T - 1)
    st2 = status_word()
    c = kvp.PagedKV.allocate(B, H, d, B * H * mp, mp)
    kvp.kvp_compact(dev_bf16(k), dev_bf16(v), dev_i32(exp), T - 1, 0, c, status=st2)
    o = kvp.kvp_decode_attn(dev_bf16(q), c, T - 1, status=st2)
    torch.cuda.synchronize()
    assert st2.item() == 0
    check_attention(o.cpu().numpy(), ref)
