"""Guard bands around every output and workspace (a substitute for a memory
checker): each buffer a call writes sits between two 4 KiB bands of a
sentinel byte, workspaces are exactly the size the library asks for, and
after the calls every band must be intact and every status word zero."""
import math

import numpy as np
import pytest
import torch

import kvp_synth as syn
import oracle as orc
from helpers import dev_bf16, dev_f32, dev_i32, status_word

pytestmark = pytest.mark.gpu

GUARD = 4096
SENTINEL = 0x5A


class Guarded:
    """A device tensor of `shape` and `dtype` between two sentinel bands."""

    bands = []

    def __init__(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((GUARD + n + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(shape)
        if fill is not None:
            self.t.fill_(fill)
        Guarded.bands.append(self)

    def intact(self):
        return bool((self.raw[:GUARD] == SENTINEL).all()) and bool((self.raw[-GUARD:] == SENTINEL).all())


def g(shape, dtype, fill=None):
    return Guarded(shape, dtype, fill).t


def ws(nbytes, zero=False):
    return g((max(int(nbytes), 16),), torch.uint8, 0 if zero else None)


def paged(kvp, B, H, d, cap, mp):
    return kvp.PagedKV(g((cap, 16, d), torch.bfloat16, 0), g((cap, 16, d), torch.bfloat16, 0),
                       g((cap, 16), torch.int32, 0), g((B, H, mp), torch.int32, -1),
                       g((B, H, mp * 16), torch.int32, -1), g((B, H), torch.int32, 0))


def check_bands():
    bad = [i for i, b in enumerate(Guarded.bands) if not b.intact()]
    Guarded.bands = []
    assert not bad, f"guard bands overwritten: buffers {bad}"


@pytest.fixture(autouse=True)
def _fresh_bands():
    """Every test starts with no guarded buffers and drops its own at the end,
    even when it fails before check_bands(): a failure is never blamed on the
    next test, and no device memory is held across tests."""
    Guarded.bands = []
    yield
    Guarded.bands = []


def test_canaries_decode_path(kvp):
    B, T, H, G, d, D, reserve = 2, 1000, 2, 4, 128, 256, 24
    n_tok = B * T
    x, w = syn.linear_inputs(3, n_tok, D, H)
    k, v = syn.kv_inputs(3, B, T + 8, H, d)
    q = syn.q_inputs(3, B, H * G, d)
    st = status_word()
    xd = dev_bf16(x)
    s = g((n_tok, H), torch.float32)
    kvp.kvp_score(xd, dev_f32(w), out=s, workspace=ws(kvp.kvp_score_workspace_bytes(kvp.KVP_SCORER_LINEAR, n_tok, D,
                                                                                   H)), status=st)
    tau = g((B, H), torch.float32)
    kvp.kvp_threshold(s.view(B, T, H), 0.75, out=tau, workspace=ws(kvp.kvp_threshold_workspace_bytes(B, H)))
    expire, bits, cnt = g((B, H, T), torch.int32), g((B, H, (T + 31) // 32), torch.int32), g((B, H), torch.int32)
    kvp.kvp_mask(mode=kvp.KVP_MASK_KVZAP, batch=B, n_kv_heads=H, n_pos=T, now=T - 1, scores=s, tau=tau,
                 expire=expire, keep_bits=bits, count=cnt)
    mp = (T + 8 + reserve + 15) // 16
    cap = B * H * mp
    kd, vd = dev_bf16(k[:, :T].copy()), dev_bf16(v[:, :T].copy())
    c = paged(kvp, B, H, d, cap, mp)
    kvp.kvp_compact(kd, vd, expire, T - 1, reserve, c, status=st,
                    workspace=ws(kvp.kvp_compact_workspace_bytes(B, H, T)))
    c2 = paged(kvp, B, H, d, cap, mp)
    kvp.kvp_compact_masked(kd, vd, T - 1, reserve, c2, mode=kvp.KVP_MASK_KVZAP, scores=s, tau=tau, status=st,
                           workspace=ws(kvp.kvp_compact_workspace_bytes(B, H, T)))
    kn, vn = dev_bf16(k[:, T:].copy()), dev_bf16(v[:, T:].copy())
    for i in range(8):
        kvp.kvp_append(c, kn[:, i].contiguous(), vn[:, i].contiguous(), T + i, mode=kvp.KVP_MASK_KVZAP,
                       score=dev_f32(np.zeros((B, H), np.float32)), tau=tau, status=st)
    out = g((B, H * G, d), torch.float32)
    kvp.kvp_decode_attn(dev_bf16(q), c, T + 7, out=out,
                        workspace=ws(kvp.kvp_decode_attn_workspace_bytes(B, H * G, H, d), zero=True), status=st)
    c3 = paged(kvp, B, H, d, cap, mp)
    kvp.kvp_compact_paged(c, T + 7, reserve, c3, status=st,
                          workspace=ws(kvp.kvp_compact_paged_workspace_bytes(B, H, mp)))
    torch.cuda.synchronize()
    assert st.item() == 0, kvp.status_string(st.item())
    check_bands()


def test_canaries_fp8_tier(kvp):
    B, T, H, G, d = 2, 900, 2, 8, 128
    k, v = syn.kv_inputs(4, B, T, H, d)
    q = syn.q_inputs(4, B, H * G, d)
    s = syn.normal_f32(4, 41, (B, T, H))
    tau = np.full((B, H), 0.7, np.float32)
    tau_q = np.full((B, H), -0.5, np.float32)
    exp = orc.mask_kvzap(s, tau, T - 1)[0].astype(np.int32)
    mp = (T + 15) // 16
    cap = B * H * mp
    st = status_word()
    kd, vd = dev_bf16(k), dev_bf16(v)
    c = paged(kvp, B, H, d, cap, mp)
    kvp.kvp_compact(kd, vd, dev_i32(exp), T - 1, 0, c, status=st)
    cq = kvp.QuantPagedKV(g((cap, 16, d), torch.uint8, 0), g((cap, 16, d), torch.uint8, 0),
                          g((cap, 3, 16), torch.int32, 0), g((B, H, mp), torch.int32, -1),
                          g((B, H, mp * 16), torch.int32, -1), g((B, H), torch.int32, 0))
    kvp.kvp_compact_quant(kd, vd, dev_f32(s), dev_f32(tau), dev_f32(tau_q), cq, status=st,
                          workspace=ws(kvp.kvp_compact_workspace_bytes(B, H, T)))
    out = g((B, H * G, d), torch.float32)
    kvp.kvp_decode_attn_two_tier(dev_bf16(q), c, cq, T - 1, out=out,
                                 workspace=ws(kvp.kvp_decode_attn_workspace_bytes(B, H * G, H, d), zero=True),
                                 status=st)
    torch.cuda.synchronize()
    assert st.item() == 0, kvp.status_string(st.item())
    check_bands()


def test_canaries_mla(kvp):
    B, T, Hq, reserve = 2, 700, 20, 20
    row = kvp.LATENT_ROW
    lat = syn.latent_inputs(6, B, T + 4, row)
    s = syn.normal_f32(6, 51, (B, T))
    tau = np.full(B, 0.5, np.float32)
    q = syn.q_inputs(6, B, Hq, row)
    mp = (T + 4 + reserve + 15) // 16
    cap = B * mp
    st = status_word()

    def latent():
        return kvp.LatentPagedKV(g((cap, 16, row), torch.bfloat16, 0), g((cap, 16), torch.int32, 0),
                                 g((B, mp), torch.int32, -1), g((B, mp * 16), torch.int32, -1),
                                 g((B,), torch.int32, 0))
    c = latent()
    kvp.kvp_compact_latent(dev_bf16(lat[:, :T].copy()), T - 1, reserve, c, mode=kvp.KVP_MASK_KVZAP,
                           scores=dev_f32(s), tau=dev_f32(tau), status=st,
                           workspace=ws(kvp.kvp_compact_workspace_bytes(B, 1, T)))
    ln = dev_bf16(lat[:, T:].copy())
    for i in range(4):
        kvp.kvp_append_latent(c, ln[:, i].contiguous(), T + i, mode=kvp.KVP_MASK_KVZAP,
                              score=dev_f32(np.zeros(B, np.float32)), tau=dev_f32(tau), status=st)
    # 16-head tiles, 64-head tiles, then the tensor-core kernel's 128-head tiles
    for hq, ns in ((Hq, 1), (Hq, 3), (40, 1), (40, 3), (72, 1), (72, 3)):
        qh = q if hq == Hq else syn.q_inputs(7, B, hq, row)
        out = g((B, hq, kvp.KVP_MLA_LATENT_DIM), torch.float32)
        kvp.kvp_decode_attn_mla(dev_bf16(qh), c, T + 3, out=out, n_splits=ns,
                                workspace=ws(kvp.kvp_decode_attn_mla_workspace_bytes(B, hq, ns), zero=True),
                                status=st)
    c2 = latent()
    kvp.kvp_compact_latent_paged(c, T + 3, reserve, c2, status=st,
                                 workspace=ws(kvp.kvp_compact_paged_workspace_bytes(B, 1, mp)))
    torch.cuda.synchronize()
    assert st.item() == 0, kvp.status_string(st.item())
    check_bands()
