"""The allocation-free compaction entry point, checked against the regular one.

Some callers of this library cannot allocate GPU memory (their runtime owns
all device memory, or their plugin interface has no workspace hook). For them
kvp_compact_noalloc runs the same compaction with its scratch in a fixed
device array inside the library. Its outputs must equal kvp_compact's, bit for
bit, on consecutive calls that share that array. This file is collected last
so that a stop at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import kvp_synth as syn
import oracle as orc
from helpers import dev_bf16, dev_i32, host_bits, status_word

pytestmark = pytest.mark.gpu

_P, _I, _L = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64


def _noalloc(lib):
    fn = lib.kvp_compact_noalloc
    fn.restype = _I
    fn.argtypes = [_I, _I, _I, _I, _P, _P, _L, _L, _L, _P, _I, _I, _P, _P, _P, _I, _P, _I, _P, _P, _P, _P]
    return fn


def _case(seed, B, T, H, d):
    if B * T * H * d > (1 << 24):   # large: the fast generator
        k = syn.fast_normal_bf16(seed, syn.S_K, (B, T, H, d))
        v = syn.fast_normal_bf16(seed, syn.S_V, (B, T, H, d))
    else:
        k, v = syn.kv_inputs(seed, B, T, H, d)
    s = syn.normal_f32(seed, 21, (B, T, H))
    tau = syn.normal_f32(seed, 22, (B, H), std=0.7)
    exp = orc.mask_kvzap(s, tau, T - 1)[0].astype(np.int32)
    return dev_bf16(k), dev_bf16(v), dev_i32(exp)


def _same(a, b):
    for name in ["count", "page_table", "remap", "expire_pool"]:
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    np.testing.assert_array_equal(host_bits(a.k_pool), host_bits(b.k_pool))
    np.testing.assert_array_equal(host_bits(a.v_pool), host_bits(b.v_pool))


def test_compact_noalloc_matches_compact_on_consecutive_calls(kvp):
    fn = _noalloc(kvp.library())
    stream = torch.cuda.current_stream().cuda_stream
    # each call reuses the scratch the one before it left behind; the third has 2,048 (b, h) pairs, above
    # the 1,024 that the copy pass's CTAs handle alone, so it also goes through the separate page-base
    # pass, whose results live in the scratch too, in words the two smaller calls never wrote
    shapes = [(2, 3000, 4, 128, 5, 1), (3, 1777, 2, 64, 0, 2), (1024, 640, 2, 64, 3, 3)]
    for B, T, H, d, reserve, seed in shapes:
        k, v, exp = _case(seed, B, T, H, d)
        mp = (T + reserve + 15) // 16
        cap = B * H * mp
        ref = kvp.PagedKV.allocate(B, H, d, cap, mp)
        st_ref = status_word()
        kvp.kvp_compact(k, v, exp, T - 1, reserve, ref, status=st_ref)
        out = kvp.PagedKV.allocate(B, H, d, cap, mp)
        st = status_word()
        code = fn(B, H, d, T, k.data_ptr(), v.data_ptr(), k.stride(0), k.stride(1), k.stride(2), exp.data_ptr(),
                  T - 1, reserve, out.k_pool.data_ptr(), out.v_pool.data_ptr(), out.expire_pool.data_ptr(), cap,
                  out.page_table.data_ptr(), mp, out.remap.data_ptr(), out.count.data_ptr(), st.data_ptr(), stream)
        torch.cuda.synchronize()
        assert code == kvp.KVP_OK, kvp.status_string(code)
        assert st.item() == 0 and st_ref.item() == 0
        _same(out, ref)


def test_compact_noalloc_rejects_oversized_scratch(kvp):
    fn = _noalloc(kvp.library())
    # 4096 (b, h) pairs x 4096 positions need 2*4096*32 + 4097 words > 1 MiB of scratch
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = dummy.data_ptr()
    code = fn(4096, 1, 128, 4096, p, p, 0, 0, 0, p, 0, 0, p, p, p, 1, p, 1, p, p, p, None)
    assert code == kvp.KVP_ERR_WORKSPACE
