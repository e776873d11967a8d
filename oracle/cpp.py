"""The C++ oracle (oracle/kvp_oracle.cpp) behind the same Python interface as
the numpy oracle (oracle/kvp_oracle.py): same function names, arguments and
results.

TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
benchmark's CPU legs use it. This module only moves arrays in and out of the
C++ library (ctypes); every step of the method is computed in C++, in double
precision, on all host cores (std::thread over (batch, kv head) units and
scorer rows).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

from .kvp_oracle import CapacityError, PagedCache, QuantPagedCache  # data containers only

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kvp_oracle.cpp")
LIB = os.path.join(HERE, "libkvp_oracle.so")

NEVER = 2**31 - 1
PAGE = 16
WINDOW = 128
E4M3_MAX = 448.0


def build(force: bool = False) -> str:
    """Compiles kvp_oracle.cpp into libkvp_oracle.so next to it (g++, plain
    IEEE arithmetic: no fused multiply-add contraction, no fast-math)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-o", tmp, SRC]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"oracle build failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


_lib = None


def _L():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _lib.kvpo_compact_dense.restype = ctypes.c_int64
        _lib.kvpo_compact_paged.restype = ctypes.c_int64
        _lib.kvpo_append.restype = ctypes.c_int64
        _lib.kvpo_compact_quant_dense.restype = ctypes.c_int64
        _lib.kvpo_append_quant.restype = ctypes.c_int64
        _lib.kvpo_kv_cache_bytes.restype = ctypes.c_int64
        _lib.kvpo_linear_projection_macs.restype = ctypes.c_int64
        _lib.kvpo_scorer_macs.restype = ctypes.c_int64
        _lib.kvpo_threads.restype = ctypes.c_int
    return _lib


def set_threads(n: int) -> None:
    """Worker threads of the C++ oracle (0 = every hardware thread)."""
    _L().kvpo_set_threads(int(n))


def threads() -> int:
    return _L().kvpo_threads()


def _c(a, dtype):
    """A C-contiguous array of dtype (copied only when needed)."""
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


_I64 = ctypes.c_int64
_D = ctypes.c_double


def widen_bf16(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, np.float64)
    _L().kvpo_widen_bf16(_p(b), _I64(b.size), _p(out))
    return out


# --------------------------------------------------------------------------- 1. score

def score_linear(x_bits, w, bias=None) -> np.ndarray:
    x = _c(x_bits, np.uint16)
    w = _c(w, np.float64)
    n, D = x.shape
    H = w.shape[0]
    b = None if bias is None else _c(bias, np.float64)
    s = np.empty((n, H), np.float64)
    _L().kvpo_score_linear(_p(x), _I64(n), ctypes.c_int(D), _p(w), ctypes.c_int(H), _p(b), _p(s))
    return s


def gelu(u) -> np.ndarray:
    u = _c(u, np.float64)
    out = np.empty(u.shape, np.float64)
    _L().kvpo_gelu(_p(u), _I64(u.size), _p(out))
    return out


def score_mlp(x_bits, w1_bits, w2_bits, b1=None, b2=None) -> np.ndarray:
    x, w1, w2 = _c(x_bits, np.uint16), _c(w1_bits, np.uint16), _c(w2_bits, np.uint16)
    n, D = x.shape
    hidden, H = w1.shape[0], w2.shape[0]
    b1c = None if b1 is None else _c(b1, np.float64)
    b2c = None if b2 is None else _c(b2, np.float64)
    s = np.empty((n, H), np.float64)
    _L().kvpo_score_mlp(_p(x), _I64(n), ctypes.c_int(D), _p(w1), ctypes.c_int(hidden), _p(w2), ctypes.c_int(H),
                        _p(b1c), _p(b2c), _p(s))
    return s


# --------------------------------------------------------------------------- 2. mask

def expire_kvzap(score, tau, pos, window: int = WINDOW):
    s, t, p = np.broadcast_arrays(np.asarray(score, np.float64), np.asarray(tau, np.float64),
                                  np.asarray(pos, np.int64))
    s, t, p = _c(s, np.float64), _c(t, np.float64), _c(p, np.int64)
    out = np.empty(s.shape, np.int64)
    _L().kvpo_expire_kvzap(_p(s), _p(t), _p(p), _I64(s.size), _I64(window), _p(out))
    return out


def expire_dms(flag_step, pos, delay: int, window: int = WINDOW):
    f, p = np.broadcast_arrays(np.asarray(flag_step, np.int64), np.asarray(pos, np.int64))
    f, p = _c(f, np.int64), _c(p, np.int64)
    out = np.empty(f.shape, np.int64)
    _L().kvpo_expire_dms(_p(f), _p(p), _I64(f.size), _I64(delay), _I64(window), _p(out))
    return out


def present(expire, now: int):
    e = _c(np.asarray(expire, np.int64), np.int64)
    out = np.empty(e.shape, np.uint8)
    _L().kvpo_present(_p(e), _I64(e.size), _I64(now), _p(out))
    return out.astype(bool)


def mask(expire_bht, now: int):
    e = _c(expire_bht, np.int64)
    B, H, T = e.shape
    keep = np.empty((B, H, T), np.uint8)
    bits = np.empty((B, H, (T + 31) // 32), np.uint32)
    count = np.empty((B, H), np.int64)
    _L().kvpo_mask(_p(e), _I64(B * H), _I64(T), _I64(now), _p(keep), _p(bits), _p(count))
    return keep.astype(bool), bits, count


def mask_kvzap(scores_bth, tau_bh, now: int, window: int = WINDOW, pos0: int = 0):
    s = np.asarray(scores_bth)
    B, T, H = s.shape
    pos = pos0 + np.arange(T)
    exp = expire_kvzap(s.transpose(0, 2, 1), np.asarray(tau_bh)[:, :, None], pos[None, None, :], window)
    return (exp,) + mask(exp, now)


def mask_dms(flag_step_bht, now: int, delay: int, window: int = WINDOW, pos0: int = 0):
    f = np.asarray(flag_step_bht)
    B, H, T = f.shape
    pos = pos0 + np.arange(T)
    exp = expire_dms(f, pos[None, None, :], delay, window)
    return (exp,) + mask(exp, now)


def threshold_at_quantile(scores_bth, q) -> np.ndarray:
    s = _c(scores_bth, np.float64)
    B, T, H = s.shape
    qh = np.broadcast_to(np.asarray(q, np.float64), (H,))
    k = _c(np.floor(qh * (T - 1)), np.int64)
    tau = np.empty((B, H), np.float32)
    _L().kvpo_threshold(_p(s), _I64(B), _I64(T), _I64(H), _p(k), _p(tau))
    return tau


# --------------------------------------------------------------------------- 3. compaction

def _check_pages(r, B, H, what):
    if r < 0:
        u = -1 - r
        raise CapacityError(f"(b={u // H}, h={u % H}) needs more {what}pages than the budget gives")


def compact_dense(k_bits, v_bits, expire_bht, now, reserve, n_pages_cap, max_pages) -> PagedCache:
    k, v = _c(k_bits, np.uint16), _c(v_bits, np.uint16)
    B, T, H, d = k.shape
    e = _c(expire_bht, np.int64)
    out = PagedCache(B, H, d, n_pages_cap, max_pages)
    r = _L().kvpo_compact_dense(_p(k), _p(v), _p(e), _I64(B), _I64(T), _I64(H), _I64(d), _I64(now), _I64(reserve),
                                _I64(n_pages_cap), _I64(max_pages), _p(out.k_pool), _p(out.v_pool),
                                _p(out.expire_pool), _p(out.page_table), _p(out.remap), _p(out.count))
    _check_pages(r, B, H, "")
    out.pages_used = int(r)
    return out


def compact_paged(src: PagedCache, now, reserve, n_pages_cap, max_pages) -> PagedCache:
    B, H, smp = src.page_table.shape
    d = src.k_pool.shape[2]
    out = PagedCache(B, H, d, n_pages_cap, max_pages)
    r = _L().kvpo_compact_paged(_p(_c(src.k_pool, np.uint16)), _p(_c(src.v_pool, np.uint16)),
                                _p(_c(src.expire_pool, np.int64)), _p(_c(src.page_table, np.int64)), _I64(smp),
                                _p(_c(src.remap, np.int64)), _p(_c(src.count, np.int64)), _I64(B * H), _I64(d),
                                _I64(now), _I64(reserve), _I64(n_pages_cap), _I64(max_pages), _p(out.k_pool),
                                _p(out.v_pool), _p(out.expire_pool), _p(out.page_table), _p(out.remap),
                                _p(out.count))
    _check_pages(r, B, H, "")
    out.pages_used = int(r)
    return out


def append(cache: PagedCache, k_new_bits, v_new_bits, pos: int, expire_new):
    B, H = cache.count.shape
    d = cache.k_pool.shape[2]
    kn, vn = _c(k_new_bits, np.uint16), _c(v_new_bits, np.uint16)
    en = _c(np.broadcast_to(np.asarray(expire_new, np.int64), (B, H)), np.int64)
    r = _L().kvpo_append(_p(cache.k_pool), _p(cache.v_pool), _p(cache.expire_pool), _p(cache.page_table),
                         _I64(cache.page_table.shape[2]), _p(cache.remap), _p(cache.count), _I64(B * H), _I64(d),
                         _p(kn), _p(vn), _I64(pos), _p(en))
    if r >= 0:
        raise CapacityError(f"(b={r // H}, h={r % H}) has no free slot")


# --------------------------------------------------------------------------- 4. attention

def decode_attention(q_bits, cache: PagedCache, now: int, scale: float | None = None) -> np.ndarray:
    q = _c(q_bits, np.uint16)
    B, Hq, d = q.shape
    H = cache.count.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = np.empty((B, Hq, d), np.float32)
    _L().kvpo_decode_attention(_p(q), _I64(B), _I64(Hq), _I64(H), _I64(d), _p(cache.k_pool), _p(cache.v_pool),
                               _p(cache.expire_pool), _p(cache.page_table), _I64(cache.page_table.shape[2]),
                               _p(cache.count), _I64(now), _D(scale), _p(out))
    return out


def decode_attention_lse(q_bits, cache: PagedCache, now: int, scale: float | None = None):
    q = _c(q_bits, np.uint16)
    B, Hq, d = q.shape
    H = cache.count.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = np.empty((B, Hq, d), np.float32)
    lse = np.empty((B, Hq), np.float64)
    _L().kvpo_decode_attention_lse(_p(q), _I64(B), _I64(Hq), _I64(H), _I64(d), _p(cache.k_pool),
                                   _p(cache.v_pool), _p(cache.expire_pool), _p(cache.page_table),
                                   _I64(cache.page_table.shape[2]), _p(cache.count), _I64(now), _D(scale), _p(out),
                                   _p(lse))
    return out, lse


def merge_attention(outs, lses):
    o = _c(outs, np.float64)
    ls = _c(lses, np.float64)
    P, d = o.shape[0], o.shape[-1]
    rows = int(np.prod(ls.shape[1:], dtype=np.int64))
    out = np.empty(o.shape[1:], np.float64)
    lse = np.empty(ls.shape[1:], np.float64)
    _L().kvpo_merge_attention(_p(o), _p(ls), _I64(P), _I64(rows), _I64(d), _p(out), _p(lse))
    return out, lse


def dense_attention(q_bits, k_bits, v_bits, now: int, scale=None, lo=None):
    q, k, v = _c(q_bits, np.uint16), _c(k_bits, np.uint16), _c(v_bits, np.uint16)
    B, Hq, d = q.shape
    T, H = k.shape[1], k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    lo = 0 if lo is None else max(0, lo)
    out = np.empty((B, Hq, d), np.float32)
    _L().kvpo_dense_attention(_p(q), _I64(B), _I64(Hq), _p(k), _p(v), _I64(T), _I64(H), _I64(d), _I64(lo),
                              _I64(now), _D(scale), _p(out))
    return out


def window_attention(q_bits, k_bits, v_bits, now: int, window: int = WINDOW, scale=None):
    return dense_attention(q_bits, k_bits, v_bits, now, scale, lo=now - window + 1)


# --------------------------------------------------------------------------- 5. fp8 tier

def e4m3_decode(codes) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _L().kvpo_e4m3_decode(_p(c), _I64(c.size), _p(out))
    return out


def e4m3_positive_values() -> np.ndarray:
    return e4m3_decode(np.arange(128, dtype=np.uint8))


def e4m3_encode(v) -> np.ndarray:
    a = _c(v, np.float64)
    out = np.empty(a.shape, np.uint8)
    _L().kvpo_e4m3_encode(_p(a), _I64(a.size), _p(out))
    return out


def quantize_rows(bits):
    b = _c(bits, np.uint16)
    d = b.shape[-1]
    n = b.size // d if d else 0
    codes = np.empty(b.shape, np.uint8)
    scale = np.empty(b.shape[:-1], np.float32)
    _L().kvpo_quantize_rows(_p(b), _I64(n), _I64(d), _p(codes), _p(scale))
    return codes, scale


def dequantize_rows(codes, scale) -> np.ndarray:
    return e4m3_decode(codes) * np.asarray(scale, dtype=np.float64)[..., None]


def quant_tier_select(scores_bth, tau_bh, tau_q_bh):
    """Entries that go to the fp8 tier: tau_q <= s < tau. [B, H, T] bool."""
    s, t, tq = np.broadcast_arrays(np.asarray(scores_bth, np.float64).transpose(0, 2, 1),
                                   np.asarray(tau_bh, np.float64)[:, :, None],
                                   np.asarray(tau_q_bh, np.float64)[:, :, None])
    s, t, tq = _c(s, np.float64), _c(t, np.float64), _c(tq, np.float64)
    out = np.empty(s.shape, np.uint8)
    _L().kvpo_quant_select(_p(s), _p(t), _p(tq), _I64(s.size), _p(out))
    return out.astype(bool)


def quant_tier_select_dms(flag_step_bht):
    return np.asarray(flag_step_bht) >= 0


def compact_quant_dense(k_bits, v_bits, scores_bth, tau_bh, tau_q_bh, reserve, n_pages_cap, max_pages,
                        window: int = WINDOW, flag_step_bht=None, delay: int = 0) -> QuantPagedCache:
    k, v = _c(k_bits, np.uint16), _c(v_bits, np.uint16)
    B, T, H, d = k.shape
    pos = np.arange(T)[None, None, :]
    if flag_step_bht is not None:
        sel = quant_tier_select_dms(flag_step_bht)
        start = expire_dms(flag_step_bht, pos, delay, window)
    else:
        sel = quant_tier_select(scores_bth, tau_bh, tau_q_bh)
        start = np.broadcast_to(pos + window, (B, H, T))
    sel = _c(sel, np.uint8)
    start = _c(start, np.int64)
    out = QuantPagedCache(B, H, d, n_pages_cap, max_pages)
    r = _L().kvpo_compact_quant_dense(_p(k), _p(v), _p(sel), _p(start), _I64(B), _I64(T), _I64(H), _I64(d),
                                      _I64(reserve), _I64(n_pages_cap), _I64(max_pages), _p(out.kq_pool),
                                      _p(out.vq_pool), _p(out.kscale), _p(out.vscale), _p(out.start_pool),
                                      _p(out.page_table), _p(out.remap), _p(out.count))
    _check_pages(r, B, H, "fp8 ")
    out.pages_used = int(r)
    return out


def append_quant(qcache: QuantPagedCache, k_new_bits, v_new_bits, pos: int, score_bh, tau_bh, tau_q_bh,
                 window: int = WINDOW, flag_bh=None, delay: int = 0):
    B, H = qcache.count.shape
    d = qcache.kq_pool.shape[2]
    if flag_bh is not None:
        sel = quant_tier_select_dms(flag_bh)
        start = expire_dms(flag_bh, pos, delay, window)
    else:
        s, t, tq = np.broadcast_arrays(np.asarray(score_bh, np.float64), np.asarray(tau_bh, np.float64),
                                       np.asarray(tau_q_bh, np.float64))
        s, t, tq = _c(s, np.float64), _c(t, np.float64), _c(tq, np.float64)
        sel = np.empty(s.shape, np.uint8)
        _L().kvpo_quant_select(_p(s), _p(t), _p(tq), _I64(s.size), _p(sel))
        start = np.full((B, H), pos + window, np.int64)
    sel = _c(np.broadcast_to(sel, (B, H)), np.uint8)
    start = _c(np.broadcast_to(start, (B, H)), np.int64)
    kn, vn = _c(k_new_bits, np.uint16), _c(v_new_bits, np.uint16)
    r = _L().kvpo_append_quant(_p(qcache.kq_pool), _p(qcache.vq_pool), _p(qcache.kscale), _p(qcache.vscale),
                               _p(qcache.start_pool), _p(qcache.page_table), _I64(qcache.page_table.shape[2]),
                               _p(qcache.remap), _p(qcache.count), _I64(B * H), _I64(d), _p(kn), _p(vn), _I64(pos),
                               _p(sel), _p(start))
    if r >= 0:
        raise CapacityError(f"(b={r // H}, h={r % H}) has no free fp8 slot")


def decode_attention_two_tier(q_bits, cache: PagedCache, qcache: QuantPagedCache, now: int,
                              scale: float | None = None) -> np.ndarray:
    q = _c(q_bits, np.uint16)
    B, Hq, d = q.shape
    H = cache.count.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = np.empty((B, Hq, d), np.float32)
    _L().kvpo_decode_attention_two_tier(
        _p(q), _I64(B), _I64(Hq), _I64(H), _I64(d), _p(cache.k_pool), _p(cache.v_pool), _p(cache.expire_pool),
        _p(cache.page_table), _I64(cache.page_table.shape[2]), _p(cache.count), _p(qcache.kq_pool),
        _p(qcache.vq_pool), _p(qcache.kscale), _p(qcache.vscale), _p(qcache.start_pool), _p(qcache.page_table),
        _I64(qcache.page_table.shape[2]), _p(qcache.count), _I64(now), _D(scale), _p(out))
    return out


# --------------------------------------------------------------------------- 6. MLA latent cache

def compact_latent_dense(lat_bits, expire_bt, now: int, reserve: int, n_pages_cap: int, max_pages: int) -> PagedCache:
    lat = _c(lat_bits, np.uint16)[:, :, None, :]
    return compact_dense(lat, lat, np.asarray(expire_bt)[:, None, :], now, reserve, n_pages_cap, max_pages)


def decode_attention_mla(q_bits, cache: PagedCache, dc: int, now: int, scale: float | None = None) -> np.ndarray:
    q = _c(q_bits, np.uint16)
    B, Hq, R = q.shape
    scale = 1.0 / math.sqrt(R) if scale is None else scale
    out = np.empty((B, Hq, dc), np.float32)
    _L().kvpo_decode_attention_mla(_p(q), _I64(B), _I64(Hq), _I64(R), _I64(dc), _p(cache.k_pool),
                                   _p(cache.expire_pool), _p(cache.page_table), _I64(cache.page_table.shape[2]),
                                   _p(cache.count), _I64(now), _D(scale), _p(out))
    return out


# --------------------------------------------------------------------------- closed forms

def kv_cache_bytes(n_layers: int, d_model: int, n_tokens: int, elem_bytes: int = 2) -> int:
    return int(_L().kvpo_kv_cache_bytes(_I64(n_layers), _I64(d_model), _I64(n_tokens), _I64(elem_bytes)))


def linear_projection_macs(d_model, n_q_heads, n_kv_heads, head_dim, ffn_hidden, gated=True) -> int:
    return int(_L().kvpo_linear_projection_macs(_I64(d_model), _I64(n_q_heads), _I64(n_kv_heads), _I64(head_dim),
                                                _I64(ffn_hidden), ctypes.c_int(1 if gated else 0)))


def scorer_macs(d_model, n_kv_heads, hidden=None) -> int:
    return int(_L().kvpo_scorer_macs(_I64(d_model), _I64(n_kv_heads), _I64(0 if hidden is None else hidden)))
