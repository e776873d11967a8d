"""Python binding of libkvp (KV-cache pruning at decode time, sm_103a).

Each function here has the name of the C entry point it calls (see
include/kvp.h) and only marshals arguments: torch tensors are checked for
dtype, device and contiguity, their device pointers and sizes are passed on,
and a non-OK status raises KvpError. Every step of the path runs in the
library's CUDA kernels; there is no other implementation to fall back on, so
importing this package fails loudly when libkvp.so has not been built.

PyTorch is used for device memory and streams only: calls are enqueued on
torch's current CUDA stream unless a stream is passed.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvp.so")

KVP_OK = 0
KVP_ERR_INVALID = 1
KVP_ERR_ALIGN = 2
KVP_ERR_CAPACITY = 3
KVP_ERR_CUDA = 4
KVP_ERR_TIMEOUT = 5
KVP_ERR_UNSUPPORTED = 6
KVP_ERR_WORKSPACE = 7
KVP_ERR_BOUNDS = 8

KVP_SCORER_LINEAR = 0
KVP_SCORER_MLP = 1
KVP_SCORER_LINEAR_SPLIT = 2
KVP_MASK_KVZAP = 0
KVP_MASK_DMS = 1
PAGE = 16
WINDOW = 128
EXPIRE_NEVER = 2**31 - 1
KVP_MLA_LATENT_DIM = 512
KVP_MLA_ROPE_DIM = 64
LATENT_ROW = KVP_MLA_LATENT_DIM + KVP_MLA_ROPE_DIM


class KvpError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn}: {status_string(code)} (status {code})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libkvp.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    return ctypes.CDLL(LIB_PATH)


_lib = _load()

_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_S = ctypes.c_size_t
_F = ctypes.c_float

_SIGS = {
    "kvp_status_string": (ctypes.c_char_p, [_I]),
    "kvp_version": (_I, []),
    "kvp_score_workspace_bytes": (_S, [_I, _L, _I, _I, _I]),
    "kvp_score_split_weight_bytes": (_S, [_I, _I]),
    "kvp_score_split_weight": (_I, [_I, _I, _P, _P, _S, _P]),
    "kvp_score": (_I, [_I, _L, _I, _I, _I, _P, _L, _P, _P, _P, _P, _P, _P, _S, _P, _P]),
    "kvp_mask": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P]),
    "kvp_threshold_workspace_bytes": (_S, [_I, _I]),
    "kvp_threshold": (_I, [_I, _I, _I, _P, ctypes.c_double, _P, _P, _S, _P]),
    "kvp_compact_workspace_bytes": (_S, [_I, _I, _I]),
    "kvp_compact": (_I, [_I, _I, _I, _I, _P, _P, _L, _L, _L, _P, _I, _I, _P, _P, _P, _I, _P, _I, _P, _P,
                         _P, _S, _P, _P]),
    "kvp_compact_masked": (_I, [_I, _I, _I, _I, _I, _P, _P, _L, _L, _L, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P,
                                _I, _P, _I, _P, _P, _P, _S, _P, _P]),
    "kvp_compact_quant": (_I, [_I, _I, _I, _I, _I, _P, _P, _L, _L, _L, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P,
                               _I, _P, _I, _P, _P, _P, _S, _P, _P]),
    "kvp_compact_noalloc": (_I, [_I, _I, _I, _I, _P, _P, _L, _L, _L, _P, _I, _I, _P, _P, _P, _I, _P, _I, _P, _P,
                                 _P, _P]),
    "kvp_compact_paged_workspace_bytes": (_S, [_I, _I, _I]),
    "kvp_compact_paged": (_I, [_I, _I, _I, _P, _P, _P, _I, _P, _I, _P, _P, _I, _I, _P, _P, _P, _I, _P, _I,
                               _P, _P, _P, _S, _P, _P]),
    "kvp_append": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _I, _P, _I, _P, _P,
                        _P, _P]),
    "kvp_append_devpos": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _I, _P, _I, _P, _P,
                               _P, _P]),
    "kvp_append_quant": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _I, _P, _I, _P, _P,
                              _P, _P]),
    "kvp_decode_attn_workspace_bytes": (_S, [_I, _I, _I, _I]),
    "kvp_decode_attn": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _I, _P, _I, _F, _P, _I, _P, _S, _P, _P]),
    "kvp_decode_attn_devpos": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _I, _P, _P, _F, _P, _I, _P, _S, _P,
                                    _P]),
    "kvp_decode_attn_lse": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _I, _P, _I, _F, _P, _P, _I, _P, _S, _P,
                                 _P]),
    "kvp_attn_merge": (_I, [_I, _L, _I, _P, _P, _P, _P, _P]),
    "kvp_decode_attn_two_tier": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _I, _P, _P, _P, _P, _I, _P, _I, _P,
                                      _I, _F, _P, _I, _P, _S, _P, _P]),
    "kvp_compact_latent": (_I, [_I, _I, _I, _I, _P, _L, _L, _P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _I, _P, _P,
                                _P, _S, _P, _P]),
    "kvp_compact_latent_paged": (_I, [_I, _I, _P, _P, _I, _P, _I, _P, _P, _I, _I, _P, _P, _I, _P, _I, _P, _P, _P,
                                      _S, _P, _P]),
    "kvp_append_latent": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _I, _I, _P, _P, _I, _P, _I, _P, _P, _P, _P]),
    "kvp_selftest_wait": (_I, [ctypes.c_uint64, _P, _P, _P]),
    "kvp_decode_attn_mla_workspace_bytes": (_S, [_I, _I, _I]),
    "kvp_decode_attn_mla": (_I, [_I, _I, _I, _I, _P, _P, _P, _I, _P, _I, _P, _I, _F, _P, _I, _P, _S, _P, _P]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


def library():
    """The loaded ctypes handle of libkvp.so."""
    return _lib


def status_string(code: int) -> str:
    return _lib.kvp_status_string(int(code)).decode()


def version() -> int:
    return _lib.kvp_version()


# --------------------------------------------------------------------------- marshalling helpers

def _ptr(t, dtype=None, name="tensor", optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(fn: str, code: int):
    if code != KVP_OK:
        raise KvpError(fn, code)


def _ws(nbytes: int, device, workspace=None):
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return workspace
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


# --------------------------------------------------------------------------- score

def kvp_score_workspace_bytes(scorer, n_tok, d_model, n_kv_heads, hidden=0) -> int:
    return _lib.kvp_score_workspace_bytes(scorer, n_tok, d_model, n_kv_heads, hidden)


def kvp_score_split_weight_bytes(d_model, n_kv_heads) -> int:
    return _lib.kvp_score_split_weight_bytes(d_model, n_kv_heads)


def kvp_score_split_weight(w, *, out=None, stream=None):
    """The KVzap-Linear weight w fp32 [H, D] as the scorer's bf16 hi/lo operand (rows 2h, 2h+1), for
    kvp_score(..., scorer=KVP_SCORER_LINEAR_SPLIT, n_kv_heads=H)."""
    H, D = w.shape
    nbytes = kvp_score_split_weight_bytes(D, H)
    if out is None:
        out = torch.empty((nbytes // (2 * D), D), dtype=torch.bfloat16, device=w.device)
    code = _lib.kvp_score_split_weight(D, H, _ptr(w, torch.float32, "w"), _ptr(out, torch.bfloat16, "out"),
                                       out.numel() * out.element_size(), _stream(stream))
    _check("kvp_score_split_weight", code)
    return out


def kvp_score(x, w, b=None, w2=None, b2=None, *, scorer=KVP_SCORER_LINEAR, n_kv_heads=None, out=None,
              workspace=None, status=None, stream=None):
    """scores[n_tok, H] from hidden states x[n_tok, D] (bf16).

    LINEAR: w fp32 [H, D], b fp32 [H] or None.
    LINEAR_SPLIT: w the bf16 operand from kvp_score_split_weight, n_kv_heads = H, b as for LINEAR.
    MLP:    w bf16 W1 [hidden, D], b fp32 b1 [hidden] or None, w2 bf16 [H, hidden], b2 fp32 [H] or None.
    """
    if x.dim() != 2:
        raise ValueError("x must be [n_tok, D]")
    n_tok, D = x.shape
    if x.stride(1) != 1:
        raise ValueError("x rows must be contiguous")
    if scorer == KVP_SCORER_LINEAR:
        H, hidden = w.shape[0], 0
        wp = _ptr(w, torch.float32, "w")
    elif scorer == KVP_SCORER_LINEAR_SPLIT:
        if n_kv_heads is None:
            raise ValueError("LINEAR_SPLIT needs n_kv_heads")
        H, hidden = int(n_kv_heads), 0
        wp = _ptr(w, torch.bfloat16, "w_split")
    else:
        hidden, H = w.shape[0], w2.shape[0]
        wp = _ptr(w, torch.bfloat16, "w1")
    if out is None:
        out = torch.empty((n_tok, H), dtype=torch.float32, device=x.device)
    need = kvp_score_workspace_bytes(scorer, n_tok, D, H, hidden)
    ws = _ws(need, x.device, workspace)
    code = _lib.kvp_score(scorer, n_tok, D, H, hidden, x.data_ptr(), x.stride(0), wp,
                          _ptr(b, torch.float32, "b", True),
                          _ptr(w2, torch.bfloat16, "w2", True), _ptr(b2, torch.float32, "b2", True),
                          _ptr(out, torch.float32, "out"), ws.data_ptr(), ws.numel() * ws.element_size(),
                          _ptr(status, torch.int32, "status", True), _stream(stream))
    _check("kvp_score", code)
    return out


# --------------------------------------------------------------------------- mask

def kvp_mask(*, mode, batch, n_kv_heads, n_pos, now, scores=None, tau=None, flag_step=None, window=WINDOW,
             delay=0, pos0=0, expire=None, keep_bits=None, count=None, want_bits=True, stream=None):
    """expire [B, H, n_pos] (+ keep_bits, count) from KVzap scores [B, n_pos, H] and tau [B, H], or from
    DMS flag steps [B, H, n_pos]."""
    dev = (scores if scores is not None else flag_step).device
    if expire is None:
        expire = torch.empty((batch, n_kv_heads, n_pos), dtype=torch.int32, device=dev)
    if want_bits and keep_bits is None:
        keep_bits = torch.empty((batch, n_kv_heads, (n_pos + 31) // 32), dtype=torch.int32, device=dev)
    if count is None:
        count = torch.empty((batch, n_kv_heads), dtype=torch.int32, device=dev)
    code = _lib.kvp_mask(mode, batch, n_kv_heads, n_pos, pos0, _ptr(scores, torch.float32, "scores", True),
                         _ptr(tau, torch.float32, "tau", True), _ptr(flag_step, torch.int32, "flag_step", True),
                         window, delay, now, _ptr(expire, torch.int32, "expire"),
                         _ptr(keep_bits, torch.int32, "keep_bits", True), _ptr(count, torch.int32, "count"),
                         _stream(stream))
    _check("kvp_mask", code)
    return expire, keep_bits, count


# --------------------------------------------------------------------------- paged cache

@dataclass
class PagedKV:
    """Device buffers of one compacted cache (allocated with torch)."""
    k_pool: torch.Tensor        # bf16 [n_pages_cap, 16, d]
    v_pool: torch.Tensor        # bf16 [n_pages_cap, 16, d]
    expire_pool: torch.Tensor   # int32 [n_pages_cap, 16]
    page_table: torch.Tensor    # int32 [B, H, max_pages]
    remap: torch.Tensor         # int32 [B, H, max_pages * 16]
    count: torch.Tensor         # int32 [B, H]

    @staticmethod
    def allocate(batch, n_kv_heads, head_dim, n_pages_cap, max_pages, device="cuda"):
        return PagedKV(
            torch.zeros((n_pages_cap, PAGE, head_dim), dtype=torch.bfloat16, device=device),
            torch.zeros((n_pages_cap, PAGE, head_dim), dtype=torch.bfloat16, device=device),
            torch.zeros((n_pages_cap, PAGE), dtype=torch.int32, device=device),
            torch.full((batch, n_kv_heads, max_pages), -1, dtype=torch.int32, device=device),
            torch.full((batch, n_kv_heads, max_pages * PAGE), -1, dtype=torch.int32, device=device),
            torch.zeros((batch, n_kv_heads), dtype=torch.int32, device=device),
        )

    @property
    def n_pages_cap(self):
        return self.k_pool.shape[0]

    @property
    def max_pages(self):
        return self.page_table.shape[2]

    @property
    def head_dim(self):
        return self.k_pool.shape[2]


@dataclass
class QuantPagedKV:
    """Device buffers of the fp8 tier (quantize instead of drop)."""
    kq_pool: torch.Tensor       # uint8 [n_pages_cap, 16, d] E4M3 codes of K rows
    vq_pool: torch.Tensor       # uint8 [n_pages_cap, 16, d] E4M3 codes of V rows
    meta_pool: torch.Tensor     # int32 [n_pages_cap, 3, 16]: start step, K scale, V scale (fp32 bits)
    page_table: torch.Tensor    # int32 [B, H, max_pages]
    remap: torch.Tensor         # int32 [B, H, max_pages * 16]
    count: torch.Tensor         # int32 [B, H]

    @staticmethod
    def allocate(batch, n_kv_heads, head_dim, n_pages_cap, max_pages, device="cuda"):
        return QuantPagedKV(
            torch.zeros((n_pages_cap, PAGE, head_dim), dtype=torch.uint8, device=device),
            torch.zeros((n_pages_cap, PAGE, head_dim), dtype=torch.uint8, device=device),
            torch.zeros((n_pages_cap, 3, PAGE), dtype=torch.int32, device=device),
            torch.full((batch, n_kv_heads, max_pages), -1, dtype=torch.int32, device=device),
            torch.full((batch, n_kv_heads, max_pages * PAGE), -1, dtype=torch.int32, device=device),
            torch.zeros((batch, n_kv_heads), dtype=torch.int32, device=device),
        )

    @property
    def n_pages_cap(self):
        return self.kq_pool.shape[0]

    @property
    def max_pages(self):
        return self.page_table.shape[2]

    @property
    def head_dim(self):
        return self.kq_pool.shape[2]

    @property
    def start_pool(self):
        return self.meta_pool[:, 0, :]

    @property
    def kscale(self):
        return self.meta_pool[:, 1, :].view(torch.float32)

    @property
    def vscale(self):
        return self.meta_pool[:, 2, :].view(torch.float32)


def kvp_threshold_workspace_bytes(batch, n_kv_heads) -> int:
    return _lib.kvp_threshold_workspace_bytes(batch, n_kv_heads)


def kvp_threshold(scores, q, *, out=None, workspace=None, stream=None):
    """Per-(b, h) threshold: the rank floor(q * (T - 1)) score of scores
    [B, T, H] along T (NaN ranked last) -> tau fp32 [B, H]."""
    if scores.dim() != 3:
        raise ValueError("scores must be [B, T, H]")
    B, T, H = scores.shape
    dev = scores.device
    tau = out if out is not None else torch.empty(B, H, dtype=torch.float32, device=dev)
    if tau.numel() != B * H:
        raise ValueError("out must hold B*H values")
    ws = _ws(kvp_threshold_workspace_bytes(B, H), dev, workspace)
    code = _lib.kvp_threshold(B, H, T, _ptr(scores, torch.float32, "scores"), float(q),
                              _ptr(tau, torch.float32, "out"), ws.data_ptr(), ws.numel() * ws.element_size(),
                              _stream(stream))
    _check("kvp_threshold", code)
    return tau


def kvp_compact_workspace_bytes(batch, n_kv_heads, n_pos) -> int:
    return _lib.kvp_compact_workspace_bytes(batch, n_kv_heads, n_pos)


def kvp_compact(k, v, expire, now, reserve, dst: PagedKV, *, status, workspace=None, stream=None):
    """Dense K, V [B, T, H, d] (any strides with d contiguous) + expire [B, H, T] -> dst."""
    B, T, H, d = k.shape
    if k.stride() != v.stride() or k.stride(3) != 1:
        raise ValueError("k and v need identical strides with the head_dim axis contiguous")
    need = kvp_compact_workspace_bytes(B, H, T)
    ws = _ws(need, k.device, workspace)
    for t, nm in ((k, "k"), (v, "v")):
        if t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{nm} must be a CUDA bf16 tensor")
    code = _lib.kvp_compact(B, H, d, T, k.data_ptr(), v.data_ptr(), k.stride(0), k.stride(1), k.stride(2),
                            _ptr(expire, torch.int32, "expire"), now, reserve,
                            _ptr(dst.k_pool, torch.bfloat16), _ptr(dst.v_pool, torch.bfloat16),
                            _ptr(dst.expire_pool, torch.int32), dst.n_pages_cap,
                            _ptr(dst.page_table, torch.int32), dst.max_pages, _ptr(dst.remap, torch.int32),
                            _ptr(dst.count, torch.int32), ws.data_ptr(), ws.numel() * ws.element_size(),
                            _ptr(status, torch.int32, "status"), _stream(stream))
    _check("kvp_compact", code)
    return dst


def kvp_compact_noalloc(k, v, expire, now, reserve, dst: PagedKV, *, status, stream=None):
    """kvp_compact with its scratch in the library's fixed device array: allocates nothing (not even through
    torch). The first call on a device looks the array's address up, so make it before any stream capture; calls
    that overlap on the GPU race on the array."""
    B, T, H, d = k.shape
    if k.stride() != v.stride() or k.stride(3) != 1:
        raise ValueError("k and v need identical strides with the head_dim axis contiguous")
    for t, nm in ((k, "k"), (v, "v")):
        if t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{nm} must be a CUDA bf16 tensor")
    code = _lib.kvp_compact_noalloc(B, H, d, T, k.data_ptr(), v.data_ptr(), k.stride(0), k.stride(1), k.stride(2),
                                    _ptr(expire, torch.int32, "expire"), now, reserve,
                                    _ptr(dst.k_pool, torch.bfloat16), _ptr(dst.v_pool, torch.bfloat16),
                                    _ptr(dst.expire_pool, torch.int32), dst.n_pages_cap,
                                    _ptr(dst.page_table, torch.int32), dst.max_pages, _ptr(dst.remap, torch.int32),
                                    _ptr(dst.count, torch.int32), _ptr(status, torch.int32, "status"),
                                    _stream(stream))
    _check("kvp_compact_noalloc", code)
    return dst


def kvp_compact_masked(k, v, now, reserve, dst: PagedKV, *, mode, scores=None, tau=None, flag_step=None,
                       window=WINDOW, delay=0, status, workspace=None, stream=None):
    """Dense K, V [B, T, H, d] with the mask applied on the fly: KVzap scores
    [B*T, H] (or [B, T, H]) + tau [B, H], or DMS flag_step [B, H, T] -> dst.
    Same result as kvp_mask (pos0 = 0) followed by kvp_compact."""
    B, T, H, d = k.shape
    if k.stride() != v.stride() or k.stride(3) != 1:
        raise ValueError("k and v need identical strides with the head_dim axis contiguous")
    for t, nm in ((k, "k"), (v, "v")):
        if t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{nm} must be a CUDA bf16 tensor")
    if scores is not None and scores.numel() != B * T * H:
        raise ValueError("scores must hold B*T*H values")
    if flag_step is not None and flag_step.numel() != B * H * T:
        raise ValueError("flag_step must hold B*H*T values")
    if tau is not None and tau.numel() != B * H:
        raise ValueError("tau must hold B*H values")
    need = kvp_compact_workspace_bytes(B, H, T)
    ws = _ws(need, k.device, workspace)
    code = _lib.kvp_compact_masked(mode, B, H, d, T, k.data_ptr(), v.data_ptr(), k.stride(0), k.stride(1),
                                   k.stride(2), _ptr(scores, torch.float32, "scores", True),
                                   _ptr(tau, torch.float32, "tau", True),
                                   _ptr(flag_step, torch.int32, "flag_step", True), window, delay, now, reserve,
                                   _ptr(dst.k_pool, torch.bfloat16), _ptr(dst.v_pool, torch.bfloat16),
                                   _ptr(dst.expire_pool, torch.int32), dst.n_pages_cap,
                                   _ptr(dst.page_table, torch.int32), dst.max_pages, _ptr(dst.remap, torch.int32),
                                   _ptr(dst.count, torch.int32), ws.data_ptr(), ws.numel() * ws.element_size(),
                                   _ptr(status, torch.int32, "status"), _stream(stream))
    _check("kvp_compact_masked", code)
    return dst


def kvp_compact_quant(k, v, scores, tau, tau_q, dst: QuantPagedKV, *, mode=KVP_MASK_KVZAP, flag_step=None, delay=0,
                      reserve=0, window=WINDOW, status, workspace=None, stream=None):
    """Dense K, V [B, T, H, d] -> the fp8 tier: entries with tau_q <= score < tau (scores [B*T, H] or
    [B, T, H]; tau, tau_q [B, H]), or with mode KVP_MASK_DMS the flagged entries (flag_step [B, H, T];
    scores, tau, tau_q None), as E4M3 codes with a per-row scale, visible from the step their bf16 copy
    is gone."""
    B, T, H, d = k.shape
    if k.stride() != v.stride() or k.stride(3) != 1:
        raise ValueError("k and v need identical strides with the head_dim axis contiguous")
    for t, nm in ((k, "k"), (v, "v")):
        if t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{nm} must be a CUDA bf16 tensor")
    if mode == KVP_MASK_KVZAP and (scores.numel() != B * T * H or tau.numel() != B * H or tau_q.numel() != B * H):
        raise ValueError("scores must hold B*T*H values, tau and tau_q B*H")
    if mode == KVP_MASK_DMS and flag_step.numel() != B * H * T:
        raise ValueError("flag_step must hold B*H*T values")
    need = kvp_compact_workspace_bytes(B, H, T)
    ws = _ws(need, k.device, workspace)
    code = _lib.kvp_compact_quant(mode, B, H, d, T, k.data_ptr(), v.data_ptr(), k.stride(0), k.stride(1),
                                  k.stride(2), _ptr(scores, torch.float32, "scores", True),
                                  _ptr(tau, torch.float32, "tau", True), _ptr(tau_q, torch.float32, "tau_q", True),
                                  _ptr(flag_step, torch.int32, "flag_step", True), window, delay, reserve,
                                  _ptr(dst.kq_pool, torch.uint8), _ptr(dst.vq_pool, torch.uint8),
                                  _ptr(dst.meta_pool, torch.int32), dst.n_pages_cap,
                                  _ptr(dst.page_table, torch.int32), dst.max_pages, _ptr(dst.remap, torch.int32),
                                  _ptr(dst.count, torch.int32), ws.data_ptr(), ws.numel() * ws.element_size(),
                                  _ptr(status, torch.int32, "status"), _stream(stream))
    _check("kvp_compact_quant", code)
    return dst


def kvp_compact_paged_workspace_bytes(batch, n_kv_heads, src_max_pages) -> int:
    return _lib.kvp_compact_paged_workspace_bytes(batch, n_kv_heads, src_max_pages)


def kvp_compact_paged(src: PagedKV, now, reserve, dst: PagedKV, *, status, workspace=None, stream=None):
    B, H, _ = src.page_table.shape
    need = kvp_compact_paged_workspace_bytes(B, H, src.max_pages)
    ws = _ws(need, src.k_pool.device, workspace)
    code = _lib.kvp_compact_paged(B, H, src.head_dim, _ptr(src.k_pool), _ptr(src.v_pool),
                                  _ptr(src.expire_pool, torch.int32), src.n_pages_cap,
                                  _ptr(src.page_table, torch.int32), src.max_pages, _ptr(src.remap, torch.int32),
                                  _ptr(src.count, torch.int32), now, reserve, _ptr(dst.k_pool), _ptr(dst.v_pool),
                                  _ptr(dst.expire_pool, torch.int32), dst.n_pages_cap,
                                  _ptr(dst.page_table, torch.int32), dst.max_pages, _ptr(dst.remap, torch.int32),
                                  _ptr(dst.count, torch.int32), ws.data_ptr(), ws.numel() * ws.element_size(),
                                  _ptr(status, torch.int32, "status"), _stream(stream))
    _check("kvp_compact_paged", code)
    return dst


# --------------------------------------------------------------------------- append

def kvp_append(cache: PagedKV, k_new, v_new, pos, *, mode, score=None, tau=None, flag_step=None,
               window=WINDOW, delay=0, status, stream=None):
    """Writes the token at position `pos` (k_new, v_new [B, H, d]) into every (b, h)'s next slot."""
    B, H, d = k_new.shape
    code = _lib.kvp_append(mode, B, H, d, pos, _ptr(k_new, torch.bfloat16, "k_new"),
                           _ptr(v_new, torch.bfloat16, "v_new"), _ptr(score, torch.float32, "score", True),
                           _ptr(tau, torch.float32, "tau", True), _ptr(flag_step, torch.int32, "flag_step", True),
                           window, delay, _ptr(cache.k_pool), _ptr(cache.v_pool),
                           _ptr(cache.expire_pool, torch.int32), cache.n_pages_cap,
                           _ptr(cache.page_table, torch.int32), cache.max_pages, _ptr(cache.remap, torch.int32),
                           _ptr(cache.count, torch.int32), _ptr(status, torch.int32, "status"), _stream(stream))
    _check("kvp_append", code)


def kvp_append_devpos(cache: PagedKV, k_new, v_new, pos_dev, *, mode, score=None, tau=None, flag_step=None,
                      window=WINDOW, delay=0, status, stream=None):
    """kvp_append with the position taken from pos_dev (a device int32 tensor of one element) when the call
    runs on the stream, so that one captured CUDA graph serves every decode step."""
    B, H, d = k_new.shape
    code = _lib.kvp_append_devpos(mode, B, H, d, _ptr(pos_dev, torch.int32, "pos_dev"),
                                  _ptr(k_new, torch.bfloat16, "k_new"),
                                  _ptr(v_new, torch.bfloat16, "v_new"), _ptr(score, torch.float32, "score", True),
                                  _ptr(tau, torch.float32, "tau", True),
                                  _ptr(flag_step, torch.int32, "flag_step", True),
                                  window, delay, _ptr(cache.k_pool), _ptr(cache.v_pool),
                                  _ptr(cache.expire_pool, torch.int32), cache.n_pages_cap,
                                  _ptr(cache.page_table, torch.int32), cache.max_pages,
                                  _ptr(cache.remap, torch.int32), _ptr(cache.count, torch.int32),
                                  _ptr(status, torch.int32, "status"), _stream(stream))
    _check("kvp_append_devpos", code)


def kvp_append_quant(qcache: QuantPagedKV, k_new, v_new, pos, *, score=None, tau=None, tau_q=None,
                     mode=KVP_MASK_KVZAP, flag_step=None, delay=0, window=WINDOW, status, stream=None):
    """Writes the token at position `pos` (k_new, v_new [B, H, d]) into the fp8 tier of every (b, h) whose
    score falls in [tau_q, tau) (or, mode KVP_MASK_DMS, whose flag_step [B, H] is >= 0)."""
    B, H, d = k_new.shape
    code = _lib.kvp_append_quant(mode, B, H, d, pos, _ptr(k_new, torch.bfloat16, "k_new"),
                                 _ptr(v_new, torch.bfloat16, "v_new"), _ptr(score, torch.float32, "score", True),
                                 _ptr(tau, torch.float32, "tau", True), _ptr(tau_q, torch.float32, "tau_q", True),
                                 _ptr(flag_step, torch.int32, "flag_step", True), window, delay,
                                 _ptr(qcache.kq_pool, torch.uint8),
                                 _ptr(qcache.vq_pool, torch.uint8), _ptr(qcache.meta_pool, torch.int32),
                                 qcache.n_pages_cap, _ptr(qcache.page_table, torch.int32), qcache.max_pages,
                                 _ptr(qcache.remap, torch.int32), _ptr(qcache.count, torch.int32),
                                 _ptr(status, torch.int32, "status"), _stream(stream))
    _check("kvp_append_quant", code)


# --------------------------------------------------------------------------- attention

def kvp_decode_attn_workspace_bytes(batch, n_q_heads, n_kv_heads, head_dim) -> int:
    return _lib.kvp_decode_attn_workspace_bytes(batch, n_q_heads, n_kv_heads, head_dim)


def kvp_decode_attn(q, cache: PagedKV, now, *, scale=0.0, out=None, grid_limit=0, workspace=None,
                    status=None, stream=None):
    """out[B, Hq, d] fp32 = attention of q [B, Hq, d] (bf16) over the slots of `cache` present at `now`.
    A caller-provided workspace must be zero-filled before its first use (torch.zeros); calls that record
    no error leave it that way."""
    B, Hq, d = q.shape
    H = cache.count.shape[1]
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    need = kvp_decode_attn_workspace_bytes(B, Hq, H, d)
    if workspace is None:
        ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=q.device)  # zero-filled before first use
    else:
        ws = _ws(need, q.device, workspace)
    code = _lib.kvp_decode_attn(B, Hq, H, d, _ptr(q, torch.bfloat16, "q"), _ptr(cache.k_pool),
                                _ptr(cache.v_pool), _ptr(cache.expire_pool, torch.int32), cache.n_pages_cap,
                                _ptr(cache.page_table, torch.int32), cache.max_pages,
                                _ptr(cache.count, torch.int32), now, float(scale), _ptr(out, torch.float32, "out"),
                                grid_limit, ws.data_ptr(), ws.numel() * ws.element_size(),
                                _ptr(status, torch.int32, "status", True), _stream(stream))
    _check("kvp_decode_attn", code)
    return out


def kvp_decode_attn_lse(q, cache: PagedKV, now, *, scale=0.0, out=None, lse=None, grid_limit=0, workspace=None,
                        status=None, stream=None):
    """(out, lse): kvp_decode_attn's out [B, Hq, d] fp32 and each row's log-sum-exp lse [B, Hq] fp32 (ln of the
    sum of exp(scale q.k) over the present slots; -inf for an empty row). Workspace rules: kvp_decode_attn's."""
    B, Hq, d = q.shape
    H = cache.count.shape[1]
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = kvp_decode_attn_workspace_bytes(B, Hq, H, d)
    if workspace is None:
        ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=q.device)  # zero-filled before first use
    else:
        ws = _ws(need, q.device, workspace)
    code = _lib.kvp_decode_attn_lse(B, Hq, H, d, _ptr(q, torch.bfloat16, "q"), _ptr(cache.k_pool),
                                    _ptr(cache.v_pool), _ptr(cache.expire_pool, torch.int32), cache.n_pages_cap,
                                    _ptr(cache.page_table, torch.int32), cache.max_pages,
                                    _ptr(cache.count, torch.int32), now, float(scale),
                                    _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"),
                                    grid_limit, ws.data_ptr(), ws.numel() * ws.element_size(),
                                    _ptr(status, torch.int32, "status", True), _stream(stream))
    _check("kvp_decode_attn_lse", code)
    return out, lse


def kvp_attn_merge(outs, lses, *, out=None, lse=None, stream=None):
    """(out, lse) of attention over the union of disjoint parts, from each part's rows: outs [P, ..., d] fp32 and
    lses [P, ...] fp32 (kvp_decode_attn_lse's, stacked). out [..., d], lse [...]."""
    n_parts, d = outs.shape[0], outs.shape[-1]
    if lses.shape != outs.shape[:-1]:
        raise ValueError("lses must have the shape of outs without its last dimension")
    rows = lses[0].numel()
    if out is None:
        out = torch.empty(outs.shape[1:], dtype=torch.float32, device=outs.device)
    if lse is None:
        lse = torch.empty(lses.shape[1:], dtype=torch.float32, device=outs.device)
    code = _lib.kvp_attn_merge(n_parts, rows, d, _ptr(outs, torch.float32, "outs"), _ptr(lses, torch.float32, "lses"),
                               _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"), _stream(stream))
    _check("kvp_attn_merge", code)
    return out, lse


def kvp_decode_attn_devpos(q, cache: PagedKV, now_dev, *, scale=0.0, out=None, grid_limit=0, workspace=None,
                           status=None, stream=None):
    """kvp_decode_attn with the decode position taken from now_dev (a device int32 tensor of one element)
    when the call runs on the stream. Workspace rules: kvp_decode_attn's."""
    B, Hq, d = q.shape
    H = cache.count.shape[1]
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    need = kvp_decode_attn_workspace_bytes(B, Hq, H, d)
    if workspace is None:
        ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=q.device)  # zero-filled before first use
    else:
        ws = _ws(need, q.device, workspace)
    code = _lib.kvp_decode_attn_devpos(B, Hq, H, d, _ptr(q, torch.bfloat16, "q"), _ptr(cache.k_pool),
                                       _ptr(cache.v_pool), _ptr(cache.expire_pool, torch.int32), cache.n_pages_cap,
                                       _ptr(cache.page_table, torch.int32), cache.max_pages,
                                       _ptr(cache.count, torch.int32), _ptr(now_dev, torch.int32, "now_dev"),
                                       float(scale), _ptr(out, torch.float32, "out"),
                                       grid_limit, ws.data_ptr(), ws.numel() * ws.element_size(),
                                       _ptr(status, torch.int32, "status", True), _stream(stream))
    _check("kvp_decode_attn_devpos", code)
    return out


def kvp_decode_attn_two_tier(q, cache: PagedKV, qcache: QuantPagedKV, now, *, scale=0.0, out=None, grid_limit=0,
                             workspace=None, status=None, stream=None):
    """Attention of q [B, Hq, d] over the bf16 tier `cache` (slots with now < expire) and the fp8 tier
    `qcache` (slots with now >= start, dequantized) -> out [B, Hq, d] fp32."""
    B, Hq, d = q.shape
    H = cache.count.shape[1]
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    need = kvp_decode_attn_workspace_bytes(B, Hq, H, d)
    if workspace is None:
        ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=q.device)  # zero-filled before first use
    else:
        ws = _ws(need, q.device, workspace)
    code = _lib.kvp_decode_attn_two_tier(
        B, Hq, H, d, _ptr(q, torch.bfloat16, "q"), _ptr(cache.k_pool), _ptr(cache.v_pool),
        _ptr(cache.expire_pool, torch.int32), cache.n_pages_cap, _ptr(cache.page_table, torch.int32),
        cache.max_pages, _ptr(cache.count, torch.int32), _ptr(qcache.kq_pool, torch.uint8),
        _ptr(qcache.vq_pool, torch.uint8), _ptr(qcache.meta_pool, torch.int32), qcache.n_pages_cap,
        _ptr(qcache.page_table, torch.int32), qcache.max_pages, _ptr(qcache.count, torch.int32), now, float(scale),
        _ptr(out, torch.float32, "out"), grid_limit, ws.data_ptr(), ws.numel() * ws.element_size(),
        _ptr(status, torch.int32, "status", True), _stream(stream))
    _check("kvp_decode_attn_two_tier", code)
    return out


def kvp_selftest_wait(limit_ns, *, status, waited_us=None, stream=None):
    """One warp waits on an mbarrier that nothing arrives on, with the bounded wait every kernel uses: after
    limit_ns it records KVP_ERR_TIMEOUT in status (device int32) and returns; waited_us (device uint32 [1], or
    None) receives how long the wait lasted."""
    code = _lib.kvp_selftest_wait(int(limit_ns), _ptr(status, torch.int32, "status"),
                                  _ptr(waited_us, None, "waited_us", True), _stream(stream))
    _check("kvp_selftest_wait", code)


# --------------------------------------------------------------------------- MLA latent cache

@dataclass
class LatentPagedKV:
    """Device buffers of one compacted MLA latent cache: one "kv head", one pool of latent rows."""
    pool: torch.Tensor          # bf16 [n_pages_cap, 16, 576]
    expire_pool: torch.Tensor   # int32 [n_pages_cap, 16]
    page_table: torch.Tensor    # int32 [B, max_pages]
    remap: torch.Tensor         # int32 [B, max_pages * 16]
    count: torch.Tensor         # int32 [B]

    @staticmethod
    def allocate(batch, n_pages_cap, max_pages, device="cuda"):
        return LatentPagedKV(
            torch.zeros((n_pages_cap, PAGE, LATENT_ROW), dtype=torch.bfloat16, device=device),
            torch.zeros((n_pages_cap, PAGE), dtype=torch.int32, device=device),
            torch.full((batch, max_pages), -1, dtype=torch.int32, device=device),
            torch.full((batch, max_pages * PAGE), -1, dtype=torch.int32, device=device),
            torch.zeros((batch,), dtype=torch.int32, device=device),
        )

    @property
    def n_pages_cap(self):
        return self.pool.shape[0]

    @property
    def max_pages(self):
        return self.page_table.shape[1]

    @property
    def batch(self):
        return self.count.shape[0]


def kvp_compact_latent(lat, now, reserve, dst: LatentPagedKV, *, mode, scores=None, tau=None, flag_step=None,
                       window=WINDOW, delay=0, status, workspace=None, stream=None):
    """Dense latent rows [B, T, 576] (row contiguous) with the mask applied on the fly: KVzap scores [B, T]
    (or [B*T, 1]) + tau [B], or DMS flag_step [B, T] -> dst."""
    B, T, R = lat.shape
    if lat.dtype != torch.bfloat16 or not lat.is_cuda or lat.stride(2) != 1:
        raise TypeError("lat must be a CUDA bf16 tensor with contiguous rows")
    if scores is not None and scores.numel() != B * T:
        raise ValueError("scores must hold B*T values")
    if flag_step is not None and flag_step.numel() != B * T:
        raise ValueError("flag_step must hold B*T values")
    if tau is not None and tau.numel() != B:
        raise ValueError("tau must hold B values")
    ws = _ws(kvp_compact_workspace_bytes(B, 1, T), lat.device, workspace)
    code = _lib.kvp_compact_latent(mode, B, R, T, lat.data_ptr(), lat.stride(0), lat.stride(1),
                                   _ptr(scores, torch.float32, "scores", True), _ptr(tau, torch.float32, "tau", True),
                                   _ptr(flag_step, torch.int32, "flag_step", True), window, delay, now, reserve,
                                   _ptr(dst.pool, torch.bfloat16), _ptr(dst.expire_pool, torch.int32),
                                   dst.n_pages_cap, _ptr(dst.page_table, torch.int32), dst.max_pages,
                                   _ptr(dst.remap, torch.int32), _ptr(dst.count, torch.int32), ws.data_ptr(),
                                   ws.numel() * ws.element_size(), _ptr(status, torch.int32, "status"),
                                   _stream(stream))
    _check("kvp_compact_latent", code)
    return dst


def kvp_compact_latent_paged(src: LatentPagedKV, now, reserve, dst: LatentPagedKV, *, status, workspace=None,
                             stream=None):
    """Re-compaction of a latent cache: its slots present at `now`, in slot order, into dst."""
    B = src.batch
    ws = _ws(kvp_compact_paged_workspace_bytes(B, 1, src.max_pages), src.pool.device, workspace)
    code = _lib.kvp_compact_latent_paged(B, src.pool.shape[2], _ptr(src.pool, torch.bfloat16),
                                         _ptr(src.expire_pool, torch.int32), src.n_pages_cap,
                                         _ptr(src.page_table, torch.int32), src.max_pages,
                                         _ptr(src.remap, torch.int32), _ptr(src.count, torch.int32), now, reserve,
                                         _ptr(dst.pool, torch.bfloat16), _ptr(dst.expire_pool, torch.int32),
                                         dst.n_pages_cap, _ptr(dst.page_table, torch.int32), dst.max_pages,
                                         _ptr(dst.remap, torch.int32), _ptr(dst.count, torch.int32), ws.data_ptr(),
                                         ws.numel() * ws.element_size(), _ptr(status, torch.int32, "status"),
                                         _stream(stream))
    _check("kvp_compact_latent_paged", code)
    return dst


def kvp_append_latent(cache: LatentPagedKV, lat_new, pos, *, mode, score=None, tau=None, flag_step=None,
                      window=WINDOW, delay=0, status, stream=None):
    """Writes the token at position `pos` (lat_new [B, 576]) into every batch element's next slot."""
    B, R = lat_new.shape
    code = _lib.kvp_append_latent(mode, B, R, pos, _ptr(lat_new, torch.bfloat16, "lat_new"),
                                  _ptr(score, torch.float32, "score", True), _ptr(tau, torch.float32, "tau", True),
                                  _ptr(flag_step, torch.int32, "flag_step", True), window, delay,
                                  _ptr(cache.pool, torch.bfloat16), _ptr(cache.expire_pool, torch.int32),
                                  cache.n_pages_cap, _ptr(cache.page_table, torch.int32), cache.max_pages,
                                  _ptr(cache.remap, torch.int32), _ptr(cache.count, torch.int32),
                                  _ptr(status, torch.int32, "status"), _stream(stream))
    _check("kvp_append_latent", code)


def kvp_decode_attn_mla_workspace_bytes(batch, n_q_heads, n_splits=0) -> int:
    return _lib.kvp_decode_attn_mla_workspace_bytes(batch, n_q_heads, n_splits)


def kvp_decode_attn_mla(q, cache: LatentPagedKV, now, *, scale=0.0, out=None, n_splits=0, workspace=None,
                        status=None, stream=None):
    """out[B, Hq, 512] fp32 = absorbed MLA attention of q [B, Hq, 576] (bf16) over the latent slots of `cache`
    present at `now`. The workspace needs no clearing between calls."""
    B, Hq, R = q.shape
    if R != LATENT_ROW:
        raise ValueError(f"q rows must hold {LATENT_ROW} values")
    if out is None:
        out = torch.empty((B, Hq, KVP_MLA_LATENT_DIM), dtype=torch.float32, device=q.device)
    need = kvp_decode_attn_mla_workspace_bytes(B, Hq, n_splits)
    ws = _ws(need, q.device, workspace)
    code = _lib.kvp_decode_attn_mla(B, Hq, KVP_MLA_LATENT_DIM, KVP_MLA_ROPE_DIM, _ptr(q, torch.bfloat16, "q"),
                                    _ptr(cache.pool, torch.bfloat16), _ptr(cache.expire_pool, torch.int32),
                                    cache.n_pages_cap, _ptr(cache.page_table, torch.int32), cache.max_pages,
                                    _ptr(cache.count, torch.int32), now, float(scale),
                                    _ptr(out, torch.float32, "out"), n_splits, ws.data_ptr(),
                                    ws.numel() * ws.element_size(), _ptr(status, torch.int32, "status", True),
                                    _stream(stream))
    _check("kvp_decode_attn_mla", code)
    return out


__all__ = [n for n in dir() if n.startswith(("kvp_", "KVP_", "PagedKV", "QuantPagedKV", "LatentPagedKV",
                                             "KvpError"))] + [
    "status_string", "version", "library", "PAGE", "WINDOW", "EXPIRE_NEVER", "LATENT_ROW"]
