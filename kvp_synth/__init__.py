"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module only draws random numbers and stores them in the dtypes the
library consumes. It holds none of the pruning method's arithmetic: no scoring,
masking, compaction or attention happens here.

Generator (counter based, so any element can be drawn without the others):

* ``splitmix64``: the SplitMix64 output function (Steele, Lea & Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014) applied to
  ``key + (i + 1) * GAMMA``, where ``key`` is derived from ``(seed, stream)``.
* uniforms in [0, 1): the top 53 bits of a draw times 2**-53.
* normals: Box-Muller on consecutive uniform pairs, in float64.
* bf16: float64 -> float32 -> bf16 with round-to-nearest-even; stored as
  ``uint16`` bit patterns so that numpy (which has no bf16) and torch can share
  the exact same bits.

Every tensor of a workload gets its own ``stream`` id, so the same seed gives
the same bits regardless of which other tensors are drawn.

Tensors of a billion elements (the full-size workloads) take minutes with the
generator above in numpy, so ``fast_normal_bf16`` draws them with numpy's
Philox4x64-10 bit generator (Salmon, Moraes, Dror & Shaw, "Parallel random
numbers: as easy as 1, 2, 3", SC 2011), also counter based, keyed by
``(seed, stream)`` and advanced to each chunk's start; its normals are
numpy's float32 ziggurat. The two generators give different numbers: a
workload uses one of them for all its draws.
"""
from __future__ import annotations

import math

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        base = np.array([(seed * 0x100000001B3 + stream * 0x9E3779B1 + 1) & 0xFFFFFFFFFFFFFFFF],
                        dtype=np.uint64)
        return _mix(base)[0]


def splitmix64(seed: int, stream: int, start: int, n: int) -> np.ndarray:
    """Draws ``start .. start+n-1`` of the counter-based sequence (uint64)."""
    key = _key(seed, stream)
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + i * GAMMA)


def uniform(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """float64 uniforms in [0, 1)."""
    out = np.empty(n, dtype=np.float64)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        r = splitmix64(seed, stream, start + c0, c1 - c0)
        out[c0:c1] = (r >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    return out


def normal(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """float64 N(mean, std^2) by Box-Muller on uniform pairs (2i, 2i+1)."""
    out = np.empty(n, dtype=np.float64)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        out[c0:c1] = _normal_slice(seed, stream, c0, c1 - c0)
    return out * std + mean


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def normal_bf16(seed: int, stream: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """N(mean, std^2) rounded to bf16, as uint16 bits of the given shape."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for c0 in range(0, n, _CHUNK * 4):
        c1 = min(n, c0 + _CHUNK * 4)
        # draw the slice c0..c1 of the same stream: Box-Muller pairs align on even c0
        z = _normal_slice(seed, stream, c0, c1 - c0) * std + mean
        out[c0:c1] = f32_to_bf16_bits(z.astype(np.float32))
    return out.reshape(shape)


def _normal_slice(seed: int, stream: int, start: int, n: int) -> np.ndarray:
    assert start % 2 == 0
    npair = (n + 1) // 2
    u = uniform(seed, stream, 2 * npair, start=start)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log1p(-u1))
    th = 2.0 * math.pi * u2
    z = np.empty(2 * npair, dtype=np.float64)
    z[0::2] = r * np.cos(th)
    z[1::2] = r * np.sin(th)
    return z[:n]


_FAST_CHUNK = 1 << 24


def _philox(seed: int, stream: int, start: int) -> np.random.Generator:
    key = np.array([seed & 0xFFFFFFFFFFFFFFFF, stream & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return np.random.Generator(np.random.Philox(key=key).advance(start * 4))


def fast_normal_bf16(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) rounded to bf16 (uint16 bits of the given shape). Chunk c
    of 2^24 values comes from a Philox4x64-10 generator keyed by (seed,
    stream) and advanced by c * 2^24 blocks (a normal uses at most a few
    draws, so chunks never overlap in practice); chunks are drawn on all host
    cores, so the result does not depend on the thread count. The float32 ->
    bf16 rounding (nearest even) is torch's conversion, multithreaded; it
    gives the same bits as f32_to_bf16_bits on finite values."""
    import concurrent.futures as cf
    import os

    import torch

    n = int(np.prod(shape))
    z = np.empty(n, dtype=np.float32)

    def chunk(c0):
        c1 = min(n, c0 + _FAST_CHUNK)
        _philox(seed, stream, c0).standard_normal(dtype=np.float32, out=z[c0:c1])
        if std != 1.0:
            z[c0:c1] *= np.float32(std)

    with cf.ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
        list(ex.map(chunk, range(0, n, _FAST_CHUNK)))
    out = torch.from_numpy(z).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return out.reshape(shape)


def fast_uniform(seed: int, stream: int, shape) -> np.ndarray:
    """float64 uniforms in [0, 1) from the same Philox keying as fast_normal_bf16."""
    return _philox(seed, stream, 0).random(int(np.prod(shape))).reshape(shape)


def normal_f32(seed: int, stream: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return normal(seed, stream, n, mean, std).astype(np.float32).reshape(shape)


def bernoulli(seed: int, stream: int, shape, p: float) -> np.ndarray:
    """Boolean array, True with probability p (u < p)."""
    n = int(np.prod(shape))
    return (uniform(seed, stream, n) < p).reshape(shape)


def beta_2_5(seed: int, stream: int, shape) -> np.ndarray:
    """Beta(2, 5) draws as the 2nd smallest of 6 iid uniforms (order statistic U(2:6))."""
    n = int(np.prod(shape))
    u = uniform(seed, stream, 6 * n).reshape(n, 6)
    return np.sort(u, axis=1)[:, 1].reshape(shape)


# ---------------------------------------------------------------------------
# Stream ids: one per tensor role, shared by every workload.
# ---------------------------------------------------------------------------
S_X, S_W, S_W1, S_W2, S_K, S_V, S_Q, S_FLAG, S_KEEPRATE, S_LAT = 1, 2, 3, 4, 5, 6, 7, 8, 9, 10
S_STEP = 1000  # + 16 * step + role, for per-decode-step tensors


def step_stream(step: int, role: int) -> int:
    return S_STEP + 16 * step + role


# ---------------------------------------------------------------------------
# Workload shapes (synthetic stand-ins for the pages' model shapes)
# ---------------------------------------------------------------------------
WORKLOADS = {
    # tiny: 1 layer, d_model 256, 4 q heads / 2 kv heads, head_dim 64, batch 1, 512 cached
    "tiny": dict(d_model=256, n_q_heads=4, n_kv_heads=2, head_dim=64, batch=1, n_pos=512,
                 scorer="linear", prune_q=0.5),
    # Llama-3-8B-shaped layer, one decode step over a 8192-token cache
    "llama3_8b_layer": dict(d_model=4096, n_q_heads=32, n_kv_heads=8, head_dim=128, batch=16,
                            n_pos=8192, scorer="linear", prune_q=0.75),
    # KVzap-MLP prefill scoring then 64 decode steps
    "mlp_prefill": dict(d_model=4096, hidden=1024, n_q_heads=32, n_kv_heads=8, head_dim=128,
                        batch=4, n_pos=32768, scorer="mlp", prune_q=0.8, steps=64, reserve=64),
    # DMS delayed-eviction decode loop, Qwen-3-8B-shaped attention
    "dms_decode": dict(n_q_heads=32, n_kv_heads=8, head_dim=128, batch=64, n_pos=4096,
                       steps=1024, evict_p=7.0 / 8.0, delay=256, recompact_every=64, reserve=64),
    # MLA latent cache (DeepSeek-V3-shaped attention: 128 query heads, latent rows of 512 + 64),
    # one decode step over a 8192-token cache
    "mla_layer": dict(n_q_heads=128, latent_dim=512, rope_dim=64, batch=16, n_pos=8192, prune_q=0.75),
    # Llama-65B-shaped MHA stress, 8 layers, 131072 cached tokens
    "llama65b_mha": dict(n_layers=8, d_model=8192, n_q_heads=64, n_kv_heads=64, head_dim=128,
                         batch=1, n_pos=131072, scorer="linear", steps=32, reserve=32),
}


def linear_inputs(seed: int, n_tok: int, d_model: int, n_kv_heads: int, layer: int = 0):
    """Hidden states x ~ N(0,1) bf16 [n_tok, D] and KVzap-Linear W ~ N(0, 1/D) fp32 [H, D]."""
    off = 100 * layer
    x = normal_bf16(seed, S_X + off, (n_tok, d_model))
    w = normal_f32(seed, S_W + off, (n_kv_heads, d_model), std=1.0 / math.sqrt(d_model))
    return x, w


def mlp_inputs(seed: int, n_tok: int, d_model: int, hidden: int, n_kv_heads: int):
    """x ~ N(0,1); W1 [hidden, D] ~ N(0, 1/D); W2 [H, hidden] ~ N(0, 1/hidden); all bf16."""
    x = normal_bf16(seed, S_X, (n_tok, d_model))
    w1 = normal_bf16(seed, S_W1, (hidden, d_model), std=1.0 / math.sqrt(d_model))
    w2 = normal_bf16(seed, S_W2, (n_kv_heads, hidden), std=1.0 / math.sqrt(hidden))
    return x, w1, w2


def kv_inputs(seed: int, batch: int, n_pos: int, n_kv_heads: int, head_dim: int, layer: int = 0):
    """Dense K, V ~ N(0,1) bf16 in [B, T, H, d] layout."""
    off = 100 * layer
    k = normal_bf16(seed, S_K + off, (batch, n_pos, n_kv_heads, head_dim))
    v = normal_bf16(seed, S_V + off, (batch, n_pos, n_kv_heads, head_dim))
    return k, v


def latent_inputs(seed: int, batch: int, n_pos: int, row: int = 576):
    """MLA latent rows (compressed KV then rotary key) ~ N(0,1) bf16 [B, T, row]."""
    return normal_bf16(seed, S_LAT, (batch, n_pos, row))


def q_inputs(seed: int, batch: int, n_q_heads: int, head_dim: int, stream: int = S_Q):
    return normal_bf16(seed, stream, (batch, n_q_heads, head_dim))
