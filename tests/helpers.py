"""Shared helpers for the GPU parity tests: moving seeded inputs between numpy
bf16 bit patterns and torch tensors, and the tolerance checks."""
import numpy as np
import torch

import oracle as orc


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev_f32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def dev_i32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def status_word(device="cuda") -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def check_scores(s_gpu: np.ndarray, s_ref: np.ndarray, scale: np.ndarray, rel=1e-3):
    """|s_gpu - s_ref| <= rel * max(|s_ref|, scale): scale is the natural size of
    the sum's terms (the 2-norm of x_t * w_h); returns the worst ratio."""
    bound = rel * np.maximum(np.abs(s_ref), scale)
    err = np.abs(s_gpu.astype(np.float64) - s_ref)
    worst = float((err / bound).max()) if err.size else 0.0
    assert (err <= bound).all(), f"score error ratio {worst:.3g} > 1"
    return worst


def check_attention(o_gpu: np.ndarray, o_ref: np.ndarray, max_abs=2e-2, mean_abs=2e-3, rel_head=1e-2):
    """Attention tolerances: max-abs 2e-2 and mean-abs 2e-3 over all elements,
    and a per-(b, head) relative 2-norm bound of 1e-2 (the absolute bounds alone
    say little when outputs are ~1/sqrt(n) small)."""
    d = np.abs(o_gpu.astype(np.float64) - o_ref.astype(np.float64))
    assert d.max() <= max_abs, f"max abs err {d.max():.3g}"
    assert d.mean() <= mean_abs, f"mean abs err {d.mean():.3g}"
    num = np.linalg.norm((o_gpu.astype(np.float64) - o_ref), axis=-1)
    den = np.linalg.norm(o_ref.astype(np.float64), axis=-1)
    rel = np.where(den > 0, num / np.maximum(den, 1e-30), num)
    assert rel.max() <= rel_head, f"per-head relative err {rel.max():.3g}"
    return float(d.max()), float(d.mean()), float(rel.max())


def oracle_linear_scores(x, w, chunk=16384):
    """The oracle's KVzap-Linear scores of every row of x, in row chunks (the
    widened float64 rows of a whole full-size x would not fit in host memory),
    and the error scale ||x_t * w_h||_2 of each score."""
    out = np.empty((x.shape[0], w.shape[0]))
    scale = np.empty_like(out)
    w64 = np.asarray(w, np.float64)
    for a in range(0, x.shape[0], chunk):
        xs = orc.widen_bf16(x[a:a + chunk])
        out[a:a + chunk] = orc.score_linear(x[a:a + chunk], w)
        scale[a:a + chunk] = np.sqrt((xs * xs) @ (w64 ** 2).T)
    return out, scale


def oracle_mlp_scores(x, w1, w2, b1=None, b2=None, chunk=8192):
    """The oracle's KVzap-MLP scores of every row of x, in row chunks, and the
    error scale of each: the 2-norm of the hidden terms z_j * w2[h, j]."""
    H = w2.shape[0]
    out = np.empty((x.shape[0], H))
    scale = np.empty_like(out)
    w1f = orc.widen_bf16(w1)
    w2f = orc.widen_bf16(w2)
    for a in range(0, x.shape[0], chunk):
        out[a:a + chunk] = orc.score_mlp(x[a:a + chunk], w1, w2, b1, b2)
        u = orc.widen_bf16(x[a:a + chunk]) @ w1f.T + (0 if b1 is None else np.asarray(b1, np.float64)[None, :])
        z = orc.gelu(u)
        scale[a:a + chunk] = np.sqrt((z * z) @ (w2f ** 2).T)
    return out, scale


def compare_paged(gpu, ref, used=None, what=""):
    """Bit-exact comparison of a compacted cache with the oracle's: counts,
    page table, remap list, and the used pages of the pools and expire_pool."""
    used = ref.pages_used if used is None else used
    np.testing.assert_array_equal(gpu.count.cpu().numpy(), ref.count, err_msg=what + " count")
    np.testing.assert_array_equal(gpu.page_table.cpu().numpy(), ref.page_table, err_msg=what + " page_table")
    np.testing.assert_array_equal(gpu.remap.cpu().numpy(), ref.remap, err_msg=what + " remap")
    np.testing.assert_array_equal(gpu.expire_pool.cpu().numpy()[:used], ref.expire_pool[:used],
                                  err_msg=what + " expire_pool")
    np.testing.assert_array_equal(host_bits(gpu.k_pool)[:used], ref.k_pool[:used], err_msg=what + " k_pool")
    np.testing.assert_array_equal(host_bits(gpu.v_pool)[:used], ref.v_pool[:used], err_msg=what + " v_pool")
