"""Shared helpers for the GPU parity tests: moving seeded inputs between numpy
bf16 bit patterns and torch tensors, and the tolerance checks."""
import numpy as np
import torch


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
