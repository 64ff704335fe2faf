"""Helpers shared by the GPU parity tests (comparison metrics and oracle calls)."""
import numpy as np
import torch

import oracle

F32 = lambda v: float(np.float32(v))


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def rel_fro(got, want) -> float:
    d = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (d if d > 0 else 1.0))


def ordered_f32(a: np.ndarray) -> np.ndarray:
    i = np.ascontiguousarray(a, dtype=np.float32).view(np.int32).astype(np.int64)
    return np.where(i < 0, -(i & 0x7FFFFFFF), i)


def ulp_diff_f32(a, b) -> np.ndarray:
    return np.abs(ordered_f32(a) - ordered_f32(b))


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def hyper(**kw) -> oracle.MuonHyper:
    """Oracle hyperparameters as the fp32 values the GPU receives."""
    base = dict(mu=0.95, gamma=0.18, lr=2.7e-4, weight_decay=0.1)
    base.update(kw)
    for k in ("mu", "gamma", "lr", "weight_decay"):
        base[k] = F32(base[k])
    return oracle.MuonHyper(**base)


def check_w(W_gpu: np.ndarray, W_ref: np.ndarray, hp: oracle.MuonHyper, scale: float, bf16: bool):
    """max|W_gpu - W_ref| <= 1e-2*lr*scale (+ half a bf16 ulp for bf16 storage)."""
    tol = 1e-2 * hp.lr * scale
    err = np.abs(W_gpu - W_ref)
    bound = tol + (0.5 * bf16_ulp(np.abs(W_ref) + tol) if bf16 else 0.0)
    worst = float(np.max(err - bound))
    assert worst <= 0.0, f"W error exceeds bound by {worst:.3e} (tol {tol:.3e})"
    return float(np.max(err))


def momentum_ref_f32(M_prev: np.ndarray, G: np.ndarray, hp: oracle.MuonHyper) -> np.ndarray:
    if hp.style == "sgd":
        return oracle.momentum_sgd(M_prev, G, hp.mu).astype(np.float32)
    return oracle.momentum_ema(M_prev, G, hp.mu).astype(np.float32)
