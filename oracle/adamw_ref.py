"""Float64 CPU oracle for the AdamW partition of a Muon optimizer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
it.  It shares no code with the CUDA path and imports nothing from it.

Sources (web pages, cited by title and section):

* "Muon 优化器" (DeepSeek-V4 tech notes), §3 "哪些参数用 Muon，哪些仍用
  AdamW": embeddings, the output head, norm scales and other vector or
  scalar parameters stay on AdamW; its hyperparameters are beta1 = 0.9,
  beta2 = 0.95, eps = 1e-20, weight decay 0.1.  The same page's reading of
  Algorithm 1 says Muon's decoupled weight decay has AdamW's form
  W <- W*(1 - lr*wd) - lr*update.
* "RFC-0023: 对齐 MaxText Muon 优化器实现与 Megatron-LM 完整行为",
  §方案 2 (Weight Decay Masking): the AdamW partition takes a per-tensor
  decay mask (biases off, norm scales configurable, embeddings and the
  output layer on, everything else on).

Reading where the pages are silent: the pages name
AdamW without writing its update; it is taken as Adam with bias correction
and decoupled decay (Loshchilov & Hutter), eps added outside the square
root, which is the form optax's ``adamw`` and PyTorch's ``AdamW`` compute:

    m_t = beta1*m + (1 - beta1)*g
    v_t = beta2*v + (1 - beta2)*g^2
    u   = (m_t / (1 - beta1^t)) / (sqrt(v_t / (1 - beta2^t)) + eps)
    W_t = W*(1 - lr*wd*mask) - lr*u

with t >= 1 counting steps including this one.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# "Muon 优化器" §3: the AdamW side of the V4 settings
BETA1 = 0.9
BETA2 = 0.95
EPS = 1e-20
WEIGHT_DECAY = 0.1


@dataclass
class AdamWHyper:
    lr: float = 2.7e-4
    beta1: float = BETA1
    beta2: float = BETA2
    eps: float = EPS
    weight_decay: float = WEIGHT_DECAY
    t: int = 1


def first_moment(m: np.ndarray, g: np.ndarray, beta1: float) -> np.ndarray:
    """Exponential average of the gradient, m_t = beta1*m + (1 - beta1)*g."""
    return beta1 * np.asarray(m, np.float64) + (1.0 - beta1) * np.asarray(g, np.float64)


def second_moment(v: np.ndarray, g: np.ndarray, beta2: float) -> np.ndarray:
    """Exponential average of the squared gradient, v_t = beta2*v + (1 - beta2)*g^2."""
    g = np.asarray(g, np.float64)
    return beta2 * np.asarray(v, np.float64) + (1.0 - beta2) * g * g


def adam_direction(m_t: np.ndarray, v_t: np.ndarray, beta1: float, beta2: float, eps: float,
                   t: int) -> np.ndarray:
    """Bias-corrected ratio m_hat / (sqrt(v_hat) + eps)."""
    if t < 1:
        raise ValueError("t counts steps from 1")
    m_hat = m_t / (1.0 - beta1 ** t)
    v_hat = v_t / (1.0 - beta2 ** t)
    return m_hat / (np.sqrt(v_hat) + eps)


def adamw_step(W: np.ndarray, G: np.ndarray, m: np.ndarray, v: np.ndarray, hp: AdamWHyper,
               decay: bool = True) -> dict:
    """One AdamW step for one tensor; returns the new m, v, W and the direction u."""
    m_t = first_moment(m, G, hp.beta1)
    v_t = second_moment(v, G, hp.beta2)
    u = adam_direction(m_t, v_t, hp.beta1, hp.beta2, hp.eps, hp.t)
    keep = 1.0 - hp.lr * hp.weight_decay if decay else 1.0
    W_t = np.asarray(W, np.float64) * keep - hp.lr * u
    return {"m": m_t, "v": v_t, "u": u, "W": W_t}
