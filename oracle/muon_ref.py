"""Float64 CPU oracle for the Muon optimizer step on 2-D weight matrices.

TEST INFRASTRUCTURE ONLY.  This module is the slow, plain statement of what
the GPU library computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  It
shares no code with the CUDA path and imports nothing from it.

Sources (web pages, cited by title and section):

* "Muon 优化器" (DeepSeek-V4 tech notes), §1 "Muon 一步在做什么",
  Algorithm 1:  G_t = grad,  M_t = mu*M_{t-1} + G_t,
  O'_t = HybridNewtonSchulz(mu*M_t + G_t),  O_t = O'_t*sqrt(max(n,m))*gamma,
  W_t = W_{t-1}*(1 - eta*lambda) - eta*O_t.
* same page, §2 "Hybrid Newton–Schulz 正交化": normalise by the Frobenius
  norm, then repeat M_k = a*M + b*(M M^T) M + c*(M M^T)^2 M; eight steps with
  (3.4445, -4.7750, 2.0315) followed by two with (2.0, -1.5, 0.5); a zero
  input is returned unchanged.
* same page, §3: mu = 0.95, weight decay 0.1, gamma = 0.18; the hybrid
  schedule's teaching code uses lr = 2.7e-4.
* "RFC-0023: 对齐 MaxText Muon 优化器实现与 Megatron-LM 完整行为", §方案 1
  (Nesterov 动量对齐): the 'sgd' style (buf = beta*buf + g; look-ahead
  g + beta*buf) and the 'ema' style (mu = beta*mu + (1-beta)*g, look-ahead
  beta*bc(mu, t+1) + (1-beta)*bc(g, t)).
* RFC-0023 §方案 2 (Weight Decay Masking): per-tensor decay on/off.
* RFC-0023 §方案 3 (consistent_rms) and §背景: spectral scale
  sqrt(max(fan_in, fan_out))*consistent_rms; with split_head the heads are a
  batch dimension and fan_out is the head size.
* "Scaling for MuP over Muon optimizer" (Megatron-LM PR #3715), "What does
  this PR do": the alternative 'unit_rms_norm' scale sqrt(fan_out / fan_in).
* RFC-0023 §方案 4 (muon_batch_update): same-shape matrices are stacked and
  orthogonalised in one batched call, chunked by a batch size.

Readings where the pages are silent:

* bias correction bc(x, k) = x / (1 - beta**k), with t >= 1 counting steps
  including the current one;
* unit_rms_norm carries no gamma; gamma multiplies only the spectral scale;
* for a tall matrix the iteration runs on the transpose (the Gram of the
  smaller side) and the result is transposed back; in exact arithmetic this is
  the same map as the page's formula (see ``newton_schulz_literal``);
* everything is float64; inputs are the exact values the GPU receives
  (bf16 / fp32 widened), hyperparameters are passed as the caller chooses
  (tests pass the fp32 values the GPU is given).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Iterable, Sequence

import numpy as np

# ---------------------------------------------------------------------------
# Newton–Schulz schedule ("Muon 优化器" §2, hybrid 8 + 2 schedule)
# ---------------------------------------------------------------------------
FAST_COEFFS = (3.4445, -4.7750, 2.0315)
STABLE_COEFFS = (2.0, -1.5, 0.5)
HYBRID_STAGES: tuple[tuple[int, tuple[float, float, float]], ...] = (
    (8, FAST_COEFFS),
    (2, STABLE_COEFFS),
)

# Default hyperparameters ("Muon 优化器" §3; the teaching step's lr).
DEFAULT_MU = 0.95
DEFAULT_GAMMA = 0.18
DEFAULT_LR = 2.7e-4
DEFAULT_WD = 0.1


def expand_stages(stages: Iterable[tuple[int, Sequence[float]]]) -> list[tuple[float, float, float]]:
    """Flatten (steps, (a, b, c)) stages into one (a, b, c) per iteration."""
    out: list[tuple[float, float, float]] = []
    for steps, (a, b, c) in stages:
        if steps < 0:
            raise ValueError("negative step count")
        out.extend([(float(a), float(b), float(c))] * int(steps))
    return out


# ---------------------------------------------------------------------------
# Momentum and the Nesterov look-ahead
# ---------------------------------------------------------------------------
def momentum_sgd(M_prev: np.ndarray, G: np.ndarray, mu: float) -> np.ndarray:
    """M_t = mu * M_{t-1} + G_t  (Algorithm 1; RFC-0023 §方案 1 'sgd')."""
    return mu * np.asarray(M_prev, np.float64) + np.asarray(G, np.float64)


def lookahead_sgd(M_t: np.ndarray, G: np.ndarray, mu: float) -> np.ndarray:
    """Nesterov look-ahead mu * M_t + G_t, no bias correction (Algorithm 1)."""
    return mu * np.asarray(M_t, np.float64) + np.asarray(G, np.float64)


def bias_correct(x: np.ndarray, beta: float, k: int) -> np.ndarray:
    """bc(x, k) = x / (1 - beta**k): Adam-style bias correction (reading of
    RFC-0023 §方案 1, which names bc without defining it)."""
    if k < 1:
        raise ValueError("bias correction needs k >= 1")
    return np.asarray(x, np.float64) / (1.0 - beta ** k)


def momentum_ema(mu_prev: np.ndarray, G: np.ndarray, beta: float) -> np.ndarray:
    """mu_t = beta * mu_{t-1} + (1 - beta) * g  (RFC-0023 §方案 1 'ema')."""
    return beta * np.asarray(mu_prev, np.float64) + (1.0 - beta) * np.asarray(G, np.float64)


def lookahead_ema(mu_t: np.ndarray, G: np.ndarray, beta: float, t: int) -> np.ndarray:
    """beta * bc(mu_t, t+1) + (1 - beta) * bc(g, t)  (RFC-0023 §方案 1 'ema')."""
    return beta * bias_correct(mu_t, beta, t + 1) + (1.0 - beta) * bias_correct(G, beta, t)


# ---------------------------------------------------------------------------
# Hybrid Newton–Schulz ("Muon 优化器" §2)
# ---------------------------------------------------------------------------
def frobenius_normalize(X: np.ndarray) -> tuple[np.ndarray, float]:
    """X / ||X||_F; a zero matrix is returned unchanged (the page's zero guard)."""
    X = np.asarray(X, np.float64)
    nrm = math.sqrt(float(np.sum(X * X)))
    if nrm == 0.0:
        return X.copy(), 0.0
    return X / nrm, nrm


def ns_iteration(X: np.ndarray, a: float, b: float, c: float) -> np.ndarray:
    """One step a*X + b*(X X^T) X + c*(X X^T)^2 X for a wide X (rows <= cols).

    Terms in the order of the equation in "Muon 优化器" §2: with
    S = X X^T, the b-term is S X and the c-term is S (S X)."""
    S = X @ X.T
    SX = S @ X
    return a * X + b * SX + c * (S @ SX)


def newton_schulz(X: np.ndarray,
                  stages: Iterable[tuple[int, Sequence[float]]] = HYBRID_STAGES,
                  normalize: bool = True) -> np.ndarray:
    """O' = HybridNewtonSchulz(X) in float64 ("Muon 优化器" §2).

    A tall matrix is iterated as its transpose (Gram of the smaller side) and
    transposed back; in exact arithmetic this equals iterating X itself.
    With ``normalize`` false the Frobenius normalisation is skipped."""
    X = np.asarray(X, np.float64)
    if X.ndim != 2:
        raise ValueError("newton_schulz takes one 2-D matrix")
    tall = X.shape[0] > X.shape[1]
    Y = X.T.copy() if tall else X.copy()
    if normalize:
        Y, nrm = frobenius_normalize(Y)
        if nrm == 0.0:
            return Y.T.copy() if tall else Y
    for a, b, c in expand_stages(stages):
        Y = ns_iteration(Y, a, b, c)
    return Y.T.copy() if tall else Y


def newton_schulz_literal(X: np.ndarray,
                          stages: Iterable[tuple[int, Sequence[float]]] = HYBRID_STAGES,
                          normalize: bool = True) -> np.ndarray:
    """Second transcription of the §2 equation for tiny inputs only.

    Always forms the Gram on the row side (X X^T, even for tall X) and the
    c-term as ((X X^T)(X X^T)) X, i.e. a different association and, for tall
    inputs, a different Gram than ``newton_schulz``.  Agreement of the two is
    a check on both."""
    X = np.asarray(X, np.float64)
    if X.size > 4096:
        raise ValueError("newton_schulz_literal is for tiny inputs")
    if normalize:
        nrm = math.sqrt(float(np.sum(X * X)))
        if nrm == 0.0:
            return X.copy()
        X = X / nrm
    for a, b, c in expand_stages(stages):
        S = X @ X.T
        X = a * X + b * (S @ X) + c * ((S @ S) @ X)
    return X


# ---------------------------------------------------------------------------
# Update scale, weight decay and the full step
# ---------------------------------------------------------------------------
SCALE_SPECTRAL = "spectral"
SCALE_UNIT_RMS_NORM = "unit_rms_norm"
SCALE_NONE = "none"


def update_scale(rows: int, cols: int, mode: str, gamma: float, fan_out_axis: int = 0) -> float:
    """Scale applied to O'.

    spectral:      sqrt(max(fan_in, fan_out)) * gamma  (Algorithm 1 of
                   "Muon 优化器"; RFC-0023 §方案 3 consistent_rms)
    unit_rms_norm: sqrt(fan_out / fan_in)  ("Scaling for MuP over Muon
                   optimizer"), no gamma (reading)
    none:          1
    ``fan_out_axis`` names the matrix axis that holds fan_out: 0 for a
    PyTorch [out, in] weight, 1 for a MaxText [in, out] kernel (and the
    split_head sub-matrices [embed, head_dim])."""
    if mode == SCALE_SPECTRAL:
        return math.sqrt(max(rows, cols)) * gamma
    if mode == SCALE_UNIT_RMS_NORM:
        if fan_out_axis not in (0, 1):
            raise ValueError("fan_out_axis must be 0 or 1")
        fan_out = rows if fan_out_axis == 0 else cols
        fan_in = cols if fan_out_axis == 0 else rows
        return math.sqrt(fan_out / fan_in)
    if mode == SCALE_NONE:
        return 1.0
    raise ValueError(f"unknown scale mode {mode!r}")


def decoupled_update(W: np.ndarray, O: np.ndarray, lr: float, weight_decay: float,
                     scale: float, decay: bool = True) -> np.ndarray:
    """W_t = W_{t-1}(1 - eta*lambda) - eta*scale*O'  (Algorithm 1); a masked-off
    tensor (RFC-0023 §方案 2) keeps W_{t-1} undecayed."""
    W = np.asarray(W, np.float64)
    keep = 1.0 - lr * weight_decay if decay else 1.0
    return W * keep - lr * (scale * np.asarray(O, np.float64))


@dataclass
class MuonHyper:
    mu: float = DEFAULT_MU
    nesterov: bool = True
    style: str = "sgd"          # 'sgd' (Megatron) or 'ema' (optax)
    t: int = 1                  # steps including this one; used by 'ema'
    scale_mode: str = SCALE_SPECTRAL
    gamma: float = DEFAULT_GAMMA
    lr: float = DEFAULT_LR
    weight_decay: float = DEFAULT_WD
    fan_out_axis: int = 0


def muon_step(W: np.ndarray, G: np.ndarray, M: np.ndarray, hp: MuonHyper,
              decay: bool = True,
              stages: Iterable[tuple[int, Sequence[float]]] = HYBRID_STAGES,
              normalize: bool = True) -> dict:
    """One Muon step on one matrix (Algorithm 1 of "Muon 优化器").

    Returns float64 arrays: 'M' (new momentum state), 'X' (the matrix handed
    to Newton–Schulz), 'O' (O'), 'W' (updated weight) and the float 'scale'."""
    G = np.asarray(G, np.float64)
    if hp.style == "sgd":
        M_t = momentum_sgd(M, G, hp.mu)
        X = lookahead_sgd(M_t, G, hp.mu) if hp.nesterov else M_t
    elif hp.style == "ema":
        M_t = momentum_ema(M, G, hp.mu)
        X = lookahead_ema(M_t, G, hp.mu, hp.t) if hp.nesterov else bias_correct(M_t, hp.mu, hp.t)
    else:
        raise ValueError(f"unknown nesterov style {hp.style!r}")
    O = newton_schulz(X, stages, normalize)
    rows, cols = np.shape(W)
    s = update_scale(rows, cols, hp.scale_mode, hp.gamma, hp.fan_out_axis)
    W_t = decoupled_update(W, O, hp.lr, hp.weight_decay, s, decay)
    return {"M": M_t, "X": X, "O": O, "W": W_t, "scale": s}


# ---------------------------------------------------------------------------
# split_head views and shape grouping (RFC-0023 §背景, §方案 3, §方案 4)
# ---------------------------------------------------------------------------
def head_slices(W: np.ndarray, n_heads: int, head_dim: int) -> list[np.ndarray]:
    """Per-head sub-matrices of a [embed, heads*head_dim] weight: head h is
    columns [h*head_dim, (h+1)*head_dim).  With split_head the heads form the
    batch dimension and fan_out is head_dim."""
    W = np.asarray(W)
    if W.shape[1] != n_heads * head_dim:
        raise ValueError("columns must equal n_heads * head_dim")
    return [W[:, h * head_dim:(h + 1) * head_dim] for h in range(n_heads)]


def row_blocks(W: np.ndarray, parts: int) -> list[np.ndarray]:
    """Sub-matrices of a weight stacked along rows, [parts*r, c] -> parts of
    [r, c] (reading of split_linear_fc1, named in RFC-0023 §实施计划 SubTask S5: a fused
    FC1 [gate; up] weight is orthogonalised as its separate blocks)."""
    W = np.asarray(W)
    if W.shape[0] % parts != 0:
        raise ValueError("rows must split into equal parts")
    r = W.shape[0] // parts
    return [W[k * r:(k + 1) * r] for k in range(parts)]


def group_by_shape(keys: Sequence[tuple], max_batch: int) -> tuple[list[int], int]:
    """Group tensors whose keys (shape, dtypes, view kind) are equal, in
    order of first appearance; each group of the same key is cut into chunks
    of at most ``max_batch`` members (0 = no limit), taken in tensor order.

    Returns (group index per tensor, number of groups)."""
    if max_batch < 0:
        raise ValueError("max_batch must be >= 0")
    order: list[tuple] = []
    members: dict[tuple, list[int]] = {}
    for i, k in enumerate(keys):
        if k not in members:
            members[k] = []
            order.append(k)
        members[k].append(i)
    group_of = [-1] * len(keys)
    g = 0
    for k in order:
        idx = members[k]
        step = len(idx) if max_batch == 0 else max_batch
        for start in range(0, len(idx), step):
            for i in idx[start:start + step]:
                group_of[i] = g
            g += 1
    return group_of, g
