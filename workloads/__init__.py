"""Seeded synthetic inputs for the Muon step (shared by tests and bench).

This module draws random inputs only; it holds none of the method's
arithmetic and imports neither the oracle nor the CUDA library.  Shapes,
value distributions and structure follow the five workloads the library is
measured on:

  single   one fp32 256x512 matrix, W ~ N(0, 0.02^2), G ~ N(0, 1e-3^2) plus a
           rank-4 spike of Frobenius norm 10x the noise's, zero momentum; seed 0
  stack    64 bf16 1024x1024 matrices, fp32 momentum carried over 5 steps of
           fresh Gaussian grads (sigma 1e-3) with per-row scales log-uniform in
           [0.1, 10] drawn once per matrix; seed 1
  heads    bf16 QKV weight 4096 x (32 heads x 128), Gaussian grads sigma 1e-3,
           orthogonalised per head; seed 2
  dense    32-layer dense transformer matrix set (hidden 4096, FFN 14336),
           Gaussian grads sigma 1e-3 plus rank-8 spikes; seed 3
  moe      256 experts x {up 2048x7168, down 7168x2048}, Student-t (nu=3)
           grads scaled 1e-3; seed 4
  adamw    the dense model's AdamW partition (embedding and head 128256 x 4096,
           65 norm scales of 4096), Gaussian grads sigma 1e-3; seed 5

A rank-k spike is U diag(s) V^T with U, V orthonormalised Gaussian columns and
equal s chosen so that its Frobenius norm is 10x the noise's.  Small and large
host workloads use numpy's PCG64 (``default_rng(seed)``); the two multi-GB
sets are drawn on the device with a seeded ``torch.Generator``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

W_STD = 0.02
G_STD = 1e-3


def _spike(rng: np.random.Generator, rows: int, cols: int, rank: int, frob: float) -> np.ndarray:
    U, _ = np.linalg.qr(rng.standard_normal((rows, rank)))
    V, _ = np.linalg.qr(rng.standard_normal((cols, rank)))
    s = frob / math.sqrt(rank)
    return (U * s) @ V.T


def to_storage(x, dtype: torch.dtype) -> torch.Tensor:
    """numpy / torch -> contiguous CPU tensor in the storage dtype (RNE)."""
    t = torch.as_tensor(np.ascontiguousarray(x)) if isinstance(x, np.ndarray) else x
    return t.to(torch.float32).to(dtype).contiguous()


# ---------------------------------------------------------------------------
@dataclass
class Single:
    W: torch.Tensor
    G: torch.Tensor
    M: torch.Tensor
    hp: dict = field(default_factory=dict)


def single_matrix(seed: int = 0, rows: int = 256, cols: int = 512, rank: int = 4,
                  dtype: torch.dtype = torch.float32) -> Single:
    """The one-matrix workload (fp32 by default)."""
    rng = np.random.default_rng(seed)
    W = rng.normal(0.0, W_STD, (rows, cols))
    noise = rng.normal(0.0, G_STD, (rows, cols))
    G = noise + _spike(rng, rows, cols, rank, 10.0 * np.linalg.norm(noise))
    return Single(W=to_storage(W, dtype), G=to_storage(G, dtype),
                  M=torch.zeros(rows, cols, dtype=torch.float32),
                  hp=dict(mu=0.95, nesterov=True, style="sgd", scale_mode="spectral",
                          gamma=0.18, lr=2.7e-4, weight_decay=0.1))


# ---------------------------------------------------------------------------
@dataclass
class Stack:
    W: torch.Tensor                  # [batch, n, n] bf16
    M: torch.Tensor                  # [batch, n, n] fp32
    row_scale: np.ndarray            # [batch, n, 1]
    seed: int
    steps: int

    def grad(self, step: int, dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
        """Fresh Gaussian grads of step ``step`` (0-based), per-row scaled."""
        if not 0 <= step:
            raise ValueError("step >= 0")
        rng = np.random.default_rng([self.seed, 1000 + step])
        z = rng.standard_normal(self.W.shape, dtype=np.float32)
        return to_storage(G_STD * self.row_scale.astype(np.float32) * z, dtype)


def stacked(seed: int = 1, batch: int = 64, n: int = 1024, steps: int = 5,
            w_dtype: torch.dtype = torch.bfloat16) -> Stack:
    """The stacked same-shape workload (64 x 1024 x 1024 by default)."""
    rng = np.random.default_rng(seed)
    W = rng.standard_normal((batch, n, n), dtype=np.float32) * np.float32(W_STD)
    row_scale = np.exp(rng.uniform(math.log(0.1), math.log(10.0), size=(batch, n, 1)))
    return Stack(W=to_storage(W, w_dtype), M=torch.zeros(batch, n, n, dtype=torch.float32),
                 row_scale=row_scale, seed=seed, steps=steps)


# ---------------------------------------------------------------------------
@dataclass
class Heads:
    W: torch.Tensor                  # [embed, heads*head_dim] bf16
    G: torch.Tensor
    M: torch.Tensor                  # fp32
    n_heads: int
    head_dim: int


def split_heads(seed: int = 2, embed: int = 4096, n_heads: int = 32, head_dim: int = 128,
                dtype: torch.dtype = torch.bfloat16) -> Heads:
    """QKV weight viewed as per-head sub-matrices [embed, head_dim]."""
    rng = np.random.default_rng(seed)
    cols = n_heads * head_dim
    W = rng.standard_normal((embed, cols), dtype=np.float32) * np.float32(W_STD)
    G = rng.standard_normal((embed, cols), dtype=np.float32) * np.float32(G_STD)
    return Heads(W=to_storage(W, dtype), G=to_storage(G, dtype),
                 M=torch.zeros(embed, cols, dtype=torch.float32), n_heads=n_heads,
                 head_dim=head_dim)


# ---------------------------------------------------------------------------
def random_case(seed: int, rows: int, cols: int, batch: int = 1, g_dtype=torch.bfloat16,
                w_dtype=torch.bfloat16, m_scale: float = 1.0):
    """Generic small case: W ~ N(0, 0.02^2), G ~ N(0, 1e-3^2), M ~ m_scale*N(0, 1e-3^2)."""
    rng = np.random.default_rng(seed)
    W = rng.normal(0.0, W_STD, (batch, rows, cols))
    G = rng.normal(0.0, G_STD, (batch, rows, cols))
    M = rng.normal(0.0, G_STD, (batch, rows, cols)) * m_scale
    return to_storage(W, w_dtype), to_storage(G, g_dtype), to_storage(M, torch.float32)


# ---------------------------------------------------------------------------
# Multi-GB sets, drawn on the device.
# ---------------------------------------------------------------------------
DENSE_SHAPES = (  # per layer, PyTorch [out, in]
    ("q", 4096, 4096), ("o", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096),
    ("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336),
)
MOE_SHAPES = (("up", 2048, 7168), ("down", 7168, 2048))


def _device_gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def dense_layers(seed: int = 3, layers: int = 32, device="cuda", spike_rank: int = 8,
                 only: tuple = ()) -> dict:
    """{name: (W bf16 [L, r, c], G bf16, M fp32)} for the dense-transformer set.
    G = N(0, 1e-3^2) + a rank-8 spike of norm 10x the noise's, per matrix."""
    gen = _device_gen(device, seed)
    out = {}
    for name, r, c in DENSE_SHAPES:
        if only and name not in only:
            continue
        W = (torch.randn(layers, r, c, generator=gen, device=device) * W_STD).to(torch.bfloat16)
        G = torch.randn(layers, r, c, generator=gen, device=device) * G_STD
        nrm = torch.linalg.vector_norm(G, dim=(1, 2))
        U = torch.linalg.qr(torch.randn(layers, r, spike_rank, generator=gen, device=device))[0]
        V = torch.linalg.qr(torch.randn(layers, c, spike_rank, generator=gen, device=device))[0]
        s = (10.0 * nrm / math.sqrt(spike_rank)).view(layers, 1, 1)
        G = G + torch.bmm(U * s, V.transpose(1, 2))
        out[name] = (W, G.to(torch.bfloat16), torch.zeros(layers, r, c, device=device))
        del G, U, V
    return out


def moe_experts(seed: int = 4, experts: int = 256, device="cuda", nu: int = 3,
                only: tuple = ()) -> dict:
    """{name: (W bf16 [E, r, c], G bf16, M fp32)}; G = 1e-3 * Student-t(nu), drawn as
    z / sqrt(chi2_nu / nu) with chi2_nu a sum of nu squared standard normals."""
    gen = _device_gen(device, seed)
    out = {}
    for name, r, c in MOE_SHAPES:
        if only and name not in only:
            continue
        W = (torch.randn(experts, r, c, generator=gen, device=device) * W_STD).to(torch.bfloat16)
        chi2 = torch.zeros(experts, r, c, device=device)
        for _ in range(int(nu)):
            chi2.add_(torch.randn(experts, r, c, generator=gen, device=device).square_())
        z = torch.randn(experts, r, c, generator=gen, device=device)
        G = (G_STD * z / torch.sqrt(chi2 / nu)).to(torch.bfloat16)
        out[name] = (W, G, torch.zeros(experts, r, c, device=device))
        del z, chi2
    return out


# ---------------------------------------------------------------------------
# AdamW partition of the dense 32-layer model (hidden 4096): token embedding
# and output head 128256 x 4096, two RMSNorm scales per layer plus the final
# one (65 x 4096).  Drawn on the device.
# ---------------------------------------------------------------------------
VOCAB = 128256
HIDDEN = 4096


def dense_adamw_partition(seed: int = 5, layers: int = 32, device="cuda",
                          vocab: int = VOCAB, hidden: int = HIDDEN) -> dict:
    """{W, G, m, v: lists of tensors, wd_mask, names}.  W bf16: embedding and
    head ~ N(0, 0.02^2), norm scales 1 + N(0, 0.02^2); G bf16 ~ N(0, 1e-3^2);
    fp32 moments start at zero.  Decay on for the embedding and head, off for
    the norm scales (the norm-parameter flag off)."""
    gen = _device_gen(device, seed)
    names = ["embed", "head"] + [f"norm{i}" for i in range(2 * layers + 1)]
    W, G, M, V, mask = [], [], [], [], []
    for nm in names:
        shape = (vocab, hidden) if nm in ("embed", "head") else (hidden,)
        w = torch.randn(shape, generator=gen, device=device) * W_STD
        if nm.startswith("norm"):
            w += 1.0
        W.append(w.to(torch.bfloat16))
        G.append((torch.randn(shape, generator=gen, device=device) * G_STD).to(torch.bfloat16))
        M.append(torch.zeros(shape, device=device))
        V.append(torch.zeros(shape, device=device))
        mask.append(not nm.startswith("norm"))
        del w
    return {"W": W, "G": G, "m": M, "v": V, "wd_mask": mask, "names": names}
