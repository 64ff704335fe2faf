"""AdamW partition kernel vs the float64 oracle (oracle/adamw_ref.py), through
the C ABI (muon_adamw_step).  Element by element on ragged small tensors and
on sampled elements of the dense model's AdamW partition.

Tolerances follow from the fp32 arithmetic the kernel does:
  m = fma(b1, m, fl((1-b1) g)):    |err| <= 2^-24 (|(1-b1) g| + |m|)  (two roundings)
  v = fma(b2, v, fl((1-b2) fl(g^2))): both terms >= 0, |err| <= 3 * 2^-24 |v|
  u = fl(fl(m c1) / (fl(sqrt(fl(v c2))) + eps)): a few roundings on top of the
      m and v errors: |err| <= 1e-6 |u| + c1 |err_m| / sqrt(v_hat)
  W = fma(-lr, u, fl(W decay)):      |err| <= lr |err_u| + 2 ulp32(W), then
      rounding to bf16 adds half a bf16 ulp.
"""
import numpy as np
import pytest
import torch

import newton_schulz_02_gb300 as m
from oracle import adamw_ref
from tests.gpu_util import F32, bf16_ulp, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
U = 2.0 ** -24


@pytest.fixture(autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()
    torch.cuda.set_device(0)


def ohyper(t, **kw):
    """Oracle hyperparameters as the fp32 values the GPU receives."""
    base = dict(lr=2.7e-4, beta1=0.9, beta2=0.95, eps=1e-20, weight_decay=0.1)
    base.update(kw)
    return adamw_ref.AdamWHyper(**{k: F32(v) for k, v in base.items()}, t=t)


def check_tensor(W0, G0, m0, v0, W1, m1, v1, hp, decay, w_bf16):
    """One tensor's step: GPU results (W1, m1, v1) vs the oracle from the same
    inputs (all float64 arrays of the exact values the GPU held)."""
    ref = adamw_ref.adamw_step(W0, G0, m0, v0, hp, decay=decay)
    tol_m = 1.01 * U * (np.abs((1 - hp.beta1) * G0) + np.abs(ref["m"])) + 1e-45
    assert np.all(np.abs(m1 - ref["m"]) <= tol_m), np.max(np.abs(m1 - ref["m"]) - tol_m)
    tol_v = 3.01 * U * np.abs(ref["v"]) + 1e-45
    assert np.all(np.abs(v1 - ref["v"]) <= tol_v), np.max(np.abs(v1 - ref["v"]) - tol_v)
    c1 = 1.0 / (1.0 - hp.beta1 ** hp.t)
    v_hat = ref["v"] / (1.0 - hp.beta2 ** hp.t)
    tol_u = 1e-6 * np.abs(ref["u"]) + c1 * tol_m / (np.sqrt(v_hat) + hp.eps + 1e-38)
    err = np.abs(W1 - ref["W"])
    bound = hp.lr * tol_u + 2.0 * np.spacing(np.abs(ref["W"]).astype(np.float32)).astype(np.float64)
    if w_bf16:
        bound = bound + 0.5 * bf16_ulp(np.abs(ref["W"]) + bound)
    worst = float(np.max(err - bound))
    assert worst <= 0.0, f"W error exceeds bound by {worst:.3e}"


def _tensors(rng, numel, w_dtype, g_dtype, state):
    W = torch.tensor(rng.normal(0, 0.02, numel), dtype=torch.float32).to(w_dtype)
    g = rng.normal(0, 1e-3, numel)
    g[rng.random(numel) < 0.01] *= 100.0          # a few large entries
    G = torch.tensor(g, dtype=torch.float32).to(g_dtype)
    if state == "zero":
        mm = torch.zeros(numel)
        vv = torch.zeros(numel)
    else:
        mm = torch.tensor(rng.normal(0, 1e-3, numel), dtype=torch.float32)
        vv = torch.tensor(np.abs(rng.normal(0, 1e-3, numel)) ** 2, dtype=torch.float32)
    return [x.to(DEV) for x in (W, G, mm, vv)]


CASES = [  # numel, W dtype, G dtype
    (1, torch.float32, torch.float32), (7, torch.bfloat16, torch.bfloat16),
    (8, torch.bfloat16, torch.float32), (9, torch.float32, torch.bfloat16),
    (4095, torch.bfloat16, torch.bfloat16), (4096, torch.bfloat16, torch.bfloat16),
    (4097, torch.float32, torch.float32), (8197, torch.bfloat16, torch.bfloat16),
    (100003, torch.bfloat16, torch.bfloat16),
]


@pytest.mark.parametrize("state", ["zero", "random"])
def test_ragged_tensors_three_steps(state):
    """Groups of ragged sizes (tails of 1..7 elements, several chunks), both
    dtypes, a decay mask; three chained steps, each checked from the GPU's own
    previous state."""
    rng = np.random.default_rng(11)
    W, G, M, V, mask = [], [], [], [], []
    for i, (n, wd, gd) in enumerate(CASES):
        for k in range(2):
            w, g, mm, vv = _tensors(rng, n, wd, gd, state)
            W.append(w); G.append(g); M.append(mm); V.append(vv)
            mask.append((i + k) % 3 != 0)
    groups = m.adamw_groups(W, G, M, V, wd_mask=mask)
    assert len(groups) == len(CASES)
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = 1 if state == "zero" else 5
    for t in range(t0, t0 + 3):
        before = [(f64(W[i]), f64(G[i]), f64(M[i]), f64(V[i])) for i in range(len(W))]
        m.muon_adamw_step(groups, m.adamw_hparams(t=t), flags)
        torch.cuda.synchronize()
        assert int(flags.item()) == 0
        for i in range(len(W)):
            check_tensor(*before[i], f64(W[i]), f64(M[i]), f64(V[i]), ohyper(t), mask[i],
                         W[i].dtype == torch.bfloat16)
        for i in range(len(G)):  # fresh gradients for the next step
            G[i].copy_(torch.tensor(rng.normal(0, 1e-3, G[i].numel()), dtype=torch.float32))


def test_more_groups_than_one_launch_holds():
    """20 groups (two launches of at most 16 groups)."""
    rng = np.random.default_rng(12)
    W, G, M, V = [], [], [], []
    for n in range(100, 120):
        w, g, mm, vv = _tensors(rng, n, torch.float32, torch.float32, "random")
        W.append(w); G.append(g); M.append(mm); V.append(vv)
    before = [(f64(W[i]), f64(G[i]), f64(M[i]), f64(V[i])) for i in range(len(W))]
    groups = m.adamw_groups(W, G, M, V)
    assert len(groups) == 20
    m.muon_adamw_step(groups, m.adamw_hparams(t=3))
    torch.cuda.synchronize()
    for i in range(len(W)):
        check_tensor(*before[i], f64(W[i]), f64(M[i]), f64(V[i]), ohyper(3), True, False)


def test_zero_gradient_only_decays():
    """g = 0 from a zero state: u = 0, so W = fp32(W * (1 - lr wd)) exactly;
    with the mask off W is bit-identical."""
    W = torch.randn(2, 5000, device=DEV) * 0.02
    W0 = W.clone()
    z = torch.zeros_like(W)
    groups = m.adamw_groups([W[0], W[1]], [z[0], z[1]], [z[0].clone(), z[1].clone()],
                            [z[0].clone(), z[1].clone()], wd_mask=[True, False])
    m.muon_adamw_step(groups, m.adamw_hparams(t=1))
    torch.cuda.synchronize()
    decay = np.float32(1.0 - np.float64(F32(2.7e-4)) * np.float64(F32(0.1)))
    want = (W0[0].cpu().numpy() * decay).astype(np.float32)
    assert np.array_equal(W[0].cpu().numpy(), want)
    assert torch.equal(W[1], W0[1])


def test_misaligned_pointer_sets_flag_and_skips_tensor():
    """A W pointer one bf16 element past a 16-byte boundary: the kernel sees it
    before any access, sets MUON_FLAG_MISALIGNED, leaves that tensor alone and
    updates the others."""
    base = torch.randn(4097, device=DEV).to(torch.bfloat16)
    Wbad = base[1:]                       # in bounds, 2-byte offset
    Wok = torch.randn(4096, device=DEV).to(torch.bfloat16)
    G = [torch.full((4096,), 1e-3, device=DEV).to(torch.bfloat16) for _ in range(2)]
    M = [torch.zeros(4096, device=DEV) for _ in range(2)]
    V = [torch.zeros(4096, device=DEV) for _ in range(2)]
    bad0, ok0 = Wbad.clone(), Wok.clone()
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.muon_adamw_step(m.adamw_groups([Wbad, Wok], G, M, V), m.adamw_hparams(t=1), flags)
    torch.cuda.synchronize()
    assert int(flags.item()) & m.MUON_FLAG_MISALIGNED
    assert torch.equal(Wbad, bad0) and torch.equal(M[0], torch.zeros_like(M[0]))
    assert not torch.equal(Wok, ok0)


def test_dense_model_adamw_partition_sampled():
    """The dense 32-layer model's AdamW partition (embedding and output head
    128256 x 4096, 65 RMSNorm scales of 4096), bf16 W and G, fp32 moments:
    three steps, step 3 checked on 2^20 sampled elements of each large tensor
    and every norm-scale element."""
    import workloads
    part = workloads.dense_adamw_partition(seed=5, device=DEV)
    W, G, M, V = part["W"], part["G"], part["m"], part["v"]
    groups = m.adamw_groups(W, G, M, V, wd_mask=part["wd_mask"])
    for t in (1, 2):
        m.muon_adamw_step(groups, m.adamw_hparams(t=t))
        for g in G:
            g.normal_(0, 1e-3)
    rng = np.random.default_rng(0)
    picks = []
    for i, w in enumerate(W):
        n = w.numel()
        idx = np.arange(n) if n <= 65536 else rng.choice(n, size=1 << 20, replace=False)
        ix = torch.tensor(idx, device=DEV)
        picks.append((i, ix, [f64(x.view(-1)[ix]) for x in (W[i], G[i], M[i], V[i])]))
    m.muon_adamw_step(groups, m.adamw_hparams(t=3))
    torch.cuda.synchronize()
    for i, ix, (w0, g0, m0, v0) in picks:
        check_tensor(w0, g0, m0, v0, f64(W[i].view(-1)[ix]), f64(M[i].view(-1)[ix]),
                     f64(V[i].view(-1)[ix]), ohyper(3), part["wd_mask"][i], True)
