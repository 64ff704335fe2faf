"""GPU parity of the split-bf16 Newton–Schulz precision (MUON_NS_BF16X3)
against the float64 oracle, through the C ABI.

Bar: relative Frobenius error of O' <= 1e-3 per matrix (the fp32-class
bound of the higher-precision path); the split-bf16 chain keeps about 16
significant bits in X, X X^T and the polynomial and sums three bf16
products per GEMM, and is expected near 1e-5.
"""
import numpy as np
import pytest
import torch

import newton_schulz_02_gb300 as m
import oracle
import workloads
from tests.gpu_util import check_w, f64, hyper, momentum_ref_f32, rel_fro, ulp_diff_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_X3 = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()
    torch.cuda.set_device(0)


def x3(stages=oracle.HYBRID_STAGES, normalize=True):
    return m.Schedule(stages, normalize=normalize, prec=m.MUON_NS_BF16X3)


def run_ns(x, schedule):
    out = torch.empty(x.shape, dtype=torch.float32, device=DEV)
    ws = m.workspace(m.newton_schulz_workspace_size(x.shape[1], x.shape[2], x.shape[0], schedule))
    m.newton_schulz_batched(x, out, ws, schedule)
    code, flags = m.muon_get_status(ws)
    assert code == m.MUON_OK and flags == 0, (code, flags)
    return out


def spiky(rng, r, c, rank=8):
    noise = rng.standard_normal((r, c))
    U, _ = np.linalg.qr(rng.standard_normal((r, rank)))
    V, _ = np.linalg.qr(rng.standard_normal((c, rank)))
    return noise + (U * (10 * np.linalg.norm(noise) / np.sqrt(rank))) @ V.T


def student(rng, r, c, nu=3):
    chi = sum(rng.standard_normal((r, c)) ** 2 for _ in range(nu))
    return rng.standard_normal((r, c)) / np.sqrt(chi / nu)


SHAPES = [(256, 512), (512, 256), (200, 328), (328, 200), (128, 128), (384, 640), (8, 8),
          (1, 64), (72, 8), (1024, 1024)]


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_x3_hybrid_gaussian(rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    x = torch.tensor(rng.standard_normal((2, rows, cols)) * 1e-3, dtype=torch.float32).to(DEV)
    got = run_ns(x, x3())
    for b in range(2):
        err = rel_fro(f64(got[b]), oracle.newton_schulz(f64(x[b])))
        assert err <= TOL_X3, (b, err)


@pytest.mark.parametrize("kind", ["spiky", "student"])
@pytest.mark.parametrize("rows,cols", [(512, 1024), (1024, 512), (1024, 1024)])
def test_x3_structured_inputs(kind, rows, cols):
    """The inputs that set the bf16 path's error: a rank-8 spike of 10x the
    noise's norm, heavy Student-t(3) tails."""
    rng = np.random.default_rng(rows + cols + (kind == "spiky"))
    gen = spiky if kind == "spiky" else student
    x = torch.tensor(np.stack([gen(rng, rows, cols) for _ in range(2)]), dtype=torch.float32).to(DEV)
    got = run_ns(x, x3())
    for b in range(2):
        err = rel_fro(f64(got[b]), oracle.newton_schulz(f64(x[b])))
        assert err <= TOL_X3, (kind, b, err)


SCHEDULES = {
    "identity": [(1, (1.0, 0.0, 0.0))],
    "gram": [(1, (0.0, 1.0, 0.0))],
    "square": [(1, (0.0, 0.0, 1.0))],
    "mixed": [(1, (0.5, -0.25, 0.125))],
    "two": [(2, (1.5, -0.5, 0.0))],
    "five": [(5, (3.4445, -4.775, 2.0315))],
}


@pytest.mark.parametrize("name", sorted(SCHEDULES))
@pytest.mark.parametrize("rows,cols", [(256, 512), (384, 256), (512, 512)])
def test_x3_isolating_schedules(name, rows, cols):
    """Single kernels and short chains (the c == 0 path, the (a - 1) I shift
    with a = 0) at the 1e-3 bar."""
    stages = SCHEDULES[name]
    rng = np.random.default_rng(5)
    x = torch.tensor(rng.standard_normal((2, rows, cols)), dtype=torch.float32).to(DEV)
    got = run_ns(x, x3(stages))
    for b in range(2):
        err = rel_fro(f64(got[b]), oracle.newton_schulz(f64(x[b]), stages))
        assert err <= TOL_X3, (name, b, err)


def test_x3_stable_stage_fixes_orthonormal_rows():
    rng = np.random.default_rng(3)
    Q, _ = np.linalg.qr(rng.standard_normal((512, 256)))
    x = torch.tensor(np.ascontiguousarray(Q.T[None]), dtype=torch.float32).to(DEV)
    got = f64(run_ns(x, x3([(2, (2.0, -1.5, 0.5))], normalize=False))[0])
    assert rel_fro(got, Q.T) <= 1e-4


def test_x3_batched_equals_unbatched_bitwise():
    rng = np.random.default_rng(13)
    x = torch.tensor(rng.standard_normal((3, 256, 640)), dtype=torch.bfloat16).to(DEV)
    whole = run_ns(x, x3())
    for b in range(3):
        assert torch.equal(run_ns(x[b:b + 1].clone(), x3())[0], whole[b])


def test_x3_workspace_is_larger():
    """Lo planes of S and P, less the ticket counters and log that only the
    fused bf16 Gram + polynomial launches use (64 counters, then 128 rows of
    one launch's 2 x 4 x 10 tickets + 2)."""
    s_bf16 = m.newton_schulz_workspace_size(1024, 1024, 4)
    s_x3 = m.newton_schulz_workspace_size(1024, 1024, 4, x3())
    log_bytes = (64 + 128 * (2 * 4 * 10 + 2)) * 4
    assert s_x3 == s_bf16 + 2 * 4 * 1024 * 1024 * 2 - (log_bytes + 255) // 256 * 256


@pytest.mark.parametrize("rows,cols", [(256, 512), (640, 384)])
def test_x3_muon_step(rows, cols):
    """A whole step with the split-bf16 chain: momentum 1 ulp, W at its bound,
    and O' (recomputed with the same chain from the oracle's look-ahead) at 1e-3."""
    W, G, M = workloads.random_case(21, rows, cols, batch=3, w_dtype=torch.float32)
    W0, G0, M0 = f64(W), f64(G), f64(M)
    Wd, Gd, Md = W.to(DEV), G.to(DEV), M.to(DEV)
    grp = m.Group.stacked(Wd, Gd, Md)
    ws = m.workspace(m.muon_step_workspace_size([grp], x3()))
    m.muon_step_batched([grp], m.hparams(), ws, x3())
    code, flags = m.muon_get_status(ws)
    assert code == m.MUON_OK and flags == 0
    hp = hyper()
    for b in range(3):
        ref = oracle.muon_step(W0[b], G0[b], M0[b], hp)
        assert np.max(ulp_diff_f32(Md[b].cpu().numpy(), momentum_ref_f32(M0[b], G0[b], hp))) <= 1
        check_w(f64(Wd[b]), ref["W"], hp, ref["scale"], bf16=False)
        xo = torch.tensor(ref["X"], dtype=torch.float32, device=DEV)[None]
        assert rel_fro(f64(run_ns(xo, x3())[0]), ref["O"]) <= TOL_X3


def test_x3_dense_shapes_sampled():
    """One matrix of each dense-set shape (q 4096^2, k 1024x4096, gate
    14336x4096, down 4096x14336) through the split-bf16 chain, at full size."""
    sets = workloads.dense_layers(seed=3, layers=2, device=DEV, only=("q", "k", "gate", "down"))
    for nm, (W, G, M) in sets.items():
        x = G[1:2].float()
        got = run_ns(x, x3())
        err = rel_fro(f64(got[0]), oracle.newton_schulz(f64(x[0])))
        assert err <= TOL_X3, (nm, err)
        print(nm, "split-bf16 O' error", err)
