"""GPU parity of the on-chip chain (iterates of one 128-row tile).

Wide iterates of at most 128 rows run every Newton–Schulz iteration in one
launch: a cluster of C CTAs per matrix keeps its columns of X on chip, adds
the CTAs' partial Grams through distributed shared memory and forms the
polynomial and the update there.  These cases cover each cluster shape (1, 2,
4, 8 and 16 CTAs; 1 to 4 update groups of 128 columns per CTA; the 128-row shapes
of the other GPU tests add 1 CTA of 128 columns), ragged rows and
columns, both orientations of W and of the output, the lo plane's hand-over
at the iteration counts where it stops, the fused W store of the last
iteration, a schedule whose polynomial has c = 0, and bit-for-bit
determinism.  Tolerances are those of the tiled chain (relative Frobenius
error of O' <= 3e-2; W as in test_gpu_parity).
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
NS_TOL = 3e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()
    torch.cuda.set_device(0)


def run_ns(x, schedule=None):
    out = torch.empty(x.shape, dtype=torch.float32, device=DEV)
    ws = m.workspace(m.newton_schulz_workspace_size(x.shape[1], x.shape[2], x.shape[0], schedule))
    m.newton_schulz_batched(x, out, ws, schedule)
    code, flags = m.muon_get_status(ws)
    assert code == m.MUON_OK and flags == 0, (code, flags)
    return out


def oracle_ns(x, stages=oracle.HYBRID_STAGES):
    return [oracle.newton_schulz(f64(x[b]), stages, True) for b in range(x.shape[0])]


# (rows, cols) -> wide n x m: CTAs per matrix x columns per CTA (the fewest
# CTAs of at most 512 columns)
#   128 x 384    1 x 384 (three update groups: the third issued after the first drains)
#   100 x 1536   4 x 384 (ragged rows)
#   128 x 768    2 x 384
#   128 x 1024   2 x 512
#   64 x 4096    8 x 512
#   4096 x 96    8 x 512 (tall: the output written transposed)
#   120 x 3000   8 x 384 (ragged columns, m padded to 3072)
#   128 x 8192   16 x 512 (a non-portable cluster size; the tiled chain where the
#                GPU cannot place one)
#   96 x 6144    16 x 384
CHAIN_SHAPES = [(128, 384), (100, 1536), (128, 768), (128, 1024), (64, 4096), (4096, 96),
                (120, 3000), (128, 8192), (96, 6144)]


@pytest.mark.parametrize("rows,cols", CHAIN_SHAPES)
def test_chain_hybrid_matches_oracle(rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    x = torch.tensor(rng.standard_normal((3, rows, cols)) * 1e-2, dtype=torch.bfloat16).to(DEV)
    got = run_ns(x)
    want = oracle_ns(x)
    for b in range(3):
        assert rel_fro(f64(got[b]), want[b]) <= NS_TOL, b


@pytest.mark.parametrize("iters", [1, 3, 4, 5])
def test_chain_lo_plane_hand_over(iters):
    """The first four iterations read the iterate's lo plane and the first
    three write it: schedules that end inside, at and past that range leave
    the final iterate with or without its lo plane in the workspace (1, 3),
    or write the output from the last update (5)."""
    stages = [(iters, (3.4445, -4.7750, 2.0315))]
    rng = np.random.default_rng(40 + iters)
    x = torch.tensor(rng.standard_normal((2, 128, 2048)), dtype=torch.bfloat16).to(DEV)
    got = run_ns(x, m.Schedule(stages))
    want = oracle_ns(x, stages)
    for b in range(2):
        assert rel_fro(f64(got[b]), want[b]) <= NS_TOL, b


def test_chain_polynomial_without_square_term():
    """c = 0 in every iteration: P = b S + (a - 1) I, no S^2 product."""
    stages = [(6, (1.5, -0.5, 0.0))]
    rng = np.random.default_rng(5)
    x = torch.tensor(rng.standard_normal((2, 96, 4096)), dtype=torch.bfloat16).to(DEV)
    got = run_ns(x, m.Schedule(stages))
    want = oracle_ns(x, stages)
    for b in range(2):
        assert rel_fro(f64(got[b]), want[b]) <= NS_TOL, b


def test_chain_repeated_calls_and_batch_bitwise():
    """The partial Grams are added in rank order: repeated calls and a matrix
    run alone give the same bits as the batched call."""
    g = torch.Generator(device=DEV).manual_seed(3)
    x = torch.randn(40, 128, 4096, device=DEV, generator=g).to(torch.bfloat16)
    first = run_ns(x)
    for _ in range(3):
        assert torch.equal(run_ns(x), first)
    for b in (0, 17, 39):
        assert torch.equal(run_ns(x[b:b + 1].clone())[0], first[b])


@pytest.mark.parametrize("rows,cols,w_dtype", [(96, 2048, torch.float32),
                                               (2048, 128, torch.bfloat16),
                                               (128, 8192, torch.float32),
                                               (8192, 120, torch.bfloat16)])
def test_chain_step_writes_w(rows, cols, w_dtype):
    """A full Muon step whose last update writes W from the cluster: wide
    fp32 W with ragged rows, and tall bf16 W (turned around through shared
    memory), on clusters of 4 and of 16 CTAs; two steps with the momentum
    carried over."""
    W, G, M = workloads.random_case(61, rows, cols, batch=2, g_dtype=torch.float32,
                                    w_dtype=w_dtype, m_scale=5.0)
    Wd, Gd, Md = W.to(DEV), G.to(DEV), M.to(DEV)
    G0 = f64(G)
    for t in (1, 2):
        Mprev, Wprev = f64(Md), f64(Wd)
        hp_kw = dict(t=t)
        ws = m.workspace(m.muon_step_workspace_size([m.Group.stacked(Wd, Gd, Md)]))
        m.muon_step_batched([m.Group.stacked(Wd, Gd, Md)], m.hparams(**hp_kw), ws)
        code, flags = m.muon_get_status(ws)
        assert code == m.MUON_OK and flags == 0
        hp = hyper(t=t)
        for b in range(2):
            ref = oracle.muon_step(Wprev[b], G0[b], Mprev[b], hp)
            assert np.max(ulp_diff_f32(Md[b].cpu().numpy(),
                                       momentum_ref_f32(Mprev[b], G0[b], hp))) <= 1
            check_w(f64(Wd[b]), ref["W"], hp, ref["scale"], bf16=(w_dtype == torch.bfloat16))


def test_chain_zero_input_gives_zero():
    """1/||X|| is 0 for a zero matrix: every iteration keeps the iterate at 0."""
    x = torch.zeros(3, 128, 2048, dtype=torch.bfloat16, device=DEV)
    assert torch.count_nonzero(run_ns(x)).item() == 0


def test_chain_without_normalisation_fixes_orthonormal_rows():
    """Stable stage alone, no normalisation, on a 96 x 2048 matrix with
    orthonormal rows: p(1) = 1 and p'(1) = 0, so the rows stay put (the
    first iteration's Gram rows travel unscaled)."""
    rng = np.random.default_rng(9)
    Q, _ = np.linalg.qr(rng.standard_normal((2048, 96)))
    x = torch.tensor(np.ascontiguousarray(Q.T[None]), dtype=torch.float32).to(DEV)
    sched = m.Schedule([(3, (2.0, -1.5, 0.5))], normalize=False)
    got = f64(run_ns(x, sched)[0])
    assert rel_fro(got, Q.T) <= 1e-2
