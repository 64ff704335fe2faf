"""Parity at the full sizes of the workloads, in the launch configuration
bench.py times: one muon_step_batched call per step with every matrix of a
shape in one group.  The oracle checks sampled matrices one by one; momentum
is checked on every matrix where that stays cheap.

Each workload runs twice from the same state: once with W in its bf16
storage (W bound 1e-2*lr*scale plus half a bf16 ulp, since rounding W to
bf16 moves it by more than the whole update), and once with the same W held
in fp32 (same groups, same kernels, the fp32-W epilogue).  In the fp32 run
the W bound is literal, and the step's own O' is read back from the update,
O' = (W_prev*(1 - lr*wd) - W_new) / (lr*scale), and checked against the
oracle's O' at the 3e-2 relative Frobenius bar; the read-back's own error is
fp32 rounding of W divided by lr*scale, two orders of magnitude below it.
"""
import gc

import numpy as np
import pytest
import torch

import newton_schulz_02_gb300 as m
import oracle
import workloads
from tests.gpu_util import F32, check_w, f64, hyper, momentum_ref_f32, rel_fro, ulp_diff_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"
NS_TOL = 3e-2


@pytest.fixture(autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()
    torch.cuda.set_device(0)
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _step(groups, **hp_kw):
    ws = m.workspace(m.muon_step_workspace_size(groups))
    m.muon_step_batched(groups, m.hparams(**hp_kw), ws)
    code, flags = m.muon_get_status(ws)
    assert code == m.MUON_OK and flags == 0, (code, flags)
    del ws


def step_o(W_prev: np.ndarray, W_new: np.ndarray, hp, scale: float) -> np.ndarray:
    """The O' an fp32-W step applied, read back from its update ("Muon 优化器"
    Algorithm 1, last line), with the fp32 decay and lr*scale the library
    forms from the fp32 hyperparameters."""
    decay = F32(1.0 - hp.lr * hp.weight_decay)
    lr_scale = F32(hp.lr * scale)
    return (W_prev * decay - W_new) / lr_scale


def _check_fp32_w(W_prev, W_new, ref, hp):
    """Literal W bound and the step's own O' at 3e-2."""
    check_w(W_new, ref["W"], hp, ref["scale"], bf16=False)
    err = rel_fro(step_o(W_prev, W_new, hp, ref["scale"]), ref["O"])
    assert err <= NS_TOL, err
    return err


def test_stack_64x1024_five_steps():
    """64 x 1024^2, five steps of fresh row-scaled grads; momentum of every
    matrix to 1 ulp each step; sampled matrices' W (bf16 and fp32 runs) and
    the fp32 run's O' against the oracle each step."""
    st = workloads.stacked(seed=1)
    Wd, Md = st.W.to(DEV), st.M.to(DEV)
    W32, M32 = Wd.float(), Md.clone()
    hp = hyper()
    sample = (0, 37)
    for t in range(st.steps):
        G = st.grad(t)
        Gd = G.to(DEV)
        M_prev = Md.cpu().numpy()
        W_prev = {b: f64(Wd[b]) for b in sample}
        W32_prev = {b: f64(W32[b]) for b in sample}
        _step([m.Group.stacked(Wd, Gd, Md)])
        _step([m.Group.stacked(W32, Gd, M32)])
        M_new = Md.cpu().numpy()
        assert torch.equal(M32, Md)            # momentum does not depend on W
        Gf = G.float().numpy()
        for b in range(Wd.shape[0]):
            want = momentum_ref_f32(M_prev[b].astype(np.float64), Gf[b].astype(np.float64), hp)
            assert np.max(ulp_diff_f32(M_new[b], want)) <= 1, (t, b)
        for b in sample:
            g, mp = Gf[b].astype(np.float64), M_prev[b].astype(np.float64)
            ref = oracle.muon_step(W_prev[b], g, mp, hp)
            check_w(f64(Wd[b]), ref["W"], hp, ref["scale"], bf16=True)
            ref32 = oracle.muon_step(W32_prev[b], g, mp, hp)
            _check_fp32_w(W32_prev[b], f64(W32[b]), ref32, hp)


def _dtype_code(dt):
    return m.MUON_BF16 if dt == torch.bfloat16 else m.MUON_F32


def _groups(sets: dict, fan_out_axis=0):
    """One group per shape (muon_group_by_shape), every matrix of the set."""
    mats, descs = [], []
    for nm, (W, G, M) in sets.items():
        for b in range(W.shape[0]):
            mats.append((nm, b))
            descs.append((W.shape[1], W.shape[2], W.shape[2], _dtype_code(W.dtype),
                          _dtype_code(G.dtype), fan_out_axis))
    gid, n_groups = m.muon_group_by_shape(descs, 0)
    groups = []
    for g in range(n_groups):
        members = [mats[i] for i in range(len(mats)) if gid[i] == g]
        groups.append(m.Group([sets[nm][0][b] for nm, b in members],
                              [sets[nm][1][b] for nm, b in members],
                              [sets[nm][2][b] for nm, b in members], fan_out_axis=fan_out_axis))
    return groups


def _grouped_step(sets: dict, sample_of: dict):
    """sets: {name: (W bf16 [B,r,c], G, M)} on the device.  Steps the set as
    the bench does (bf16 W), and a copy of it with fp32 W from the same
    state; checks one sampled matrix per name in both (one oracle step each:
    both runs start from the same values)."""
    sets32 = {nm: (W.float(), G, M.clone()) for nm, (W, G, M) in sets.items()}
    before = {}
    for nm, b in sample_of.items():
        W, G, M = sets[nm]
        before[nm] = (f64(W[b]), f64(G[b]), M[b].cpu().numpy().astype(np.float64))
    groups = _groups(sets)
    _step(groups)
    _step(_groups(sets32))
    hp = hyper()
    errs = {}
    for nm, b in sample_of.items():
        Wp, Gp, Mp = before[nm]
        ref = oracle.muon_step(Wp, Gp, Mp, hp)
        M_new = sets[nm][2][b].cpu().numpy()
        assert np.max(ulp_diff_f32(M_new, momentum_ref_f32(Mp, Gp, hp))) <= 1
        assert torch.equal(sets32[nm][2][b], sets[nm][2][b])
        check_w(f64(sets[nm][0][b]), ref["W"], hp, ref["scale"], bf16=True)
        errs[nm] = _check_fp32_w(Wp, f64(sets32[nm][0][b]), ref, hp)
    return len(groups), errs


def test_dense_transformer_matrix_set():
    """32 layers x {q, o 4096^2; k, v 1024x4096; gate, up 14336x4096; down
    4096x14336}: four shape groups in one call; one matrix per shape checked."""
    sets = workloads.dense_layers(seed=3, device=DEV)
    n_groups, errs = _grouped_step(sets, {"q": 5, "k": 17, "gate": 30, "down": 2})
    assert n_groups == 4
    print("dense O' errors (step's own, fp32 W)", errs)


def test_moe_expert_stack():
    """256 experts x {up 2048x7168, down 7168x2048}: two shape groups."""
    sets = workloads.moe_experts(seed=4, device=DEV)
    n_groups, errs = _grouped_step(sets, {"up": 201, "down": 9})
    assert n_groups == 2
    print("moe O' errors (step's own, fp32 W)", errs)


@pytest.mark.parametrize("scale_mode", ["spectral", "unit_rms_norm"])
def test_split_head_attention_weight_fp32_w(scale_mode):
    """QKV weight 4096 x (32 x 128) with fp32 W, orthogonalised per head
    (heads = batch, fan_out = head size 128): every head's momentum (1 ulp),
    W (literal bound) and the step's own O' (3e-2)."""
    h = workloads.split_heads(seed=2)
    W0, G0, M0 = f64(h.W), f64(h.G), f64(h.M)
    Wd, Gd, Md = h.W.to(DEV).float(), h.G.to(DEV), h.M.to(DEV)
    _step([m.Group.split_head(Wd, Gd, Md, h.n_heads, h.head_dim)], scale_mode=scale_mode)
    hp = hyper(scale_mode=scale_mode, fan_out_axis=1)
    Wg, Mg = f64(Wd), Md.cpu().numpy()
    errs = []
    for k in range(h.n_heads):
        s = slice(k * h.head_dim, (k + 1) * h.head_dim)
        ref = oracle.muon_step(W0[:, s], G0[:, s], M0[:, s], hp)
        assert np.max(ulp_diff_f32(Mg[:, s], momentum_ref_f32(M0[:, s], G0[:, s], hp))) <= 1
        errs.append(_check_fp32_w(W0[:, s], Wg[:, s], ref, hp))
    print(scale_mode, "worst head O' error", max(errs))
