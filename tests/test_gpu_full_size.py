"""Parity at the full sizes of the workloads, in the launch configuration
bench.py times: one muon_step_batched call per step with every matrix of a
shape in one group.  The oracle checks sampled matrices one by one (each
sampled matrix fully: momentum to 1 ulp, W to its tolerance, O' to 3e-2 via
newton_schulz_batched on the oracle's look-ahead); momentum is checked on
every matrix where that stays cheap.
"""
import gc

import numpy as np
import pytest
import torch

import newton_schulz_02_gb300 as m
import oracle
import workloads
from tests.gpu_util import check_w, f64, hyper, momentum_ref_f32, rel_fro, ulp_diff_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


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


def _check_sample(W_prev, G, M_prev, W_new, M_new, hp, fan_out_axis=0):
    """One matrix: momentum (1 ulp), W (tolerance), O' (3e-2)."""
    hp.fan_out_axis = fan_out_axis
    ref = oracle.muon_step(W_prev, G, M_prev, hp)
    assert np.max(ulp_diff_f32(M_new, momentum_ref_f32(M_prev, G, hp))) <= 1
    check_w(W_new, ref["W"], hp, ref["scale"], bf16=True)
    x = torch.tensor(ref["X"], dtype=torch.float32, device=DEV)[None]
    out = torch.empty_like(x)
    ws = m.workspace(m.newton_schulz_workspace_size(x.shape[1], x.shape[2], 1))
    m.newton_schulz_batched(x, out, ws)
    torch.cuda.synchronize()
    err = rel_fro(f64(out[0]), ref["O"])
    assert err <= 3e-2, err
    return err


def test_stack_64x1024_five_steps():
    st = workloads.stacked(seed=1)
    Wd, Md = st.W.to(DEV), st.M.to(DEV)
    hp = hyper()
    sample = (0, 37)
    for t in range(st.steps):
        G = st.grad(t)
        Gd = G.to(DEV)
        M_prev = Md.cpu().numpy()
        W_prev = {b: f64(Wd[b]) for b in sample}
        _step([m.Group.stacked(Wd, Gd, Md)])
        M_new = Md.cpu().numpy()
        Gf = G.float().numpy()
        for b in range(Wd.shape[0]):
            want = momentum_ref_f32(M_prev[b].astype(np.float64), Gf[b].astype(np.float64), hp)
            assert np.max(ulp_diff_f32(M_new[b], want)) <= 1, (t, b)
        for b in sample:
            _check_sample(W_prev[b], Gf[b].astype(np.float64), M_prev[b].astype(np.float64),
                          f64(Wd[b]), M_new[b], hyper())


def _grouped_step(sets: dict, sample_of: dict, fan_out_axis=0):
    """sets: {name: (W [B,r,c], G, M)} on the device.  Groups by shape with
    muon_group_by_shape, steps once, then checks one sampled matrix per name."""
    names = list(sets)
    mats, descs = [], []
    for nm in names:
        W, G, M = sets[nm]
        for b in range(W.shape[0]):
            mats.append((nm, b))
            descs.append((W.shape[1], W.shape[2], W.shape[2], m.MUON_BF16, m.MUON_BF16, fan_out_axis))
    gid, n_groups = m.muon_group_by_shape(descs, 0)
    groups = []
    for g in range(n_groups):
        members = [mats[i] for i in range(len(mats)) if gid[i] == g]
        groups.append(m.Group([sets[nm][0][b] for nm, b in members],
                              [sets[nm][1][b] for nm, b in members],
                              [sets[nm][2][b] for nm, b in members], fan_out_axis=fan_out_axis))
    before = {}
    for nm, b in sample_of.items():
        W, G, M = sets[nm]
        before[nm] = (f64(W[b]), f64(G[b]), M[b].cpu().numpy().astype(np.float64))
    _step(groups)
    errs = {}
    for nm, b in sample_of.items():
        W, G, M = sets[nm]
        Wp, Gp, Mp = before[nm]
        errs[nm] = _check_sample(Wp, Gp, Mp, f64(W[b]), M[b].cpu().numpy(), hyper(),
                                 fan_out_axis)
    return n_groups, errs


def test_dense_transformer_matrix_set():
    """32 layers x {q, o 4096^2; k, v 1024x4096; gate, up 14336x4096; down
    4096x14336}: four shape groups in one call; one matrix per shape checked."""
    sets = workloads.dense_layers(seed=3, device=DEV)
    n_groups, errs = _grouped_step(sets, {"q": 5, "k": 17, "gate": 30, "down": 2})
    assert n_groups == 4
    print("dense O' errors", errs)


def test_moe_expert_stack():
    """256 experts x {up 2048x7168, down 7168x2048}: two shape groups."""
    sets = workloads.moe_experts(seed=4, device=DEV)
    n_groups, errs = _grouped_step(sets, {"up": 201, "down": 9})
    assert n_groups == 2
    print("moe O' errors", errs)
