"""The step completes while other work holds most of the GPU's SMs.

The fused Gram + polynomial launch hands its work units out by tickets, so a
polynomial unit only ever waits for Gram units of CTA pairs that are
running.  Here a kernel on a second stream holds all but a few SMs for
200 ms (it ends by itself, by the global timer) while a 64 x 1024^2 step runs
with every bounded wait limited to 50 ms: the step must finish before the
SMs are given back, report no timeout, and give bit for bit what it gives
on an idle GPU.
"""
import pytest
import torch

import newton_schulz_02_gb300 as m
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()
    torch.cuda.set_device(0)
    yield
    m.muon_set_wait_timeout_ns(2_000_000_000)


def _state():
    st = workloads.stacked(seed=11)
    return st.W.to(DEV), st.grad(0).to(DEV), st.M.to(DEV)


def test_step_progresses_while_most_sms_are_held():
    W, G, M = _state()
    grp = [m.Group.stacked(W, G, M)]
    ws = m.workspace(m.muon_step_workspace_size(grp))
    m.muon_step_batched(grp, m.hparams(), ws)
    code, flags = m.muon_get_status(ws)
    assert code == m.MUON_OK and flags == 0
    W_solo, M_solo = W.clone(), M.clone()

    W2, G2, M2 = _state()
    grp2 = [m.Group.stacked(W2, G2, M2)]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    held = sms - 24
    m.muon_set_wait_timeout_ns(50_000_000)
    busy = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    t0, t_step, t_busy = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    torch.cuda.synchronize()
    t0.record(main)
    busy.wait_event(t0)
    m.muon_occupy_sms(held, 200 << 10, 200_000_000, stream=busy)
    t_busy.record(busy)
    m.muon_step_batched(grp2, m.hparams(), ws)
    t_step.record(main)
    torch.cuda.synchronize()
    code, flags = m.muon_get_status(ws)
    assert code == m.MUON_OK and flags == 0, (code, flags)
    step_ms, busy_ms = t0.elapsed_time(t_step), t0.elapsed_time(t_busy)
    print(f"step done at {step_ms:.1f} ms, SMs held until {busy_ms:.1f} ms")
    assert busy_ms >= 190.0
    assert step_ms < busy_ms, "the step waited for the SMs to be given back"
    assert torch.equal(W2, W_solo) and torch.equal(M2, M_solo)


def test_cluster_chain_completes_correctly_while_most_sms_are_held():
    """The split_head set runs its whole chain as clusters of 8 CTAs that wait
    only on one another (never on another cluster).  With all but a few SMs
    held by a kernel on a second stream, each cluster starts once the GPU can
    place it: the step must report no timeout (every wait limited to 50 ms)
    and give bit for bit what it gives on an idle GPU."""
    h = workloads.split_heads(seed=2)
    W, G, M = h.W.to(DEV), h.G.to(DEV), h.M.to(DEV)
    grp = [m.Group.split_head(W, G, M, h.n_heads, h.head_dim)]
    ws = m.workspace(m.muon_step_workspace_size(grp))
    m.muon_step_batched(grp, m.hparams(), ws)
    code, flags = m.muon_get_status(ws)
    assert code == m.MUON_OK and flags == 0
    W_solo, M_solo = W.clone(), M.clone()

    W2, G2, M2 = h.W.to(DEV), h.G.to(DEV), h.M.to(DEV)
    grp2 = [m.Group.split_head(W2, G2, M2, h.n_heads, h.head_dim)]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    m.muon_set_wait_timeout_ns(50_000_000)
    busy = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(main)
    busy.wait_event(t0)
    m.muon_occupy_sms(sms - 24, 200 << 10, 100_000_000, stream=busy)
    m.muon_step_batched(grp2, m.hparams(), ws)
    torch.cuda.synchronize()
    code, flags = m.muon_get_status(ws)
    assert code == m.MUON_OK and flags == 0, (code, flags)
    assert torch.equal(W2, W_solo) and torch.equal(M2, M_solo)
