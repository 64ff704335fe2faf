"""The allocation-free Newton–Schulz entry point (newton_schulz_batched_noalloc).

It exists for callers that cannot get device memory from cudaMalloc (code
inside a framework whose allocator owns the device memory, loops that cannot
afford the synchronisation an allocation may cause).  It must give what
newton_schulz_batched gives on the same input, within the Newton–Schulz
tolerance of the other tests, on consecutive calls that share its static
scratch.  This file is collected last so a failure here leaves every other
test already run.
"""
import numpy as np
import pytest
import torch

import newton_schulz_02_gb300 as m

pytestmark = pytest.mark.gpu

NS_TOL = 3e-2   # relative Frobenius tolerance of the bf16 Newton–Schulz path


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()
    torch.cuda.set_device(0)


def _with_workspace(x):
    out = torch.empty(x.shape, dtype=torch.float32, device="cuda")
    ws = m.workspace(m.newton_schulz_workspace_size(x.shape[1], x.shape[2], x.shape[0]))
    m.newton_schulz_batched(x, out, ws)
    code, flags = m.muon_get_status(ws)
    assert code == m.MUON_OK and flags == 0
    return out


def _rel(a, b):
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    rng = np.random.default_rng(2024)
    # a larger call first, then a smaller ragged one that reuses the stale scratch
    cases = [torch.tensor(rng.standard_normal((2, 256, 384)) * 1e-3, dtype=torch.bfloat16),
             torch.tensor(rng.standard_normal((3, 200, 328)) * 1e-3, dtype=torch.bfloat16)]
    flags = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
    for x in cases:
        x = x.cuda()
        out = torch.empty(x.shape, dtype=torch.float32, device="cuda")
        code = m.newton_schulz_batched_noalloc(x, out, device_flags=flags)
        assert code == m.MUON_OK, m.status_string(code)
        torch.cuda.synchronize()
        assert int(flags.item()) == 0
        ref = _with_workspace(x)
        for b in range(x.shape[0]):
            assert _rel(out[b], ref[b]) <= NS_TOL


def test_noalloc_rejects_requests_beyond_its_scratch():
    x = torch.zeros(64, 1024, 1024, dtype=torch.bfloat16, device="cuda")   # needs ~512 MiB
    out = torch.empty(x.shape, dtype=torch.float32, device="cuda")
    out.fill_(7.0)
    code = m.newton_schulz_batched_noalloc(x, out)
    assert code == m.MUON_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())          # nothing was enqueued
