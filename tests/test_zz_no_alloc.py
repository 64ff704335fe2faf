"""The allocation-free Newton–Schulz entry point (newton_schulz_batched_noalloc).

It exists for callers that cannot get device memory from cudaMalloc (code
inside a framework whose allocator owns the device memory, loops that cannot
afford the synchronisation an allocation may cause).  It runs the same
deterministic kernels as newton_schulz_batched, only on the library's static
scratch instead of a caller workspace, so on the same input its output must
be bit-identical to that entry point's, on consecutive calls that share the
scratch; both are also checked against the float64 oracle at the bf16
Newton–Schulz tolerance.  Its only error channel, the copy of the scratch's
status word into the caller's device word, is checked with a non-finite
input.  This file is collected last so a failure here leaves every other
test already run.
"""
import numpy as np
import pytest
import torch

import newton_schulz_02_gb300 as m
import oracle
from tests.gpu_util import f64, rel_fro

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


def _noalloc(x, flags):
    out = torch.empty(x.shape, dtype=torch.float32, device="cuda")
    code = m.newton_schulz_batched_noalloc(x, out, device_flags=flags)
    assert code == m.MUON_OK, m.status_string(code)
    torch.cuda.synchronize()
    return out


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    rng = np.random.default_rng(2024)
    # a larger call first (pair-wide kernels, ten iterations), then a smaller
    # ragged one (one-CTA kernels, a tall input) that reuses the stale scratch
    cases = [torch.tensor(rng.standard_normal((2, 256, 512)) * 1e-3, dtype=torch.bfloat16),
             torch.tensor(rng.standard_normal((3, 328, 200)) * 1e-3, dtype=torch.bfloat16)]
    flags = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
    for x in cases:
        x = x.cuda()
        out = _noalloc(x, flags)
        assert int(flags.item()) == 0
        ref = _with_workspace(x)
        assert torch.equal(out, ref), "no-alloc output differs from newton_schulz_batched's"
        for b in range(x.shape[0]):
            assert rel_fro(f64(out[b]), oracle.newton_schulz(f64(x[b]))) <= NS_TOL


def test_noalloc_status_word_reaches_the_caller():
    """A non-finite input sets MUON_FLAG_NONFINITE in the scratch's status
    word; the call's closing copy must deliver it to device_flags, and the
    next clean call must clear it again."""
    rng = np.random.default_rng(7)
    x = torch.tensor(rng.standard_normal((2, 128, 256)) * 1e-3, dtype=torch.bfloat16).cuda()
    bad = x.clone()
    bad[1, 5, 9] = float("nan")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    _noalloc(bad, flags)
    assert int(flags.item()) & m.MUON_FLAG_NONFINITE
    out = _noalloc(x, flags)
    assert int(flags.item()) == 0
    assert torch.equal(out, _with_workspace(x))


def test_noalloc_rejects_requests_beyond_its_scratch():
    x = torch.zeros(64, 1024, 1024, dtype=torch.bfloat16, device="cuda")   # needs ~512 MiB
    out = torch.empty(x.shape, dtype=torch.float32, device="cuda")
    out.fill_(7.0)
    code = m.newton_schulz_batched_noalloc(x, out)
    assert code == m.MUON_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())          # nothing was enqueued


def test_noalloc_binding_rejects_a_bad_flags_tensor():
    x = torch.zeros(1, 64, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(x.shape, dtype=torch.float32, device="cuda")
    for bad in (torch.zeros(1, dtype=torch.int32),                     # host memory
                torch.zeros(0, dtype=torch.int32, device="cuda"),     # empty
                torch.zeros(1, dtype=torch.int16, device="cuda")):    # 2-byte word
        with pytest.raises(ValueError):
            m.newton_schulz_batched_noalloc(x, out, device_flags=bad)
