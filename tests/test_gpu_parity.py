"""GPU parity: the CUDA path through the C ABI against the float64 oracle on
the same seeded inputs.

Tolerances (element by element, per matrix):
  O'  (bf16 Newton–Schulz)  relative Frobenius error <= 3e-2
  M   (fp32 momentum)       within 1 ulp of the correctly rounded oracle value
  W                         max-abs <= 1e-2*lr*scale, plus half a bf16 ulp when
                            W is stored in bf16 (the rounding of the store)
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


def run_ns(x: torch.Tensor, schedule=None, out_dtype=torch.float32):
    """x: [batch, rows, cols] on the device."""
    out = torch.empty(x.shape, dtype=out_dtype, device=DEV)
    ws = m.workspace(m.newton_schulz_workspace_size(x.shape[1], x.shape[2], x.shape[0], schedule))
    m.newton_schulz_batched(x, out, ws, schedule)
    code, flags = m.muon_get_status(ws)
    assert code == m.MUON_OK and flags == 0, (code, flags)
    return out


def oracle_ns_batch(x: torch.Tensor, stages=oracle.HYBRID_STAGES, normalize=True):
    return [oracle.newton_schulz(f64(x[b]), stages, normalize) for b in range(x.shape[0])]


# ---------------------------------------------------------------------------
# Newton–Schulz alone
# ---------------------------------------------------------------------------
NS_SHAPES = [(256, 512), (512, 256), (200, 328), (328, 200), (128, 128), (384, 640),
             (640, 384), (8, 8), (1, 64), (72, 8), (1024, 1024)]


@pytest.mark.parametrize("rows,cols", NS_SHAPES)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_ns_hybrid_matches_oracle(rows, cols, dtype):
    rng = np.random.default_rng(rows * 1000 + cols)
    batch = 3 if rows * cols <= 400_000 else 2
    x = torch.tensor(rng.standard_normal((batch, rows, cols)) * 1e-3, dtype=dtype).to(DEV)
    got = run_ns(x)
    want = oracle_ns_batch(x)
    for b in range(batch):
        err = rel_fro(f64(got[b]), want[b])
        assert err <= NS_TOL, (b, err)


ISOLATING_SCHEDULES = {
    "identity": [(1, (1.0, 0.0, 0.0))],        # X/||X||: load, norm, update epilogue
    "gram": [(1, (0.0, 1.0, 0.0))],            # (X X^T) X: Gram + update (poly skipped)
    "square": [(1, (0.0, 0.0, 1.0))],          # (X X^T)^2 X: Gram + poly + update
    "mixed": [(1, (0.5, -0.25, 0.125))],
    "two": [(2, (1.5, -0.5, 0.0))],
}


@pytest.mark.parametrize("name", sorted(ISOLATING_SCHEDULES))
@pytest.mark.parametrize("rows,cols", [(256, 512), (384, 256), (512, 512)])
def test_ns_single_stage_schedules(name, rows, cols):
    """One-iteration schedules that isolate the kernels, at the O' bar.  The
    library evaluates X + (bS + cS^2 + (a-1)I) X, so schedules with a = 0
    (gram, square) cancel X against -X and keep fewer digits than the
    hybrid schedule does."""
    stages = ISOLATING_SCHEDULES[name]
    sched = m.Schedule(stages)
    rng = np.random.default_rng(7)
    x = torch.tensor(rng.standard_normal((2, rows, cols)), dtype=torch.bfloat16).to(DEV)
    got = run_ns(x, sched)
    want = oracle_ns_batch(x, stages)
    for b in range(2):
        assert rel_fro(f64(got[b]), want[b]) <= NS_TOL


def test_ns_without_normalisation_fixes_orthonormal_rows():
    """Stable stage alone, no normalisation: rows of Q orthonormal stay put
    (p(1) = 1, p'(1) = 0)."""
    rng = np.random.default_rng(3)
    Q, _ = np.linalg.qr(rng.standard_normal((512, 256)))
    x = torch.tensor(np.ascontiguousarray(Q.T[None]), dtype=torch.float32).to(DEV)  # 256 x 512
    sched = m.Schedule([(2, (2.0, -1.5, 0.5))], normalize=False)
    got = f64(run_ns(x, sched)[0])
    assert rel_fro(got, Q.T) <= 1e-2


def test_ns_zero_input_gives_zero():
    x = torch.zeros(2, 256, 384, dtype=torch.bfloat16, device=DEV)
    got = run_ns(x)
    assert torch.count_nonzero(got).item() == 0


def test_ns_zero_iterations_is_normalisation():
    rng = np.random.default_rng(11)
    x = torch.tensor(rng.standard_normal((1, 128, 256)), dtype=torch.float32).to(DEV)
    got = f64(run_ns(x, m.Schedule([]))[0])
    want = f64(x[0]) / np.linalg.norm(f64(x[0]))
    assert rel_fro(got, want) <= 5e-3


def test_ns_strided_input_view():
    """Matrices read through a view with row_stride > cols and a batch stride."""
    rng = np.random.default_rng(12)
    big = torch.tensor(rng.standard_normal((512, 1024)), dtype=torch.bfloat16).to(DEV)
    view = m.muon_view_t(512, 256, 1024, 256, 0)          # 4 heads of 512 x 256
    out = torch.empty(4, 512, 256, dtype=torch.float32, device=DEV)
    ws = m.workspace(m.newton_schulz_workspace_size(512, 256, 4))
    m.newton_schulz_batched(big, out, ws, view=view, batch=4)
    torch.cuda.synchronize()
    for h in range(4):
        want = oracle.newton_schulz(f64(big[:, 256 * h:256 * (h + 1)]))
        assert rel_fro(f64(out[h]), want) <= NS_TOL


def test_ns_batched_equals_unbatched_bitwise():
    rng = np.random.default_rng(13)
    x = torch.tensor(rng.standard_normal((5, 256, 640)), dtype=torch.bfloat16).to(DEV)
    whole = run_ns(x)
    for b in range(5):
        one = run_ns(x[b:b + 1].clone())
        assert torch.equal(one[0], whole[b])


@pytest.mark.parametrize("batch,rows,cols", [(16, 1024, 1024), (4, 2048, 7168)])
def test_ns_repeated_calls_bitwise(batch, rows, cols):
    """Shapes whose Gram and polynomial share a launch (per-matrix hand-over
    between CTAs through arrival counters): repeated calls on one input give
    bit-identical results, whatever order the CTAs reach the counters in."""
    g = torch.Generator(device=DEV).manual_seed(batch + rows)
    x = torch.randn(batch, rows, cols, device=DEV, generator=g).to(torch.bfloat16)
    first = run_ns(x)
    for _ in range(4):
        assert torch.equal(run_ns(x), first)


# Grams of at most 128 rows over a long K: the on-chip chain up to K = 8192
# (test_gpu_cluster_chain.py covers it in detail), beyond that the tiled chain,
# whose split-K Gram adds K-slices in a separate pass (8 slices at K = 16384).
SPLIT_SHAPES = [(128, 2048), (96, 4096), (4096, 120), (128, 8192), (128, 16384)]


@pytest.mark.parametrize("rows,cols", SPLIT_SHAPES)
def test_ns_split_k_gram_matches_oracle(rows, cols):
    rng = np.random.default_rng(rows + cols)
    x = torch.tensor(rng.standard_normal((3, rows, cols)), dtype=torch.bfloat16).to(DEV)
    got = run_ns(x)
    want = oracle_ns_batch(x)
    for b in range(3):
        assert rel_fro(f64(got[b]), want[b]) <= NS_TOL, b


@pytest.mark.parametrize("name", ["gram", "square", "mixed"])
def test_ns_split_k_single_stage_schedules(name):
    """The split Gram's epilogue pass: 1/||X||^2 scale, and with c = 0 the
    (a - 1) shift and P's diagonal residual written by that pass."""
    stages = ISOLATING_SCHEDULES[name]
    rng = np.random.default_rng(11)
    x = torch.tensor(rng.standard_normal((2, 128, 4096)), dtype=torch.bfloat16).to(DEV)
    got = run_ns(x, m.Schedule(stages))
    want = oracle_ns_batch(x, stages)
    for b in range(2):
        assert rel_fro(f64(got[b]), want[b]) <= NS_TOL


@pytest.mark.parametrize("rows,cols", [(256, 512), (128, 2048)])
def test_long_schedule_beyond_the_fused_launch_limit(rows, cols):
    """70 iterations with c != 0.  On pair-wide 256 x 512 matrices the first
    64 Gram + polynomial pairs of the chain run as fused launches handing out
    their units by tickets, the last 6 as separate Gram and polynomial
    launches; 128 x 2048 matrices, whose chain would otherwise run on chip
    (at most 64 iterations), take the tiled chain.  The stable stage repeated
    keeps every singular value at 1, so the result must still match the
    oracle at the bf16 bar."""
    stages = [(8, (3.4445, -4.7750, 2.0315)), (62, (2.0, -1.5, 0.5))]
    rng = np.random.default_rng(71)
    x = torch.tensor(rng.standard_normal((2, rows, cols)) * 1e-3, dtype=torch.bfloat16).to(DEV)
    got = run_ns(x, m.Schedule(stages))
    want = oracle_ns_batch(x, stages)
    for b in range(2):
        assert rel_fro(f64(got[b]), want[b]) <= NS_TOL, b


def test_ns_split_k_batched_equals_unbatched_bitwise():
    rng = np.random.default_rng(17)
    x = torch.tensor(rng.standard_normal((6, 128, 4096)), dtype=torch.bfloat16).to(DEV)
    whole = run_ns(x)
    for b in (0, 3, 5):
        one = run_ns(x[b:b + 1].clone())
        assert torch.equal(one[0], whole[b])


# ---------------------------------------------------------------------------
# the full step
# ---------------------------------------------------------------------------
def step_once(groups, hp_kw, schedule=None):
    hp = m.hparams(**hp_kw)
    ws = m.workspace(m.muon_step_workspace_size(groups, schedule))
    m.muon_step_batched(groups, hp, ws, schedule)
    code, flags = m.muon_get_status(ws)
    return code, flags


def test_single_fp32_matrix_step():
    """One fp32 256x512 matrix with a rank-4 spike, zero momentum, spectral."""
    case = workloads.single_matrix(seed=0)
    W0, G0, M0 = f64(case.W), f64(case.G), f64(case.M)
    W, G, M = case.W.to(DEV), case.G.to(DEV), case.M.to(DEV)
    code, flags = step_once([m.Group([W], [G], [M])], case.hp)
    assert code == m.MUON_OK and flags == 0
    hp = hyper()
    ref = oracle.muon_step(W0, G0, M0, hp)
    assert np.max(ulp_diff_f32(M.cpu().numpy(), momentum_ref_f32(M0, G0, hp))) <= 1
    check_w(f64(W), ref["W"], hp, ref["scale"], bf16=False)


@pytest.mark.parametrize("style,nesterov,scale_mode", [
    ("sgd", True, "spectral"), ("sgd", False, "unit_rms_norm"), ("ema", True, "spectral"),
    ("ema", False, "none")])
@pytest.mark.parametrize("rows,cols", [(256, 384), (384, 256)])
def test_step_variants_fp32(style, nesterov, scale_mode, rows, cols):
    W, G, M = workloads.random_case(21, rows, cols, batch=2, g_dtype=torch.float32,
                                    w_dtype=torch.float32, m_scale=5.0)
    W0, G0, M0 = f64(W), f64(G), f64(M)
    Wd, Gd, Md = W.to(DEV), G.to(DEV), M.to(DEV)
    for t in (1, 2):
        kw = dict(style=style, nesterov=nesterov, scale_mode=scale_mode, t=t)
        Mprev = f64(Md)
        Wprev = f64(Wd)
        code, flags = step_once([m.Group.stacked(Wd, Gd, Md)], kw)
        assert code == m.MUON_OK and flags == 0
        hp = hyper(style=style, nesterov=nesterov, scale_mode=scale_mode, t=t)
        for b in range(2):
            ref = oracle.muon_step(Wprev[b], G0[b], Mprev[b], hp)
            assert np.max(ulp_diff_f32(Md[b].cpu().numpy(),
                                       momentum_ref_f32(Mprev[b], G0[b], hp))) <= 1
            check_w(f64(Wd[b]), ref["W"], hp, ref["scale"], bf16=False)


def test_stacked_bf16_steps_and_ragged_shapes():
    """Several groups in one call (square, wide ragged, tall ragged), bf16 W/G,
    two steps with the state carried over."""
    shapes = [(4, 512, 512), (3, 200, 328), (2, 328, 200)]
    cases = [workloads.random_case(30 + i, r, c, batch=b) for i, (b, r, c) in enumerate(shapes)]
    dev = [(W.to(DEV), G.to(DEV), M.to(DEV)) for W, G, M in cases]
    groups = [m.Group.stacked(W, G, M) for W, G, M in dev]
    hp = hyper()
    for step in range(2):
        prev = [(f64(W), f64(G), f64(M)) for W, G, M in dev]
        code, flags = step_once(groups, {})
        assert code == m.MUON_OK and flags == 0
        for (W, G, M), (W0, G0, M0) in zip(dev, prev):
            for b in range(W.shape[0]):
                ref = oracle.muon_step(W0[b], G0[b], M0[b], hp)
                assert np.max(ulp_diff_f32(M[b].cpu().numpy(), momentum_ref_f32(M0[b], G0[b], hp))) <= 1
                check_w(f64(W[b]), ref["W"], hp, ref["scale"], bf16=True)


@pytest.mark.parametrize("offset", [0, 8])
def test_w_rows_not_32_byte_aligned(offset):
    """W, G and M as views with a padded row stride (520 elements: bf16 rows
    alternate between 32- and 16-byte alignment) and, with offset 8, a base
    16 bytes past a 32-byte boundary: the last update's W read-modify-write
    takes its 16-byte path and must give the same result as the oracle."""
    W0, G0, M0 = workloads.random_case(44, 256, 512, batch=2)
    pad = 520

    def padded(t):
        big = torch.zeros(t.shape[0], t.shape[1], pad + offset, dtype=t.dtype, device=DEV)
        v = big[:, :, offset:offset + t.shape[2]]
        v.copy_(t.to(DEV))
        return big, v

    (Wb, W), (Gb, G), (Mb, M) = padded(W0), padded(G0), padded(M0)
    assert (W.data_ptr() % 32 == 0) == (offset == 0) and W.stride(2) == 1
    group = m.Group([W[0], W[1]], [G[0], G[1]], [M[0], M[1]])
    hp = hyper()
    code, flags = step_once([group], {})
    assert code == m.MUON_OK and flags == 0
    for b in range(2):
        ref = oracle.muon_step(f64(W0[b]), f64(G0[b]), f64(M0[b]), hp)
        check_w(f64(W[b]), ref["W"], hp, ref["scale"], bf16=True)
        # the padding around each row is untouched
        assert float(Wb[b, :, :offset].abs().sum()) == 0.0
        assert float(Wb[b, :, offset + 512:].abs().sum()) == 0.0


def test_empty_call_is_a_no_op():
    """No groups: the call succeeds, clears the status word and touches nothing."""
    W, G, M = workloads.random_case(45, 64, 64, batch=1)
    Wd = W.to(DEV)
    before = Wd.clone()
    hp = m.hparams()
    ws = m.workspace(m.muon_step_workspace_size([m.Group.stacked(Wd, G.to(DEV), M.to(DEV))]))
    ws.fill_(0xFF)                                   # a stale status word
    m.muon_step_batched([], hp, ws)
    code, flags = m.muon_get_status(ws)
    assert code == m.MUON_OK and flags == 0
    assert torch.equal(Wd, before)


def test_weight_decay_mask():
    W, G, M = workloads.random_case(40, 256, 256, batch=2, w_dtype=torch.float32)
    W0, G0, M0 = f64(W), f64(G), f64(M)
    Wd, Gd, Md = W.to(DEV), G.to(DEV), M.to(DEV)
    code, flags = step_once([m.Group.stacked(Wd, Gd, Md, wd_mask=[True, False])], {})
    assert code == m.MUON_OK and flags == 0
    hp = hyper()
    for b, decay in enumerate([True, False]):
        ref = oracle.muon_step(W0[b], G0[b], M0[b], hp, decay=decay)
        check_w(f64(Wd[b]), ref["W"], hp, ref["scale"], bf16=False)


def test_zero_gradient_is_pure_weight_decay():
    W = torch.tensor(np.random.default_rng(41).normal(0, 0.02, (1, 256, 512)), dtype=torch.float32)
    Wd = W.to(DEV)
    Gd = torch.zeros_like(Wd)
    Md = torch.zeros_like(Wd)
    code, flags = step_once([m.Group.stacked(Wd, Gd, Md)], {})
    assert code == m.MUON_OK and flags == 0
    decay = np.float32(1.0 - float(np.float32(2.7e-4)) * float(np.float32(0.1)))
    want = (W.numpy() * decay).astype(np.float32)
    assert np.max(ulp_diff_f32(Wd.cpu().numpy(), want)) <= 1
    assert torch.count_nonzero(Md).item() == 0


def test_batched_equals_unbatched_and_chunking_bitwise():
    W, G, M = workloads.random_case(42, 256, 384, batch=6)
    runs = []
    for chunks in ([6], [1] * 6, [2, 2, 2], [4, 2]):
        Wd, Gd, Md = W.clone().to(DEV), G.to(DEV), M.clone().to(DEV)
        groups, start = [], 0
        for c in chunks:
            groups.append(m.Group.stacked(Wd[start:start + c], Gd[start:start + c], Md[start:start + c]))
            start += c
        code, flags = step_once(groups, {})
        assert code == m.MUON_OK and flags == 0
        runs.append((Wd.cpu(), Md.cpu()))
    for Wr, Mr in runs[1:]:
        assert torch.equal(Wr, runs[0][0]) and torch.equal(Mr, runs[0][1])


@pytest.mark.parametrize("scale_mode", ["spectral", "unit_rms_norm"])
def test_split_head_attention_weight(scale_mode):
    """QKV weight 4096 x (32 x 128), orthogonalised per head (heads = batch,
    fan_out = head size 128)."""
    h = workloads.split_heads(seed=2)
    W0, G0, M0 = f64(h.W), f64(h.G), f64(h.M)
    Wd, Gd, Md = h.W.to(DEV), h.G.to(DEV), h.M.to(DEV)
    code, flags = step_once([m.Group.split_head(Wd, Gd, Md, h.n_heads, h.head_dim)],
                            dict(scale_mode=scale_mode))
    assert code == m.MUON_OK and flags == 0
    hp = hyper(scale_mode=scale_mode, fan_out_axis=1)
    Wg, Mg = f64(Wd), Md.cpu().numpy()
    for k in range(h.n_heads):
        s = slice(k * h.head_dim, (k + 1) * h.head_dim)
        ref = oracle.muon_step(W0[:, s], G0[:, s], M0[:, s], hp)
        assert np.max(ulp_diff_f32(Mg[:, s], momentum_ref_f32(M0[:, s], G0[:, s], hp))) <= 1
        check_w(Wg[:, s], ref["W"], hp, ref["scale"], bf16=True)


def test_split_linear_fc1_rows():
    """Fused [gate; up] FC1 weight (2 x 512 rows, 384 columns, fp32 W):
    each row block is orthogonalised on its own (fan_out = its rows)."""
    W, G, M = workloads.random_case(60, 1024, 384, batch=1, w_dtype=torch.float32)
    W, G, M = W[0], G[0], M[0]
    W0, G0, M0 = f64(W), f64(G), f64(M)
    Wd, Gd, Md = W.to(DEV), G.to(DEV), M.to(DEV)
    for mode in ("spectral", "unit_rms_norm"):
        Wp, Mp = f64(Wd), Md.cpu().numpy().astype(np.float64)
        code, flags = step_once([m.Group.split_rows(Wd, Gd, Md, 2)], dict(scale_mode=mode))
        assert code == m.MUON_OK and flags == 0
        hp = hyper(scale_mode=mode)
        for k, (w, g, mm) in enumerate(zip(oracle.row_blocks(Wp, 2), oracle.row_blocks(G0, 2),
                                           oracle.row_blocks(Mp, 2))):
            ref = oracle.muon_step(w, g, mm, hp)
            check_w(f64(Wd[512 * k:512 * (k + 1)]), ref["W"], hp, ref["scale"], bf16=False)


# ---------------------------------------------------------------------------
# device status
# ---------------------------------------------------------------------------
def test_nonfinite_gradient_is_flagged():
    W, G, M = workloads.random_case(50, 128, 256, batch=1)
    G[0, 3, 5] = float("nan")
    code, flags = step_once([m.Group.stacked(W.to(DEV), G.to(DEV), M.to(DEV))], {})
    assert code == m.MUON_OK and (flags & m.MUON_FLAG_NONFINITE)


def test_misaligned_pointer_in_device_array_is_flagged_and_skipped():
    """A matrix whose pointer is not 16-byte aligned is detected by the kernel
    before any access, flagged, and left untouched; the others are updated."""
    W, G, M = workloads.random_case(51, 128, 256, batch=2)
    Wd, Gd, Md = W.to(DEV), G.to(DEV), M.to(DEV)
    grp = m.Group.stacked(Wd, Gd, Md)
    grp.ptrs[1, 1] += 2                       # G of matrix 1 shifted by one bf16 element
    W1, M1 = Wd[1].clone(), Md[1].clone()
    code, flags = step_once([grp], {})
    assert code == m.MUON_OK and (flags & m.MUON_FLAG_MISALIGNED)
    assert torch.equal(Wd[1], W1) and torch.equal(Md[1], M1)
    assert not torch.equal(Md[0], M[0].to(DEV))


def test_bounded_wait_times_out_and_context_survives():
    ws = m.workspace(256)
    m.muon_check_wait_timeout(ws, 2_000_000)           # 2 ms
    code, flags = m.muon_get_status(ws)
    assert code == m.MUON_ERR_TIMEOUT and (flags & m.MUON_FLAG_TIMEOUT)
    x = torch.randn(1, 128, 256, device=DEV)
    got = run_ns(x)
    assert rel_fro(f64(got[0]), oracle.newton_schulz(f64(x[0]))) <= NS_TOL


# ---------------------------------------------------------------------------
# groups sharing one Newton–Schulz chain (merge_groups)
# ---------------------------------------------------------------------------
HYBRID = [(8, (3.4445, -4.7750, 2.0315)), (2, (2.0, -1.5, 0.5))]


def _merge_sets(seed):
    """Groups: 3 wide 512x768 bf16, 2 tall 768x512 bf16, 2 of 256x384, 1 wide
    512x768 fp32 W (four groups share the 512 x 768 wide shape)."""
    specs = [(3, 512, 768, torch.bfloat16), (2, 768, 512, torch.bfloat16),
             (2, 256, 384, torch.bfloat16), (1, 512, 768, torch.float32)]
    out = []
    for k, (b, r, c, wdt) in enumerate(specs):
        W, G, M = workloads.random_case(seed + k, r, c, batch=b, w_dtype=wdt, m_scale=1.0)
        out.append((W, G, M))
    return out


def _run_sets(sets, schedule, masks=None):
    dev = [(W.to(DEV), G.to(DEV), M.to(DEV)) for W, G, M in sets]
    groups = [m.Group.stacked(W, G, M, wd_mask=None if masks is None else masks[i])
              for i, (W, G, M) in enumerate(dev)]
    code, flags = step_once(groups, {}, schedule)
    assert code == m.MUON_OK and flags == 0, (code, flags)
    return [(W.cpu(), M.cpu()) for W, _, M in dev]


@pytest.mark.parametrize("stages", [HYBRID, [(3, (3.4445, -4.7750, 2.0315))]],
                         ids=["hybrid-fused-store", "three-iterations-apply-pass"])
def test_merged_chains_equal_separate_chains_bitwise(stages):
    """A tall and a wide group of one wide shape (and a same-shape fp32 group)
    in one chain give bit-identical W and M to one chain per group; the
    unmerged run is itself checked against the oracle."""
    sets = _merge_sets(70)
    masks = [[True, False, True], [False, True], None, [True]]
    merged = _run_sets(sets, m.Schedule(stages, merge_groups=True), masks)
    plain = _run_sets(sets, m.Schedule(stages), masks)
    for (Wm, Mm), (Wp, Mp) in zip(merged, plain):
        assert torch.equal(Wm, Wp) and torch.equal(Mm, Mp)
    hp = hyper()
    for gi, (W, G, M) in enumerate(sets):
        for b in range(W.shape[0]):
            decay_on = masks[gi] is None or masks[gi][b]
            ref = oracle.muon_step(f64(W[b]), f64(G[b]), f64(M[b]), hp, decay=decay_on,
                                   stages=stages)
            check_w(f64(plain[gi][0][b]), ref["W"], hp, ref["scale"],
                    bf16=W.dtype == torch.bfloat16)


def test_more_groups_than_one_chain_holds():
    """Five groups of one shape: chains of at most four groups."""
    sets = [workloads.random_case(80 + k, 256, 512, batch=2) for k in range(5)]
    merged = _run_sets(sets, m.Schedule(HYBRID, merge_groups=True))
    plain = _run_sets(sets, m.Schedule(HYBRID))
    for (Wm, Mm), (Wp, Mp) in zip(merged, plain):
        assert torch.equal(Wm, Wp) and torch.equal(Mm, Mp)
