"""Pins for the float64 oracle (CPU only).

Each check ties the oracle to something other than itself: the page's printed
constants, hand-worked examples (tests/golden/), the closed form of an odd
matrix polynomial through the SVD, textbook special cases, invariants, and a
BLAS-free C transcription.  The last block plants mistakes in the oracle and
asserts that the pins catch each one.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import muon_ref
from tests.conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------------------
# page constants
# ---------------------------------------------------------------------------
def golden_stages():
    return tuple((int(r[0]), (float(r[1]), float(r[2]), float(r[3])))
                 for r in read_golden("hybrid_schedule.txt"))


def test_schedule_matches_page():
    assert tuple(oracle.HYBRID_STAGES) == golden_stages()


def test_hyperparameters_match_page():
    g = {r[0]: float(r[1]) for r in read_golden("hyperparameters.txt")}
    assert oracle.DEFAULT_MU == g["mu"]
    assert oracle.DEFAULT_WD == g["weight_decay"]
    assert oracle.DEFAULT_GAMMA == g["gamma"]
    assert oracle.DEFAULT_LR == g["lr"]


# ---------------------------------------------------------------------------
# P1: closed form through the SVD.  An odd polynomial a x + b (x x^T) x +
# c (x x^T)^2 x maps each singular value s to a s + b s^3 + c s^5 and keeps
# the singular vectors, so the whole schedule acts as a scalar map on the
# normalised spectrum.
# ---------------------------------------------------------------------------
def scalar_map(sig, stages):
    out = []
    for s in sig:
        for steps, (a, b, c) in stages:
            for _ in range(steps):
                s = a * s + b * s ** 3 + c * s ** 5
        out.append(s)
    return np.array(out)


def svd_closed_form(X, stages, normalize=True):
    U, sig, Vt = np.linalg.svd(X, full_matrices=False)
    if normalize:
        sig = sig / math.sqrt(float(np.sum(sig ** 2)))
    return (U * scalar_map(sig, stages)) @ Vt


SVD_SHAPES = [(8, 16), (16, 8), (64, 32), (32, 64), (100, 100), (1, 7), (7, 1), (3, 3)]


def check_svd_closed_form(ns, stages=None, seed=0):
    stages = golden_stages() if stages is None else stages
    rng = np.random.default_rng(seed)
    for shape in SVD_SHAPES:
        X = rng.standard_normal(shape)
        got = ns(X, stages, True)
        want = svd_closed_form(X, stages)
        assert got.shape == want.shape
        assert np.max(np.abs(got - want)) < 1e-10, shape


def test_p1_svd_closed_form():
    check_svd_closed_form(oracle.newton_schulz)


def test_p1_svd_closed_form_custom_schedules():
    rng = np.random.default_rng(5)
    for stages in [((1, (1.0, 0.0, 0.0)),), ((1, (0.0, 1.0, 0.0)),), ((1, (0.0, 0.0, 1.0)),),
                   ((3, (1.5, -0.5, 0.0)),), ((2, (2.0, -1.5, 0.5)), (1, (3.4445, -4.775, 2.0315)))]:
        for shape in [(5, 9), (9, 5), (12, 12)]:
            X = rng.standard_normal(shape)
            X = X / (1.1 * np.linalg.norm(X, 2))          # spectrum inside (0, 1)
            for norm in (True, False):
                got = oracle.newton_schulz(X, stages, norm)
                U, sig, Vt = np.linalg.svd(X, full_matrices=False)
                if norm:
                    sig = sig / np.linalg.norm(sig)
                want = (U * scalar_map(sig, stages)) @ Vt
                assert np.max(np.abs(got - want)) < 1e-11


# ---------------------------------------------------------------------------
# P2: near the polar factor U V^T on well-conditioned inputs
# ---------------------------------------------------------------------------
def test_p2_polar_factor_well_conditioned():
    rng = np.random.default_rng(1)
    for (r, c) in [(8, 16), (16, 8), (24, 24)]:
        k = min(r, c)
        U, _ = np.linalg.qr(rng.standard_normal((r, k)))
        V, _ = np.linalg.qr(rng.standard_normal((c, k)))
        sig = rng.uniform(0.05, 1.0, size=k)          # sigma/||sigma|| >= ~1e-2
        X = (U * sig) @ V.T
        O = oracle.newton_schulz(X)
        polar = U @ V.T
        assert np.linalg.norm(O - polar, 2) < 3e-3
        s = np.linalg.svd(O, compute_uv=False)
        assert np.all(np.abs(s - 1.0) < 3e-3)


# ---------------------------------------------------------------------------
# P3: zero in -> zero out; pure weight decay
# ---------------------------------------------------------------------------
def test_p3_zero_input():
    Z = np.zeros((6, 10))
    assert np.array_equal(oracle.newton_schulz(Z), Z)
    W = np.random.default_rng(2).standard_normal((6, 10))
    hp = oracle.MuonHyper(lr=2.7e-4, weight_decay=0.1)
    out = oracle.muon_step(W, Z, Z, hp)
    assert np.array_equal(out["O"], Z)
    assert np.array_equal(out["M"], Z)
    assert np.array_equal(out["W"], W * (1.0 - 2.7e-4 * 0.1))


# ---------------------------------------------------------------------------
# P4: the stable stage fixes a matrix with orthonormal rows (p(1) = 1);
# one fast step scales it by q(1) = a + b + c.
# ---------------------------------------------------------------------------
def test_p4_stable_stage_fixes_orthonormal_rows():
    rng = np.random.default_rng(3)
    Q, _ = np.linalg.qr(rng.standard_normal((20, 7)))
    Q = Q.T.copy()                                    # 7 x 20, orthonormal rows
    stable = golden_stages()[1]
    out = oracle.newton_schulz(Q, (stable,), normalize=False)
    assert np.max(np.abs(out - Q)) < 1e-14
    out_t = oracle.newton_schulz(Q.T, (stable,), normalize=False)
    assert np.max(np.abs(out_t - Q.T)) < 1e-14


def test_p4_fast_step_scales_orthonormal_rows():
    rng = np.random.default_rng(4)
    Q, _ = np.linalg.qr(rng.standard_normal((9, 9)))
    steps, (a, b, c) = golden_stages()[0]
    out = oracle.newton_schulz(Q, ((1, (a, b, c)),), normalize=False)
    assert np.max(np.abs(out - 0.701 * Q)) < 1e-13


# ---------------------------------------------------------------------------
# P5: equivariances
# ---------------------------------------------------------------------------
def test_p5_equivariances():
    rng = np.random.default_rng(6)
    X = rng.standard_normal((12, 20))
    O = oracle.newton_schulz(X)
    assert np.max(np.abs(oracle.newton_schulz(X.T) - O.T)) < 1e-12
    assert np.max(np.abs(oracle.newton_schulz(37.5 * X) - O)) < 1e-12
    assert np.max(np.abs(oracle.newton_schulz(-X) + O)) < 1e-12
    P, _ = np.linalg.qr(rng.standard_normal((12, 12)))
    R, _ = np.linalg.qr(rng.standard_normal((20, 20)))
    assert np.max(np.abs(oracle.newton_schulz(P @ X @ R) - P @ O @ R)) < 1e-11


# ---------------------------------------------------------------------------
# P6: 1 x 1 input -> sign(x) f(1)
# ---------------------------------------------------------------------------
def test_p6_scalar_case():
    f1 = scalar_map([1.0], golden_stages())[0]
    for x in (3.0, -0.25, 1e-30):
        out = oracle.newton_schulz(np.array([[x]]))
        assert abs(out[0, 0] - math.copysign(f1, x)) < 1e-15


# ---------------------------------------------------------------------------
# P7: hand-worked momentum / look-ahead values
# ---------------------------------------------------------------------------
def check_momentum_golden(step_fn):
    for style, nest, t, M_want, X_want in read_golden("momentum_hand.txt"):
        t = int(t)
        M = np.zeros((2, 3))
        G = np.ones((2, 3))
        for k in range(1, t + 1):
            hp = oracle.MuonHyper(mu=0.95, style=style, nesterov=bool(int(nest)), t=k)
            out = step_fn(np.zeros((2, 3)), G, M, hp)
            M = out["M"]
        assert np.allclose(out["M"], float(M_want), rtol=1e-13, atol=0), (style, t)
        assert np.allclose(out["X"], float(X_want), rtol=1e-13, atol=0), (style, t)


def test_p7_momentum_hand_examples():
    check_momentum_golden(oracle.muon_step)


def test_p7_ema_tends_to_sgd_direction():
    """EMA look-ahead is proportional to beta*buf/(1-beta^{t+1}) + g/(1-beta^t)
    with buf the SGD buffer (mu_ema = (1-beta) buf), so its direction tends to
    the SGD look-ahead's as t grows (RFC-0023 §方案 1, both styles)."""
    rng = np.random.default_rng(7)
    beta = 0.95
    buf = np.zeros((4, 4))
    mu = np.zeros((4, 4))
    for t in range(1, 400):
        g = rng.standard_normal((4, 4))
        buf = oracle.momentum_sgd(buf, g, beta)
        mu = oracle.momentum_ema(mu, g, beta)
        x_sgd = oracle.lookahead_sgd(buf, g, beta)
        x_ema = oracle.lookahead_ema(mu, g, beta, t)
        assert np.allclose(mu, (1 - beta) * buf, rtol=1e-12, atol=1e-14)
        want = beta * buf / (1 - beta ** (t + 1)) + g / (1 - beta ** t)
        assert np.allclose(x_ema / (1 - beta), want, rtol=1e-10, atol=1e-12)
    cos = np.sum(x_sgd * x_ema) / (np.linalg.norm(x_sgd) * np.linalg.norm(x_ema))
    assert cos > 1 - 1e-12


# ---------------------------------------------------------------------------
# P8: scale and weight-decay examples
# ---------------------------------------------------------------------------
def check_scale_golden(scale_fn):
    for r, c, mode, gamma, axis, want in read_golden("scale_examples.txt"):
        got = scale_fn(int(r), int(c), mode, float(gamma), int(axis))
        assert abs(got - float(want)) <= 1e-14 * max(1.0, abs(float(want))), (r, c, mode)


def test_p8_scale_examples():
    check_scale_golden(oracle.update_scale)


def check_weight_decay_golden(fn):
    for W, O, lr, wd, s, decay, want in read_golden("weight_decay_examples.txt"):
        got = fn(np.array([[float(W)]]), np.array([[float(O)]]),
                 float(lr), float(wd), float(s), bool(int(decay)))
        assert abs(got[0, 0] - float(want)) < 1e-15


def test_p8_weight_decay_examples():
    check_weight_decay_golden(oracle.decoupled_update)


def test_full_step_composition():
    """muon_step is the page's composition: momentum, look-ahead, NS, scale, decay."""
    rng = np.random.default_rng(8)
    W, G, M = (rng.standard_normal((10, 6)) for _ in range(3))
    hp = oracle.MuonHyper()
    out = oracle.muon_step(W, G, M, hp)
    M_t = 0.95 * M + G
    X = 0.95 * M_t + G
    O = svd_closed_form(X, golden_stages())
    W_t = W * (1 - 2.7e-4 * 0.1) - 2.7e-4 * math.sqrt(10) * 0.18 * O
    assert np.max(np.abs(out["W"] - W_t)) < 1e-13
    assert np.max(np.abs(out["O"] - O)) < 1e-10


# ---------------------------------------------------------------------------
# cross-checks: literal transcription and plain C
# ---------------------------------------------------------------------------
def test_literal_transcription_agrees():
    rng = np.random.default_rng(9)
    for shape in [(4, 9), (9, 4), (16, 16), (1, 30), (30, 1)]:
        X = rng.standard_normal(shape)
        a = oracle.newton_schulz(X)
        b = oracle.newton_schulz_literal(X)
        assert np.max(np.abs(a - b)) <= 1e-12


def test_plain_c_transcription_agrees():
    try:
        from oracle.c_ref import ns_iterate_c
        ns_iterate_c(np.ones((1, 1)), [(1.0, 0.0, 0.0)])
    except Exception as e:  # pragma: no cover - no compiler
        pytest.skip(f"C oracle unavailable: {e}")
    rng = np.random.default_rng(10)
    coeffs = oracle.expand_stages(golden_stages())
    for shape in [(5, 11), (11, 5), (17, 17), (2, 40)]:
        X = rng.standard_normal(shape)
        assert np.max(np.abs(ns_iterate_c(X, coeffs) - oracle.newton_schulz(X))) <= 1e-12
        Y = X / (2.0 * np.linalg.norm(X))
        want = oracle.newton_schulz(Y, golden_stages(), False)
        assert np.max(np.abs(ns_iterate_c(Y, coeffs, False) - want)) <= 1e-12


# ---------------------------------------------------------------------------
# split_head and grouping
# ---------------------------------------------------------------------------
def test_split_head_slices_are_columns():
    W = np.arange(4 * 6, dtype=np.float64).reshape(4, 6)
    heads = oracle.head_slices(W, 3, 2)
    assert len(heads) == 3
    assert np.array_equal(heads[1], W[:, 2:4])
    with pytest.raises(ValueError):
        oracle.head_slices(W, 4, 2)


def test_split_head_fan_rule():
    """With split_head the heads are the batch dimension and fan_out is the
    head size (RFC-0023 §背景 consistent_rms; §方案 3)."""
    assert oracle.update_scale(4096, 128, "spectral", 0.18, 1) == pytest.approx(11.52, rel=1e-15)
    assert oracle.update_scale(4096, 128, "unit_rms_norm", 0.18, 1) == pytest.approx(
        math.sqrt(128 / 4096), rel=1e-15)


def test_row_blocks_are_contiguous_row_ranges():
    W = np.arange(6 * 4, dtype=np.float64).reshape(6, 4)
    gate, up = oracle.row_blocks(W, 2)
    assert np.array_equal(gate, W[:3]) and np.array_equal(up, W[3:])
    with pytest.raises(ValueError):
        oracle.row_blocks(W, 4)


def test_group_by_shape_golden():
    K0, K1, K2 = (1024, 1024, 0, 0, 0), (1024, 4096, 0, 0, 0), (8, 16, 0, 0, 0)
    keys = [K0, K1, K0, K0, K2, K1]
    for row in read_golden("group_by_shape.txt"):
        mb, ng = int(row[0]), int(row[1])
        want = [int(v) for v in row[2:]]
        got, n = oracle.group_by_shape(keys, mb)
        assert n == ng and got == want, mb


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------
_REAL_NS = muon_ref.ns_iteration


def _ns_drop_c(X, a, b, c):
    S = X @ X.T
    return a * X + b * (S @ X)


def _ns_sign_b(X, a, b, c):
    S = X @ X.T
    SX = S @ X
    return a * X - b * SX + c * (S @ SX)


def _ns_wrong_side(X, a, b, c):
    """(X^T X) X in place of (X X^T) X; differs only for square inputs."""
    if X.shape[0] != X.shape[1]:
        return _REAL_NS(X, a, b, c)
    S = X.T @ X
    SX = S @ X
    return a * X + b * SX + c * (S @ SX)


def _ns_transposed_operand(X, a, b, c):
    """X^T in place of X inside the b-term; differs only for square inputs."""
    if X.shape[0] != X.shape[1]:
        return _REAL_NS(X, a, b, c)
    S = X @ X.T
    return a * X + b * (S @ X.T) + c * (S @ (S @ X))


@pytest.mark.parametrize("bad", [_ns_drop_c, _ns_sign_b, _ns_wrong_side, _ns_transposed_operand])
def test_planted_ns_mistakes_are_caught(monkeypatch, bad):
    monkeypatch.setattr(muon_ref, "ns_iteration", bad)
    with pytest.raises(AssertionError):
        check_svd_closed_form(muon_ref.newton_schulz)


def test_planted_missing_normalisation_is_caught(monkeypatch):
    real = muon_ref.newton_schulz

    def no_norm(X, stages=muon_ref.HYBRID_STAGES, normalize=True):
        return real(X, stages, False)
    with pytest.raises(AssertionError):
        check_svd_closed_form(no_norm)


def test_planted_stage_order_is_caught():
    swapped = (golden_stages()[1], golden_stages()[0])
    with pytest.raises(AssertionError):
        check_svd_closed_form(lambda X, st, n: oracle.newton_schulz(X, swapped, n))


def test_planted_momentum_mistakes_are_caught(monkeypatch):
    monkeypatch.setattr(muon_ref, "lookahead_sgd", lambda M_t, G, mu: np.asarray(M_t, float))
    with pytest.raises(AssertionError):
        check_momentum_golden(muon_ref.muon_step)


def test_planted_bias_correction_off_by_one_is_caught(monkeypatch):
    monkeypatch.setattr(muon_ref, "lookahead_ema",
                        lambda mu_t, G, beta, t: beta * mu_t / (1 - beta ** t)
                        + (1 - beta) * G / (1 - beta ** t))
    with pytest.raises(AssertionError):
        check_momentum_golden(muon_ref.muon_step)


def test_planted_scale_mistake_is_caught():
    def bad_scale(r, c, mode, gamma, axis):
        if mode == "spectral":
            return math.sqrt(min(r, c)) * gamma
        return oracle.update_scale(r, c, mode, gamma, axis)
    with pytest.raises(AssertionError):
        check_scale_golden(bad_scale)

    def bad_axis(r, c, mode, gamma, axis):
        return oracle.update_scale(r, c, mode, gamma, 1 - axis)
    with pytest.raises(AssertionError):
        check_scale_golden(bad_axis)


def _wd_without_lr(W, O, lr, wd, scale, decay=True):
    """Decay by (1 - lambda) in place of (1 - eta*lambda)."""
    return W * ((1.0 - wd) if decay else 1.0) - lr * scale * O


def _wd_mask_ignored(W, O, lr, wd, scale, decay=True):
    return W * (1.0 - lr * wd) - lr * scale * O


def _wd_sign_of_step(W, O, lr, wd, scale, decay=True):
    return W * ((1.0 - lr * wd) if decay else 1.0) + lr * scale * O


def _wd_coupled(W, O, lr, wd, scale, decay=True):
    """Decay folded into the scaled step (lambda*W added to O before the scale)."""
    return W - lr * scale * (O + (wd * W if decay else 0.0))


@pytest.mark.parametrize("bad", [_wd_without_lr, _wd_mask_ignored, _wd_sign_of_step, _wd_coupled])
def test_planted_weight_decay_mistakes_are_caught(bad):
    with pytest.raises(AssertionError):
        check_weight_decay_golden(bad)
