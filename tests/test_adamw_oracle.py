"""Pins of the AdamW oracle (CPU): hand-worked values, closed forms of Adam's
first steps, invariances, and planted mistakes that each must fail a pin."""
import numpy as np
import pytest

from oracle import adamw_ref
from oracle.adamw_ref import AdamWHyper, adamw_step
from tests.conftest import read_golden


def check_hand_values(step=adamw_step):
    """Golden: g = 1, -1, 2 from a zero state (tests/golden/adamw_hand.txt)."""
    rows = read_golden("adamw_hand.txt")
    m = v = np.zeros(1)
    W = np.zeros(1)
    for t, g, m_w, v_w, mh_w, vh_w, u_w in rows:
        hp = AdamWHyper(lr=0.0, t=int(t))
        out = step(W, np.array([float(g)]), m, v, hp)
        m, v = out["m"], out["v"]
        assert m[0] == pytest.approx(float(m_w), rel=1e-14, abs=1e-16)
        assert v[0] == pytest.approx(float(v_w), rel=1e-14)
        assert out["u"][0] == pytest.approx(float(u_w), rel=1e-13)
        b1, b2 = hp.beta1, hp.beta2
        assert m[0] / (1 - b1 ** hp.t) == pytest.approx(float(mh_w), rel=1e-13)
        assert v[0] / (1 - b2 ** hp.t) == pytest.approx(float(vh_w), rel=1e-13)


def check_first_step_is_sign_descent(step=adamw_step):
    """Adam's bias correction makes step 1 from a zero state m_hat = g,
    v_hat = g^2, so u = g/(|g| + eps) = sign(g) for |g| >> eps and
    W_1 = W(1 - lr wd) - lr sign(g)."""
    rng = np.random.default_rng(7)
    g = rng.standard_normal(64) * np.exp(rng.uniform(-8, 3, 64))
    W = rng.standard_normal(64) * 0.02
    hp = AdamWHyper(lr=1e-3, weight_decay=0.1, t=1)
    out = step(W, g, np.zeros(64), np.zeros(64), hp)
    np.testing.assert_allclose(out["u"], np.sign(g), rtol=1e-14, atol=0)
    np.testing.assert_allclose(out["W"], W * (1 - 1e-4) - 1e-3 * np.sign(g), rtol=1e-14, atol=1e-18)


def check_constant_gradient(step=adamw_step, steps=6):
    """A constant gradient gives m_t = g(1 - b1^t), v_t = g^2(1 - b2^t), so the
    bias-corrected direction is sign(g) at every step t."""
    g = np.array([3e-3, -2.5, 7.0, -1e-6])
    m = v = np.zeros(4)
    W = np.zeros(4)
    for t in range(1, steps + 1):
        out = step(W, g, m, v, AdamWHyper(lr=0.0, t=t))
        m, v = out["m"], out["v"]
        np.testing.assert_allclose(m, g * (1 - 0.9 ** t), rtol=1e-13)
        np.testing.assert_allclose(v, g * g * (1 - 0.95 ** t), rtol=1e-13)
        np.testing.assert_allclose(out["u"], np.sign(g), rtol=1e-12)


def check_scale_invariance(step=adamw_step):
    """Scaling every gradient of a history by k > 0 scales m by k and v by k^2,
    leaving u unchanged (eps negligible)."""
    rng = np.random.default_rng(3)
    gs = rng.standard_normal((4, 32))
    for k in (1e-3, 10.0):
        m1 = v1 = m2 = v2 = np.zeros(32)
        for t, g in enumerate(gs, start=1):
            a = step(np.zeros(32), g, m1, v1, AdamWHyper(lr=0.0, t=t))
            b = step(np.zeros(32), k * g, m2, v2, AdamWHyper(lr=0.0, t=t))
            m1, v1, m2, v2 = a["m"], a["v"], b["m"], b["v"]
            np.testing.assert_allclose(b["u"], a["u"], rtol=1e-12)


def check_zero_gradient_and_mask(step=adamw_step):
    """g = 0 from a zero state gives u = 0/(0 + eps) = 0: W only decays, and
    with the decay masked off W is unchanged."""
    W = np.array([0.5, -0.25, 1.0])
    z = np.zeros(3)
    hp = AdamWHyper(lr=0.1, weight_decay=0.1, t=1)
    on = step(W, z, z, z, hp, decay=True)
    off = step(W, z, z, z, hp, decay=False)
    np.testing.assert_array_equal(on["W"], W * (1 - 0.01))
    np.testing.assert_array_equal(off["W"], W)


PINS = (check_hand_values, check_first_step_is_sign_descent, check_constant_gradient,
        check_scale_invariance, check_zero_gradient_and_mask)


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_adamw_pin(pin):
    pin()


def test_defaults_are_the_v4_settings():
    """"Muon 优化器" §3: beta1 0.9, beta2 0.95, eps 1e-20, weight decay 0.1."""
    hp = AdamWHyper()
    assert (hp.beta1, hp.beta2, hp.eps, hp.weight_decay) == (0.9, 0.95, 1e-20, 0.1)


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------
def _no_bias_correction(m_t, v_t, beta1, beta2, eps, t):
    return m_t / (np.sqrt(v_t) + eps)


def _bias_correction_off_by_one(m_t, v_t, beta1, beta2, eps, t):
    return (m_t / (1 - beta1 ** (t + 1))) / (np.sqrt(v_t / (1 - beta2 ** (t + 1))) + eps)


def _no_sqrt(m_t, v_t, beta1, beta2, eps, t):
    return (m_t / (1 - beta1 ** t)) / (v_t / (1 - beta2 ** t) + eps)


def _swapped_betas_first(m, g, beta1):
    return 0.95 * np.asarray(m, float) + 0.05 * np.asarray(g, float)


def _sign_flip(m_t, v_t, beta1, beta2, eps, t):
    return -(m_t / (1 - beta1 ** t)) / (np.sqrt(v_t / (1 - beta2 ** t)) + eps)


def _square_missing(v, g, beta2):
    return beta2 * np.asarray(v, float) + (1 - beta2) * np.abs(np.asarray(g, float))


@pytest.mark.parametrize("name,bad", [
    ("adam_direction", _no_bias_correction),
    ("adam_direction", _bias_correction_off_by_one),
    ("adam_direction", _no_sqrt),
    ("adam_direction", _sign_flip),
    ("first_moment", _swapped_betas_first),
    ("second_moment", _square_missing),
])
def test_planted_adamw_mistakes_are_caught(monkeypatch, name, bad):
    monkeypatch.setattr(adamw_ref, name, bad)
    failed = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1


def test_planted_coupled_decay_is_caught(monkeypatch):
    """L2-style decay (wd*W added to the gradient) instead of decoupled decay."""
    real = adamw_ref.adamw_step

    def coupled(W, G, m, v, hp, decay=True):
        G2 = np.asarray(G, float) + (hp.weight_decay * np.asarray(W, float) if decay else 0.0)
        out = real(W, G2, m, v, AdamWHyper(hp.lr, hp.beta1, hp.beta2, hp.eps, 0.0, hp.t))
        return out
    failed = 0
    for pin in PINS:
        try:
            pin(coupled)
        except AssertionError:
            failed += 1
    assert failed >= 1
