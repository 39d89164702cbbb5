"""Pins of the fp64 Adam oracle (the optimizer of the embedding, head and scalars).

Closed forms derived by hand, properties of the update, a second pure-Python
implementation and the pages' constants -- chosen so that a wrong bias
correction, a misplaced eps, swapped betas or a dropped L2 term fail one of
them.
"""

import os

import numpy as np
import pytest

import oracle
from tests import adam_bruteforce_py

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "adam_groups.txt")


def _golden():
    out = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            out[k] = float(v)
    return out


G = _golden()


def test_page_constants_match_defaults():
    assert oracle.ADAM_BETAS == (G["p50b.beta1"], G["p50b.beta2"]) == (G["flex.beta1"], G["flex.beta2"])
    assert oracle.AdamConfig().weight_decay == G["p50b.weight_decay"]
    assert oracle.ADAM_EPS == 1e-8


def _run(p0, grads, lr, cfg=oracle.AdamConfig()):
    orc = oracle.AdamOracle([p0.size], cfg)
    p = p0.copy()
    for g in grads:
        (p,) = orc.step([p], [g], [lr])
    return p, orc


@pytest.mark.parametrize("k", [1, 2, 7, 40])
def test_constant_gradient_closed_form(k):
    # m_t = (1 - b1^t) g and v_t = (1 - b2^t) g^2, so every step moves p by lr * g / (|g| + eps)
    rng = np.random.default_rng(k)
    p0 = rng.normal(size=37)
    g = rng.normal(size=37) * 10.0 ** rng.uniform(-6, 1, size=37)
    lr = 0.3
    p, orc = _run(p0, [g] * k, lr)
    expect = p0 - k * lr * g / (np.abs(g) + oracle.ADAM_EPS)
    assert np.allclose(p, expect, rtol=1e-13, atol=1e-15)
    assert np.allclose(orc.m[0], (1 - 0.9 ** k) * g, rtol=1e-13, atol=0)
    assert np.allclose(orc.v[0], (1 - 0.95 ** k) * g * g, rtol=1e-13, atol=0)


@pytest.mark.parametrize("k", [1, 2, 3, 10])
def test_alternating_gradient_closed_form(k):
    # g_t = (-1)^(t+1) c:  m_t = (1-b1) c (-1)^(t+1) (1 - (-b1)^t) / (1 + b1),  v_t = (1 - b2^t) c^2
    b1, b2, c, lr = 0.9, 0.95, 0.7, 0.002
    p0 = np.array([0.25, -1.5])
    grads = [np.full(2, c * (-1) ** (t + 1)) for t in range(1, k + 1)]
    p, orc = _run(p0, grads, lr)
    total = 0.0
    for t in range(1, k + 1):
        m_t = (1 - b1) * c * (-1) ** (t + 1) * (1 - (-b1) ** t) / (1 + b1)
        total += lr * (m_t / (1 - b1 ** t)) / (c + oracle.ADAM_EPS)
    assert np.allclose(p, p0 - total, rtol=0, atol=1e-15)
    assert np.allclose(orc.v[0], (1 - b2 ** k) * c * c, rtol=1e-14, atol=0)


def test_zero_gradient_is_a_fixed_point():
    p0 = np.linspace(-1, 1, 9)
    p, orc = _run(p0, [np.zeros(9)] * 3, 0.6)
    assert np.array_equal(p, p0) and not orc.m[0].any() and not orc.v[0].any()


def test_update_is_scale_invariant_without_eps():
    rng = np.random.default_rng(5)
    p0 = rng.normal(size=20)
    grads = [rng.normal(size=20) for _ in range(4)]
    cfg = oracle.AdamConfig(eps=0.0)
    a, _ = _run(p0, grads, 0.04, cfg)
    b, _ = _run(p0, [1e3 * g for g in grads], 0.04, cfg)
    assert np.allclose(a, b, rtol=1e-14, atol=1e-15)


def test_l2_term_on_a_zero_gradient():
    # g = wd p on the first step: p moves by lr * sign(p) * |wd p| / (|wd p| + eps)
    p0 = np.array([0.5, -2.0, 1e-9])
    wd, lr = 0.1, 0.01
    p, _ = _run(p0, [np.zeros(3)], lr, oracle.AdamConfig(weight_decay=wd))
    gw = wd * p0
    assert np.allclose(p, p0 - lr * gw / (np.abs(gw) + oracle.ADAM_EPS), rtol=1e-14, atol=0)


@pytest.mark.parametrize("wd", [0.0, 0.05])
def test_matches_pure_python(wd):
    rng = np.random.default_rng(11)
    p0 = rng.normal(size=6)
    grads = [rng.normal(size=6) * 1e-3 for _ in range(5)]
    p, orc = _run(p0, grads, 0.3, oracle.AdamConfig(weight_decay=wd))
    bp, bm, bv = adam_bruteforce_py.adam_steps(p0.tolist(), [g.tolist() for g in grads], 0.3, 0.9, 0.95, 1e-8, wd)
    assert np.allclose(p, bp, rtol=1e-13, atol=1e-16)
    assert np.allclose(orc.m[0], bm, rtol=1e-13, atol=1e-20)
    assert np.allclose(orc.v[0], bv, rtol=1e-13, atol=1e-24)


def test_rejects_step_zero():
    with pytest.raises(ValueError):
        oracle.adam_param_update(np.zeros(1), np.zeros(1), np.zeros(1), 0, 0.1, 0.9, 0.95, 1e-8)


def test_mutations_are_caught():
    """Plausible mistakes fail the closed forms above."""
    g = np.array([0.3, -2.0, 3e-6, -2e-5])  # small entries make the place of eps visible
    p0 = np.zeros(4)
    lr, k = 0.3, 3
    expect = p0 - k * lr * g / (np.abs(g) + 1e-8)

    def run(update):
        m = np.zeros(4)
        v = np.zeros(4)
        p = p0.copy()
        for t in range(1, k + 1):
            m, v = oracle.adam_moments(m, v, g, 0.9, 0.95)
            p = update(p, m, v, t)
        return p

    good = run(lambda p, m, v, t: oracle.adam_param_update(p, m, v, t, lr, 0.9, 0.95, 1e-8))
    assert np.allclose(good, expect, rtol=1e-13)
    shifted_t = run(lambda p, m, v, t: oracle.adam_param_update(p, m, v, t + 1, lr, 0.9, 0.95, 1e-8))
    eps_inside = run(lambda p, m, v, t: p - lr * (m / (1 - 0.9 ** t)) / np.sqrt(v / (1 - 0.95 ** t) + 1e-8))
    swapped = run(lambda p, m, v, t: oracle.adam_param_update(p, m, v, t, lr, 0.95, 0.9, 1e-8))
    no_bc2 = run(lambda p, m, v, t: p - lr * (m / (1 - 0.9 ** t)) / (np.sqrt(v) + 1e-8))
    for bad in (shifted_t, eps_inside, swapped, no_bc2):
        assert not np.allclose(bad, expect, rtol=1e-6)
