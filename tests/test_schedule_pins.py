"""Pins of the oracle's step schedules (learning-rate multiplier, momentum warm-up).

The constants come from tests/golden/schedule_points.txt (printed on the
pages, cited there); the checks are properties those pages fix -- where the
schedule starts and ends, that it is a straight line in between (constant
per-step change), its area, and flatness after the end -- so that a dropped
clamp, an off-by-one at either end or a floor applied relative to the
decayed value fails one of them.
"""

import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "schedule_points.txt")


def _points():
    out = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = line.split()
        out[k] = float(v)
    return out


P = _points()


def test_flex_warmdown_boundaries_and_linearity():
    n, w, start = int(P["flex.num_iterations"]), int(P["flex.warmdown_iters"]), int(P["flex.warmdown_start"])
    assert n - w == start  # the page's own numbers agree
    m = np.array([oracle.lr_multiplier(s, start, n, P["flex.lr_end"]) for s in range(n + 1)])
    assert np.all(m[: start + 1] == 1.0)        # constant phase, including the last full step
    assert m[n] == 0.0                          # reaches zero at the last iteration
    steps = np.diff(m[start: n + 1])
    assert np.allclose(steps, -1.0 / w, rtol=0, atol=1e-15)  # a straight line: 1/562 per step
    assert np.all(np.diff(m) <= 0)


def test_fixmuonlr_cooldown_floor_and_extension():
    frac, floor, ext = P["fix.cooldown_frac"], P["fix.lr_floor"], int(P["fix.extension_steps"])
    for n in (1000, 1645, 2290):  # main-phase lengths (the page fixes the shape, not N)
        cs, ce = round(n * (1.0 - frac)), n
        m = np.array([oracle.lr_multiplier(s, cs, ce, floor) for s in range(n + ext + 1)])
        assert m.max() == 1.0 and m.min() == floor             # clamped above by 1, floor is absolute
        assert np.all(m[: cs + 1] == 1.0)
        assert np.all(m[n:] == floor)                          # flat through every extension step
        assert len(m[n:]) == ext + 1
        seg = m[cs: ce + 1]
        assert np.allclose(np.diff(seg), -(1.0 - floor) / (ce - cs), rtol=0, atol=1e-15)
        # trapezoid: the mean multiplier over the cool-down is (1 + floor) / 2
        assert abs((seg[:-1] + seg[1:]).mean() / 2 - (1.0 + floor) / 2) < 1e-12
        assert oracle.scheduled_lr(ce, 0.03, cs, ce, floor) == pytest.approx(0.03 * floor, rel=1e-15)


def test_flex_momentum_warmup():
    mu0, mu1, w = P["flex.momentum_start"], P["flex.momentum_end"], int(P["flex.momentum_warmup"])
    mu = np.array([oracle.scheduled_momentum(s, mu0, mu1, w) for s in range(3 * w)])
    assert mu[0] == pytest.approx(mu0, abs=1e-15)
    assert mu[w] == pytest.approx(mu1, abs=1e-15)
    assert np.all(mu[w:] == mu[w])                              # frac is clamped at 1
    assert np.allclose(np.diff(mu[: w + 1]), (mu1 - mu0) / w, rtol=0, atol=1e-15)
    assert mu[w // 2] == pytest.approx((mu0 + mu1) / 2, abs=1e-15)
    assert oracle.scheduled_momentum(7, mu0, mu1, 0) == mu1     # no warm-up


def test_schedule_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.lr_multiplier(0, 10, 10, 0.3)
    with pytest.raises(ValueError):
        oracle.scheduled_momentum(0, 0.85, 0.95, -1)


def test_schedule_mutations_are_caught():
    """Plausible mistakes in a schedule fail the properties above."""
    n, w, start = 1875, 562, 1313

    def off_by_one(s, cs, ce, fl):  # decays one step early
        return oracle.lr_multiplier(s + 1, cs, ce, fl)

    def relative_floor(s, cs, ce, fl):  # floor applied as a factor of the decayed value
        return max(oracle.lr_multiplier(s, cs, ce, 0.0), 0.0) * (1 - fl) + fl * oracle.lr_multiplier(s, cs, ce, 0.0)

    def unclamped(s, cs, ce, fl):  # keeps decaying after the end
        return fl + (1 - fl) * (ce - s) / (ce - cs) if s > cs else 1.0

    assert off_by_one(start, start, n, 0.0) != 1.0
    assert relative_floor(n + 5, int(0.2 * 1000), 1000, 0.3) != 0.3
    assert unclamped(n + 5, start, n, 0.3) != 0.3
