"""Step-indexed learning-rate and momentum schedules (fp64 reference).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Two schedules are described on the pages:

* Momentum warm-up -- "modded-nanogpt 的 FlexAttention 记录解析", section
  "优化器分工" (optimizer split): the training loop moves Muon's momentum
  linearly from 0.85 to 0.95 with ``frac = min(step / 500, 1)``.
* Learning-rate multiplier -- the same page, hyper-parameter table
  (``num_iterations`` 1875, ``warmdown_iters`` 562, no warm-up): constant,
  then a linear warmdown that starts at step 1313 and reaches 0 at the last
  step; and the 2025-10-27 FixMuonLR write-up, change 3 (the two hidden
  schedule bugs): a linear cool-down over the last ``LR_COOLDOWN_FRAC`` (0.80)
  of the main phase, clamped so it never exceeds 1, ending at an absolute
  floor (``LR_FLOOR`` 0.30) that stays flat through the extension steps; the
  learning rate actually used is the base lr times that multiplier.

One piecewise-linear multiplier covers both readings: 1 up to and including
``cooldown_start``, then a straight line to ``floor`` at ``cooldown_end``,
then ``floor`` for every later step.  The Flex schedule is
(1313, 1875, 0.0); FixMuonLR with a main phase of N steps is
(N - 0.8 N, N, 0.3).  Step indices count optimizer steps from 0.
"""

from __future__ import annotations


def lr_multiplier(step: int, cooldown_start: int, cooldown_end: int, floor: float) -> float:
    """Multiplier of the base learning rate at ``step`` (see the module docstring)."""
    if cooldown_end <= cooldown_start:
        raise ValueError("cooldown_end must be greater than cooldown_start")
    if step <= cooldown_start:
        return 1.0
    if step >= cooldown_end:
        return float(floor)
    frac_left = (cooldown_end - step) / (cooldown_end - cooldown_start)  # 1 at the start, 0 at the end
    return float(floor) + (1.0 - float(floor)) * frac_left


def scheduled_lr(step: int, lr_base: float, cooldown_start: int, cooldown_end: int, floor: float) -> float:
    """Learning rate at ``step``: the base lr times :func:`lr_multiplier`."""
    return float(lr_base) * lr_multiplier(step, cooldown_start, cooldown_end, floor)


def scheduled_momentum(step: int, momentum_start: float, momentum_end: float, warmup: int) -> float:
    """Momentum at ``step``: linear from ``momentum_start`` to ``momentum_end`` over ``warmup`` steps.

    ``warmup == 0`` means no warm-up (``momentum_end`` from the first step).
    """
    if warmup < 0:
        raise ValueError("warmup must be >= 0")
    frac = 1.0 if warmup == 0 else min(step / warmup, 1.0)
    return float(momentum_start) + (float(momentum_end) - float(momentum_start)) * frac
