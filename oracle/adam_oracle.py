"""fp64 Adam for the parameters Muon does not take (embedding, head, scalars).

TEST INFRASTRUCTURE ONLY (see the package docstring).

What the pages fix:

* "modded-nanogpt 50B-token 长时程训练实验解析：Muon vs Adam 与数据复用策略的实证对比",
  section "优化器三件套" (the optimizer trio): the token embedding and the
  output head are trained by the library Adam with ``betas=(0.9, 0.95)`` and
  ``fused=True`` -- lr 0.3 for ``wte.weight``, 0.002 for ``lm_head.weight`` --
  while Muon takes the transformer body; weight decay is 0; one WSD schedule
  (no warm-up for the Muon runs, constant, linear warmdown to 0) scales every
  optimizer's learning rate.
* "modded-nanogpt 的 FlexAttention 记录解析", section "优化器分工": the same split
  with lr 0.6 (embedding), 0.008 (head) and 0.04 for a group of scalar
  parameters, betas (0.9, 0.95).

The pages pass only ``lr`` and ``betas``, so everything else is the library
default: eps = 1e-8 added to the square root of the bias-corrected second
moment, no AMSGrad, and an optional L2 term ``g + wd * p`` (0 on the pages).
The update is Adam as published (Kingma & Ba, "Adam: A Method for
Stochastic Optimization", Algorithm 1), with the step counter t starting at 1:

    m <- beta1 m + (1 - beta1) g
    v <- beta2 v + (1 - beta2) g^2
    p <- p - lr * (m / (1 - beta1^t)) / (sqrt(v / (1 - beta2^t)) + eps)
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np

ADAM_BETAS = (0.9, 0.95)
ADAM_EPS = 1e-8


@dataclass
class AdamConfig:
    beta1: float = ADAM_BETAS[0]
    beta2: float = ADAM_BETAS[1]
    eps: float = ADAM_EPS
    weight_decay: float = 0.0


def adam_moments(m: np.ndarray, v: np.ndarray, g: np.ndarray, beta1: float, beta2: float):
    """New first and second moments (exponential moving averages of g and g^2)."""
    m_new = beta1 * m + (1.0 - beta1) * g
    v_new = beta2 * v + (1.0 - beta2) * g * g
    return m_new, v_new


def adam_param_update(p: np.ndarray, m: np.ndarray, v: np.ndarray, t: int, lr: float, beta1: float, beta2: float,
                      eps: float) -> np.ndarray:
    """Parameter after step t (t >= 1) given the already-updated moments."""
    if t < 1:
        raise ValueError("the Adam step counter starts at 1")
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    return p - lr * m_hat / (np.sqrt(v_hat) + eps)


class AdamOracle:
    """Adam state (m, v per tensor, one shared step counter) and step."""

    def __init__(self, numels: Sequence[int], cfg: AdamConfig = AdamConfig()):
        self.numels = [int(n) for n in numels]
        self.cfg = cfg
        self.reset()

    def reset(self):
        self.m = [np.zeros(n) for n in self.numels]
        self.v = [np.zeros(n) for n in self.numels]
        self.t = 0

    def step(self, params: Sequence[np.ndarray], grads: Sequence[np.ndarray], lrs: Sequence[float],
             weight_decays: Optional[Sequence[float]] = None) -> List[np.ndarray]:
        """One step for every tensor; ``lrs`` are the learning rates of this step.

        ``weight_decays`` gives each tensor its own L2 coefficient (the
        library Adam's per-group ``weight_decay``); by default every tensor
        uses ``cfg.weight_decay``.  Arrays are flattened; the new parameters
        are returned (inputs untouched).
        """
        c = self.cfg
        self.t += 1
        out = []
        for i, (p, g, lr) in enumerate(zip(params, grads, lrs)):
            wd = c.weight_decay if weight_decays is None else float(weight_decays[i])
            p = np.asarray(p, dtype=np.float64).reshape(-1)
            g = np.asarray(g, dtype=np.float64).reshape(-1)
            if wd != 0.0:
                g = g + wd * p
            self.m[i], self.v[i] = adam_moments(self.m[i], self.v[i], g, c.beta1, c.beta2)
            out.append(adam_param_update(p, self.m[i], self.v[i], self.t, lr, c.beta1, c.beta2, c.eps))
        return out
