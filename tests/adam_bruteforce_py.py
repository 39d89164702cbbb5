"""A second, independent Adam written with Python floats and lists only.

It follows the library formulation (step size lr / (1 - beta1^t), denominator
sqrt(v) / sqrt(1 - beta2^t) + eps) rather than the bias-corrected moments of
the oracle, so that the two agree only if both are right.
"""

import math


def adam_steps(p0, grads, lr, beta1, beta2, eps, weight_decay=0.0):
    p = list(p0)
    m = [0.0] * len(p)
    v = [0.0] * len(p)
    for t, g in enumerate(grads, start=1):
        step_size = lr / (1.0 - beta1 ** t)
        root_bc2 = math.sqrt(1.0 - beta2 ** t)
        for i in range(len(p)):
            gi = g[i] + weight_decay * p[i]
            m[i] = m[i] + (1.0 - beta1) * (gi - m[i])
            v[i] = beta2 * v[i] + (1.0 - beta2) * gi * gi
            p[i] = p[i] - step_size * m[i] / (math.sqrt(v[i]) / root_bc2 + eps)
    return p, m, v
