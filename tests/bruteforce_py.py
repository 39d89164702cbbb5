"""A second, independent implementation of one Muon/NorMuon step in pure Python.

Lists of floats and explicit loops only (no numpy), written separately from
the oracle so the two can check each other on tiny matrices.  It follows the
same page definitions: lerp momentum, lerp Nesterov, Frobenius normalisation
with eps, transpose to the short side, the quintic iteration
``A = X X^T; B = A X; X = a X + b B + c A B``, NorMuon lane scaling with norm
preservation, decoupled weight decay and the lr write-back.
"""

import math


def _matmul(p, q):
    n, k, m = len(p), len(q), len(q[0])
    out = [[0.0] * m for _ in range(n)]
    for i in range(n):
        row = p[i]
        for t in range(k):
            pit = row[t]
            if pit == 0.0:
                continue
            qt = q[t]
            o = out[i]
            for j in range(m):
                o[j] += pit * qt[j]
    return out


def _transpose(p):
    return [list(col) for col in zip(*p)]


def _axpby(alpha, p, beta, q):
    return [[alpha * x + beta * y for x, y in zip(rp, rq)] for rp, rq in zip(p, q)]


def step_one_matrix(p, g, buf, v, *, lr, mu, beta2, coeffs, steps, eps, normuon,
                    lr_mul=1.0, wd=0.0, wd_mul=1.0, v_floor=1e-10):
    """Returns (new_p, new_buf, new_v, o_wide).  All inputs are lists of lists (v: list)."""
    rows, cols = len(p), len(p[0])
    new_buf = [[b + (1.0 - mu) * (gg - b) for b, gg in zip(rb, rg)] for rb, rg in zip(buf, g)]
    u = [[gg + mu * (b - gg) for b, gg in zip(rb, rg)] for rb, rg in zip(new_buf, g)]
    fro = math.sqrt(sum(x * x for row in u for x in row))
    x = [[e / (fro + eps) for e in row] for row in u]
    transposed = rows > cols
    if transposed:
        x = _transpose(x)
    a, b, c = coeffs
    for _ in range(steps):
        A = _matmul(x, _transpose(x))
        B = _matmul(A, x)
        AB = _matmul(A, B)
        x = [[a * x0 + b * b0 + c * c0 for x0, b0, c0 in zip(rx, rb, rc)] for rx, rb, rc in zip(x, B, AB)]
    o = x
    m, n = len(o), len(o[0])
    if normuon:
        new_v = []
        scaled = []
        for i in range(m):
            r_i = sum(e * e for e in o[i]) / n
            vi = v[i] + (1.0 - beta2) * (r_i - v[i])
            new_v.append(vi)
            qi = 1.0 / math.sqrt(max(vi, v_floor))
            scaled.append([e * qi for e in o[i]])
        before = math.sqrt(sum(e * e for row in o for e in row))
        after = math.sqrt(sum(e * e for row in scaled for e in row))
        k = before / max(after, v_floor)
        upd = [[e * k for e in row] for row in scaled]
        scale = 1.0
    else:
        new_v = list(v)
        upd = o
        scale = max(1.0, rows / cols) ** 0.5
    if transposed:
        upd = _transpose(upd)
    eff = lr * lr_mul
    decay = 1.0 - eff * wd * wd_mul
    new_p = _axpby(decay, p, -eff * scale, upd)
    return new_p, new_buf, new_v, o
