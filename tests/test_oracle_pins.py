"""Pins of the fp64 oracle against things other than itself (CPU only).

* closed form: an odd matrix polynomial acts on singular values only, so
  k quintic steps equal ``U f^k(S) V^T`` with ``f(s) = a s + b s^3 + c s^5``
  (SVD from LAPACK via numpy);
* textbook special case: coefficients (1.5, -0.5, 0) are classic
  Newton-Schulz, whose limit is the polar factor ``U V^T``;
* invariants: the singular-value band after 5 steps, preserved singular
  vectors, NorMuon norm preservation;
* hand-derived recurrences (momentum / Nesterov for a constant gradient),
  a hand-worked NorMuon example and the page's printed constants
  (``tests/golden``);
* a second, pure-Python implementation (``bruteforce_py``) on 8 x 16 and
  16 x 8 matrices;
* mutation checks: plausible mistakes planted in the oracle make a pin fail.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests import bruteforce_py

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = [s.strip() for s in line.split("=", 1)]
            out[k] = v
    return out


def _matrix(text):
    return np.array([[float(x) for x in row.split()] for row in text.split(";")])


def _rand_with_spectrum(rng, m, n, s):
    u, _ = np.linalg.qr(rng.standard_normal((m, len(s))))
    v, _ = np.linalg.qr(rng.standard_normal((n, len(s))))
    return (u * s) @ v.T


def _f_iter(s, coeffs, steps):
    a, b, c = coeffs
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# ---------------------------------------------------------------------------
# constants printed on the pages
# ---------------------------------------------------------------------------

def test_page_constants():
    kv = _load_kv("page_constants.txt")
    assert oracle.NS_COEFFS == (float(kv["ns_a"]), float(kv["ns_b"]), float(kv["ns_c"]))
    assert oracle.NORM_EPS == float(kv["norm_eps"])
    cfg = oracle.OracleConfig()
    assert cfg.ns_steps == int(kv["ns_steps"])
    assert cfg.momentum == float(kv["momentum"])
    assert cfg.lr == float(kv["muon_lr_50b"])
    # lr_mul = sqrt(output_dim ratio): 768 -> 3072 gives 2.0
    assert math.sqrt(3072 / 768) == float(kv["c_fc_lr_mul"])
    from workloads import workload
    wl = workload("gpt2-124m")
    assert wl.lr == float(kv["normuon_lr"])
    assert {m.lr_mul for m in wl.matrices if "c_fc" in m.name} == {float(kv["c_fc_lr_mul"])}
    # f(1) = a + b + c
    assert abs(sum(oracle.NS_COEFFS) - 0.701) < 1e-12


# ---------------------------------------------------------------------------
# Newton-Schulz: closed form, textbook limit, band
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("m,n", [(64, 256), (32, 32), (48, 16), (5, 9)])
@pytest.mark.parametrize("form", ["page", "poly"])
def test_ns_matches_svd_closed_form(m, n, form):
    rng = np.random.default_rng(m * 1000 + n)
    g = rng.standard_normal((m, n))
    x0 = g / (np.linalg.norm(g) + oracle.NORM_EPS)
    out = oracle.zeropower_via_newtonschulz5(g, steps=5, form=form)
    u, s, vt = np.linalg.svd(x0, full_matrices=False)
    expect = (u * _f_iter(s, oracle.NS_COEFFS, 5)) @ vt
    assert out.shape == g.shape
    assert _rel(out, expect) < 1e-12


def test_ns_per_iteration_coefficients_closed_form():
    rng = np.random.default_rng(7)
    table = [(3.4445, -4.7750, 2.0315), (2.0, -1.5, 0.5), (1.5, -0.5, 0.0)]
    x = rng.standard_normal((12, 20))
    x /= np.linalg.norm(x) + 1e-7
    out = oracle.newton_schulz(x, steps=3, coeffs=table)
    u, s, vt = np.linalg.svd(x, full_matrices=False)
    for a, b, c in table:
        s = a * s + b * s ** 3 + c * s ** 5
    assert _rel(out, (u * s) @ vt) < 1e-12


def _gram_pairs_fp64(x, coeffs):
    """The order of operations of the GPU path's Gram-pair form (``MUON_NS_GRAM_PAIRS``),
    restated in fp64 from two identities of the iteration X_{k+1} = P_k X_k with
    P_k = a_k I + b_k A_k + c_k A_k^2 and A_k = X_k X_k^T: A_{k+1} = P_k A_k P_k, and
    P_k commutes with A_k, so A_{k+1} = (A_k P_k) P_k and X_{k+2} = (P_{k+1} P_k) X_k.
    The first iteration and a single one left at the end run in the plain form."""
    m = x.shape[0]

    def poly(A, t):
        a, b, c = t
        return a * np.eye(m) + b * A + c * (A @ A)

    x = poly(x @ x.T, coeffs[0]) @ x
    k = 1
    while k < len(coeffs):
        A = x @ x.T
        P = poly(A, coeffs[k])
        if k + 1 < len(coeffs):
            A2 = (A @ P) @ P
            x = (poly(A2, coeffs[k + 1]) @ P) @ x
            k += 2
        else:
            x = P @ x
            k += 1
    return x


@pytest.mark.parametrize("steps", [3, 4, 5, 6])
def test_gram_pairs_equal_the_iteration(steps):
    # Exact-arithmetic identity, checked in fp64 on a spectrum from 1e-4 to 1 with the
    # pages' coefficients and with a per-iteration table.
    rng = np.random.default_rng(100 + steps)
    x = _rand_with_spectrum(rng, 24, 96, np.geomspace(1e-4, 1.0, 24))
    x /= np.linalg.norm(x)
    plain = [tuple(oracle.NS_COEFFS)] * steps
    cycle = [(3.0, -3.2, 1.2), (2.0, -1.5, 0.5), (1.875, -1.25, 0.375), (3.4445, -4.7750, 2.0315)]
    table = [cycle[k % 4] for k in range(steps)]
    for coeffs in (plain, table):
        ref = oracle.newton_schulz(x, steps=steps, coeffs=coeffs, form="poly")
        assert _rel(_gram_pairs_fp64(x, coeffs), ref) < 1e-11


def test_gram_pair_products_are_symmetric_in_exact_arithmetic():
    # T = A_k P_k and Q = P_{k+1} P_k are symmetric: P_k is a polynomial in A_k, so it commutes
    # with A_k, and A_{k+1} = T P_k is a polynomial in A_k too, so P_{k+1} commutes with P_k.
    # This is what allows a symmetric product to be stored as one triangle; a product of two
    # symmetric matrices that do not commute is not symmetric (the last check).
    rng = np.random.default_rng(11)
    x = _rand_with_spectrum(rng, 20, 64, np.geomspace(1e-3, 1.0, 20))
    x /= np.linalg.norm(x)
    a, b, c = oracle.NS_COEFFS
    m = x.shape[0]

    def poly(A):
        return a * np.eye(m) + b * A + c * (A @ A)

    A = x @ x.T
    P = poly(A)
    T = A @ P
    A2 = T @ P
    Q = poly(A2) @ P
    for M in (T, A2, Q):
        assert _rel(M, M.T) < 1e-13
    S = rng.standard_normal((m, m))
    S = S + S.T
    assert _rel(S @ P, (S @ P).T) > 1e-2


def test_gram_pairs_identity_catches_a_wrong_order():
    # The pin above is not vacuous: pairing the polynomials in the other order
    # (P_k P_{k+1} built from A_k alone) differs from the iteration.
    rng = np.random.default_rng(5)
    x = _rand_with_spectrum(rng, 16, 48, np.geomspace(1e-3, 1.0, 16))
    x /= np.linalg.norm(x)
    a, b, c = oracle.NS_COEFFS
    m = x.shape[0]
    A = x @ x.T
    P = a * np.eye(m) + b * A + c * A @ A
    wrong = (P @ P) @ x  # uses A_k for both iterations
    ref = oracle.newton_schulz(x, steps=2, form="poly")
    assert _rel(wrong, ref) > 1e-2


@pytest.mark.parametrize("m,n", [(16, 40), (24, 24), (8, 200)])
def test_closed_form_matches_iteration(m, n):
    rng = np.random.default_rng(m + n)
    s = np.geomspace(1e-5, 1.0, m)
    x = _rand_with_spectrum(rng, m, n, s) * 0.5
    it = oracle.newton_schulz(x, steps=5)
    cf = oracle.newton_schulz_closed_form(x, steps=5)
    assert _rel(cf, it) < 1e-9
    table = [(3.0, -3.2, 1.2), (2.0, -1.5, 0.5)]
    assert _rel(oracle.newton_schulz_closed_form(x, 2, table), oracle.newton_schulz(x, 2, table)) < 1e-9


def test_classic_newton_schulz_converges_to_polar_factor():
    rng = np.random.default_rng(11)
    s = np.linspace(0.05, 1.0, 24)
    x = _rand_with_spectrum(rng, 24, 40, s)
    out = oracle.newton_schulz(x, steps=40, coeffs=(1.5, -0.5, 0.0))
    u, _, vt = np.linalg.svd(x, full_matrices=False)
    assert _rel(out, u @ vt) < 1e-10


def test_singular_value_band_after_five_steps():
    # The band itself, computed by scalar iteration on a fine grid.
    grid = np.geomspace(2e-3, 1.0, 20001)
    f5 = _f_iter(grid, oracle.NS_COEFFS, 5)
    assert f5.min() > 0.68 and f5.max() < 1.21
    # The oracle's matrix output has its singular values in that band and keeps
    # the input's singular vectors.
    rng = np.random.default_rng(3)
    s = np.geomspace(2e-3, 1.0, 32)
    x = _rand_with_spectrum(rng, 32, 96, s)
    out = oracle.newton_schulz(x, steps=5)
    sv = np.linalg.svd(out, compute_uv=False)
    assert sv.min() > 0.68 and sv.max() < 1.21
    u, _, vt = np.linalg.svd(x, full_matrices=False)
    core = u.T @ out @ vt.T
    off = core - np.diag(np.diag(core))
    assert np.abs(off).max() < 1e-12


def test_normalisation_uses_eps():
    u = np.zeros((3, 4))
    u[0, 0] = 1e-7  # ||u|| = 1e-7 -> X = u / (2e-7) has norm exactly 0.5
    x = oracle.frobenius_normalise(u)
    assert abs(np.linalg.norm(x) - 0.5) < 1e-15


def test_transpose_rule_short_side():
    x, t = oracle.orient_wide(np.zeros((7, 3)))
    assert t and x.shape == (3, 7)
    x, t = oracle.orient_wide(np.zeros((3, 7)))
    assert not t and x.shape == (3, 7)
    x, t = oracle.orient_wide(np.zeros((4, 4)))
    assert not t


# ---------------------------------------------------------------------------
# Momentum and Nesterov by hand
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("k", [1, 2, 7])
def test_momentum_recurrence_lerp_form(k):
    mu = 0.95
    g = np.array([[1.0, -2.0], [0.5, 3.0]])
    buf = np.zeros_like(g)
    for _ in range(k):
        buf = oracle.momentum_update(buf, g, mu, lerp_form=True)
    assert np.allclose(buf, (1 - mu ** k) * g, rtol=0, atol=1e-15)
    u = oracle.nesterov_direction(g, buf, mu, lerp_form=True)
    assert np.allclose(u, (1 - mu) * g + mu * (1 - mu ** k) * g, rtol=0, atol=1e-15)
    assert np.allclose(oracle.nesterov_direction(g, buf, mu, True, nesterov=False), buf)


@pytest.mark.parametrize("k", [1, 3])
def test_momentum_recurrence_mul_add_form(k):
    mu = 0.95
    g = np.array([[1.0, -2.0, 4.0]])
    buf = np.zeros_like(g)
    for _ in range(k):
        buf = oracle.momentum_update(buf, g, mu, lerp_form=False)
    assert np.allclose(buf, g * (1 - mu ** k) / (1 - mu), rtol=1e-14, atol=0)
    u = oracle.nesterov_direction(g, buf, mu, lerp_form=False)
    assert np.allclose(u, g + mu * buf, rtol=1e-15)


def test_momentum_forms_give_same_orthogonalised_direction():
    # lerp and mul/add differ by the factor (1 - mu) on buf and u; the
    # normalisation removes it, so the Newton-Schulz outputs agree.
    rng = np.random.default_rng(5)
    gs = [rng.standard_normal((6, 10)) for _ in range(4)]
    b1 = np.zeros((6, 10))
    b2 = np.zeros((6, 10))
    for g in gs:
        b1 = oracle.momentum_update(b1, g, 0.95, True)
        b2 = oracle.momentum_update(b2, g, 0.95, False)
    u1 = oracle.nesterov_direction(gs[-1], b1, 0.95, True)
    u2 = oracle.nesterov_direction(gs[-1], b2, 0.95, False)
    assert _rel(u1, 0.05 * u2) < 1e-14
    o1 = oracle.zeropower_via_newtonschulz5(u1)
    o2 = oracle.zeropower_via_newtonschulz5(u2)
    assert _rel(o1, o2) < 1e-6


# ---------------------------------------------------------------------------
# NorMuon
# ---------------------------------------------------------------------------

def test_normuon_hand_example():
    kv = _load_kv("normuon_hand_2x4.txt")
    o = _matrix(kv["O"])
    out, v = oracle.normuon_scale(o, np.zeros(2), float(kv["beta2"]))
    assert np.allclose(v, [float(x) for x in kv["v"].split()], rtol=0, atol=1e-15)
    expect = _matrix(kv["O_prime_over_sqrt_5_8"]) * math.sqrt(5 / 8)
    assert np.allclose(out, expect, rtol=0, atol=1e-14)


def test_normuon_orthogonal_square_is_identity_map():
    rng = np.random.default_rng(9)
    q, _ = np.linalg.qr(rng.standard_normal((16, 16)))
    out, v = oracle.normuon_scale(q, np.zeros(16), 0.95)
    assert np.allclose(v, 0.05 / 16, rtol=1e-13)
    assert _rel(out, q) < 1e-14


def test_normuon_constant_update_second_moment_and_norm():
    rng = np.random.default_rng(10)
    o = rng.standard_normal((8, 24))
    v = np.zeros(8)
    beta2 = 0.95
    for k in range(1, 6):
        out, v = oracle.normuon_scale(o, v, beta2)
        r = np.mean(o * o, axis=1)
        assert np.allclose(v, (1 - beta2 ** k) * r, rtol=1e-13)
        assert abs(np.linalg.norm(out) - np.linalg.norm(o)) < 1e-12 * np.linalg.norm(o)


def test_normuon_zero_update_gives_zero():
    out, v = oracle.normuon_scale(np.zeros((4, 8)), np.zeros(4), 0.95)
    assert np.all(out == 0) and np.all(v == 0)


def test_normuon_column_lanes_hand_example_transposed():
    # The 2 x 4 hand example, transposed: with one lane per column of the 4 x 2
    # matrix the lanes, v and the scaled update are those of the example, transposed.
    kv = _load_kv("normuon_hand_2x4.txt")
    o = _matrix(kv["O"])
    out, v = oracle.normuon_scale(o.T.copy(), np.zeros(2), float(kv["beta2"]), lanes="cols")
    assert np.allclose(v, [float(x) for x in kv["v"].split()], rtol=0, atol=1e-15)
    expect = _matrix(kv["O_prime_over_sqrt_5_8"]) * math.sqrt(5 / 8)
    assert np.allclose(out, expect.T, rtol=0, atol=1e-14)


@pytest.mark.parametrize("lanes", ["short_side", "rows", "cols"])
@pytest.mark.parametrize("rows,cols", [(12, 6), (6, 12), (8, 8)])
def test_normuon_lane_choice_per_matrix(lanes, rows, cols):
    # Whatever orientation the iteration runs in, "rows" / "cols" must give one lane per
    # row / column of the matrix as the caller stores it, and "short_side" one per row of
    # the short side: checked against normuon_scale applied to the stored orientation.
    rng = np.random.default_rng(13)
    g = rng.standard_normal((rows, cols))
    cfg = oracle.OracleConfig(lr=0.03, normuon_lanes=lanes, beta2=0.9)
    orc = oracle.MuonOracle([(rows, cols, 1, 1.0, 1.0)], cfg)
    orc.step([np.zeros((rows, cols))], [g])
    rec = orc.records[0][0]
    o_stored = rec.o.T if rec.transposed else rec.o
    axis = {"short_side": "rows" if rows <= cols else "cols", "rows": "rows", "cols": "cols"}[lanes]
    out, v = oracle.normuon_scale(o_stored, np.zeros(rows if axis == "rows" else cols), 0.9, lanes=axis)
    got = rec.o_scaled.T if rec.transposed else rec.o_scaled
    assert _rel(got, out) < 1e-14 and _rel(rec.v, v) < 1e-14


# ---------------------------------------------------------------------------
# non-finite gradients (the library's own failure handling; the pages give none)
# ---------------------------------------------------------------------------

def test_nonfinite_gradient_skips_only_its_matrix():
    rng = np.random.default_rng(14)
    shapes = [(6, 10, 1, 1.0, 1.0), (10, 6, 1, 1.0, 1.0), (4, 16, 2, 1.0, 1.0)]
    params = [rng.standard_normal((r, c)) for r, c, *_ in shapes]
    g0 = [rng.standard_normal((r, c)) for r, c, *_ in shapes]
    g1 = [x.copy() for x in g0]
    g1[0][2, 3] = np.nan
    g1[2][3, 9] = np.inf   # the second half of the contiguous bank split (rows 2-3)
    cfg = oracle.OracleConfig(lr=0.03)
    bad = oracle.MuonOracle(shapes, cfg)
    good = oracle.MuonOracle(shapes, cfg)
    bad.step(params, g0)
    good.step(params, g0)
    mom0 = [m.copy() for m in bad.momentum]
    v0 = [[v.copy() for v in vs] for vs in bad.v]
    out = bad.step(params, g1)
    ref = good.step(params, g0)
    # matrix 0 and the second block of matrix 2 are skipped, all else steps as usual
    assert np.array_equal(out[0], params[0])
    assert np.array_equal(bad.v[0][0], v0[0][0]) and bad.records[0][0].skipped
    assert _rel(out[1], ref[1]) == 0.0 and not bad.records[1][0].skipped
    assert [r.skipped for r in bad.records[2]] == [False, True]
    assert np.array_equal(out[2][2:], params[2][2:]) and np.array_equal(out[2][:2], ref[2][:2])
    # the momentum keeps its old value exactly at the non-finite elements only
    assert bad.momentum[0][2, 3] == mom0[0][2, 3]
    mask = np.ones_like(g1[0], dtype=bool)
    mask[2, 3] = False
    assert np.array_equal(bad.momentum[0][mask], good.momentum[0][mask])
    assert bad.momentum[2][3, 9] == mom0[2][3, 9]


def test_momentum_overflow_keeps_the_old_value():
    # mul/add form: mu * b + g beyond the fp32 range is not stored, and the matrix is skipped
    cfg = oracle.OracleConfig(lr=0.03, lerp_form=False)
    orc = oracle.MuonOracle([(2, 4, 1, 1.0, 1.0)], cfg)
    orc.momentum[0][...] = 3.0e38
    g = np.full((2, 4), 1.0)
    g[1, 1] = 3.0e38
    p = np.ones((2, 4))
    out = orc.step([p], [g])
    assert orc.momentum[0][1, 1] == 3.0e38 and orc.records[0][0].skipped
    assert np.array_equal(out[0], p)


# ---------------------------------------------------------------------------
# write-back, split
# ---------------------------------------------------------------------------

def test_write_back_delta_and_weight_decay():
    rng = np.random.default_rng(12)
    p = rng.standard_normal((4, 6))
    upd = rng.standard_normal((4, 6))
    new = oracle.write_back(p, upd, lr=0.03, lr_mul=2.0)
    assert np.allclose(new - p, -0.06 * upd, rtol=1e-12, atol=1e-15)
    decayed = oracle.write_back(p, np.zeros_like(p), lr=0.03, lr_mul=2.0, weight_decay=0.1, wd_mul=0.5)
    assert np.allclose(decayed, p * (1 - 0.06 * 0.05), rtol=1e-15)
    assert oracle.shape_scale(3072, 768) == 2.0 and oracle.shape_scale(768, 3072) == 1.0


def test_split_contiguous_and_columns():
    w = np.arange(16.0).reshape(2, 8)
    subs = oracle.split_matrix(w, 4, "contiguous")
    assert [s.tolist() for s in subs] == [[[0, 1], [2, 3]], [[4, 5], [6, 7]],
                                          [[8, 9], [10, 11]], [[12, 13], [14, 15]]]
    assert np.array_equal(oracle.merge_matrix(subs, 2, 8, "contiguous"), w)
    subs = oracle.split_matrix(w, 4, "columns")
    assert subs[1].tolist() == [[2, 3], [10, 11]]
    assert np.array_equal(oracle.merge_matrix(subs, 2, 8, "columns"), w)


# ---------------------------------------------------------------------------
# bf16 emulation vs a library cast
# ---------------------------------------------------------------------------

def test_fp16_round_exact_cases():
    # binary16: 11 significant bits, ties to even, max 65504, subnormal step 2^-24
    cases = [(1.0 + 2.0 ** -11, 1.0), (1.0 + 3 * 2.0 ** -12, 1.0 + 2.0 ** -10), (1.0 + 2.0 ** -10, 1.0 + 2.0 ** -10),
             (65504.0, 65504.0), (3 * 2.0 ** -25, 2.0 ** -23), (2.0 ** -25, 0.0), (-0.1, -0.0999755859375)]
    for x, want in cases:
        assert oracle.fp16_round(np.array([x]))[0] == want, x


def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(10000) * 10.0 ** rng.integers(-8, 8, 10000),
                        [1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -1 - 2 ** -8, 0.0]]).astype(np.float32)
    ours = oracle.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)
    assert oracle.bf16_round(np.array([1 + 2 ** -8]))[0] == 1.0           # tie -> even
    assert oracle.bf16_round(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6


# ---------------------------------------------------------------------------
# brute force against the pure-Python second implementation
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rows,cols,normuon", [(8, 16, True), (16, 8, True), (8, 16, False), (12, 12, True)])
def test_full_step_matches_pure_python(rows, cols, normuon):
    rng = np.random.default_rng(rows * 31 + cols)
    cfg = oracle.OracleConfig(lr=0.03, normuon=normuon, weight_decay=0.01)
    orc = oracle.MuonOracle([(rows, cols, 1, 1.5, 2.0)], cfg)
    p = rng.standard_normal((rows, cols)) * 0.02
    buf = [[0.0] * cols for _ in range(rows)]
    v = [0.0] * min(rows, cols)
    pl = p.tolist()
    for step in range(3):
        g = rng.standard_normal((rows, cols))
        (p_new,) = orc.step([p], [g])
        pl, buf, v, o = bruteforce_py.step_one_matrix(
            pl, g.tolist(), buf, v, lr=0.03, mu=0.95, beta2=0.95, coeffs=oracle.NS_COEFFS, steps=5,
            eps=1e-7, normuon=normuon, lr_mul=1.5, wd=0.01, wd_mul=2.0)
        assert _rel(np.array(buf), orc.momentum[0]) < 1e-14
        assert _rel(np.array(o), orc.records[0][0].o) < 1e-12
        if normuon:
            assert _rel(np.array(v), orc.v[0][0]) < 1e-12
        assert _rel(np.array(pl) - p, p_new - p) < 1e-11
        p = p_new


def test_bank_split_step_matches_per_matrix_steps():
    # A bank of 4 contiguous blocks steps exactly like 4 separate matrices.
    rng = np.random.default_rng(21)
    cfg = oracle.OracleConfig(lr=0.03)
    bank = oracle.MuonOracle([(8, 32, 4, 1.0, 1.0)], cfg)
    single = oracle.MuonOracle([(8, 8, 1, 1.0, 1.0)] * 4, cfg)
    p = rng.standard_normal((8, 32))
    g = rng.standard_normal((8, 32))
    (pb,) = bank.step([p], [g])
    ps = single.step(oracle.split_matrix(p, 4), oracle.split_matrix(g, 4))
    assert np.array_equal(pb, oracle.merge_matrix(ps, 8, 32))


def test_zero_gradient_leaves_params():
    cfg = oracle.OracleConfig(lr=0.03)
    orc = oracle.MuonOracle([(6, 10, 1, 1.0, 1.0)], cfg)
    p = np.ones((6, 10))
    (pn,) = orc.step([p], [np.zeros((6, 10))])
    assert np.array_equal(pn, p)


def test_reset_zeroes_state():
    cfg = oracle.OracleConfig(lr=0.03)
    orc = oracle.MuonOracle([(6, 10, 2, 1.0, 1.0)], cfg)
    rng = np.random.default_rng(0)
    orc.step([rng.standard_normal((6, 10))], [rng.standard_normal((6, 10))])
    assert np.abs(orc.momentum[0]).sum() > 0 and np.abs(orc.v[0][1]).sum() > 0
    orc.reset()
    assert np.abs(orc.momentum[0]).sum() == 0 and all(np.abs(v).sum() == 0 for v in orc.v[0])


# ---------------------------------------------------------------------------
# mutation checks: a planted mistake in the oracle must fail a pin
# ---------------------------------------------------------------------------

def _closed_form_error(ns, m=10, n=14):
    rng = np.random.default_rng(99)
    g = rng.standard_normal((m, n))
    x0 = g / (np.linalg.norm(g) + 1e-7)
    u, s, vt = np.linalg.svd(x0, full_matrices=False)
    return _rel(ns(x0), (u * _f_iter(s, oracle.NS_COEFFS, 5)) @ vt)


def test_mutations_are_caught():
    a, b, c = oracle.NS_COEFFS

    def dropped_term(x):
        for _ in range(5):
            A = x @ x.T
            B = A @ x
            x = a * x + b * B  # c * A @ B dropped
        return x

    def wrong_sign(x):
        for _ in range(5):
            A = x @ x.T
            B = A @ x
            x = a * x - b * B + c * (A @ B)
        return x

    def transposed_operand(x):
        for _ in range(5):
            A = x.T @ x  # X^T X where X X^T belongs
            B = A @ x
            x = a * x + b * B + c * (A @ B)
        return x

    def wrong_index(x):
        for _ in range(5):
            A = x @ x.T
            B = A @ x
            x = a * x + c * B + b * (A @ B)  # coefficients b and c swapped
        return x
    assert _closed_form_error(lambda x: oracle.newton_schulz(x, 5)) < 1e-12
    for bad in (dropped_term, wrong_sign, wrong_index):
        assert _closed_form_error(bad) > 1e-5
    assert _closed_form_error(transposed_operand, 12, 12) > 1e-3

    # A NorMuon lane-axis mistake (mean along the short side) fails the hand example.
    kv = _load_kv("normuon_hand_2x4.txt")
    o = _matrix(kv["O"])
    r_bad = np.mean(o * o, axis=0)
    assert r_bad.shape != (2,) or not np.allclose(0.25 * r_bad, [0.25, 1])
