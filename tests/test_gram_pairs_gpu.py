"""GPU parity of the Gram-pair order of the Newton-Schulz work (MUON_NS_GRAM_PAIRS).

For wide matrices that tile by 256 (n >= 2m) the iterations after the first run two
at a time in Gram space: one Gram matrix and one update per pair plus three m x m
products, equal to the iteration in exact arithmetic (pinned in fp64 by
tests/test_oracle_pins.py).  Here the CUDA path in that order is held to the same
tolerances against the fp64 oracle as the standard order, on the three spectra of
the synthetic workloads, for ns_steps from 3 to 6 (a pair, a pair plus a single
iteration, two pairs, two pairs plus a single one), with matrices of the standard
form (a square one, a narrow one and one that does not tile by 256) in the same
handle.
"""

import numpy as np
import pytest
import torch

from tests.parity_util import Shape, make_optimizer, rel, run_parity
from workloads.generators import _rng, gaussian_params, log_uniform_spectrum, lowrank_plus_noise, power_law_spectrum

pytestmark = pytest.mark.gpu

SHAPES = [Shape(256, 512), Shape(768, 3072), Shape(1536, 512), Shape(512, 512), Shape(512, 768), Shape(320, 640)]
GEN = {"lowrank": lowrank_plus_noise, "powerlaw": power_law_spectrum, "loguniform": log_uniform_spectrum}


def _inputs(kind, seed):
    params = [gaussian_params(_rng(seed + 7777, i), s.rows, s.cols) for i, s in enumerate(SHAPES)]
    grads = [GEN[kind](_rng(seed, i), s.rows, s.cols).to(torch.bfloat16).contiguous()
             for i, s in enumerate(SHAPES)]
    return params, grads


@pytest.mark.parametrize("ns_steps", [3, 4, 5, 6])
@pytest.mark.parametrize("kind", ["lowrank", "powerlaw", "loguniform"])
def test_gram_pairs_match_the_oracle(kind, ns_steps):
    params, grads = _inputs(kind, 9100 + ns_steps)
    opt = make_optimizer(SHAPES, ns_steps=ns_steps, ns_form="gram_pairs", lr=0.03)
    errs, opt, _ = run_parity(SHAPES, params, [grads], ns_steps=ns_steps, lr=0.03, opt=opt)
    errs.assert_within()
    work = opt.stage_work()
    # the wide groups take the Gram-pair order: a pair adds one launch of its own (Q = P'' P');
    # T = A P' and A <- T P' ride along with the update and Gram launches
    pairs = (ns_steps - 1) // 2
    assert work["product"][2] == pairs, work
    opt.close()


def test_gram_pairs_and_standard_order_agree():
    """Both orders on the same input: each within the oracle bound, and close to each other."""
    from optimizer_nesterov_momentum_gb300 import MUON_STATE_ORTHO

    params, grads = _inputs("powerlaw", 9300)
    outs = {}
    for form in ("standard", "gram_pairs"):
        opt = make_optimizer(SHAPES, ns_form=form, lr=0.03)
        errs, opt, _ = run_parity(SHAPES, [p.clone() for p in params], [grads], lr=0.03, opt=opt)
        errs.assert_within()
        outs[form] = [opt.get_state(MUON_STATE_ORTHO, k).double().cpu().numpy() for k in range(opt.num_matrices())]
        if form == "standard":
            assert opt.stage_work()["product"][2] == 0
        opt.close()
    for a, b in zip(outs["standard"], outs["gram_pairs"]):
        assert rel(b, a) < 1e-2


def test_gram_pairs_launch_plan():
    """The step's launch count and per-stage work follow the plan of both orders."""
    from optimizer_nesterov_momentum_gb300 import MatrixSpec, Muon

    specs = [MatrixSpec(768, 3072), MatrixSpec(768, 768)]
    std = Muon(specs, ns_form="standard")
    gp = Muon(specs, ns_form="gram_pairs")
    ws, wg = std.stage_work(), gp.stage_work()
    m, n = 768, 3072
    # standard: five Gram matrices, polynomials and updates per matrix
    assert ws["gram"][0] == 5 * (m * (m + 1) * n + m * (m + 1) * m)
    assert ws["update"][0] == 5 * (2 * m * m * n + 2 * m * m * m)
    # Gram pairs (five iterations: one plain, two pairs): the wide matrix forms three Gram
    # matrices and three updates; per pair A <- T P' runs in a Gram launch (symmetric, m^2(m+1)),
    # T = A P' in an update launch (its 256 x 256 blocks on or above the diagonal: 6 of 9) and
    # Q = P'' P' in a launch of its own (full tiles on the update kernel)
    assert wg["gram"][0] == 3 * m * (m + 1) * n + 5 * m * (m + 1) * m + 2 * m * m * (m + 1)
    assert wg["update"][0] == 3 * 2 * m * m * n + 5 * 2 * m * m * m + 2 * 2 * m * m * m * 6 // 9
    assert wg["product"][0] == 2 * 2 * m * m * m  # Q as a full product (update kernel)
    assert wg["poly"][0] == ws["poly"][0]
    # the square matrix keeps its Gram and update launches in every iteration, so the pairs
    # only add their Q launches
    assert gp.launch_count() == std.launch_count() + 2
    std.close()
    gp.close()


def test_q_launch_takes_standard_tiles_to_fill_its_last_wave():
    """With the GPT-2-124M shapes the launch of Q = P'' P' (216 tiles) leaves its last wave of
    SM pairs part empty while the update launch after it (1296 tiles) starts a wave for a few
    tiles: the plan moves the fewest standard-form update tiles that save that wave into Q's
    launch.  The work moves between the two stages; the sum stays the same."""
    from optimizer_nesterov_momentum_gb300 import MatrixSpec, Muon

    specs = [MatrixSpec(768, 768)] * 48 + [MatrixSpec(768, 3072)] * 24
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    m = 768
    nq, nu, n_std = 24 * 9, 48 * 9 + 24 * 36, 48 * 9

    def waves(x):
        return -(-x // pairs)

    best = 0
    for s in range(1, min(n_std, pairs - 1) + 1):
        if waves(nq + s) + waves(nu - s) < waves(nq + best) + waves(nu - best):
            best = s
    gp = Muon(specs, ns_form="gram_pairs")
    w = gp.stage_work()
    q_fl = 2 * 24 * 2 * m ** 3                # two Q launches, full m x m products
    tile_fl = 2 * m * m * m / 9               # one 256 x 256 tile of a square matrix's update
    assert w["product"][0] == pytest.approx(q_fl + 2 * best * tile_fl, rel=1e-9)
    upd_all = 48 * 5 * 2 * m ** 3 + 24 * (3 * 2 * m * m * 3072 + 2 * 2 * m ** 3 * 6 // 9)
    assert w["update"][0] + w["product"][0] == pytest.approx(upd_all + q_fl, rel=1e-9)
    assert w["product"][2] == 2
    gp.close()
