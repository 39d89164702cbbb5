"""The allocation-free entry point against the regular step.

``muon_nesterov_normalize_noalloc`` serves callers that cannot allocate
device memory where they run (a framework that owns all device memory in its
own pool, code where cudaMalloc would synchronise the device or is not
allowed, a memory budget fixed at load time): it keeps its scratch in a
static device array.  Here its momentum and normalised direction are compared
with what ``muon_step`` (through a regular handle) produces for the same
gradients, over two calls in a row, within the elementwise-state tolerance
of the other parity tests.  This file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

from tests.parity_util import TOL_STATE, make_optimizer, rel, Shape
from workloads.generators import _rng, lowrank_plus_noise

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,cols", [(192, 320), (320, 192), (100, 70)])
def test_noalloc_matches_step_two_calls(rows, cols):
    from optimizer_nesterov_momentum_gb300 import MUON_STATE_DIRECTION, MUON_STATE_MOMENTUM, _abi

    opt = make_optimizer([Shape(rows, cols)], lr=0.03)
    params = [torch.zeros(rows, cols, device="cuda")]
    mom = torch.zeros(rows, cols, device="cuda")
    x0 = torch.empty(rows, cols, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for k in range(2):
        g = lowrank_plus_noise(_rng(900 + k, 0), rows, cols).to(torch.bfloat16).cuda().contiguous()
        opt.step(params, [g])
        _abi.muon_nesterov_normalize_noalloc(g.data_ptr(), _abi.MUON_GRAD_BF16, mom.data_ptr(), x0.data_ptr(),
                                             rows, cols, 0.95, True, True, stream)
        torch.cuda.synchronize()
        ref_mom = opt.get_state(MUON_STATE_MOMENTUM, 0).double().cpu().numpy()
        u = opt.get_state(MUON_STATE_DIRECTION, 0).double().cpu().numpy()
        if rows > cols:
            u = u.T
        ref_x0 = u / (np.linalg.norm(u) + 1e-7)
        assert rel(mom.double().cpu().numpy(), ref_mom) <= TOL_STATE
        assert rel(x0.double().cpu().numpy(), ref_x0) <= TOL_STATE
    opt.close()


def test_noalloc_rejects_oversized_and_bad_arguments():
    from optimizer_nesterov_momentum_gb300 import _abi

    lib = _abi.load_library()
    t = torch.zeros(8, device="cuda")
    p = t.data_ptr()
    side = 64 * 257  # 257 x 257 tiles > MUON_NOALLOC_MAX_TILES
    assert lib.muon_nesterov_normalize_noalloc(p, 0, p, p, side, side, 0.95, 1, 1, None) == _abi.MUON_ERR_SHAPE
    assert lib.muon_nesterov_normalize_noalloc(None, 0, p, p, 8, 8, 0.95, 1, 1, None) == _abi.MUON_ERR_ARG
    assert lib.muon_nesterov_normalize_noalloc(p, 5, p, p, 8, 8, 0.95, 1, 1, None) == _abi.MUON_ERR_ARG
