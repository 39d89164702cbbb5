"""The allocation-free entry point against the fp64 oracle.

``muon_nesterov_normalize_noalloc`` is for callers that cannot allocate
device memory where they run the step: a framework that owns all device
memory in its own pool or arena, code in which cudaMalloc would synchronise
the device or is not allowed at all, a device-memory budget fixed when the
library is loaded.  It keeps its scratch in a static device array instead.
Its momentum and normalised Nesterov direction are compared here with the
oracle's ``momentum_update``, ``nesterov_direction`` and
``frobenius_normalise`` fed the same gradient bits, over two calls in a row,
within the elementwise-state tolerance of the other parity tests; a call
must also leave the device's free memory exactly as it was.  This file is
collected last on purpose.
"""

import numpy as np
import pytest
import torch

import oracle
from tests.parity_util import TOL_STATE, rel
from workloads.generators import _rng, lowrank_plus_noise

pytestmark = pytest.mark.gpu


def _call(g, mom, x0, rows, cols, mu, lerp_form, nesterov):
    from optimizer_nesterov_momentum_gb300 import _abi

    dt = _abi.MUON_GRAD_BF16 if g.dtype == torch.bfloat16 else _abi.MUON_GRAD_F32
    _abi.muon_nesterov_normalize_noalloc(g.data_ptr(), dt, mom.data_ptr(), x0.data_ptr(), rows, cols, mu,
                                         lerp_form, nesterov, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("rows,cols,grad_dtype,lerp_form,nesterov", [
    (192, 320, "bf16", True, True),
    (320, 192, "bf16", True, True),
    (100, 70, "bf16", True, True),
    (192, 320, "f32", True, True),
    (192, 320, "bf16", False, True),
    (100, 70, "f32", True, False),
    (192, 320, "bf16", False, False),
])
def test_noalloc_matches_oracle_two_calls(rows, cols, grad_dtype, lerp_form, nesterov):
    mu = 0.95
    dt = torch.bfloat16 if grad_dtype == "bf16" else torch.float32
    mom = torch.zeros(rows, cols, device="cuda")
    x0 = torch.empty(rows, cols, device="cuda")
    buf = np.zeros((rows, cols))
    for k in range(2):
        g = lowrank_plus_noise(_rng(900 + k, 0), rows, cols).to(dt).contiguous()
        _call(g.cuda(), mom, x0, rows, cols, mu, lerp_form, nesterov)
        torch.cuda.synchronize()
        g64 = g.double().numpy()
        buf = oracle.momentum_update(buf, g64, mu, lerp_form)
        u = oracle.nesterov_direction(g64, buf, mu, lerp_form, nesterov)
        assert rel(mom.double().cpu().numpy(), buf) <= TOL_STATE
        assert rel(x0.double().cpu().numpy(), oracle.frobenius_normalise(u)) <= TOL_STATE


def test_noalloc_largest_accepted_matrix():
    """16384 x 16384 needs exactly MUON_NOALLOC_MAX_TILES tiles of 64 x 64 and is accepted;
    the normalisation over all of it is checked, the elements on sampled rows."""
    from optimizer_nesterov_momentum_gb300 import _abi

    n = 16384
    assert (n // 64) ** 2 == _abi.MUON_NOALLOC_MAX_TILES
    gen = torch.Generator().manual_seed(5)
    g = (torch.randn(n, n, generator=gen) * 1e-2).to(torch.bfloat16)
    mom = torch.zeros(n, n, device="cuda")
    x0 = torch.empty(n, n, device="cuda")
    _call(g.cuda(), mom, x0, n, n, 0.95, True, True)
    torch.cuda.synchronize()
    # the oracle's elementwise steps row block by row block; ||u|| from the blocks' sums
    sq = 0.0
    for r0 in range(0, n, 1024):
        g64 = g[r0:r0 + 1024].double().numpy()
        u = oracle.nesterov_direction(g64, oracle.momentum_update(np.zeros_like(g64), g64, 0.95), 0.95)
        sq += float(np.sum(u * u))
    scale = 1.0 / (np.sqrt(sq) + oracle.NORM_EPS)
    rows = np.random.default_rng(6).choice(n, 24, replace=False)
    for r in rows:
        g64 = g[r].double().numpy()
        b = oracle.momentum_update(np.zeros_like(g64), g64, 0.95)
        u = oracle.nesterov_direction(g64, b, 0.95)
        assert rel(mom[r].double().cpu().numpy(), b) <= TOL_STATE
        assert rel(x0[r].double().cpu().numpy(), u * scale) <= TOL_STATE


def test_noalloc_allocates_nothing():
    rows, cols = 320, 192
    g = lowrank_plus_noise(_rng(950, 0), rows, cols).to(torch.bfloat16).cuda().contiguous()
    mom = torch.zeros(rows, cols, device="cuda")
    x0 = torch.empty(rows, cols, device="cuda")
    _call(g, mom, x0, rows, cols, 0.95, True, True)  # warm: the device address lookup happens here
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        _call(g, mom, x0, rows, cols, 0.95, True, True)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0 and torch.cuda.memory_allocated() == alloc0


def test_noalloc_rejects_oversized_and_bad_arguments():
    from optimizer_nesterov_momentum_gb300 import _abi

    lib = _abi.load_library()
    t = torch.zeros(64, device="cuda")
    p, q, r = t.data_ptr(), t[16:].data_ptr(), t[32:].data_ptr()
    side = 64 * 257  # 257 x 257 tiles > MUON_NOALLOC_MAX_TILES
    assert lib.muon_nesterov_normalize_noalloc(p, 0, q, r, side, side, 0.95, 1, 1, None) == _abi.MUON_ERR_SHAPE
    assert lib.muon_nesterov_normalize_noalloc(p, 0, q, r, 16384, 16385, 0.95, 1, 1, None) == _abi.MUON_ERR_SHAPE
    assert lib.muon_nesterov_normalize_noalloc(p, 0, q, r, 1 << 40, 1 << 40, 0.95, 1, 1, None) == _abi.MUON_ERR_SHAPE
    assert lib.muon_nesterov_normalize_noalloc(None, 0, q, r, 8, 8, 0.95, 1, 1, None) == _abi.MUON_ERR_ARG
    assert lib.muon_nesterov_normalize_noalloc(p, 5, q, r, 8, 8, 0.95, 1, 1, None) == _abi.MUON_ERR_ARG
    # aliasing buffers
    assert lib.muon_nesterov_normalize_noalloc(p, 0, q, q, 8, 8, 0.95, 1, 1, None) == _abi.MUON_ERR_ARG
    assert lib.muon_nesterov_normalize_noalloc(q, 1, q, r, 8, 8, 0.95, 1, 1, None) == _abi.MUON_ERR_ARG
