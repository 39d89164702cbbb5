"""Failure handling on the GPU, without a fault: a bounded wait that gives up.

``muon_debug_inject_stall`` (test support only) makes the next step's first
polynomial launch -- a one-SM tcgen05 kernel -- wait on an mbarrier that
nothing arrives on.  After its 2 s limit the wait gives up: the kernel sets
the device status word, lets the copies it issued land, frees its TMEM and
returns, and the GPU stays usable.  What the test checks:

* the failed step reports MUON_ERR_TIMEOUT through muon_sync_status;
* neither that step nor a step enqueued after it (before the status is read)
  changes the parameters or the second moment; the failed step has folded its
  gradient into the momentum, the step after it has not;
* once the status is cleared, the next step matches the fp64 oracle started
  from that state.
"""

import numpy as np
import pytest
import torch

import oracle
from tests.parity_util import TOL_STATE, Shape, make_optimizer, ns_tolerance, rel
from workloads.generators import _rng, gaussian_params, lowrank_plus_noise

pytestmark = pytest.mark.gpu


def test_timeout_leaves_parameters_and_state_untouched_then_recovers():
    from optimizer_nesterov_momentum_gb300 import (MUON_ERR_TIMEOUT, MUON_STATE_MOMENTUM, MUON_STATE_ORTHO,
                                                   MUON_STATE_SECOND_MOMENT, MuonError)

    shapes = [Shape(128, 384), Shape(384, 128)]  # not multiples of 256: every product on one SM
    lr, mu, beta2 = 0.03, 0.95, 0.95
    params_cpu = [gaussian_params(_rng(8100, i), s.rows, s.cols) for i, s in enumerate(shapes)]
    g = [[lowrank_plus_noise(_rng(8101 + k, i), s.rows, s.cols).to(torch.bfloat16) for i, s in enumerate(shapes)]
         for k in range(4)]
    opt = make_optimizer(shapes, lr=lr, momentum=mu, beta2=beta2)
    params = [p.cuda() for p in params_cpu]
    orc = oracle.MuonOracle([(s.rows, s.cols, 1, 1.0, 1.0) for s in shapes],
                            oracle.OracleConfig(lr=lr, momentum=mu, beta2=beta2))

    # step 0: normal
    opt.step(params, [x.cuda() for x in g[0]])
    opt.sync_status()
    orc.step([p.double().numpy() for p in params_cpu], [x.double().numpy() for x in g[0]])
    p_before = [p.clone() for p in params]
    v_before = [opt.get_state(MUON_STATE_SECOND_MOMENT, k).clone() for k in range(2)]

    # step 1 stalls; step 2 is enqueued behind it before anyone reads the status
    opt.debug_inject_stall()
    opt.step(params, [x.cuda() for x in g[1]])
    opt.step(params, [x.cuda() for x in g[2]])
    with pytest.raises(MuonError) as ei:
        opt.sync_status()
    assert ei.value.code == MUON_ERR_TIMEOUT
    for p, p0 in zip(params, p_before):
        assert torch.equal(p, p0)
    for k in range(2):
        assert torch.equal(opt.get_state(MUON_STATE_SECOND_MOMENT, k), v_before[k])
    # the failed step consumed its gradient into the momentum; the one behind it did nothing
    for i in range(2):
        orc.momentum[i] = oracle.momentum_update(orc.momentum[i], g[1][i].double().numpy(), mu)
        assert rel(opt.get_state(MUON_STATE_MOMENTUM, i).double().cpu().numpy(), orc.momentum[i]) <= TOL_STATE
    opt.sync_status()  # the word was cleared by the read above

    # step 3: normal again, against the oracle continued from that state
    p_old = [p.double().cpu().numpy() for p in params]
    opt.step(params, [x.cuda() for x in g[3]])
    opt.sync_status()
    expect = orc.step(p_old, [x.double().numpy() for x in g[3]])
    for i in range(2):
        assert rel(opt.get_state(MUON_STATE_MOMENTUM, i).double().cpu().numpy(), orc.momentum[i]) <= TOL_STATE
        rec = orc.records[i][0]
        o_gpu = opt.get_state(MUON_STATE_ORTHO, i).double().cpu().numpy()
        assert rel(o_gpu, rec.o) <= ns_tolerance(rec.u, rec.o, 5, None)
        d_gpu = params[i].double().cpu().numpy() - p_old[i]
        assert rel(d_gpu, expect[i] - p_old[i]) <= ns_tolerance(rec.u, rec.o, 5, None)
        assert rel(opt.get_state(MUON_STATE_SECOND_MOMENT, i).double().cpu().numpy(), rec.v) <= 2e-2
    opt.close()


def test_stall_needs_the_tensor_core_engine():
    from optimizer_nesterov_momentum_gb300 import MuonError

    opt = make_optimizer([Shape(64, 128)], gemm_engine="simt")
    with pytest.raises(MuonError):
        opt.debug_inject_stall()
    opt.close()
