"""GPU parity of the fused Adam step (embedding, head, scalars) against the fp64 oracle.

Per step and per tensor (relative Frobenius errors, fp32 state bound 1e-5):
the parameter change (the oracle is fed the GPU's parameters before the
step), and m and v end to end (the oracle keeps its own state).
"""

import numpy as np
import pytest
import torch

import oracle
from optimizer_nesterov_momentum_gb300 import MUON_ADAM_M, MUON_ADAM_V, AdamGroup, AdamTensorSpec, MuonError
from tests.parity_util import TOL_STATE, rel
from workloads import adam_grads_for, adam_params_for, adam_workload

pytestmark = pytest.mark.gpu


def _group(wl, dtype=None, **kw):
    specs = [AdamTensorSpec(t.numel, t.lr, t.weight_decay) for t in wl.tensors]
    return AdamGroup(specs, grad_dtype=dtype or wl.grad_dtype, **kw)


def _run(wl, steps, *, dtype=None, lr_scale=None, grp=None, orc=None, params=None, step0=0):
    """Steps the GPU group and the oracle together; returns the worst errors."""
    grp = grp or _group(wl, dtype)
    orc = orc or oracle.AdamOracle([t.numel for t in wl.tensors])
    if params is None:
        params = [p.reshape(-1).cuda() for p in adam_params_for(wl)]
    worst = dict(delta=0.0, m=0.0, v=0.0)
    for k in range(steps):
        grads = adam_grads_for(wl, step0 + k, dtype=dtype)
        scale = 1.0 if lr_scale is None else lr_scale[k]
        p_old = [p.double().cpu().numpy() for p in params]
        grp.step(params, [g.reshape(-1).cuda() for g in grads])
        torch.cuda.synchronize()
        expect = orc.step(p_old, [g.double().reshape(-1).numpy() for g in grads],
                          [t.lr * scale for t in wl.tensors], [t.weight_decay for t in wl.tensors])
        for i in range(len(wl.tensors)):
            d_gpu = params[i].double().cpu().numpy() - p_old[i]
            worst["delta"] = max(worst["delta"], rel(d_gpu, expect[i] - p_old[i]))
            worst["m"] = max(worst["m"], rel(grp.get_state(MUON_ADAM_M, i).double().cpu().numpy(), orc.m[i]))
            worst["v"] = max(worst["v"], rel(grp.get_state(MUON_ADAM_V, i).double().cpu().numpy(), orc.v[i]))
    return worst, grp, orc, params


def _assert_ok(worst):
    assert all(e <= TOL_STATE for e in worst.values()), worst


def test_gpt2_embedding_head_and_scalars_full_size():
    wl = adam_workload("gpt2-124m-adam")
    worst, grp, _, _ = _run(wl, 2)
    _assert_ok(worst)
    assert grp.step_count() == 2 and grp.launch_count() == 2


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ragged_tensors_and_l2_terms(dtype):
    wl = adam_workload("adam-ragged")
    worst, _, _, _ = _run(wl, 4, dtype=dtype)
    _assert_ok(worst)


def test_lr_scale_and_device_schedule():
    wl = adam_workload("adam-ragged")
    grp = _group(wl)
    grp.set_lr_scale(0.5)
    worst, grp, orc, params = _run(wl, 2, grp=grp, lr_scale=[0.5, 0.5])
    _assert_ok(worst)
    # schedule: multiplier 2.0 * m(s), cool-down from s = 0 to s = 3, floor 0.1
    grp.set_schedule(2.0, cooldown_start=0, cooldown_end=3, lr_floor=0.1)
    scales = [2.0 * oracle.lr_multiplier(s, 0, 3, 0.1) for s in range(5)]
    worst, _, _, _ = _run(wl, 5, grp=grp, orc=orc, params=params, lr_scale=scales, step0=2)
    _assert_ok(worst)
    grp.clear_schedule()
    worst, _, _, _ = _run(wl, 1, grp=grp, orc=orc, params=params, lr_scale=[0.5], step0=7)
    _assert_ok(worst)


def test_reset_and_resume_from_saved_state():
    wl = adam_workload("adam-ragged")
    worst, grp, orc, params = _run(wl, 3)
    _assert_ok(worst)
    saved = [(grp.get_state(MUON_ADAM_M, i).clone(), grp.get_state(MUON_ADAM_V, i).clone()) for i in range(len(wl.tensors))]
    t = grp.step_count()
    grp.reset()
    assert grp.step_count() == 0
    assert all(not grp.get_state(MUON_ADAM_M, i).any() for i in range(len(wl.tensors)))
    for i, (m, v) in enumerate(saved):
        grp.set_state(MUON_ADAM_M, i, m)
        grp.set_state(MUON_ADAM_V, i, v)
    grp.set_step_count(t)
    worst, _, _, _ = _run(wl, 2, grp=grp, orc=orc, params=params, step0=3)
    _assert_ok(worst)
    assert grp.step_count() == 5


def test_zero_gradient_leaves_parameters_unchanged():
    wl = adam_workload("adam-ragged")
    grp = _group(wl)
    params = [p.reshape(-1).cuda() for p in adam_params_for(wl)]
    before = [p.clone() for p in params]
    zeros = [torch.zeros(t.numel, dtype=torch.bfloat16, device="cuda") for t in wl.tensors]
    grp.step(params, zeros)
    torch.cuda.synchronize()
    for i, t in enumerate(wl.tensors):
        if t.weight_decay == 0.0:
            assert torch.equal(params[i], before[i])
        assert torch.isfinite(params[i]).all()


def test_graph_replays_match_eager_bitwise():
    wl = adam_workload("adam-ragged")
    eager, graphed = _group(wl), _group(wl)
    graphed.set_schedule(1.0, cooldown_start=1, cooldown_end=4, lr_floor=0.3)
    eager.set_schedule(1.0, cooldown_start=1, cooldown_end=4, lr_floor=0.3)
    p0 = [p.reshape(-1).cuda() for p in adam_params_for(wl)]
    pe = [p.clone() for p in p0]
    pg = [p.clone() for p in p0]
    gbuf = [g.reshape(-1).cuda() for g in adam_grads_for(wl, 0)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        graphed.step(pg, gbuf)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        graphed.step(pg, gbuf)
    graphed.reset()
    for a, b in zip(pg, p0):
        a.copy_(b)
    for k in range(5):
        for dst, src in zip(gbuf, adam_grads_for(wl, k)):
            dst.copy_(src.reshape(-1).cuda())
        graph.replay()
        eager.step(pe, gbuf)
    torch.cuda.synchronize()
    assert graphed.step_count() == eager.step_count() == 5
    for a, b in zip(pe, pg):
        assert torch.equal(a, b)


def test_bad_pointers_and_sizes_are_rejected():
    wl = adam_workload("adam-ragged")
    grp = _group(wl)
    params = [p.reshape(-1).cuda() for p in adam_params_for(wl)]
    grads = [g.reshape(-1).cuda() for g in adam_grads_for(wl, 0)]
    big = torch.zeros(wl.tensors[3].numel + 1, device="cuda")
    params_mis = list(params)
    params_mis[3] = big[1:]  # 4-byte offset: not 16-byte aligned
    with pytest.raises(MuonError) as ei:
        grp.step(params_mis, grads)
    assert ei.value.code == -2
    with pytest.raises(ValueError):
        grp.step(params[:-1], grads[:-1])
