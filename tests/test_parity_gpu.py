"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Every case compares, per step and per matrix (tolerances in parity_util):
momentum (1e-5), the Newton-Schulz output O (2e-2), the second moment
stage-wise (1e-5, oracle fed the GPU's O) and end to end (2e-2), the
parameter update stage-wise (1e-5) and end to end (2e-2).
"""

import numpy as np
import pytest
import torch

from tests.parity_util import Shape, TOL_NS, TOL_STATE, make_optimizer, rel, run_parity
from workloads import grads_for, params_for, workload
from workloads.generators import _rng, gaussian_params, lowrank_plus_noise

pytestmark = pytest.mark.gpu


def _inputs(shapes, steps, seed, grad_dtype="bf16"):
    dt = torch.bfloat16 if grad_dtype == "bf16" else torch.float32
    params = [gaussian_params(_rng(seed + 7777, i), s.rows, s.cols) for i, s in enumerate(shapes)]
    grads = [[lowrank_plus_noise(_rng(seed + k, i), s.rows, s.cols).to(dt).contiguous()
              for i, s in enumerate(shapes)] for k in range(steps)]
    return params, grads


def _wl_shapes(wl):
    return [Shape(m.rows, m.cols, m.split, m.lr_mul, m.wd_mul) for m in wl.matrices]


# ----------------------------------------------------------------- named workloads

def test_tiny_plain_muon_fp32_grads():
    wl = workload("tiny")
    errs, opt, _ = run_parity(_wl_shapes(wl), params_for(wl), [grads_for(wl, 0)], lr=wl.lr,
                              normuon=False, grad_dtype="f32")
    errs.assert_within(normuon=False)


def test_gpt2_124m_normuon_full_step():
    """The timed workload, every matrix, in the launch configuration the benchmark uses."""
    wl = workload("gpt2-124m")
    errs, _, _ = run_parity(_wl_shapes(wl), params_for(wl), [grads_for(wl, 0)], lr=wl.lr, normuon=True)
    errs.assert_within()


def test_gpt2_124m_plain_muon():
    wl = workload("gpt2-124m-plain")
    sample = [0, 1, 2, 33, 34, 35]
    errs, _, _ = run_parity(_wl_shapes(wl), params_for(wl), [grads_for(wl, 0)], lr=wl.lr, normuon=False,
                            check_parents=sample)
    errs.assert_within(normuon=False)


def test_gpt2_medium_sampled():
    wl = workload("gpt2-medium")
    sample = [0, 1, 2, 70, 71]
    grads = [g.cpu() for g in grads_for(wl, 0, device="cuda")]
    errs, _, _ = run_parity(_wl_shapes(wl), params_for(wl), [grads], lr=wl.lr, check_parents=sample)
    errs.assert_within()


def test_stress_sampled_closed_form():
    """4096-wide stress set (ill-conditioned spectrum); a square and a tall matrix checked."""
    wl = workload("stress")
    sample = [0, 20]
    grads = [g.cpu() for g in grads_for(wl, 0, device="cuda")]
    errs, _, _ = run_parity(_wl_shapes(wl), params_for(wl), [grads], lr=wl.lr, check_parents=sample,
                            ns_impl="closed_form")
    errs.assert_within()


# ----------------------------------------------------------------- shapes and edges

RAGGED = [Shape(96, 200), Shape(200, 96), Shape(130, 300), Shape(8, 40), Shape(33, 70), Shape(70, 33),
          Shape(256, 1024, split=4, lr_mul=2.0), Shape(300, 520), Shape(1, 17), Shape(5, 5),
          Shape(64, 512, split=4, split_mode="columns", wd_mul=0.5)]


@pytest.mark.parametrize("engine", ["tcgen05", "simt"])
def test_ragged_shapes_three_steps(engine):
    params, grads = _inputs(RAGGED, 3, seed=11)
    errs, _, _ = run_parity(RAGGED, params, grads, lr=0.03, gemm_engine=engine, weight_decay=0.01)
    errs.assert_within()


def test_ragged_shapes_fp32_grads_plain():
    params, grads = _inputs(RAGGED, 2, seed=12, grad_dtype="f32")
    errs, _, _ = run_parity(RAGGED, params, grads, lr=0.02, normuon=False, grad_dtype="f32")
    errs.assert_within(normuon=False)


@pytest.mark.parametrize("lerp_form,nesterov", [(False, True), (True, False), (False, False)])
def test_momentum_variants(lerp_form, nesterov):
    shapes = [Shape(128, 384), Shape(384, 128)]
    params, grads = _inputs(shapes, 3, seed=13)
    errs, _, _ = run_parity(shapes, params, grads, lr=0.03, lerp_form=lerp_form, nesterov=nesterov)
    errs.assert_within()


def test_per_iteration_coefficients_and_step_counts():
    shapes = [Shape(192, 320), Shape(256, 256)]
    params, grads = _inputs(shapes, 1, seed=14)
    table = [(3.4445, -4.7750, 2.0315), (3.0, -3.2, 1.2), (2.0, -1.5, 0.5)]
    errs, _, _ = run_parity(shapes, params, grads, ns_steps=3, ns_coeffs=table)
    errs.assert_within()
    errs, _, _ = run_parity(shapes, params, grads, ns_steps=1)
    errs.assert_within()
    # a coefficient table whose middle iteration has no linear term (a = 0)
    table0 = [(3.4445, -4.7750, 2.0315), (0.0, 1.2, -0.4), (2.0, -1.5, 0.5)]
    errs, _, _ = run_parity(shapes, params, grads, ns_steps=3, ns_coeffs=table0)
    errs.assert_within()


def test_lr_schedule_through_device_scalars():
    shapes = [Shape(128, 512), Shape(512, 128)]
    params, grads = _inputs(shapes, 3, seed=15)
    errs, _, _ = run_parity(shapes, params, grads, lr=0.03, lr_schedule=[0.03, 0.01, 0.002])
    errs.assert_within()


SCHED = dict(lr_base=0.03, cooldown_start=1, cooldown_end=4, lr_floor=0.3,
             momentum_start=0.85, momentum_end=0.95, momentum_warmup=3)


def test_device_schedule_cooldown_and_momentum_warmup():
    """Six steps cross the whole cool-down and the momentum warm-up on the device."""
    shapes = [Shape(128, 384), Shape(256, 256), Shape(384, 128, split=2)]
    params, grads = _inputs(shapes, 6, seed=21)
    errs, opt, _ = run_parity(shapes, params, grads, lr=0.5, momentum=0.5, device_schedule=SCHED)
    errs.assert_within()
    assert opt.schedule_step() == 6
    # resuming mid-schedule: steps 2..4 only
    params, grads = _inputs(shapes, 3, seed=22)
    errs, opt, _ = run_parity(shapes, params, grads, device_schedule=dict(SCHED, start_step=2))
    errs.assert_within()
    assert opt.schedule_step() == 5


def test_device_schedule_counter_reset_and_removal():
    shapes = [Shape(64, 192)]
    params, grads = _inputs(shapes, 1, seed=23)
    opt = make_optimizer(shapes, lr=0.03)
    base = opt.launch_count()
    opt.set_schedule(**SCHED, start_step=7)
    assert opt.launch_count() == base + 1
    assert opt.schedule_step() == 7
    p = [params[0].cuda()]
    opt.step(p, [grads[0][0].cuda()])
    assert opt.schedule_step() == 8
    opt.reset()
    assert opt.schedule_step() == 0
    opt.clear_schedule(start_step=3)
    assert opt.launch_count() == base
    opt.step(p, [grads[0][0].cuda()])
    assert opt.schedule_step() == 3  # no schedule kernel, counter untouched
    from optimizer_nesterov_momentum_gb300 import MuonError
    with pytest.raises(MuonError):
        opt.set_schedule(0.03, cooldown_start=5, cooldown_end=5)
    with pytest.raises(MuonError):
        opt.set_schedule(0.03, cooldown_start=1, cooldown_end=4, momentum_warmup=-1)


def test_device_schedule_followed_by_graph_replays():
    """A graph captured once follows the schedule on every replay, bitwise like eager steps."""
    shapes = [Shape(128, 384), Shape(384, 128), Shape(128, 512, split=4)]
    params, grads = _inputs(shapes, 5, seed=24)
    eager = make_optimizer(shapes, lr=0.5)
    graphed = make_optimizer(shapes, lr=0.5)
    eager.set_schedule(**SCHED)
    graphed.set_schedule(**SCHED)
    pe = [p.cuda() for p in params]
    pg = [p.cuda() for p in params]
    gbuf = [g.cuda() for g in grads[0]]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        graphed.step(pg, gbuf)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        graphed.step(pg, gbuf)
    graphed.reset()
    for p, p0 in zip(pg, params):
        p.copy_(p0.cuda())
    for k in range(5):
        for dst, src in zip(gbuf, grads[k]):
            dst.copy_(src.cuda())
        graph.replay()
        eager.step(pe, gbuf)
    torch.cuda.synchronize()
    assert graphed.schedule_step() == 5 and eager.schedule_step() == 5
    for a, b in zip(pe, pg):
        assert torch.equal(a, b)
    # and the eager run itself follows the oracle schedule
    params2 = [p.clone() for p in params]
    errs, _, _ = run_parity(shapes, params2, grads, device_schedule=SCHED)
    errs.assert_within()


@pytest.mark.parametrize("gscale", [1e-12, 1e-9, 1e4])
def test_extreme_gradient_scales(gscale):
    """X0 = u / (||u|| + 1e-7) is far from unit norm when ||u|| is tiny; the fp16
    iterate is stored divided by ||X0|| so such inputs keep their precision."""
    shapes = [Shape(256, 512), Shape(512, 256), Shape(192, 192)]
    params, grads = _inputs(shapes, 2, seed=25, grad_dtype="f32")
    grads = [[(g * gscale).contiguous() for g in gs] for gs in grads]
    # zero parameters: an update of ~1e-7 would otherwise be measured against the
    # fp32 rounding of parameters of size ~0.02, not against the kernels
    params = [torch.zeros_like(p) for p in params]
    errs, _, _ = run_parity(shapes, params, grads, grad_dtype="f32")
    errs.assert_within()


def test_sm_pair_update_shapes_two_steps():
    """Every group tiles into 256 x 256 blocks, so the updates after the first run on
    SM pairs (tcgen05.mma.cta_group::2); tall and wide matrices, NorMuon row sums."""
    shapes = [Shape(256, 512), Shape(512, 256), Shape(256, 256), Shape(512, 1024, lr_mul=2.0)]
    params, grads = _inputs(shapes, 2, seed=31)
    errs, _, _ = run_parity(shapes, params, grads)
    errs.assert_within()


def test_sm_pair_step_counts_and_coefficient_tables():
    """The pair kernels with one Newton-Schulz step (the first update is also the last,
    so it writes the NorMuon row sums) and with per-iteration coefficients, including
    an iteration without a linear term (a = 0 on the folded diagonal).  The 192 x 320
    matrix runs on the one-SM kernels in a chunk of its own."""
    shapes = [Shape(256, 512), Shape(256, 256), Shape(192, 320)]
    params, grads = _inputs(shapes, 1, seed=41)
    for steps, table in [(1, None), (3, [(3.4445, -4.7750, 2.0315), (3.0, -3.2, 1.2), (2.0, -1.5, 0.5)]),
                         (3, [(3.4445, -4.7750, 2.0315), (0.0, 1.2, -0.4), (2.0, -1.5, 0.5)])]:
        errs, _, _ = run_parity(shapes, params, grads, ns_steps=steps, ns_coeffs=table)
        errs.assert_within()


@pytest.mark.parametrize("gscale", [1e-12, 1e4])
def test_sm_pair_update_extreme_scales(gscale):
    shapes = [Shape(256, 512), Shape(512, 256)]
    params, grads = _inputs(shapes, 2, seed=37, grad_dtype="f32")
    grads = [[(g * gscale).contiguous() for g in gs] for gs in grads]
    params = [torch.zeros_like(p) for p in params]
    errs, _, _ = run_parity(shapes, params, grads, grad_dtype="f32")
    errs.assert_within()


def test_zero_gradient_keeps_params_and_is_finite():
    shapes = [Shape(64, 192), Shape(192, 64)]
    opt = make_optimizer(shapes, lr=0.03)
    params = [torch.randn(s.rows, s.cols, device="cuda") for s in shapes]
    before = [p.clone() for p in params]
    grads = [torch.zeros(s.rows, s.cols, device="cuda", dtype=torch.bfloat16) for s in shapes]
    opt.step(params, grads)
    opt.sync_status()
    for a, b in zip(params, before):
        assert torch.equal(a, b)


# ----------------------------------------------------------------- state handling

def test_reset_restores_fresh_state():
    shapes = [Shape(128, 256), Shape(256, 128, split=2)]
    params, grads = _inputs(shapes, 2, seed=16)
    errs, opt, _ = run_parity(shapes, params, grads[:1], lr=0.03)
    opt.reset()
    # after reset, a step from the same params must match a fresh optimizer's step
    fresh = make_optimizer(shapes, lr=0.03)
    pa = [p.cuda() for p in params]
    pb = [p.cuda() for p in params]
    g = [x.cuda() for x in grads[1]]
    opt.step(pa, g)
    fresh.step(pb, g)
    torch.cuda.synchronize()
    for a, b in zip(pa, pb):
        assert torch.equal(a, b)


def test_runs_are_bitwise_reproducible():
    shapes = [Shape(256, 768), Shape(768, 256), Shape(128, 512, split=4)]
    params, grads = _inputs(shapes, 1, seed=17)
    outs = []
    for _ in range(2):
        opt = make_optimizer(shapes, lr=0.03)
        p = [x.cuda() for x in params]
        opt.step(p, [x.cuda() for x in grads[0]])
        torch.cuda.synchronize()
        outs.append([x.cpu() for x in p])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_gpt2_124m_steps_are_bitwise_reproducible():
    """The timed workload twice from the same state: every parameter and every Newton-Schulz
    output bit for bit equal.  A race between a kernel's roles that only shows under the full
    workload's traffic makes two runs differ in a few matrices long before it moves an error
    bound."""
    from optimizer_nesterov_momentum_gb300 import MUON_STATE_ORTHO

    wl = workload("gpt2-124m")
    shapes = _wl_shapes(wl)
    outs = []
    for _ in range(2):
        opt = make_optimizer(shapes, lr=wl.lr)
        params = [p.cuda() for p in params_for(wl)]
        for k in range(6):
            opt.step(params, grads_for(wl, k, device="cuda"))
        opt.sync_status()
        torch.cuda.synchronize()
        outs.append(([p.clone() for p in params],
                     [opt.get_state(MUON_STATE_ORTHO, i).clone() for i in range(opt.num_matrices())]))
        opt.close()
    bad_p = [i for i, (a, b) in enumerate(zip(outs[0][0], outs[1][0])) if not torch.equal(a, b)]
    bad_o = [i for i, (a, b) in enumerate(zip(outs[0][1], outs[1][1])) if not torch.equal(a, b)]
    assert not bad_p and not bad_o, (bad_p, bad_o)


def test_launch_overlap_changes_no_bit():
    """Launches that overlap the previous kernel's tail (muon_config.launch_overlap) wait in
    the kernel for its results: every parameter equals, bit for bit, a run in plain stream
    order, eager and under graph replay, over one-SM, SM-pair and Gram-pair shapes."""
    shapes = [Shape(256, 768), Shape(768, 256), Shape(128, 512, split=4), Shape(512, 1024), Shape(320, 96)]
    params, grads = _inputs(shapes, 3, seed=29)
    outs = []
    for ov in (False, True):
        opt = make_optimizer(shapes, lr=0.03, launch_overlap=ov)
        p = [x.cuda() for x in params]
        gs = [[x.cuda() for x in g] for g in grads]
        for k in range(2):
            opt.step(p, gs[k])
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            opt.step(p, gs[2])  # warm the allocator-free path on the capture stream
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            opt.step(p, gs[2])
        g.replay()
        torch.cuda.synchronize()
        opt.sync_status()
        outs.append([x.cpu() for x in p])
        opt.close()
    bad = [i for i, (a, b) in enumerate(zip(*outs)) if not torch.equal(a, b)]
    assert not bad, bad


def test_state_roundtrip_checkpoint():
    from optimizer_nesterov_momentum_gb300 import MUON_STATE_MOMENTUM, MUON_STATE_SECOND_MOMENT

    shapes = [Shape(128, 256), Shape(64, 256, split=2)]
    params, grads = _inputs(shapes, 2, seed=18)
    _, opt, p_gpu = run_parity(shapes, params, grads[:1], lr=0.03)
    saved_m = [opt.get_state(MUON_STATE_MOMENTUM, i).clone() for i in range(len(shapes))]
    saved_v = [opt.get_state(MUON_STATE_SECOND_MOMENT, k).clone() for k in range(opt.num_matrices())]
    other = make_optimizer(shapes, lr=0.03)
    for i, t in enumerate(saved_m):
        other.set_state(MUON_STATE_MOMENTUM, i, t)
    for k, t in enumerate(saved_v):
        other.set_state(MUON_STATE_SECOND_MOMENT, k, t)
    pa = [p.clone() for p in p_gpu]
    pb = [p.clone() for p in p_gpu]
    g = [x.cuda() for x in grads[1]]
    opt.step(pa, g)
    other.step(pb, g)
    torch.cuda.synchronize()
    for a, b in zip(pa, pb):
        assert torch.equal(a, b)


def test_bad_pointer_alignment_is_rejected():
    from optimizer_nesterov_momentum_gb300 import MuonError

    shapes = [Shape(64, 64)]
    opt = make_optimizer(shapes)
    buf = torch.zeros(64 * 64 + 4, device="cuda")
    p = buf[1:1 + 64 * 64].view(64, 64)  # 4-byte offset
    g = torch.zeros(64, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(MuonError) as ei:
        opt.step([p], [g])
    assert ei.value.code == -2


def test_graph_capture_replay_matches_eager():
    shapes = [Shape(128, 384), Shape(384, 128), Shape(128, 512, split=4)]
    params, grads = _inputs(shapes, 3, seed=19)
    eager = make_optimizer(shapes, lr=0.03)
    graphed = make_optimizer(shapes, lr=0.03)
    pe = [p.cuda() for p in params]
    pg = [p.cuda() for p in params]
    gbuf = [g.cuda() for g in grads[0]]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        graphed.step(pg, gbuf)  # warm-up (also exercises the pointer cache)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        graphed.step(pg, gbuf)
    graphed.reset()
    for p, p0 in zip(pg, params):
        p.copy_(p0.cuda())
    for k in range(3):
        for dst, src in zip(gbuf, grads[k]):
            dst.copy_(src.cuda())
        graph.replay()
        eager.step(pe, gbuf)
    torch.cuda.synchronize()
    for a, b in zip(pe, pg):
        assert torch.equal(a, b)


# ----------------------------------------------------------------- caller row strides

def _guarded(rows, cols, ld, dtype, sentinel, guard_rows=8):
    """A rows x cols view with row stride ld inside a buffer of sentinels: guard_rows
    full rows before and after it and ld - cols columns after every row.  8 guard
    rows keep the view's first element 16-byte aligned for 2- and 4-byte types."""
    buf = torch.full((rows + 2 * guard_rows, ld), sentinel, dtype=dtype, device="cuda")
    view = buf[guard_rows:guard_rows + rows, :cols]
    mask = torch.ones_like(buf, dtype=torch.bool)
    mask[guard_rows:guard_rows + rows, :cols] = False
    return buf, view, mask


@pytest.mark.parametrize("pad,grad_dtype", [(8, "bf16"), (3, "bf16"), (8, "f32"), (3, "f32")])
def test_strided_caller_buffers_with_guard_bands(pad, grad_dtype):
    """Parameters and gradients as row-strided views (ld = cols + pad) inside sentinel-filled
    buffers: parity with the oracle, and not one sentinel changed.  pad = 8 keeps the 8-wide
    vector path where cols allows it; pad = 3 forces the scalar path everywhere.  A bank split
    into column blocks is included (a contiguous split needs ld == cols)."""
    shapes = [Shape(96, 200), Shape(200, 96), Shape(130, 300), Shape(64, 512, split=4, split_mode="columns"),
              Shape(256, 512)]
    lds = [s.cols + pad for s in shapes]
    params, grads = _inputs(shapes, 2, seed=51, grad_dtype=grad_dtype)
    p_sent, g_sent = 12345.0, -777.0
    gdt = torch.bfloat16 if grad_dtype == "bf16" else torch.float32
    p_bufs, p_views, p_masks = zip(*[_guarded(s.rows, s.cols, ld, torch.float32, p_sent) for s, ld in zip(shapes, lds)])
    for v, p0 in zip(p_views, params):
        v.copy_(p0.cuda())
    g_store = [_guarded(s.rows, s.cols, ld, gdt, g_sent) for s, ld in zip(shapes, lds)]

    def grads_gpu_fn(step, grads_cpu):
        out = []
        for (buf, view, mask), g in zip(g_store, grads_cpu):
            view.copy_(g.cuda())
            out.append(view)
        return out

    opt = make_optimizer(shapes, ld=lds, lr=0.03, weight_decay=0.01, grad_dtype=grad_dtype)
    errs, _, _ = run_parity(shapes, params, grads, lr=0.03, weight_decay=0.01, opt=opt, params_gpu=list(p_views),
                            grads_gpu_fn=grads_gpu_fn, grad_dtype=grad_dtype)
    errs.assert_within()
    torch.cuda.synchronize()
    for buf, mask in zip(p_bufs, p_masks):
        assert torch.all(buf[mask] == p_sent)
    for buf, _, mask in g_store:
        assert torch.all(buf[mask] == g_sent)


# ----------------------------------------------------------------- NorMuon lanes

@pytest.mark.parametrize("lanes,engine", [("rows", "tcgen05"), ("cols", "tcgen05"), ("cols", "simt")])
def test_normuon_lane_axis_flag(lanes, engine):
    """One second-moment entry per row (or per column) of every matrix as stored, instead of
    per row of the short side: tall, wide and square matrices on both tensor-core kernel families,
    and on the CUDA-core cross-check engine."""
    shapes = [Shape(128, 384), Shape(384, 128), Shape(192, 192), Shape(256, 512), Shape(512, 256),
              Shape(256, 1024, split=4)]
    params, grads = _inputs(shapes, 3, seed=61)
    errs, opt, _ = run_parity(shapes, params, grads, lr=0.03, normuon_lanes=lanes, gemm_engine=engine)
    errs.assert_within()
    for k in range(opt.num_matrices()):
        info = opt.matrix_info(k)
        assert info["lanes"] == (info["rows"] if lanes == "rows" else info["cols"])


# ----------------------------------------------------------------- non-finite gradients

def test_nonfinite_gradients_skip_only_their_matrices():
    """A NaN in one matrix's gradient and an infinity in one block of a split bank: those two
    matrices keep their parameters and second moment, their momentum keeps its old value at
    the bad elements, every other matrix steps as usual, the step reports
    MUON_ERR_NONFINITE, and the next step with finite gradients is normal again."""
    shapes = [Shape(128, 384), Shape(384, 128), Shape(256, 1024, split=4), Shape(256, 512)]
    params, grads = _inputs(shapes, 3, seed=71, grad_dtype="f32")
    grads[1][0][5, 7] = float("nan")
    # the contiguous split views the [256, 1024] bank as four [256, 256] blocks of consecutive
    # memory: parent rows 128..191 hold the third block
    grads[1][2][130, 11] = float("inf")
    grads[1][2][131, 600] = float("-inf")
    errs, _, _ = run_parity(shapes, params, grads, lr=0.03, grad_dtype="f32")
    errs.assert_within()
