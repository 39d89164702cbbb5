"""Runs the CUDA path and the fp64 oracle on the same seeded inputs and
measures their disagreement, stage by stage.

Tolerances (relative Frobenius error):
  * fp32 elementwise state -- momentum, second moment -- and the write-back
    given the GPU's own Newton-Schulz output: 1e-5;
  * anything downstream of the bf16 Newton-Schulz iteration (its output O,
    the parameter update end to end): 2e-2.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

import oracle

TOL_STATE = 1e-5
TOL_NS = 2e-2
# Below this short side the relative Frobenius error of a bf16 iteration is
# dominated by a few singular values and can exceed TOL_NS by itself.  There
# the bound comes from the pages' own arithmetic: the orthogonalisation run in
# bf16 as the "modded-nanogpt 50B-token" write-up runs it (section "Muon from
# the source": bf16 input, bf16 normalisation, every product stored in bf16),
# measured against the fp64 iteration on the same input; the GPU must be
# within twice that error, and never held to less than TOL_NS.
TINY_SIDE = 32


def ns_tolerance(u_sub: np.ndarray, o_ref: np.ndarray, ns_steps: int, ns_coeffs) -> float:
    if min(u_sub.shape) >= TINY_SIDE:
        return TOL_NS
    pages_bf16, _ = oracle.orient_wide(oracle.zeropower_via_newtonschulz5(u_sub, ns_steps, coeffs=ns_coeffs,
                                                                           bf16=True))
    return max(TOL_NS, 2.0 * rel(pages_bf16, o_ref))


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    if nb == 0.0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


@dataclass
class Shape:
    rows: int
    cols: int
    split: int = 1
    lr_mul: float = 1.0
    wd_mul: float = 1.0
    split_mode: str = "contiguous"


@dataclass
class Errors:
    momentum: float = 0.0
    ortho: float = 0.0
    v_stage: float = 0.0
    v_e2e: float = 0.0
    delta_stage: float = 0.0
    delta_e2e: float = 0.0
    # NS-dependent errors divided by their per-matrix bound (<= 1 passes)
    ortho_ratio: float = 0.0
    v_e2e_ratio: float = 0.0
    delta_e2e_ratio: float = 0.0
    per_matrix: List[Dict] = field(default_factory=list)

    worst: Dict = field(default_factory=dict)

    def update(self, where=None, **kw):
        for k, v in kw.items():
            if not v <= getattr(self, k):  # also catches NaN
                setattr(self, k, v)
                self.worst[k] = where

    def assert_within(self, state_tol=TOL_STATE, ns_tol=TOL_NS, normuon=True, v_e2e=True):
        """``v_e2e=False``: the end-to-end second moment (which accumulates the
        Newton-Schulz rounding of every earlier step) is reported, not gated."""
        msg = repr(self)
        assert self.momentum <= state_tol, msg
        assert self.ortho_ratio <= 1.0, msg
        assert self.delta_stage <= state_tol, msg
        assert self.delta_e2e_ratio <= 1.0, msg
        if normuon:
            assert self.v_stage <= state_tol, msg
            if v_e2e:
                assert self.v_e2e_ratio <= 1.0, msg

    def __repr__(self):
        return (f"Errors(momentum={self.momentum:.2e}, ortho={self.ortho:.2e}, v_stage={self.v_stage:.2e}, "
                f"v_e2e={self.v_e2e:.2e}, delta_stage={self.delta_stage:.2e}, delta_e2e={self.delta_e2e:.2e}, "
                f"ratios(ortho={self.ortho_ratio:.2f}, v={self.v_e2e_ratio:.2f}, delta={self.delta_e2e_ratio:.2f}), "
                f"worst={self.worst})")


def make_optimizer(shapes: Sequence[Shape], ld: Optional[Sequence[int]] = None, **kw):
    from optimizer_nesterov_momentum_gb300 import MUON_SPLIT_COLUMNS, MUON_SPLIT_CONTIGUOUS, MatrixSpec, Muon

    specs = [MatrixSpec(s.rows, s.cols, s.split, s.lr_mul, s.wd_mul, 0 if ld is None else ld[i],
                        MUON_SPLIT_COLUMNS if s.split_mode == "columns" else MUON_SPLIT_CONTIGUOUS)
             for i, s in enumerate(shapes)]
    return Muon(specs, **kw)


def run_parity(shapes: Sequence[Shape], params_cpu: List[torch.Tensor], grads_steps: List[List[torch.Tensor]],
               *, lr=0.02, momentum=0.95, beta2=0.95, weight_decay=0.0, ns_steps=5, nesterov=True,
               lerp_form=True, normuon=True, grad_dtype="bf16", gemm_engine="tcgen05", ns_coeffs=None,
               ns_impl="iterate", check_parents: Optional[Sequence[int]] = None, opt=None,
               lr_schedule: Optional[Sequence[float]] = None, device_schedule: Optional[dict] = None,
               normuon_lanes: str = "short_side", params_gpu: Optional[List[torch.Tensor]] = None,
               grads_gpu_fn=None, step_fn=None) -> Errors:
    """Steps the GPU optimizer over ``grads_steps`` and compares every step.

    The oracle keeps its own momentum and second moment (they are compared
    end to end); the parameters are re-synced from the GPU before each step so
    that per-step updates are compared.  ``check_parents`` restricts the
    oracle to a sample of the parameters (each parameter is an independent
    unit of the step).  ``device_schedule`` (keyword arguments of
    ``Muon.set_schedule``) installs a device-side step schedule; the oracle
    then takes each step's lr and momentum from ``oracle.scheduled_lr`` /
    ``oracle.scheduled_momentum``.  ``params_gpu`` (device tensors, possibly
    strided views) replaces the copies of ``params_cpu``; ``grads_gpu_fn(step,
    grads_cpu)`` builds each step's device gradients (default: dense copies);
    ``step_fn(opt, params, grads)`` runs the step (default: ``opt.step``, e.g.
    a graph replay instead).  A matrix the oracle skips (non-finite
    direction) must be left exactly as it was, and the step must then report
    MUON_ERR_NONFINITE.
    """
    from optimizer_nesterov_momentum_gb300 import (MUON_ERR_NONFINITE, MUON_STATE_MOMENTUM, MUON_STATE_ORTHO,
                                                   MUON_STATE_SECOND_MOMENT, MuonError)

    if opt is None:
        opt = make_optimizer(shapes, lr=lr, momentum=momentum, beta2=beta2, weight_decay=weight_decay,
                             ns_steps=ns_steps, nesterov=nesterov, lerp_form=lerp_form, normuon=normuon,
                             grad_dtype=grad_dtype, gemm_engine=gemm_engine, ns_coeffs=ns_coeffs,
                             normuon_lanes=normuon_lanes)
    parents = list(range(len(shapes))) if check_parents is None else list(check_parents)
    cfg = oracle.OracleConfig(lr=lr, momentum=momentum, beta2=beta2, weight_decay=weight_decay,
                              ns_steps=ns_steps, nesterov=nesterov, lerp_form=lerp_form, normuon=normuon,
                              ns_coeffs=ns_coeffs, ns_impl=ns_impl, normuon_lanes=normuon_lanes)
    orc = oracle.MuonOracle([(shapes[i].rows, shapes[i].cols, shapes[i].split, shapes[i].lr_mul,
                              shapes[i].wd_mul, shapes[i].split_mode) for i in parents], cfg)
    # which GPU matrix index holds (parent, split index)
    where = {}
    for k in range(opt.num_matrices()):
        info = opt.matrix_info(k)
        where[(info["parent"], info["split_index"])] = (k, info)

    params = [p.cuda() for p in params_cpu] if params_gpu is None else params_gpu
    errs = Errors()
    if device_schedule is not None:
        opt.set_schedule(**device_schedule)
    for step, grads_cpu in enumerate(grads_steps):
        if device_schedule is not None:
            d = device_schedule
            s_idx = d.get("start_step", 0) + step
            orc.cfg.lr = oracle.scheduled_lr(s_idx, d["lr_base"], d["cooldown_start"], d["cooldown_end"],
                                             d.get("lr_floor", 0.0))
            orc.cfg.momentum = oracle.scheduled_momentum(s_idx, d.get("momentum_start", 0.95),
                                                         d.get("momentum_end", 0.95), d.get("momentum_warmup", 0))
        if lr_schedule is not None:
            opt.set_hparams(lr_schedule[step], momentum, beta2, weight_decay)
            orc.cfg.lr = lr_schedule[step]
        cur_lr = orc.cfg.lr
        grads = [g.cuda() for g in grads_cpu] if grads_gpu_fn is None else grads_gpu_fn(step, grads_cpu)
        p_old = {i: params[i].double().cpu().numpy() for i in parents}
        v_old = {}
        for i in parents:
            for q in range(shapes[i].split):
                k, _ = where[(i, q)]
                v_old[(i, q)] = opt.get_state(MUON_STATE_SECOND_MOMENT, k).double().cpu().numpy()
        if step_fn is None:
            opt.step(params, grads)
        else:
            step_fn(opt, params, grads)
        status = 0
        try:
            opt.sync_status()
        except MuonError as e:
            status = e.code
        torch.cuda.synchronize()
        expect = orc.step([p_old[i] for i in parents], [grads_cpu[i].double().numpy() for i in parents])
        any_skipped = any(rec.skipped for recs in orc.records for rec in recs)
        assert status == (MUON_ERR_NONFINITE if any_skipped else 0), (step, status)
        for j, i in enumerate(parents):
            sh = shapes[i]
            mom_gpu = opt.get_state(MUON_STATE_MOMENTUM, i).double().cpu().numpy()
            errs.update(where=(step, i), momentum=rel(mom_gpu, orc.momentum[j]))
            p_new = params[i].double().cpu().numpy()
            d_gpu = p_new - p_old[i]
            live = [rec for rec in orc.records[j] if not rec.skipped]
            tol_parent = max([ns_tolerance(rec.u, rec.o, ns_steps, ns_coeffs) for rec in live] or [TOL_NS])
            e_d = rel(d_gpu, expect[j] - p_old[i])
            errs.update(where=(step, i), delta_e2e=e_d, delta_e2e_ratio=e_d / tol_parent)
            subs_p = oracle.split_matrix(p_old[i], sh.split, sh.split_mode)
            subs_d = oracle.split_matrix(d_gpu, sh.split, sh.split_mode)
            for q in range(sh.split):
                k, info = where[(i, q)]
                rec = orc.records[j][q]
                if rec.skipped:
                    # a skipped matrix keeps its parameters and second moment bit for bit
                    assert np.array_equal(subs_d[q], np.zeros_like(subs_d[q])), (step, i, q)
                    if normuon:
                        v_gpu = opt.get_state(MUON_STATE_SECOND_MOMENT, k).double().cpu().numpy()
                        assert np.array_equal(v_gpu, v_old[(i, q)]), (step, i, q)
                    continue
                tol = ns_tolerance(rec.u, rec.o, ns_steps, ns_coeffs)
                o_gpu = opt.get_state(MUON_STATE_ORTHO, k).double().cpu().numpy()
                e_o = rel(o_gpu, rec.o)
                errs.update(where=(step, i, q), ortho=e_o, ortho_ratio=e_o / tol)
                # stage-wise: NorMuon and write-back fed with the GPU's own O
                if normuon:
                    lanes = "cols" if orc.lane_cols(info["rows"], info["cols"]) else "rows"
                    o_sc, v_exp = oracle.normuon_scale(o_gpu, v_old[(i, q)], beta2, lanes=lanes)
                    v_gpu = opt.get_state(MUON_STATE_SECOND_MOMENT, k).double().cpu().numpy()
                    e_v = rel(v_gpu, rec.v)
                    errs.update(where=(step, i, q), v_stage=rel(v_gpu, v_exp), v_e2e=e_v,
                                v_e2e_ratio=e_v / (tol if tol > TOL_NS else TOL_NS))
                    scale = 1.0
                else:
                    o_sc = o_gpu
                    scale = oracle.shape_scale(info["rows"], info["cols"])
                upd = o_sc.T if info["transposed"] else o_sc
                exp_sub = oracle.write_back(subs_p[q], upd, cur_lr, sh.lr_mul, weight_decay, sh.wd_mul, scale)
                errs.update(where=(step, i, q), delta_stage=rel(subs_d[q], exp_sub - subs_p[q]))
                errs.per_matrix.append(dict(step=step, parent=i, q=q, ortho=e_o, tol=tol))
    return errs, opt, params
