"""Plain fp64 implementation of one Muon / NorMuon optimizer step.

TEST INFRASTRUCTURE ONLY -- see the package docstring.  Written for a reader
to check against the web pages by eye: no blocking, no fusion, no reordering
beyond what the pages state.  All arithmetic is float64 unless the optional
bf16 emulation is switched on (a diagnostic that rounds the iterates to
bfloat16 the way a bf16 matmul pipeline stores them).

Sources (web pages about the modded-nanogpt speedrun, cited by title and
section):

* [50B] "modded-nanogpt 50B-token 长时程训练实验解析：Muon vs Adam 与数据复用策略的实证对比"
  (m.mzlw.cn/news/234117), section "从源码看 Muon 的分布式正交化实现"
  (Muon from the source): the ``zeropower_via_newtonschulz5`` routine --
  coefficients (a, b, c) = (3.4445, -4.7750, 2.0315), eps = 1e-7, bf16,
  Frobenius normalisation so the top singular value is <= 1, transpose so the
  iteration runs on the shorter side, ``A = X X^T; B = A X;
  X = a X + b B + c A B`` -- and the ``Muon.step`` flow: momentum buffer
  ``buf.mul_(momentum).add_(g)``, a Nesterov correction, the factor
  ``max(1, rows/cols)^0.5``, ``p.add_(g, alpha=-lr)``.  Section "优化器三件套"
  (the optimizer trio): ``Muon(..., lr=0.02, momentum=0.95)``, Nesterov on by
  default.
* [FixMuonLR] "2025-10-27_FixMuonLR" record write-up (nxmr.cn/news/120724):
  background -- NorMuon adds an Adafactor-like low-rank variance estimate
  ``second_momentum_buffer``; change 1 -- per-matrix ``lr_mul`` / ``wd_mul``,
  ``c_fc.lr_mul = 2.0`` from effective lr proportional to sqrt(output_dim);
  change 2 -- the momentum buffer lives with the parameter group and is
  updated in place with ``lerp_``, a ``reset()`` clears it, and the attention
  bank is ``view``-ed as four matrices before momentum / NorMuon; the
  second-moment estimate averages along the matrix's longer dimension and
  then scales every lane by ``rsqrt``.

Readings where the pages are garbled or silent (each also listed in the
design notes):

* The printed Newton-Schulz body lost its operators; it is read as
  ``A = X @ X.T; B = A @ X; X = a*X + b*B + c*(A @ B)``.
* "transpose if G.size(0) ? G.size(1)" lost its comparison; read as rows >
  cols, which is what "iterate on the shorter dimension" needs.
* Nesterov in the lerp form: ``u = lerp(g, buf, mu)``; in the mul/add form:
  ``u = g + mu * buf``.  Without Nesterov, ``u = buf``.
* NorMuon: lanes are the rows of the wide orientation (the shorter side), the
  mean of the squared update is taken along the longer side; square matrices
  use rows.  ``v <- lerp(v, r, 1 - beta2)`` from v = 0, no bias correction,
  lane scale ``rsqrt(max(v, 1e-10))``, then the scaled update is rescaled to
  the Frobenius norm it had before the lane scaling.  The same write-up says
  the early attention reshape makes NorMuon act per column (per output
  dimension); ``OracleConfig.normuon_lanes`` = "rows" / "cols" selects one
  lane per row / per column of each matrix as stored instead.
* Weight decay is decoupled: ``p <- p * (1 - lr*lr_mul*wd*wd_mul)`` before
  the update.
* NorMuon mode scales the update by ``lr * lr_mul``; plain-Muon mode by
  ``lr * lr_mul * max(1, rows/cols)^0.5`` (rows/cols of the matrix as the
  optimizer sees it, i.e. after the bank split).

Failure handling (not from the pages, which give none; the library's
definition, mirrored here): a momentum element whose new value is not finite
in the fp32 buffer keeps its previous value and makes the direction u
non-finite there; a matrix whose u has a non-finite element, or whose
||u||_F^2 exceeds the fp32 range, is skipped for the step (parameters and
second moment unchanged).
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np

# [50B] Muon from the source: quintic coefficients and the normalisation epsilon.
NS_COEFFS: Tuple[float, float, float] = (3.4445, -4.7750, 2.0315)
NORM_EPS: float = 1e-7
# Floor under the second moment before the rsqrt (reading; the pages give none).
V_FLOOR: float = 1e-10
# Largest finite fp32 value: the momentum buffer and the squared norm of u are fp32.
FP32_MAX: float = 3.4028234663852886e38


# ---------------------------------------------------------------------------
# bf16 emulation (diagnostic only)
# ---------------------------------------------------------------------------

def fp16_round(x: np.ndarray) -> np.ndarray:
    """Round to IEEE binary16 (round-to-nearest-even, subnormals kept) via float32, return float64."""
    f = np.asarray(np.asarray(x, dtype=np.float32), dtype=np.float16)
    return f.astype(np.float64)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round to bfloat16 (round-to-nearest-even) via float32, return float64.

    Goes through float32 first because a GPU epilogue holds its accumulator
    in fp32 before it stores bf16.
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    bits = (bits + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


def _id(x):
    return x


# ---------------------------------------------------------------------------
# S1 / S2: momentum buffer and Nesterov correction
# ---------------------------------------------------------------------------

def momentum_update(buf: np.ndarray, g: np.ndarray, mu: float, lerp_form: bool = True) -> np.ndarray:
    """New momentum buffer.

    lerp form ([FixMuonLR] change 2): ``buf.lerp_(g, 1 - mu)``, i.e.
    ``buf + (1 - mu) * (g - buf)``.  mul/add form ([50B] Muon.step):
    ``buf * mu + g``.
    """
    if lerp_form:
        return buf + (1.0 - mu) * (g - buf)
    return buf * mu + g


def nesterov_direction(g: np.ndarray, buf: np.ndarray, mu: float, lerp_form: bool = True,
                       nesterov: bool = True) -> np.ndarray:
    """Update direction handed to the orthogonalisation ([50B]: Nesterov on by default)."""
    if not nesterov:
        return buf.copy()
    if lerp_form:
        return g + mu * (buf - g)  # lerp(g, buf, mu)
    return g + mu * buf


# ---------------------------------------------------------------------------
# S3: bank split and orientation
# ---------------------------------------------------------------------------

def split_matrix(w: np.ndarray, split: int, mode: str = "contiguous") -> List[np.ndarray]:
    """The matrices the optimizer sees in one [rows, cols] parameter.

    ``contiguous`` ([FixMuonLR] change 2, attention reshape): the ``view`` of
    a contiguous [rows, cols] tensor as [split, rows, cols/split], i.e.
    ``split`` consecutive memory blocks.  ``columns``: column blocks.
    """
    rows, cols = w.shape
    if split == 1:
        return [w.copy()]
    if cols % split:
        raise ValueError("cols must be divisible by split")
    c = cols // split
    if mode == "contiguous":
        flat = np.ascontiguousarray(w).reshape(-1)
        return [flat[q * rows * c:(q + 1) * rows * c].reshape(rows, c).copy() for q in range(split)]
    if mode == "columns":
        return [w[:, q * c:(q + 1) * c].copy() for q in range(split)]
    raise ValueError(mode)


def merge_matrix(subs: Sequence[np.ndarray], rows: int, cols: int, mode: str = "contiguous") -> np.ndarray:
    """Inverse of :func:`split_matrix`."""
    split = len(subs)
    if split == 1:
        return subs[0].copy()
    if mode == "contiguous":
        return np.concatenate([s.reshape(-1) for s in subs]).reshape(rows, cols)
    return np.concatenate(list(subs), axis=1)


def orient_wide(m: np.ndarray) -> Tuple[np.ndarray, bool]:
    """Transpose when rows > cols so the iteration runs on the shorter side ([50B])."""
    if m.shape[0] > m.shape[1]:
        return m.T.copy(), True
    return m.copy(), False


# ---------------------------------------------------------------------------
# S4-S7: normalisation and the Newton-Schulz iteration
# ---------------------------------------------------------------------------

def frobenius_normalise(u: np.ndarray, eps: float = NORM_EPS, rnd=_id) -> np.ndarray:
    """``X = G / (||G||_F + eps)`` so the top singular value is at most 1 ([50B])."""
    return rnd(u / (np.sqrt(np.sum(u * u)) + eps))


def _coeff_list(coeffs, steps: int):
    if coeffs is None:
        coeffs = NS_COEFFS
    coeffs = list(coeffs)
    if len(coeffs) == 3 and not isinstance(coeffs[0], (tuple, list, np.ndarray)):
        return [tuple(float(c) for c in coeffs)] * steps
    if len(coeffs) != steps:
        raise ValueError("need one (a, b, c) triple per iteration")
    return [tuple(float(c) for c in t) for t in coeffs]


def newton_schulz(x: np.ndarray, steps: int = 5, coeffs=None, form: str = "page",
                  bf16: bool = False) -> np.ndarray:
    """``steps`` quintic iterations on a wide (rows <= cols) matrix.

    ``form="page"`` follows [50B] literally: ``A = X X^T; B = A X;
    X = a X + b B + c A B``.  ``form="poly"`` is the same map grouped as
    ``X = a X + (b A + c A A) X`` (equal in exact arithmetic; it only moves
    the bf16 rounding points when ``bf16`` is on).
    """
    rnd = bf16_round if bf16 else _id
    for a, b, c in _coeff_list(coeffs, steps):
        A = rnd(x @ x.T)
        if form == "page":
            B = rnd(A @ x)
            x = rnd(a * x + b * B + c * rnd(A @ B))
        elif form == "poly":
            P = rnd(b * A + c * (A @ A))
            x = rnd(a * x + P @ x)
        else:
            raise ValueError(form)
    return x


def zeropower_via_newtonschulz5(g: np.ndarray, steps: int = 5, eps: float = NORM_EPS, coeffs=None,
                                form: str = "page", bf16: bool = False) -> np.ndarray:
    """The [50B] orthogonalisation of one matrix, result in the input's orientation."""
    rnd = bf16_round if bf16 else _id
    x = frobenius_normalise(rnd(g), eps, rnd)
    x, transposed = orient_wide(x)
    x = newton_schulz(x, steps, coeffs, form, bf16)
    return x.T.copy() if transposed else x


def newton_schulz_closed_form(x: np.ndarray, steps: int = 5, coeffs=None) -> np.ndarray:
    """The exact value of ``steps`` quintic iterations on a wide matrix, from the spectrum.

    Every iterate is an odd polynomial of X0, so with X0 = U S V^T the result is
    ``U f(S) V^T = U diag(f(s)/s) U^T X0`` where f composes the per-iteration
    maps ``s -> a s + b s^3 + c s^5``.  U and s^2 come from the symmetric
    eigendecomposition of the Gram matrix X0 X0^T (LAPACK via numpy).  Equal
    to :func:`newton_schulz` in exact arithmetic; much cheaper for tall
    matrices (one Gram, one eigendecomposition, one product).
    """
    gram = x @ x.T
    lam, u = np.linalg.eigh(gram)
    s = np.sqrt(np.maximum(lam, 0.0))
    g = np.empty_like(s)
    small = s < 1e-150
    f = s.copy()
    for a, b, c in _coeff_list(coeffs, steps):
        f = a * f + b * f ** 3 + c * f ** 5
    g[~small] = f[~small] / s[~small]
    slope = 1.0
    for a, _b, _c in _coeff_list(coeffs, steps):
        slope *= a
    g[small] = slope  # limit of f(s)/s at s -> 0
    return (u * g[None, :]) @ (u.T @ x)


# ---------------------------------------------------------------------------
# S8 / S9: NorMuon second moment and lane scaling
# ---------------------------------------------------------------------------

def normuon_scale(o_wide: np.ndarray, v: np.ndarray, beta2: float, norm_preserve: bool = True,
                  v_floor: float = V_FLOOR, lanes: str = "rows") -> Tuple[np.ndarray, np.ndarray]:
    """One NorMuon update of the per-lane second moment and the scaled update.

    ``o_wide`` is m x n with m <= n.  With ``lanes="rows"`` the lanes are its
    rows ([FixMuonLR]: mean along the longer dimension, then a per-lane
    rsqrt); with ``lanes="cols"`` they are its columns (mean along the
    shorter dimension).  Returns ``(o_scaled, v_new)``.
    """
    axis = {"rows": 1, "cols": 0}[lanes]
    r = np.mean(o_wide * o_wide, axis=axis)               # mean square across each lane
    v_new = v + (1.0 - beta2) * (r - v)                   # v.lerp_(r, 1 - beta2)
    q = 1.0 / np.sqrt(np.maximum(v_new, v_floor))         # per-lane rsqrt
    o_scaled = o_wide * (q[:, None] if axis == 1 else q[None, :])
    if norm_preserve:
        before = np.sqrt(np.sum(o_wide * o_wide))
        after = np.sqrt(np.sum(o_scaled * o_scaled))
        o_scaled = o_scaled * (before / max(after, v_floor))
    return o_scaled, v_new


# ---------------------------------------------------------------------------
# S10: write-back
# ---------------------------------------------------------------------------

def shape_scale(rows: int, cols: int) -> float:
    """``max(1, rows/cols)^0.5`` ([50B] Muon.step)."""
    return max(1.0, rows / cols) ** 0.5


def write_back(p: np.ndarray, update: np.ndarray, lr: float, lr_mul: float = 1.0,
               weight_decay: float = 0.0, wd_mul: float = 1.0, scale: float = 1.0) -> np.ndarray:
    """``p <- p * (1 - lr*lr_mul*wd*wd_mul) - lr*lr_mul*scale*update``."""
    eff = lr * lr_mul
    return p * (1.0 - eff * weight_decay * wd_mul) - (eff * scale) * update


# ---------------------------------------------------------------------------
# The whole step
# ---------------------------------------------------------------------------

@dataclass
class OracleConfig:
    lr: float = 0.02
    momentum: float = 0.95
    beta2: float = 0.95
    weight_decay: float = 0.0
    ns_steps: int = 5
    nesterov: bool = True
    lerp_form: bool = True
    normuon: bool = True
    norm_preserve: bool = True
    ns_coeffs: Optional[Sequence] = None
    eps: float = NORM_EPS
    split_mode: str = "contiguous"
    ns_form: str = "page"
    ns_impl: str = "iterate"  # or "closed_form" (exact spectral value; large matrices)
    bf16: bool = False
    normuon_lanes: str = "short_side"  # or "rows" / "cols" of each matrix as stored


@dataclass
class SubRecord:
    """Intermediates of one optimizer matrix (after the bank split)."""

    u: np.ndarray          # Nesterov direction, original orientation
    o: Optional[np.ndarray]         # Newton-Schulz output, wide orientation (None when skipped)
    o_scaled: Optional[np.ndarray]  # after NorMuon (== o in plain mode), wide orientation
    v: Optional[np.ndarray]
    transposed: bool
    skipped: bool = False  # the direction was not finite: parameters and v left unchanged


class MuonOracle:
    """State (momentum per parameter, second moment per optimizer matrix) + step.

    ``shapes``: list of (rows, cols, split, lr_mul, wd_mul[, split_mode]); the
    split mode defaults to ``cfg.split_mode``.
    """

    def __init__(self, shapes, cfg: OracleConfig):
        self.cfg = cfg
        self.shapes = [tuple(s[:5]) for s in shapes]
        self.split_modes = [s[5] if len(s) > 5 else cfg.split_mode for s in shapes]
        self.momentum = [np.zeros((r, c)) for (r, c, *_rest) in self.shapes]
        self.v = []
        for (r, c, split, *_rest) in self.shapes:
            sr, sc = r, c // split
            nl = max(sr, sc) if self.lane_cols(sr, sc) else min(sr, sc)
            self.v.append([np.zeros(nl) for _ in range(split)])
        self.records: List[List[SubRecord]] = []

    def lane_cols(self, rows: int, cols: int) -> bool:
        """Whether the NorMuon lanes of a rows x cols matrix are the columns of its wide orientation."""
        transposed = rows > cols
        lanes = self.cfg.normuon_lanes
        if lanes not in ("short_side", "rows", "cols"):
            raise ValueError(lanes)
        return (lanes == "rows" and transposed) or (lanes == "cols" and not transposed)

    def reset(self):
        """Zero the momentum and second-moment buffers ([FixMuonLR] change 2, reset())."""
        for b in self.momentum:
            b[...] = 0.0
        for vs in self.v:
            for v in vs:
                v[...] = 0.0

    def step(self, params: Sequence[np.ndarray], grads: Sequence[np.ndarray]) -> List[np.ndarray]:
        cfg = self.cfg
        out = []
        self.records = []
        for i, (r, c, split, lr_mul, wd_mul) in enumerate(self.shapes):
            g = np.asarray(grads[i], dtype=np.float64)
            p = np.asarray(params[i], dtype=np.float64)
            new_buf = momentum_update(self.momentum[i], g, cfg.momentum, cfg.lerp_form)
            # an element whose new value is not finite in the fp32 buffer keeps its old value
            with np.errstate(invalid="ignore", over="ignore"):
                kept = np.isfinite(new_buf) & (np.abs(new_buf) <= FP32_MAX)
            self.momentum[i] = np.where(kept, new_buf, self.momentum[i])
            with np.errstate(invalid="ignore", over="ignore"):
                u = nesterov_direction(g, self.momentum[i], cfg.momentum, cfg.lerp_form, cfg.nesterov)
            u = np.where(kept, u, np.nan)
            mode = self.split_modes[i]
            subs_u = split_matrix(u, split, mode)
            subs_p = split_matrix(p, split, mode)
            new_subs, recs = [], []
            for q, (su, sp) in enumerate(zip(subs_u, subs_p)):
                with np.errstate(invalid="ignore", over="ignore"):
                    bad = not np.all(np.isfinite(su)) or not np.sum(su * su) <= FP32_MAX
                if bad:
                    # skipped for this step: parameters and second moment unchanged
                    new_subs.append(sp.copy())
                    vrec = self.v[i][q].copy() if cfg.normuon else None
                    recs.append(SubRecord(su, None, None, vrec, su.shape[0] > su.shape[1], skipped=True))
                    continue
                rnd = bf16_round if cfg.bf16 else _id
                x = frobenius_normalise(rnd(su), cfg.eps, rnd)
                x, transposed = orient_wide(x)
                if cfg.ns_impl == "closed_form" and not cfg.bf16:
                    o = newton_schulz_closed_form(x, cfg.ns_steps, cfg.ns_coeffs)
                else:
                    o = newton_schulz(x, cfg.ns_steps, cfg.ns_coeffs, cfg.ns_form, cfg.bf16)
                if cfg.normuon:
                    lanes = "cols" if self.lane_cols(*su.shape) else "rows"
                    o_scaled, self.v[i][q] = normuon_scale(o, self.v[i][q], cfg.beta2, cfg.norm_preserve,
                                                           lanes=lanes)
                    scale = 1.0
                    vrec = self.v[i][q].copy()
                else:
                    o_scaled = o
                    scale = shape_scale(*su.shape)
                    vrec = None
                upd = o_scaled.T if transposed else o_scaled
                new_subs.append(write_back(sp, upd, cfg.lr, lr_mul, cfg.weight_decay, wd_mul, scale))
                recs.append(SubRecord(su, o, o_scaled, vrec, transposed))
            out.append(merge_matrix(new_subs, r, c, mode))
            self.records.append(recs)
        return out
