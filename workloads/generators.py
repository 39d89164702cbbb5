"""Seeded synthetic parameters and gradients.

Every draw comes from ``numpy.random.Generator(PCG64([seed, index]))`` so a
(seed, matrix index) pair always gives the same numbers on any machine.  The
only floating-point work here is building a matrix with a prescribed
spectrum, ``U diag(s) V^T`` with orthonormal ``U, V`` taken from the QR
factorisation of a Gaussian matrix, and the final cast of gradients to the
dtype the optimizer is handed (bf16 or fp32, via ``torch``'s round-to-nearest
cast).  None of the optimizer's own arithmetic lives here.

Gradient families (one per workload):

* ``lowrank``: ``U diag(1/i) V^T`` of rank 16 plus N(0, 1e-3) noise (std).
* ``powerlaw``: full rank, singular values ``s_i = i^-0.5``.
* ``loguniform``: full rank, singular values log-uniform on [1e-4, 1].

Parameters are N(0, 0.02) in fp32.
"""

from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np
import torch

from .shapes import MatrixShape, Workload


def seed_for(wl: Workload, step: int) -> int:
    """Seed of the gradients of ``step`` (0-based) of workload ``wl``."""
    return wl.base_seed + step


def _rng(seed: int, index: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(index)]))


def _orthonormal_columns(rng: np.random.Generator, n: int, k: int, device: Optional[str]) -> torch.Tensor:
    """n x k matrix with orthonormal columns (Haar-distributed up to the sign fix)."""
    g = rng.standard_normal((n, k))
    if device is None or device == "cpu" or k <= 64:
        q, r = np.linalg.qr(g)
        q = q * np.sign(np.diag(r))[None, :]
        return torch.from_numpy(q)
    gt = torch.from_numpy(g.astype(np.float32)).to(device)
    q, r = torch.linalg.qr(gt)
    return q * torch.sign(torch.diagonal(r))[None, :]


def _spectral(rng, rows, cols, s: np.ndarray, device) -> torch.Tensor:
    k = s.shape[0]
    u = _orthonormal_columns(rng, rows, k, device)
    v = _orthonormal_columns(rng, cols, k, device)
    st = torch.from_numpy(s).to(u.device, u.dtype)
    return (u * st[None, :]) @ v.T


def lowrank_plus_noise(rng, rows: int, cols: int, rank: int = 16, noise_std: float = 1e-3,
                       device: Optional[str] = None) -> torch.Tensor:
    rank = min(rank, rows, cols)
    s = 1.0 / np.arange(1, rank + 1, dtype=np.float64)
    low = _spectral(rng, rows, cols, s, device)
    noise = torch.from_numpy(rng.standard_normal((rows, cols)) * noise_std).to(low.device, low.dtype)
    return low + noise


def power_law_spectrum(rng, rows: int, cols: int, power: float = 0.5,
                       device: Optional[str] = None) -> torch.Tensor:
    k = min(rows, cols)
    s = np.arange(1, k + 1, dtype=np.float64) ** (-power)
    return _spectral(rng, rows, cols, s, device)


def log_uniform_spectrum(rng, rows: int, cols: int, lo: float = 1e-4, hi: float = 1.0,
                         device: Optional[str] = None) -> torch.Tensor:
    k = min(rows, cols)
    s = np.exp(rng.uniform(np.log(lo), np.log(hi), size=k))
    s = np.sort(s)[::-1].copy()
    return _spectral(rng, rows, cols, s, device)


def gaussian_params(rng, rows: int, cols: int, std: float = 0.02) -> torch.Tensor:
    return torch.from_numpy((rng.standard_normal((rows, cols)) * std).astype(np.float32))


_KINDS = {
    "lowrank": lowrank_plus_noise,
    "powerlaw": power_law_spectrum,
    "loguniform": log_uniform_spectrum,
}

_DTYPES = {"bf16": torch.bfloat16, "f32": torch.float32}


def grads_for(wl: Workload, step: int = 0, device: Optional[str] = None,
              indices: Optional[Sequence[int]] = None, seed: Optional[int] = None) -> List[torch.Tensor]:
    """Gradients of one step, in the workload's gradient dtype, contiguous.

    ``device`` selects where the spectral factors are built (``None``/"cpu":
    numpy fp64; a CUDA device: torch fp32, for the large stress shapes).  The
    returned tensors live on ``device`` (CPU when ``None``).  ``indices``
    restricts the draw to a subset of matrices; each matrix's numbers depend
    only on (seed, index), never on which other matrices were drawn.
    """
    make = _KINDS[wl.grad_kind]
    dt = _DTYPES[wl.grad_dtype]
    s = seed_for(wl, step) if seed is None else seed
    idx = range(len(wl.matrices)) if indices is None else indices
    out = []
    for i in idx:
        m: MatrixShape = wl.matrices[i]
        g = make(_rng(s, i), m.rows, m.cols, device=device)
        if device is not None:
            g = g.to(device)
        out.append(g.to(dt).contiguous())
    return out


def params_for(wl: Workload, indices: Optional[Sequence[int]] = None) -> List[torch.Tensor]:
    """fp32 parameters N(0, 0.02) on the CPU (seed = base seed + 10^6)."""
    idx = range(len(wl.matrices)) if indices is None else indices
    return [gaussian_params(_rng(wl.base_seed + 1_000_000, i), wl.matrices[i].rows, wl.matrices[i].cols)
            for i in idx]
