"""GB300 (sm_103a) Muon / NorMuon optimizer step behind a C ABI.

``Muon`` owns one ``muon_handle`` of ``libmuon_gb300.so``.  PyTorch is used
for device memory and the current stream only; ``step()`` passes raw device
pointers to ``muon_step`` and every stage of the step runs in this package's
CUDA kernels.  There is no CPU path: if the library is missing or the device
is not an sm_103 GPU, construction raises.
"""

from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional, Sequence

from . import _abi
from ._abi import (  # noqa: F401  (re-exported names of the C ABI)
    MUON_ERR_NONFINITE,
    MUON_ERR_TIMEOUT,
    MUON_GEMM_SIMT,
    MUON_GEMM_TCGEN05,
    MUON_LANES_COLS,
    MUON_LANES_ROWS,
    MUON_LANES_SHORT_SIDE,
    MUON_NS_GRAM_PAIRS,
    MUON_NS_STANDARD,
    MUON_SPLIT_COLUMNS,
    MUON_SPLIT_CONTIGUOUS,
    MUON_STATE_DIRECTION,
    MUON_STATE_MOMENTUM,
    MUON_STATE_ORTHO,
    MUON_STATE_SECOND_MOMENT,
    MuonError,
    load_library,
)

from .adam import MUON_ADAM_M, MUON_ADAM_V, AdamGroup, AdamTensorSpec  # noqa: E402

__all__ = ["Muon", "MatrixSpec", "MuonError", "load_library", "AdamGroup", "AdamTensorSpec", "MUON_ADAM_M",
           "MUON_ADAM_V"]


@dataclass(frozen=True)
class MatrixSpec:
    """One parameter matrix: row-major rows x cols; ``split`` > 1 views it as a bank."""

    rows: int
    cols: int
    split: int = 1
    lr_mul: float = 1.0
    wd_mul: float = 1.0
    ld: int = 0
    split_mode: int = MUON_SPLIT_CONTIGUOUS


def _stream_ptr(stream) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


class Muon:
    """Muon / NorMuon step for a fixed list of 2-D parameter matrices.

    Hyper-parameters follow the C ABI's ``muon_config``.  ``grad_dtype`` is
    "bf16" or "f32"; ``gemm_engine`` is "tcgen05" (the product path) or
    "simt" (a slow cross-check engine for debugging); ``normuon_lanes`` is
    "short_side" (default: one second-moment entry per row of the short side),
    "rows" or "cols" (per row / per column of each matrix as stored);
    ``ns_form`` is "gram_pairs" (default: wide matrices take the Newton-Schulz
    iterations after the first two at a time in Gram space) or "standard" (every
    iteration as the write-ups order it; see MUON_NS_* in include/muon.h).
    ``launch_overlap`` (default True) lets each launch of a step after the first
    begin while the previous kernel finishes (``muon_config.launch_overlap``).
    """

    def __init__(self, specs: Sequence, *, lr: float = 0.02, momentum: float = 0.95, beta2: float = 0.95,
                 weight_decay: float = 0.0, ns_steps: int = 5, nesterov: bool = True, lerp_form: bool = True,
                 normuon: bool = True, norm_preserve: bool = True, grad_dtype: str = "bf16",
                 gemm_engine: str = "tcgen05", ns_coeffs: Optional[Sequence[Sequence[float]]] = None,
                 normuon_lanes: str = "short_side", ns_form: str = "gram_pairs", launch_overlap: bool = True,
                 device: Optional[int] = None):
        import torch

        self.specs = [s if isinstance(s, MatrixSpec) else MatrixSpec(*s) for s in specs]
        if device is None:
            device = torch.cuda.current_device()
        self.device = int(device)
        self.grad_dtype = {"bf16": torch.bfloat16, "f32": torch.float32}[grad_dtype]
        cfg = _abi.muon_config_default()
        cfg.lr, cfg.momentum, cfg.beta2, cfg.weight_decay = lr, momentum, beta2, weight_decay
        cfg.ns_steps = ns_steps
        cfg.nesterov, cfg.lerp_form, cfg.normuon = int(nesterov), int(lerp_form), int(normuon)
        cfg.norm_preserve = int(norm_preserve)
        cfg.grad_dtype = _abi.MUON_GRAD_BF16 if grad_dtype == "bf16" else _abi.MUON_GRAD_F32
        cfg.gemm_engine = {"tcgen05": MUON_GEMM_TCGEN05, "simt": MUON_GEMM_SIMT}[gemm_engine]
        cfg.normuon_lanes = {"short_side": MUON_LANES_SHORT_SIDE, "rows": MUON_LANES_ROWS,
                             "cols": MUON_LANES_COLS}[normuon_lanes]
        cfg.ns_form = {"standard": MUON_NS_STANDARD, "gram_pairs": MUON_NS_GRAM_PAIRS}[ns_form]
        cfg.launch_overlap = int(bool(launch_overlap))
        n = len(self.specs)
        self._lr_mul = (ctypes.c_float * n)(*[s.lr_mul for s in self.specs])
        self._wd_mul = (ctypes.c_float * n)(*[s.wd_mul for s in self.specs])
        cfg.lr_mul = ctypes.cast(self._lr_mul, ctypes.POINTER(ctypes.c_float))
        cfg.wd_mul = ctypes.cast(self._wd_mul, ctypes.POINTER(ctypes.c_float))
        if ns_coeffs is not None:
            flat = [float(c) for t in ns_coeffs for c in t]
            if len(flat) != 3 * ns_steps:
                raise ValueError("ns_coeffs needs one (a, b, c) triple per iteration")
            self._coeffs = (ctypes.c_float * len(flat))(*flat)
            cfg.ns_coeffs = ctypes.cast(self._coeffs, ctypes.POINTER(ctypes.c_float))
        shapes = [_abi.muon_shape(s.rows, s.cols, s.ld, s.split, s.split_mode) for s in self.specs]
        self.handle = _abi.muon_create(shapes, cfg, self.device)
        self._ptr_cache = None

    # -------------------------------------------------------------- the step
    def _pointer_arrays(self, params, grads):
        key = tuple(p.data_ptr() for p in params) + tuple(g.data_ptr() for g in grads)
        if self._ptr_cache is None or self._ptr_cache[0] != key:
            n = len(self.specs)
            if len(params) != n or len(grads) != n:
                raise ValueError(f"expected {n} params and grads")
            import torch

            for i, (s, p, g) in enumerate(zip(self.specs, params, grads)):
                ld = s.ld or s.cols
                for t, dt, what in ((p, torch.float32, "param"), (g, self.grad_dtype, "grad")):
                    if not t.is_cuda or t.dtype != dt:
                        raise ValueError(f"{what} {i}: expected a CUDA {dt} tensor")
                    if t.dim() != 2 or tuple(t.shape) != (s.rows, s.cols) or t.stride() != (ld, 1):
                        raise ValueError(f"{what} {i}: expected shape {(s.rows, s.cols)} with row stride {ld}")
            pa = (ctypes.c_void_p * n)(*[p.data_ptr() for p in params])
            ga = (ctypes.c_void_p * n)(*[g.data_ptr() for g in grads])
            self._ptr_cache = (key, pa, ga)
        return self._ptr_cache[1], self._ptr_cache[2]

    def step(self, params, grads, stream=None) -> None:
        """One optimizer step, enqueued on ``stream`` (default: torch's current stream)."""
        pa, ga = self._pointer_arrays(params, grads)
        _abi.muon_step(self.handle, pa, ga, _stream_ptr(stream))

    def reset(self, stream=None) -> None:
        _abi.muon_reset(self.handle, _stream_ptr(stream))

    def set_hparams(self, lr: float, momentum: float = 0.95, beta2: float = 0.95, weight_decay: float = 0.0,
                    stream=None) -> None:
        _abi.muon_set_hparams(self.handle, lr, momentum, beta2, weight_decay, _stream_ptr(stream))

    def set_schedule(self, lr_base: float, cooldown_start: int, cooldown_end: int, lr_floor: float = 0.0,
                     momentum_start: float = 0.95, momentum_end: float = 0.95, momentum_warmup: int = 0,
                     start_step: int = 0, stream=None) -> None:
        """Installs a device-side step schedule (see muon_set_schedule in include/muon.h).

        Every later step writes lr(s) and mu(s) on the device before it runs,
        so a CUDA graph captured afterwards follows the schedule by itself.
        """
        sc = _abi.muon_schedule(lr_base, lr_floor, cooldown_start, cooldown_end, momentum_start, momentum_end,
                                momentum_warmup)
        _abi.muon_set_schedule(self.handle, sc, start_step, _stream_ptr(stream))

    def clear_schedule(self, start_step: int = 0, stream=None) -> None:
        """Removes the step schedule; later steps use the muon_set_hparams scalars."""
        _abi.muon_set_schedule(self.handle, None, start_step, _stream_ptr(stream))

    def schedule_step(self, stream=None) -> int:
        """Schedule index the next step will use (synchronises ``stream``)."""
        return _abi.muon_get_step(self.handle, _stream_ptr(stream))

    def sync_status(self, stream=None) -> None:
        """Synchronises ``stream`` and raises MuonError if a kernel reported a failure
        (MUON_ERR_TIMEOUT, MUON_ERR_NONFINITE, ...); clears the device status word."""
        _abi.muon_sync_status(self.handle, _stream_ptr(stream))

    def debug_inject_stall(self) -> None:
        """Test support: the next step's first polynomial launch waits on an mbarrier
        that nothing arrives on until its bounded wait gives up (see muon.h)."""
        _abi.muon_debug_inject_stall(self.handle)

    # -------------------------------------------------------------- introspection
    def num_matrices(self) -> int:
        return _abi.muon_num_matrices(self.handle)

    def matrix_info(self, index: int) -> dict:
        parent, q, rows, cols, transposed, m, n, lanes = _abi.muon_matrix_info(self.handle, index)
        return dict(parent=parent, split_index=q, rows=rows, cols=cols, transposed=bool(transposed), m=m, n=n,
                    lanes=lanes)

    def workspace_bytes(self) -> int:
        return _abi.muon_workspace_bytes(self.handle)

    def launch_count(self) -> int:
        """Kernel launches one step enqueues."""
        return _abi.muon_launch_count(self.handle)

    def set_profiling(self, enable: bool) -> None:
        _abi.muon_set_profiling(self.handle, enable)

    def stage_work(self) -> dict:
        """Per stage: (algorithmic flops, algorithmic DRAM bytes, launches) of one step."""
        return _abi.muon_stage_work(self.handle)

    def stage_times(self) -> dict:
        """Device ms per stage of the most recent profiled step."""
        return _abi.muon_get_stage_times(self.handle)

    def get_state(self, which: int, index: int):
        """A device copy of one state array (see include/muon.h for layouts)."""
        import torch

        dev = torch.device("cuda", self.device)
        if which == MUON_STATE_MOMENTUM:
            s = self.specs[index]
            out = torch.empty((s.rows, s.cols), dtype=torch.float32, device=dev)
        else:
            info = self.matrix_info(index)
            if which == MUON_STATE_SECOND_MOMENT:
                out = torch.empty((info["lanes"],), dtype=torch.float32, device=dev)
            elif which == MUON_STATE_ORTHO:
                out = torch.empty((info["m"], info["n"]), dtype=torch.float32, device=dev)
            elif which == MUON_STATE_DIRECTION:
                out = torch.empty((info["m"], info["n"]), dtype=torch.float32, device=dev)
            else:
                raise ValueError(which)
        _abi.muon_get_state(self.handle, which, index, out.data_ptr(), _stream_ptr(None))
        return out

    def set_state(self, which: int, index: int, tensor) -> None:
        t = tensor.contiguous()
        _abi.muon_set_state(self.handle, which, index, t.data_ptr(), _stream_ptr(None))
        import torch

        torch.cuda.current_stream().synchronize()

    def close(self) -> None:
        if getattr(self, "handle", None) is not None:
            _abi.muon_destroy(self.handle)
            self.handle = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass
