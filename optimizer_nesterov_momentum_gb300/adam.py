"""Fused Adam for the tensors Muon does not take (embedding, head, scalars).

``AdamGroup`` owns one ``muon_adam_handle`` of ``libmuon_gb300.so``
(include/muon_adam.h).  ``step()`` passes raw device pointers; the update runs
in the library's CUDA kernels and there is no CPU path.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Sequence

from . import _abi

MUON_ADAM_M = 0
MUON_ADAM_V = 1


@dataclass(frozen=True)
class AdamTensorSpec:
    numel: int
    lr: float
    weight_decay: float = 0.0


def _stream_ptr(stream) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


class AdamGroup:
    """Adam over a fixed list of tensors (fp32 parameters, contiguous)."""

    def __init__(self, tensors: Sequence[AdamTensorSpec], beta1: float = 0.9, beta2: float = 0.95, eps: float = 1e-8,
                 grad_dtype: str = "bf16", device: int = 0):
        cfg = _abi.muon_adam_config_default()
        cfg.beta1, cfg.beta2, cfg.eps = beta1, beta2, eps
        cfg.grad_dtype = {"bf16": _abi.MUON_GRAD_BF16, "f32": _abi.MUON_GRAD_F32}[grad_dtype]
        self.specs = list(tensors)
        self.grad_dtype = grad_dtype
        arr = [_abi.muon_adam_tensor(t.numel, t.lr, t.weight_decay) for t in self.specs]
        self.handle = _abi.muon_adam_create(arr, cfg, device)

    def step(self, params, grads, stream=None) -> None:
        """One Adam step; ``params`` fp32 and ``grads`` (bf16 / fp32) CUDA tensors, contiguous."""
        import torch

        want = torch.bfloat16 if self.grad_dtype == "bf16" else torch.float32
        if len(params) != len(self.specs) or len(grads) != len(self.specs):
            raise ValueError("one parameter and one gradient per tensor")
        for p, g, s in zip(params, grads, self.specs):
            if p.dtype != torch.float32 or g.dtype != want or p.numel() != s.numel or g.numel() != s.numel:
                raise ValueError("parameter / gradient dtype or size does not match the group")
            if not (p.is_contiguous() and g.is_contiguous() and p.is_cuda and g.is_cuda):
                raise ValueError("tensors must be contiguous CUDA tensors")
        _abi.muon_adam_step(self.handle, [p.data_ptr() for p in params], [g.data_ptr() for g in grads],
                            _stream_ptr(stream))

    def reset(self, stream=None) -> None:
        _abi.muon_adam_reset(self.handle, _stream_ptr(stream))

    def set_lr_scale(self, scale: float, stream=None) -> None:
        _abi.muon_adam_set_lr_scale(self.handle, scale, _stream_ptr(stream))

    def set_schedule(self, lr_base: float, cooldown_start: int, cooldown_end: int, lr_floor: float = 0.0,
                     start_step: int = 0, stream=None) -> None:
        sc = _abi.muon_schedule(lr_base, lr_floor, cooldown_start, cooldown_end, 0.0, 0.0, 0)
        _abi.muon_adam_set_schedule(self.handle, sc, start_step, _stream_ptr(stream))

    def clear_schedule(self, stream=None) -> None:
        _abi.muon_adam_set_schedule(self.handle, None, 0, _stream_ptr(stream))

    def step_count(self, stream=None) -> int:
        return _abi.muon_adam_get_step(self.handle, _stream_ptr(stream))

    def set_step_count(self, t: int, stream=None) -> None:
        _abi.muon_adam_set_step(self.handle, t, _stream_ptr(stream))

    def get_state(self, which: int, index: int):
        import torch

        out = torch.empty(self.specs[index].numel, dtype=torch.float32, device="cuda")
        _abi.muon_adam_get_state(self.handle, which, index, out.data_ptr(), _stream_ptr(None))
        return out

    def set_state(self, which: int, index: int, src) -> None:
        import torch

        if src.dtype != torch.float32 or src.numel() != self.specs[index].numel or not src.is_contiguous():
            raise ValueError("state must be a contiguous fp32 tensor of the tensor's size")
        _abi.muon_adam_set_state(self.handle, which, index, src.data_ptr(), _stream_ptr(None))

    def launch_count(self) -> int:
        return _abi.muon_adam_launch_count(self.handle)

    def close(self) -> None:
        if getattr(self, "handle", None) is not None:
            _abi.muon_adam_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
