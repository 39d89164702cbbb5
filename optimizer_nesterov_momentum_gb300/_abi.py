"""ctypes binding of include/muon.h (argument marshalling only).

Every function here has the name of the C entry point it wraps and only
converts arguments; all work of the optimizer step happens in the CUDA
kernels of ``libmuon_gb300.so``.  Loading fails loudly when the library has
not been built: there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int32, c_int64, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmuon_gb300.so")

MUON_OK = 0
MUON_ERR_ARG = -1
MUON_ERR_ALIGN = -2
MUON_ERR_SHAPE = -3
MUON_ERR_CUDA = -4
MUON_ERR_TIMEOUT = -5
MUON_ERR_DESTROYED = -6
MUON_ERR_NOMEM = -7
MUON_ERR_UNSUPPORTED = -8
MUON_ERR_NONFINITE = -9

MUON_GRAD_BF16 = 0
MUON_GRAD_F32 = 1
MUON_SPLIT_CONTIGUOUS = 0
MUON_SPLIT_COLUMNS = 1
MUON_GEMM_TCGEN05 = 0
MUON_GEMM_SIMT = 1
MUON_LANES_SHORT_SIDE = 0
MUON_LANES_ROWS = 1
MUON_LANES_COLS = 2
MUON_NS_STANDARD = 0
MUON_NS_GRAM_PAIRS = 1
MUON_MAX_MATRICES = 1024
MUON_MAX_NS_STEPS = 16

MUON_STATE_MOMENTUM = 0
MUON_STATE_SECOND_MOMENT = 1
MUON_STATE_ORTHO = 2
MUON_STATE_DIRECTION = 3

MUON_STAGE_NAMES = ("momentum", "norm_scale", "gram", "poly", "update", "lane_stats", "apply", "product")
MUON_NUM_STAGES = len(MUON_STAGE_NAMES)

# Every entry point declared in include/muon.h.
EXPORTED = (
    "muon_config_default",
    "muon_create",
    "muon_step",
    "muon_reset",
    "muon_set_hparams",
    "muon_set_schedule",
    "muon_get_step",
    "muon_sync_status",
    "muon_destroy",
    "muon_error_string",
    "muon_last_error",
    "muon_num_matrices",
    "muon_matrix_info",
    "muon_workspace_bytes",
    "muon_launch_count",
    "muon_stage_work",
    "muon_set_profiling",
    "muon_get_stage_times",
    "muon_get_state",
    "muon_set_state",
    "muon_debug_inject_stall",
    "muon_nesterov_normalize_noalloc",
    # include/muon_adam.h
    "muon_adam_config_default",
    "muon_adam_create",
    "muon_adam_step",
    "muon_adam_reset",
    "muon_adam_set_lr_scale",
    "muon_adam_set_schedule",
    "muon_adam_get_step",
    "muon_adam_set_step",
    "muon_adam_get_state",
    "muon_adam_set_state",
    "muon_adam_launch_count",
    "muon_adam_last_error",
    "muon_adam_destroy",
)

MUON_ADAM_MAX_TENSORS = 1024

MUON_NOALLOC_MAX_TILES = 65536


class muon_shape(ctypes.Structure):
    _fields_ = [("rows", c_int64), ("cols", c_int64), ("ld", c_int64), ("split", c_int32), ("flags", c_int32)]


class muon_schedule(ctypes.Structure):
    _fields_ = [
        ("lr_base", c_float),
        ("lr_floor", c_float),
        ("cooldown_start", c_int64),
        ("cooldown_end", c_int64),
        ("momentum_start", c_float),
        ("momentum_end", c_float),
        ("momentum_warmup", c_int64),
    ]


class muon_adam_tensor(ctypes.Structure):
    _fields_ = [("numel", c_int64), ("lr", c_float), ("weight_decay", c_float)]


class muon_adam_config(ctypes.Structure):
    _fields_ = [("beta1", c_float), ("beta2", c_float), ("eps", c_float), ("grad_dtype", c_int32)]


class muon_config(ctypes.Structure):
    _fields_ = [
        ("lr", c_float),
        ("momentum", c_float),
        ("beta2", c_float),
        ("weight_decay", c_float),
        ("ns_steps", c_int32),
        ("nesterov", c_int32),
        ("lerp_form", c_int32),
        ("normuon", c_int32),
        ("norm_preserve", c_int32),
        ("grad_dtype", c_int32),
        ("gemm_engine", c_int32),
        ("lr_mul", POINTER(c_float)),
        ("wd_mul", POINTER(c_float)),
        ("ns_coeffs", POINTER(c_float)),
        ("normuon_lanes", c_int32),
        ("ns_form", c_int32),
        ("launch_overlap", c_int32),
    ]


class MuonError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{message} (code {code})")
        self.code = code


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads the C-ABI library once; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m optimizer_nesterov_momentum_gb300.build` "
            "(the optimizer has no CPU or fallback path)")
    lib = ctypes.CDLL(path)
    lib.muon_config_default.argtypes = [POINTER(muon_config)]
    lib.muon_config_default.restype = None
    lib.muon_create.argtypes = [POINTER(muon_shape), c_int32, POINTER(muon_config), c_int32, POINTER(c_void_p)]
    lib.muon_step.argtypes = [c_void_p, POINTER(c_void_p), POINTER(c_void_p), c_void_p]
    lib.muon_reset.argtypes = [c_void_p, c_void_p]
    lib.muon_set_hparams.argtypes = [c_void_p, c_float, c_float, c_float, c_float, c_void_p]
    lib.muon_sync_status.argtypes = [c_void_p, c_void_p]
    lib.muon_destroy.argtypes = [c_void_p]
    lib.muon_error_string.argtypes = [c_int32]
    lib.muon_error_string.restype = c_char_p
    lib.muon_last_error.argtypes = [c_void_p]
    lib.muon_last_error.restype = c_char_p
    lib.muon_num_matrices.argtypes = [c_void_p, POINTER(c_int32)]
    lib.muon_matrix_info.argtypes = [c_void_p, c_int32, POINTER(c_int64)]
    lib.muon_workspace_bytes.argtypes = [c_void_p, POINTER(c_int64)]
    lib.muon_launch_count.argtypes = [c_void_p, POINTER(c_int32)]
    lib.muon_stage_work.argtypes = [c_void_p, POINTER(c_int64), POINTER(c_int64), POINTER(c_int32)]
    lib.muon_set_schedule.argtypes = [c_void_p, POINTER(muon_schedule), c_int64, c_void_p]
    lib.muon_get_step.argtypes = [c_void_p, POINTER(c_int64), c_void_p]
    lib.muon_adam_config_default.argtypes = [POINTER(muon_adam_config)]
    lib.muon_adam_config_default.restype = None
    lib.muon_adam_create.argtypes = [POINTER(muon_adam_tensor), c_int32, POINTER(muon_adam_config), c_int32,
                                     POINTER(c_void_p)]
    lib.muon_adam_step.argtypes = [c_void_p, POINTER(c_void_p), POINTER(c_void_p), c_void_p]
    lib.muon_adam_reset.argtypes = [c_void_p, c_void_p]
    lib.muon_adam_set_lr_scale.argtypes = [c_void_p, c_float, c_void_p]
    lib.muon_adam_set_schedule.argtypes = [c_void_p, POINTER(muon_schedule), c_int64, c_void_p]
    lib.muon_adam_get_step.argtypes = [c_void_p, POINTER(c_int64), c_void_p]
    lib.muon_adam_set_step.argtypes = [c_void_p, c_int64, c_void_p]
    lib.muon_adam_get_state.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_void_p]
    lib.muon_adam_set_state.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_void_p]
    lib.muon_adam_launch_count.argtypes = [c_void_p, POINTER(c_int32)]
    lib.muon_adam_last_error.argtypes = [c_void_p]
    lib.muon_adam_last_error.restype = c_char_p
    lib.muon_adam_destroy.argtypes = [c_void_p]
    lib.muon_set_profiling.argtypes = [c_void_p, c_int32]
    lib.muon_get_stage_times.argtypes = [c_void_p, POINTER(c_float)]
    lib.muon_get_state.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_void_p]
    lib.muon_set_state.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_void_p]
    lib.muon_debug_inject_stall.argtypes = [c_void_p]
    lib.muon_nesterov_normalize_noalloc.argtypes = [c_void_p, c_int32, c_void_p, c_void_p, c_int64, c_int64,
                                                    c_float, c_int32, c_int32, c_void_p]
    for name in EXPORTED:
        if name not in ("muon_config_default", "muon_error_string", "muon_last_error", "muon_adam_config_default",
                        "muon_adam_last_error"):
            getattr(lib, name).restype = c_int32
    _lib = lib
    return lib


def _check(rc: int, handle=None) -> int:
    if rc < 0:
        lib = load_library()
        msg = lib.muon_last_error(handle).decode() or lib.muon_error_string(rc).decode()
        raise MuonError(rc, msg)
    return rc


def muon_config_default() -> muon_config:
    cfg = muon_config()
    load_library().muon_config_default(ctypes.byref(cfg))
    return cfg


def muon_create(shapes, cfg: muon_config, device: int) -> c_void_p:
    arr = (muon_shape * len(shapes))(*shapes)
    h = c_void_p()
    _check(load_library().muon_create(arr, len(shapes), ctypes.byref(cfg), device, ctypes.byref(h)))
    return h


def muon_step(h, params_ptrs, grads_ptrs, stream: int) -> None:
    _check(load_library().muon_step(h, params_ptrs, grads_ptrs, c_void_p(stream)), h)


def muon_reset(h, stream: int) -> None:
    _check(load_library().muon_reset(h, c_void_p(stream)), h)


def muon_set_hparams(h, lr, momentum, beta2, weight_decay, stream: int) -> None:
    _check(load_library().muon_set_hparams(h, lr, momentum, beta2, weight_decay, c_void_p(stream)), h)


def muon_set_schedule(h, sched, start_step: int, stream: int) -> None:
    ref = ctypes.byref(sched) if sched is not None else None
    _check(load_library().muon_set_schedule(h, ref, c_int64(start_step), c_void_p(stream)), h)


def muon_get_step(h, stream: int) -> int:
    out = c_int64()
    _check(load_library().muon_get_step(h, ctypes.byref(out), c_void_p(stream)), h)
    return out.value


def muon_sync_status(h, stream: int) -> int:
    return _check(load_library().muon_sync_status(h, c_void_p(stream)), h)


def muon_destroy(h) -> None:
    _check(load_library().muon_destroy(h), h)


def muon_error_string(code: int) -> str:
    return load_library().muon_error_string(code).decode()


def muon_last_error(h) -> str:
    return load_library().muon_last_error(h).decode()


def muon_num_matrices(h) -> int:
    out = c_int32()
    _check(load_library().muon_num_matrices(h, ctypes.byref(out)), h)
    return out.value


def muon_matrix_info(h, index: int):
    out = (c_int64 * 8)()
    _check(load_library().muon_matrix_info(h, index, out), h)
    return tuple(out)


def muon_debug_inject_stall(h) -> None:
    _check(load_library().muon_debug_inject_stall(h), h)


def muon_workspace_bytes(h) -> int:
    out = c_int64()
    _check(load_library().muon_workspace_bytes(h, ctypes.byref(out)), h)
    return out.value


def muon_launch_count(h) -> int:
    out = c_int32()
    _check(load_library().muon_launch_count(h, ctypes.byref(out)), h)
    return out.value


def muon_stage_work(h):
    """Per stage name: (algorithmic flops, algorithmic DRAM bytes, launches) of one step."""
    fl = (c_int64 * MUON_NUM_STAGES)()
    by = (c_int64 * MUON_NUM_STAGES)()
    ln = (c_int32 * MUON_NUM_STAGES)()
    _check(load_library().muon_stage_work(h, fl, by, ln), h)
    return {name: (fl[k], by[k], ln[k]) for k, name in enumerate(MUON_STAGE_NAMES)}


def muon_set_profiling(h, enable: bool) -> None:
    _check(load_library().muon_set_profiling(h, int(enable)), h)


def muon_get_stage_times(h):
    out = (c_float * MUON_NUM_STAGES)()
    _check(load_library().muon_get_stage_times(h, out), h)
    return dict(zip(MUON_STAGE_NAMES, list(out)))


def muon_get_state(h, which: int, index: int, dst_ptr: int, stream: int) -> None:
    _check(load_library().muon_get_state(h, which, index, c_void_p(dst_ptr), c_void_p(stream)), h)


def muon_set_state(h, which: int, index: int, src_ptr: int, stream: int) -> None:
    _check(load_library().muon_set_state(h, which, index, c_void_p(src_ptr), c_void_p(stream)), h)


def muon_nesterov_normalize_noalloc(grad_ptr: int, grad_dtype: int, momentum_ptr: int, x0_ptr: int, rows: int,
                                    cols: int, mu: float, lerp_form: bool, nesterov: bool, stream: int) -> None:
    """Allocation-free momentum + Nesterov + normalisation of one dense matrix (see include/muon.h)."""
    rc = load_library().muon_nesterov_normalize_noalloc(
        c_void_p(grad_ptr), grad_dtype, c_void_p(momentum_ptr), c_void_p(x0_ptr), rows, cols, mu, int(lerp_form),
        int(nesterov), c_void_p(stream))
    if rc < 0:
        raise MuonError(rc, muon_error_string(rc))


# ---------------------------------------------------------------- include/muon_adam.h


def _adam_check(rc: int, handle=None) -> int:
    if rc < 0:
        lib = load_library()
        msg = lib.muon_adam_last_error(handle).decode() or lib.muon_error_string(rc).decode()
        raise MuonError(rc, msg)
    return rc


def muon_adam_config_default() -> muon_adam_config:
    cfg = muon_adam_config()
    load_library().muon_adam_config_default(ctypes.byref(cfg))
    return cfg


def muon_adam_create(tensors, cfg: muon_adam_config, device: int):
    arr = (muon_adam_tensor * len(tensors))(*tensors)
    out = c_void_p()
    _adam_check(load_library().muon_adam_create(arr, len(tensors), ctypes.byref(cfg), device, ctypes.byref(out)))
    return out


def muon_adam_step(h, params, grads, stream: int) -> None:
    n = len(params)
    pa = (c_void_p * n)(*params)
    ga = (c_void_p * n)(*grads)
    _adam_check(load_library().muon_adam_step(h, pa, ga, c_void_p(stream)), h)


def muon_adam_reset(h, stream: int) -> None:
    _adam_check(load_library().muon_adam_reset(h, c_void_p(stream)), h)


def muon_adam_set_lr_scale(h, scale: float, stream: int) -> None:
    _adam_check(load_library().muon_adam_set_lr_scale(h, scale, c_void_p(stream)), h)


def muon_adam_set_schedule(h, sched, start_step: int, stream: int) -> None:
    ref = ctypes.byref(sched) if sched is not None else None
    _adam_check(load_library().muon_adam_set_schedule(h, ref, c_int64(start_step), c_void_p(stream)), h)


def muon_adam_get_step(h, stream: int) -> int:
    out = c_int64()
    _adam_check(load_library().muon_adam_get_step(h, ctypes.byref(out), c_void_p(stream)), h)
    return out.value


def muon_adam_set_step(h, t: int, stream: int) -> None:
    _adam_check(load_library().muon_adam_set_step(h, c_int64(t), c_void_p(stream)), h)


def muon_adam_get_state(h, which: int, index: int, dst_ptr: int, stream: int) -> None:
    _adam_check(load_library().muon_adam_get_state(h, which, index, c_void_p(dst_ptr), c_void_p(stream)), h)


def muon_adam_set_state(h, which: int, index: int, src_ptr: int, stream: int) -> None:
    _adam_check(load_library().muon_adam_set_state(h, which, index, c_void_p(src_ptr), c_void_p(stream)), h)


def muon_adam_launch_count(h) -> int:
    out = c_int32()
    _adam_check(load_library().muon_adam_launch_count(h, ctypes.byref(out)), h)
    return out.value


def muon_adam_destroy(h) -> None:
    _adam_check(load_library().muon_adam_destroy(h), h)
