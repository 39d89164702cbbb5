"""The C-ABI library on the host: it loads, exports every entry point that
include/*.h declare, and rejects bad arguments before any device work.
No kernel runs here (there is no GPU in the build container)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from optimizer_nesterov_momentum_gb300 import _abi, build

    build.build()
    return _abi.load_library()


def _declared_entry_points():
    text = ""
    for name in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if name.endswith(".h"):
            with open(os.path.join(ROOT, "include", name)) as f:
                text += f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(muon_[a-z_]+)\s*\(", text)))


def test_header_and_binding_agree():
    from optimizer_nesterov_momentum_gb300 import _abi

    assert _declared_entry_points() == sorted(_abi.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_entry_points():
        assert hasattr(lib, name), name


def test_struct_layouts_match_header():
    from optimizer_nesterov_momentum_gb300 import _abi

    assert ctypes.sizeof(_abi.muon_shape) == 32
    assert _abi.muon_config.lr_mul.offset == 48
    assert _abi.muon_config.normuon_lanes.offset == 72
    assert _abi.muon_config.ns_form.offset == 76
    assert _abi.muon_config.launch_overlap.offset == 80
    assert ctypes.sizeof(_abi.muon_config) == 88
    assert ctypes.sizeof(_abi.muon_schedule) == 40
    assert [getattr(_abi.muon_schedule, f).offset for f, _ in _abi.muon_schedule._fields_] == [0, 4, 8, 16, 24, 28, 32]
    assert ctypes.sizeof(_abi.muon_adam_tensor) == 16 and ctypes.sizeof(_abi.muon_adam_config) == 16


def test_struct_layouts_match_a_c_compiler(tmp_path):
    """Every field offset and struct size of the ctypes mirrors, against what a C
    compiler makes of include/*.h."""
    import shutil
    import subprocess

    from optimizer_nesterov_momentum_gb300 import _abi

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"muon_shape": _abi.muon_shape, "muon_config": _abi.muon_config,
               "muon_schedule": _abi.muon_schedule, "muon_adam_tensor": _abi.muon_adam_tensor,
               "muon_adam_config": _abi.muon_adam_config}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "muon.h"', '#include "muon_adam.h"',
             'int main(void) {']
    expect = []
    for name, cls in structs.items():
        lines.append(f'  printf("%zu\\n", sizeof({name}));')
        expect.append(ctypes.sizeof(cls))
        for field, _ in cls._fields_:
            lines.append(f'  printf("%zu\\n", offsetof({name}, {field}));')
            expect.append(getattr(cls, field).offset)
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    assert got == expect


def test_config_default(lib):
    from optimizer_nesterov_momentum_gb300 import _abi

    cfg = _abi.muon_config_default()
    assert abs(cfg.lr - 0.02) < 1e-9 and abs(cfg.momentum - 0.95) < 1e-7
    assert cfg.ns_steps == 5 and cfg.nesterov == 1 and cfg.lerp_form == 1 and cfg.normuon == 1
    assert not cfg.lr_mul and not cfg.ns_coeffs


def _create(lib, shapes, cfg=None, n=None, out=True):
    from optimizer_nesterov_momentum_gb300 import _abi

    arr = (_abi.muon_shape * max(len(shapes), 1))(*shapes)
    h = ctypes.c_void_p()
    return lib.muon_create(arr, len(shapes) if n is None else n, ctypes.byref(cfg) if cfg else None, 0,
                           ctypes.byref(h) if out else None)


def test_create_rejects_bad_arguments_on_the_host(lib):
    from optimizer_nesterov_momentum_gb300 import _abi as A

    good = [A.muon_shape(64, 256, 0, 1, 0)]
    assert _create(lib, good, out=False) == A.MUON_ERR_ARG
    assert _create(lib, good, n=0) == A.MUON_ERR_ARG
    assert _create(lib, good, n=A.MUON_MAX_MATRICES + 1) == A.MUON_ERR_ARG
    cfg = A.muon_config_default()
    cfg.ns_steps = 0
    assert _create(lib, good, cfg) == A.MUON_ERR_ARG
    cfg = A.muon_config_default()
    cfg.ns_steps = A.MUON_MAX_NS_STEPS + 1
    assert _create(lib, good, cfg) == A.MUON_ERR_ARG
    cfg = A.muon_config_default()
    cfg.grad_dtype = 7
    assert _create(lib, good, cfg) == A.MUON_ERR_ARG
    assert _create(lib, [A.muon_shape(0, 256, 0, 1, 0)]) == A.MUON_ERR_SHAPE
    assert _create(lib, [A.muon_shape(64, 256, 100, 1, 0)]) == A.MUON_ERR_SHAPE      # ld < cols
    assert _create(lib, [A.muon_shape(64, 250, 0, 4, 0)]) == A.MUON_ERR_SHAPE        # cols % split
    assert _create(lib, [A.muon_shape(64, 256, 512, 4, 0)]) == A.MUON_ERR_SHAPE      # contiguous split, ld != cols
    assert _create(lib, [A.muon_shape(64, 256, 0, 1, 9)]) == A.MUON_ERR_ARG          # bad flags
    assert "split" in lib.muon_last_error(None).decode() or "flags" in lib.muon_last_error(None).decode()


def test_create_without_a_device_reports_cuda_error(lib):
    import torch
    from optimizer_nesterov_momentum_gb300 import _abi as A

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _create(lib, [A.muon_shape(64, 256, 0, 1, 0)]) == A.MUON_ERR_CUDA
    assert "device" in lib.muon_last_error(None).decode().lower()


def test_calls_on_invalid_handles(lib):
    from optimizer_nesterov_momentum_gb300 import _abi as A

    assert lib.muon_step(None, None, None, None) == A.MUON_ERR_ARG
    assert lib.muon_reset(None, None) == A.MUON_ERR_ARG
    assert lib.muon_destroy(None) == A.MUON_ERR_ARG
    bogus = ctypes.c_void_p(0x1234)
    assert lib.muon_step(bogus, None, None, None) == A.MUON_ERR_ARG
    assert lib.muon_sync_status(bogus, None) == A.MUON_ERR_ARG
    sc = A.muon_schedule(0.03, 0.3, 10, 20, 0.85, 0.95, 5)
    assert lib.muon_set_schedule(None, ctypes.byref(sc), ctypes.c_int64(0), None) == A.MUON_ERR_ARG
    assert lib.muon_set_schedule(bogus, None, ctypes.c_int64(0), None) == A.MUON_ERR_ARG
    step = ctypes.c_int64()
    assert lib.muon_get_step(bogus, ctypes.byref(step), None) == A.MUON_ERR_ARG
    n = ctypes.c_int32()
    assert lib.muon_num_matrices(bogus, ctypes.byref(n)) == A.MUON_ERR_ARG


def test_adam_rejects_bad_arguments_on_the_host(lib):
    A = __import__("optimizer_nesterov_momentum_gb300._abi", fromlist=["x"])
    cfg = A.muon_adam_config_default()
    assert (cfg.beta1, cfg.beta2, cfg.grad_dtype) == (pytest.approx(0.9), pytest.approx(0.95), A.MUON_GRAD_BF16)
    assert cfg.eps == pytest.approx(1e-8)
    good = (A.muon_adam_tensor * 1)(A.muon_adam_tensor(10, 0.1, 0.0))
    out = ctypes.c_void_p()
    assert lib.muon_adam_create(good, 1, ctypes.byref(cfg), 0, None) == A.MUON_ERR_ARG
    assert lib.muon_adam_create(good, 0, ctypes.byref(cfg), 0, ctypes.byref(out)) == A.MUON_ERR_ARG
    assert lib.muon_adam_create(good, A.MUON_ADAM_MAX_TENSORS + 1, ctypes.byref(cfg), 0, ctypes.byref(out)) == A.MUON_ERR_ARG
    bad = A.muon_adam_config_default()
    bad.beta1 = 1.0
    assert lib.muon_adam_create(good, 1, ctypes.byref(bad), 0, ctypes.byref(out)) == A.MUON_ERR_ARG
    bad = A.muon_adam_config_default()
    bad.grad_dtype = 7
    assert lib.muon_adam_create(good, 1, ctypes.byref(bad), 0, ctypes.byref(out)) == A.MUON_ERR_ARG
    for t in (A.muon_adam_tensor(0, 0.1, 0.0), A.muon_adam_tensor(4, -1.0, 0.0), A.muon_adam_tensor(4, float("nan"), 0.0)):
        arr = (A.muon_adam_tensor * 1)(t)
        assert lib.muon_adam_create(arr, 1, ctypes.byref(cfg), 0, ctypes.byref(out)) in (A.MUON_ERR_ARG, A.MUON_ERR_SHAPE)
    assert lib.muon_adam_last_error(None).decode()
    # no GPU here: a valid request fails at the device, loudly
    assert lib.muon_adam_create(good, 1, ctypes.byref(cfg), 0, ctypes.byref(out)) == A.MUON_ERR_CUDA
    assert lib.muon_adam_step(None, None, None, None) == A.MUON_ERR_ARG
    assert lib.muon_adam_reset(ctypes.c_void_p(0x1234), None) == A.MUON_ERR_ARG
    assert lib.muon_adam_destroy(None) == A.MUON_ERR_ARG


def test_error_strings(lib):
    from optimizer_nesterov_momentum_gb300 import _abi as A

    for code in range(0, -9, -1):
        assert lib.muon_error_string(code).decode() != "unknown error"
    assert lib.muon_error_string(-99).decode() == "unknown error"
    assert A.muon_error_string(A.MUON_ERR_TIMEOUT) == "device wait timed out"


def test_missing_library_fails_loudly(tmp_path):
    from optimizer_nesterov_momentum_gb300 import _abi

    saved = _abi._lib
    _abi._lib = None
    try:
        with pytest.raises(RuntimeError, match="no CPU or fallback path"):
            _abi.load_library(str(tmp_path / "absent.so"))
    finally:
        _abi._lib = saved


def test_noalloc_rejects_bad_arguments_on_the_host(lib):
    """Checked before any CUDA call, so no device is needed (the pointers are never used)."""
    from optimizer_nesterov_momentum_gb300 import _abi as A

    f = lib.muon_nesterov_normalize_noalloc
    g, m, x = 0x10000, 0x20000, 0x30000
    assert f(None, 0, m, x, 8, 8, 0.95, 1, 1, None) == A.MUON_ERR_ARG
    assert f(g, 0, None, x, 8, 8, 0.95, 1, 1, None) == A.MUON_ERR_ARG
    assert f(g, 2, m, x, 8, 8, 0.95, 1, 1, None) == A.MUON_ERR_ARG
    assert f(g, 0, m, m, 8, 8, 0.95, 1, 1, None) == A.MUON_ERR_ARG          # x0 aliases the momentum
    assert f(m, A.MUON_GRAD_F32, m, x, 8, 8, 0.95, 1, 1, None) == A.MUON_ERR_ARG  # fp32 grad aliases it
    assert f(g, 0, m, x, 0, 8, 0.95, 1, 1, None) == A.MUON_ERR_SHAPE
    assert f(g, 0, m, x, 16384, 16385, 0.95, 1, 1, None) == A.MUON_ERR_SHAPE  # 256 x 257 tiles
    assert f(g, 0, m, x, 1 << 40, 1 << 40, 0.95, 1, 1, None) == A.MUON_ERR_SHAPE  # would overflow a product
    assert f(g, 0, m, x, 1, (1 << 22) + 1, 0.95, 1, 1, None) == A.MUON_ERR_SHAPE


def test_normuon_lanes_is_validated(lib):
    from optimizer_nesterov_momentum_gb300 import _abi as A

    cfg = A.muon_config_default()
    assert cfg.normuon_lanes == A.MUON_LANES_SHORT_SIDE
    cfg.normuon_lanes = 3
    assert _create(lib, [A.muon_shape(64, 256, 0, 1, 0)], cfg) == A.MUON_ERR_ARG


def test_ns_form_is_validated(lib):
    from optimizer_nesterov_momentum_gb300 import _abi as A

    cfg = A.muon_config_default()
    assert cfg.ns_form == A.MUON_NS_GRAM_PAIRS
    cfg.ns_form = 2
    assert _create(lib, [A.muon_shape(64, 256, 0, 1, 0)], cfg) == A.MUON_ERR_ARG


def test_launch_overlap_is_validated(lib):
    from optimizer_nesterov_momentum_gb300 import _abi as A

    cfg = A.muon_config_default()
    assert cfg.launch_overlap == 1
    cfg.launch_overlap = 2
    assert _create(lib, [A.muon_shape(64, 256, 0, 1, 0)], cfg) == A.MUON_ERR_ARG


def test_stage_names_follow_the_header():
    from optimizer_nesterov_momentum_gb300 import _abi as A

    hdr = open(os.path.join(ROOT, "include", "muon.h")).read()
    ids = {}
    for line in hdr.splitlines():
        parts = line.split()
        if len(parts) >= 3 and parts[0] == "#define" and parts[1].startswith("MUON_STAGE_"):
            ids[parts[1]] = int(parts[2])
        if len(parts) >= 3 and parts[0] == "#define" and parts[1] == "MUON_NUM_STAGES":
            assert int(parts[2]) == A.MUON_NUM_STAGES
    names = {"MUON_STAGE_MOMENTUM": "momentum", "MUON_STAGE_NORM": "norm_scale", "MUON_STAGE_GRAM": "gram",
             "MUON_STAGE_POLY": "poly", "MUON_STAGE_UPDATE": "update", "MUON_STAGE_LANE": "lane_stats",
             "MUON_STAGE_APPLY": "apply", "MUON_STAGE_PRODUCT": "product"}
    assert set(ids) == set(names)
    for macro, k in ids.items():
        assert A.MUON_STAGE_NAMES[k] == names[macro]
