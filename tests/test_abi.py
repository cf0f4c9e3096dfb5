"""The C ABI library builds, loads without a GPU and exports every entry
point declared in include/*.h (CPU only: no compute calls)."""
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(hdr).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[\w\s\*]+?\b(mlora_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import rl_step_gb300
    return rl_step_gb300.load_library()


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("mlora_create", "mlora_forward", "mlora_forward_backward",
              "mlora_forward_backward_custom", "mlora_optim_step", "mlora_save_state",
              "mlora_destroy", "mlora_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import rl_step_gb300
    out = subprocess.run(["nm", "-D", "--defined-only", rl_step_gb300.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = _declared() - exported
    assert not missing, f"declared but not exported: {sorted(missing)}"
    for n in _declared():
        assert hasattr(lib, n)


def test_library_has_no_unresolved_internal_symbols(lib):
    import rl_step_gb300
    out = subprocess.run(["nm", "-D", "--undefined-only", rl_step_gb300.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    bad = [ln for ln in out.splitlines() if "mlk" in ln or "mlora" in ln]
    assert not bad, bad


def test_argument_errors_need_no_gpu(lib):
    import ctypes
    import rl_step_gb300 as m
    out = ctypes.c_void_p()
    rc = lib.mlora_create(None, None, ctypes.byref(out))
    assert rc == -1
    assert b"NULL" in lib.mlora_last_error()
    assert lib.mlora_forward(None, None, None, None) == -1
    assert lib.mlora_kernel_launches(None) == 0


def test_build_is_for_sm103a():
    src = open(os.path.join(ROOT, "rl_step_gb300", "_build.py")).read()
    assert "arch=compute_103a,code=sm_103a" in src


def test_transformer_entry_points_reject_bad_arguments_without_a_gpu(lib):
    import ctypes
    import rl_step_gb300.transformer as t
    tl = t._lib()
    out = ctypes.c_void_p()
    assert tl.mlora_tf_create(None, None, ctypes.byref(out)) == -1
    assert b"NULL" in tl.mlora_last_error()
    ranks = (ctypes.c_int32 * 1)(8)
    alphas = (ctypes.c_float * 1)(16.0)
    cfg = t._TfConfig(100, 256, 4, 3, 128, 512, 2, 1, ranks, alphas, 1e6, 1e-6, 64)   # 3 does not divide 4
    init = t._TfInit()
    assert tl.mlora_tf_create(ctypes.byref(cfg), ctypes.byref(init), ctypes.byref(out)) == -1
    cfg = t._TfConfig(100, 256, 4, 2, 64, 512, 2, 1, ranks, alphas, 1e6, 1e-6, 64)    # head_dim 64
    assert tl.mlora_tf_create(ctypes.byref(cfg), ctypes.byref(init), ctypes.byref(out)) == -1
    assert b"head_dim" in tl.mlora_last_error()
    assert tl.mlora_tf_forward(None, None, None, None) == -1
    assert tl.mlora_tf_kernel_launches(None) == 0
