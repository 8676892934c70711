"""The C-ABI library loads and exports every function include/lmce.h declares.

No compute call is made: only entry points that reject their arguments before
touching a device are exercised, so this runs without a GPU.
"""

import ctypes
import os
import re

import pytest

from grad_lmce_microstep_gb300 import build as B
from grad_lmce_microstep_gb300 import lmce as M

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "lmce.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(M.LIB_PATH):
        B.build()
    return M.load()


def declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"LMCE_API\s+[\w\s\*]+?\b(lmce_\w+)\s*\(", txt)))


def test_header_declares_the_binding_exports():
    assert declared() == sorted(M.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_status_strings(lib):
    for code in range(9):
        assert M.status_string(code) and M.status_string(code) != "unknown status"
    assert M.status_string(99) == "unknown status"


def test_argument_errors_before_any_device_call(lib):
    cfg = M.Config(768, 50304, 1024, 0, -100, 0, 1, 0, 0)
    h = ctypes.c_void_p()
    # null dW / null cfg / null out
    assert lib.lmce_create(ctypes.byref(cfg), None, ctypes.byref(h)) == M.ERR_ARG
    assert lib.lmce_create(None, ctypes.c_void_p(16), ctypes.byref(h)) == M.ERR_ARG
    for bad in (dict(C=0), dict(V=-1), dict(max_N=-5), dict(dtype=7), dict(norm=3), dict(path=9),
                dict(path=5), dict(C=100, path=4), dict(dtype=1, path=2),
                dict(grad_accum_steps=0), dict(flags=8), dict(C=4096, path=1)):
        c = M.Config(768, 50304, 1024, 0, -100, 0, 1, 0, 0)
        for k, v in bad.items():
            setattr(c, k, v)
        assert lib.lmce_create(ctypes.byref(c), ctypes.c_void_p(16), ctypes.byref(h)) == M.ERR_ARG, bad
    assert lib.lmce_microstep(None, None, None, None, 0, 0, None, None, None) == M.ERR_ARG
    assert lib.lmce_finalize(None, None, None, None, None) == M.ERR_ARG
    assert lib.lmce_dw_sumsq(None, None, None) == M.ERR_ARG
    assert lib.lmce_microstep_compact(None, None, None, None, 0, 0, 1, None, None, None) == M.ERR_ARG
    assert lib.lmce_microstep_ln(None, None, None, None, 0, 1e-5, None, None, 0, 1, None, None, None, None, None) == M.ERR_ARG
    assert lib.lmce_microstep_ln_compact(None, None, None, None, 0, 1e-5, None, None, 0, 0, 1, None, None, None, None, None) == M.ERR_ARG
    assert lib.lmce_adamw(None, None, None, None, None, 1, 1e-3, 0.9, 0.95, 1e-8, 0.1, 1.0, None) == M.ERR_ARG
    assert lib.lmce_destroy(None) == M.OK
    assert lib.lmce_profile(None, 1) == M.ERR_ARG
    assert lib.lmce_launch_count(None) == 0


def test_clip_coef_behind_the_c_abi():
    # lmce_clip_coef (host only) is the oracle's global-norm clip rule, rounded to float32
    import numpy as np
    from oracle import lmce_oracle as O
    for sumsq, mx in ((4.0, 1.0), (0.25, 1.0), (0.0, 1.0), (1e6, 0.5), (1.0, 1.0), (3.7e-3, 0.05)):
        assert M.clip_coef(sumsq, mx) == float(np.float32(O.clip_coef(sumsq, mx)))
    lib = M.load()
    c = ctypes.c_float()
    for sumsq, mx in ((-1.0, 1.0), (float("nan"), 1.0), (1.0, 0.0), (1.0, float("inf")), (float("inf"), 1.0)):
        assert lib.lmce_clip_coef(sumsq, mx, ctypes.byref(c)) == M.ERR_ARG
    assert lib.lmce_clip_coef(1.0, 1.0, None) == M.ERR_ARG


def test_header_compiles_as_c_and_links(lib, tmp_path):
    # a C99 program with warnings as errors, linked against the in-tree library, run on the CPU
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    here = os.path.dirname(os.path.abspath(__file__))
    libdir = os.path.dirname(M.LIB_PATH)
    exe = str(tmp_path / "c_abi_check")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.dirname(HEADER),
                    os.path.join(here, "c_abi_check.c"), "-o", exe, "-L" + libdir, "-llmce",
                    "-Wl,-rpath," + libdir], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok"


def test_binding_fails_loudly_without_the_library_or_a_device(tmp_path):
    # no CPU fallback: a missing library is an error, and so is a handle on host memory
    import torch
    with pytest.raises(RuntimeError):
        saved, M._lib = M._lib, None
        try:
            M.load(str(tmp_path / "missing.so"))
        finally:
            M._lib = saved
    with pytest.raises(ValueError):
        M.Lmce(64, 65, 16, torch.zeros(65, 64), "fp32")


def test_cuda_failure_reaches_the_caller_as_a_status(lib):
    # a host-side fault: on a machine without a usable device the runtime call in lmce_create
    # fails, and the library returns LMCE_ERR_CUDA with no handle instead of crashing
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    cfg = M.Config(768, 50304, 1024, 0, -100, 0, 1, 0, 0)
    h = ctypes.c_void_p(123)
    assert lib.lmce_create(ctypes.byref(cfg), ctypes.c_void_p(256), ctypes.byref(h)) == M.ERR_CUDA
    assert h.value is None
    # every valid path, the recompute path (4) included, gets past the argument checks
    for path in (1, 2, 3, 4):
        cfg = M.Config(768, 50304, 1024, 0, -100, 0, 1, path, 0)
        assert lib.lmce_create(ctypes.byref(cfg), ctypes.c_void_p(256), ctypes.byref(h)) == M.ERR_CUDA, path
    assert M.status_string(M.ERR_CUDA) != "unknown status"


def test_release_build_has_no_bounds_checks(lib):
    assert lib.lmce_debug_bounds() == 0
    assert lib.lmce_test_bounds_limit(None, 0) == M.ERR_ARG


def test_debug_build_compiles_the_bounds_checks():
    # the debug build (LMCE_DEBUG_BOUNDS=1) cross-compiles here like the release one, exports the
    # same entry points, and says it is the debug build (a host call: no device needed)
    path = B.build(debug_bounds=True)
    assert os.path.basename(path) == "liblmce_dbg.so"
    dbg = ctypes.CDLL(path)
    for name in declared():
        assert hasattr(dbg, name), name
    assert dbg.lmce_debug_bounds() == 1
    assert dbg.lmce_test_bounds_limit(None, 0) == M.ERR_ARG
