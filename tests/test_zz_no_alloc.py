"""The allocation-free entry point (lmce_microstep_noalloc) against the handle-based one.

lmce_microstep_noalloc exists for callers that cannot call cudaMalloc (a runtime that
owns all device memory through its own pool, or a path that must not stall on cudaFree's
device-wide synchronisation); its scratch is a fixed array inside the library.  Two
calls in a row -- the second one accumulating into dW -- must give what lmce_create /
lmce_microstep / lmce_finalize give on the same micro-batches.  This file is collected
last so that a run stopping at the first failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

from grad_lmce_microstep_gb300 import inputs as I
from grad_lmce_microstep_gb300 import lmce as M

from gpu_util import GRAD_REL, LOSS_REL, max_rel_err, to_dev

pytestmark = pytest.mark.gpu


def _noalloc_step(w, W, mbs, gv):
    lib = M.load()
    cfg = M.Config(w.C, w.V, 0, M.DTYPES[w.dtype], -100, M.NORMS["global"], len(mbs), M.PATHS["auto"], 0)
    dW = torch.full((w.V, w.C), float("nan"), dtype=torch.float32, device="cuda")
    out = []
    stream = M._stream(None)
    for k, (h, y) in enumerate(mbs):
        dh = torch.empty_like(h)
        ls = torch.zeros(1, dtype=torch.float64, device="cuda")
        cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
        st = lib.lmce_microstep_noalloc(ctypes.byref(cfg), M._ptr(h), M._ptr(W), M._ptr(y), int(y.numel()), gv,
                                        M._ptr(dh), M._ptr(dW), 1 if k else 0, None, M._ptr(ls), M._ptr(cnt),
                                        stream)
        assert st == M.OK, M.status_string(st)
        out.append((dh, ls, cnt))
    torch.cuda.synchronize()
    return dW, out


@pytest.mark.parametrize("kind", ["bf16_ragged", "fp32_tiny_char"])
def test_noalloc_matches_handle_api_on_two_calls(kind):
    w = I.custom([300, 213], 256, 1000, "bf16", seed=11, ignore_frac=0.1) if kind == "bf16_ragged" \
        else I.tiny_char(seed=3)
    W, mbs = to_dev(w)
    gv = sum(w.valid_counts())
    dW_ref, dhs_ref, _, (ls_ref, cnt_ref, _, st_ref) = M.run_step(W, mbs, w.dtype, path="simt")
    assert st_ref == M.OK
    dW, out = _noalloc_step(w, W, mbs, gv)
    tol = GRAD_REL[w.dtype]
    assert max_rel_err(dW.double().cpu().numpy(), dW_ref.double().cpu().numpy()) <= tol
    for (dh, ls, cnt), dh_ref in zip(out, dhs_ref):
        assert max_rel_err(dh.double().cpu().numpy(), dh_ref.double().cpu().numpy()) <= tol
    assert sum(int(c.item()) for _, _, c in out) == cnt_ref
    ls_sum = sum(float(l.item()) for _, l, _ in out)
    assert abs(ls_sum - ls_ref) <= LOSS_REL * abs(ls_ref)


def test_noalloc_rejects_oversize():
    lib = M.load()
    cfg = M.Config(64, 100, 0, 0, -100, 0, 1, 0, 0)
    big = M.NOALLOC_MAX_N + 1
    dW = torch.zeros(100, 64, dtype=torch.float32, device="cuda")
    st = lib.lmce_microstep_noalloc(ctypes.byref(cfg), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                    ctypes.c_void_p(16), big, big, ctypes.c_void_p(16), M._ptr(dW), 0, None, None,
                                    None, M._stream(None))
    assert st == M.ERR_ARG
    assert float(dW.abs().max()) == 0.0
