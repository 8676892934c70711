"""The allocation-free entry point (lmce_microstep_noalloc) against the float64 oracle.

lmce_microstep_noalloc exists for callers that cannot call cudaMalloc (a runtime that
owns all device memory through its own pool, or a path that must not stall on cudaFree's
device-wide synchronisation); its scratch is a fixed array inside the library.  Two
calls in a row -- the second one accumulating into dW -- must give the oracle's optimizer
step on the same micro-batches, under both normalisations, and also what the handle
API's micro-step gives.  This file is collected last so that a run stopping at the first
failure has already run every other test.
"""

import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from grad_lmce_microstep_gb300 import inputs as I
from grad_lmce_microstep_gb300 import lmce as M

from gpu_util import GRAD_REL, LOSS_REL, max_rel_err, run_oracle, to_dev

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _noalloc_step(w, W, mbs, gv, norm="global"):
    lib = M.load()
    cfg = M.Config(w.C, w.V, 0, M.DTYPES[w.dtype], -100, M.NORMS[norm], len(mbs), M.PATHS["auto"], 0)
    dW = torch.full((w.V, w.C), float("nan"), dtype=torch.float32, device="cuda")
    out = []
    stream = M._stream(None)
    for k, (h, y) in enumerate(mbs):
        dh = torch.empty_like(h)
        rl = torch.empty(y.numel(), dtype=torch.float32, device="cuda")
        ls = torch.zeros(1, dtype=torch.float64, device="cuda")
        cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
        st = lib.lmce_microstep_noalloc(ctypes.byref(cfg), M._ptr(h), M._ptr(W), M._ptr(y), int(y.numel()), gv,
                                        M._ptr(dh), M._ptr(dW), 1 if k else 0, M._ptr(rl), M._ptr(ls), M._ptr(cnt),
                                        stream)
        assert st == M.OK, M.status_string(st)
        out.append((dh, rl, ls, cnt))
    torch.cuda.synchronize()
    return dW, out


def _check_against_oracle(w, dW, out, norm):
    ref = run_oracle(w, norm=norm)
    tol = GRAD_REL[w.dtype]
    e = max_rel_err(dW.double().cpu().numpy(), ref.dW)
    assert e <= tol, f"dW max err {e:.3e}"
    for (dh, rl, ls, cnt), m in zip(out, ref.micro):
        e = max_rel_err(dh.double().cpu().numpy(), m.dh)
        assert e <= tol, f"dh max err {e:.3e}"
        assert int(cnt.item()) == m.count
        assert abs(float(ls.item()) - m.loss_sum) <= LOSS_REL * abs(m.loss_sum)
        d = np.abs(rl.double().cpu().numpy() - m.row_loss)
        assert float(d.max()) <= LOSS_REL * max(1.0, float(np.abs(m.row_loss).max()))


@pytest.mark.parametrize("norm", ["global", "micro_mean"])
@pytest.mark.parametrize("kind", ["bf16_ragged", "fp32_tiny_char"])
def test_noalloc_two_calls_match_oracle(kind, norm):
    w = I.custom([300, 213], 256, 1000, "bf16", seed=11, ignore_frac=0.1) if kind == "bf16_ragged" \
        else I.tiny_char(seed=3)
    W, mbs = to_dev(w)
    gv = sum(w.valid_counts())
    dW, out = _noalloc_step(w, W, mbs, gv, norm)
    _check_against_oracle(w, dW, out, norm)
    # and the handle API's micro-step on the same inputs (the same normalisation)
    dW_h, dhs_h, _, (ls_h, cnt_h, _, st_h) = M.run_step(W, mbs, w.dtype, norm=norm, path="simt")
    assert st_h == M.OK
    tol = GRAD_REL[w.dtype]
    assert max_rel_err(dW.double().cpu().numpy(), dW_h.double().cpu().numpy()) <= tol
    for (dh, _, _, _), d_h in zip(out, dhs_h):
        assert max_rel_err(dh.double().cpu().numpy(), d_h.double().cpu().numpy()) <= tol
    assert sum(int(c.item()) for *_, c in out) == cnt_h


def test_noalloc_at_its_row_limit():
    # N == LMCE_NOALLOC_MAX_N fills the logsumexp and partial slots of the fixed array to the end:
    # the exact valid count (per-block count partials, the last block holding 13 valid rows) and
    # every row's loss (its logsumexp slot) are checked.  bf16 inputs: a float32 sum over ~98k
    # tokens is itself accurate only to about 1e-5, the tolerance the float32 check uses at its
    # 256-token size
    C, V, N = 64, 65, M.NOALLOC_MAX_N
    g = torch.Generator().manual_seed(5)
    W = (0.3 * torch.randn(V, C, generator=g)).to(torch.bfloat16)
    hs = [torch.randn(N, C, generator=g).to(torch.bfloat16), torch.randn(N // 2 + 7, C, generator=g).to(torch.bfloat16)]
    ys = [torch.randint(0, V, (h.shape[0],), generator=g, dtype=torch.int32) for h in hs]
    ys[0][-3:] = -100
    w = I.Workload("noalloc_limit", C, V, "bf16", W, list(zip(hs, ys)))
    Wd, mbs = to_dev(w)
    gv = sum(w.valid_counts())
    dW, out = _noalloc_step(w, Wd, mbs, gv, "micro_mean")
    _check_against_oracle(w, dW, out, "micro_mean")


def test_noalloc_rejects_oversize_and_misaligned():
    lib = M.load()
    cfg = M.Config(64, 100, 0, 0, -100, 0, 1, 0, 0)
    big = M.NOALLOC_MAX_N + 1
    dW = torch.zeros(100, 64, dtype=torch.float32, device="cuda")
    st = lib.lmce_microstep_noalloc(ctypes.byref(cfg), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                    ctypes.c_void_p(16), big, big, ctypes.c_void_p(16), M._ptr(dW), 0, None, None,
                                    None, M._stream(None))
    assert st == M.ERR_ARG
    h = torch.zeros(2 * 64 + 1, dtype=torch.bfloat16, device="cuda")
    st = lib.lmce_microstep_noalloc(ctypes.byref(cfg), ctypes.c_void_p(h.data_ptr() + 1), ctypes.c_void_p(16),
                                    ctypes.c_void_p(16), 2, 2, ctypes.c_void_p(16), M._ptr(dW), 0, None, None,
                                    None, M._stream(None))
    assert st == M.ERR_ARG
    torch.cuda.synchronize()
    assert float(dW.abs().max()) == 0.0


_FRESH = r"""
import ctypes, sys, torch
sys.path.insert(0, sys.argv[1])
from grad_lmce_microstep_gb300 import lmce as M
lib = M.load()
torch.cuda.set_device(0)
g = torch.Generator().manual_seed(2)
cases = []
for dt, C, V, N in (("fp32", 64, 65, 128), ("bf16", 256, 1000, 200)):
    tdt = M.TORCH_DTYPES[dt]
    h = torch.randn(N, C, generator=g).to(tdt).cuda()
    W = (0.02 * torch.randn(V, C, generator=g)).to(tdt).cuda()
    y = torch.randint(0, V, (N,), generator=g, dtype=torch.int32).cuda()
    cfg = M.Config(C, V, 0, M.DTYPES[dt], -100, 0, 1, 0, 0)
    cases.append((cfg, h, W, y, torch.empty_like(h), torch.empty(V, C, device="cuda"),
                  torch.zeros(1, dtype=torch.float64, device="cuda")))
torch.cuda.synchronize()
s = M._stream(None)
def call(c, n):
    cfg, h, W, y, dh, dW, ls = c
    return lib.lmce_microstep_noalloc(ctypes.byref(cfg), M._ptr(h), M._ptr(W), M._ptr(y), n, int(y.numel()),
                                      M._ptr(dh), M._ptr(dW), 0, None, M._ptr(ls), None, s)
assert call(cases[1], 0) == M.OK          # the first call: N == 0, bf16
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
for c in (cases[0], cases[1], cases[0]):   # fp32 first, then bf16, each with rows
    assert call(c, int(c[3].numel())) == M.OK
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
print("FREE", free0, free1, float(cases[0][6].item()), float(cases[1][6].item()))
"""


def test_noalloc_first_empty_call_then_both_dtypes_allocate_nothing():
    # In a fresh process: after a first call with N == 0, micro-steps of either dtype must not
    # change the device's free memory (no module load, no allocation).
    r = subprocess.run([sys.executable, "-c", _FRESH, ROOT], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("FREE")][-1].split()
    free0, free1 = int(line[1]), int(line[2])
    assert free1 == free0, f"free device memory moved from {free0} to {free1} bytes"
    assert np.isfinite(float(line[3])) and np.isfinite(float(line[4]))
