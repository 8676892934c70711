"""The debug build's device bounds checks (liblmce_dbg.so, LMCE_DEBUG_BOUNDS=1) on the GPU.

Every kernel of the debug build checks the indices it computes before the accesses they guard
and reports a failed check in the step's error word (lmce_finalize: LMCE_ERR_INTERNAL) instead
of trapping.  Clean runs over ragged shapes, split tiles, the compaction and ln_f must report
nothing and match the oracle; a full-size micro-step of the GPT-2 124M head must equal the
release build's bit for bit (the checks change no arithmetic); and the compaction's check,
given a smaller buffer than it has by the test hook, must report without reading or writing
outside the real buffers.

The binding loads one library per process, so each part runs in a child process."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")

PRELUDE = r"""
import json, os, sys
sys.path.insert(0, __ROOT__)
sys.path.insert(0, __TESTS__)
import torch
from grad_lmce_microstep_gb300 import build as B
from grad_lmce_microstep_gb300 import inputs as I
from grad_lmce_microstep_gb300 import lmce as M
if __DBG__:
    if not os.path.exists(M.DEBUG_LIB_PATH):
        B.build(debug_bounds=True)
    M.load(M.DEBUG_LIB_PATH)
else:
    M.load()
assert M._lib.lmce_debug_bounds() == (1 if __DBG__ else 0)
"""

CLEAN = r"""
from gpu_util import assert_parity, run_lib, run_oracle
cases = [
    (I.custom([300, 213], 256, 1000, "bf16", seed=61, ignore_frac=0.1), dict()),
    (I.custom([300, 213], 256, 1000, "bf16", seed=61, ignore_frac=0.1), dict(norm="micro_mean")),
    (I.custom([520, 130], 768, 3001, "bf16", seed=62, ignore_frac=0.2), dict()),
    (I.custom([520, 130], 768, 3001, "bf16", seed=62, ignore_frac=0.3), dict(compact=True)),
    (I.custom([200, 77], 1024, 1500, "bf16", seed=63, ignore_frac=0.1), dict(path="tcgen05_two_pass")),
    (I.tiny_char(), dict()),
]
for w, kw in cases:
    got = run_lib(w, **kw)
    assert got["status"] == M.OK, (kw, M.status_string(got["status"]))
    assert_parity(got, run_oracle(w, norm=kw.get("norm", "global")), w.dtype)
# ln_f fused with the compaction
from oracle import lmce_oracle as O
import numpy as np
w = I.custom([300, 173], 768, 1000, "bf16", seed=64, ignore_frac=0.4)
xs = [((h.float() * 1.7 + 0.4).to(torch.bfloat16), y) for h, y in w.micro]
g = torch.Generator().manual_seed(64)
gamma, beta = 1 + 0.1 * torch.randn(w.C, generator=g), 0.1 * torch.randn(w.C, generator=g)
dW = torch.empty(w.V, w.C, device="cuda")
dgamma, dbeta = torch.empty(w.C, device="cuda"), torch.empty(w.C, device="cuda")
L = M.Lmce(w.C, w.V, 300, dW, "bf16", grad_accum_steps=2, compact=True, final_norm=True)
gv = sum(w.valid_counts())
for (x, y), nv in zip(xs, w.valid_counts()):
    L.microstep_ln(x.cuda(), gamma.cuda(), beta.cuda(), w.W.cuda(), y.cuda(), gv, torch.empty_like(x.cuda()),
                   dgamma, dbeta, n_valid=nv)
ls, cnt, mean, st = L.finalize(check=False)
L.close()
assert st == M.OK, M.status_string(st)
rnd = lambda h: torch.from_numpy(h).to(torch.bfloat16).double().numpy()
ref = O.step_ln(xs, gamma.double().numpy(), beta.double().numpy(), w.W, "layernorm", 1e-5, h_round=rnd)
assert cnt == ref.head.count and abs(mean - ref.head.objective) <= 1e-3 * abs(ref.head.objective)
print("RESULT ok")
"""

FULL = r"""
w = I.make("gpt2_124m_head")
W = w.W.cuda()
h, y = w.micro[0]
dW = torch.empty(w.V, w.C, device="cuda")
dh = torch.empty_like(h.cuda())
L = M.Lmce(w.C, w.V, h.shape[0], dW, "bf16", grad_accum_steps=1)
L.microstep(h.cuda(), W, y.cuda(), int(y.numel()), dh)
ls, cnt, mean, st = L.finalize(check=False)
L.close()
torch.cuda.synchronize()
print("RESULT " + json.dumps({"status": st, "loss": ls, "dW": int(dW.view(torch.int32).long().sum()),
                              "dW2": float(dW.double().pow(2).sum()), "dh": int(dh.view(torch.int16).long().sum())}))
"""

HOOK = r"""
from gpu_util import assert_parity, run_oracle
w = I.custom([384, 256], 256, 1000, "bf16", seed=65, ignore_frac=0.3)
W = w.W.cuda()
mbs = [(h.cuda(), y.cuda()) for h, y in w.micro]
dW = torch.empty(w.V, w.C, device="cuda")
L = M.Lmce(w.C, w.V, 384, dW, "bf16", grad_accum_steps=2, compact=True)
gv = sum(w.valid_counts())
assert L.test_bounds_limit(385) == M.ERR_ARG
# the checks see 10 compact rows: the positions past them are reported and skipped
assert L.test_bounds_limit(10) == M.OK
for (h, y), nv in zip(mbs, w.valid_counts()):
    L.microstep_compact(h, W, y, nv, gv, torch.empty_like(h))
*_, st = L.finalize(check=False)
assert st == M.ERR_INTERNAL, M.status_string(st)
# restored: the next step is clean and matches the oracle
assert L.test_bounds_limit(384) == M.OK
dhs, rls = [], []
for (h, y), nv in zip(mbs, w.valid_counts()):
    dh = torch.empty_like(h)
    rl = torch.empty(y.numel(), device="cuda")
    L.microstep_compact(h, W, y, nv, gv, dh, row_loss=rl)
    dhs.append(dh)
    rls.append(rl)
ls, cnt, mean, st = L.finalize(check=False)
L.close()
assert st == M.OK, M.status_string(st)
got = {"dW": dW.double().cpu().numpy(), "dh": [d.double().cpu().numpy() for d in dhs],
       "row_loss": [r.double().cpu().numpy() for r in rls], "loss_sum": ls, "count": cnt, "loss_mean": mean}
assert_parity(got, run_oracle(w), "bf16")
print("RESULT ok")
"""


def _child(body: str, debug: bool, timeout: int = 900) -> str:
    code = PRELUDE.replace("__ROOT__", repr(ROOT)).replace("__TESTS__", repr(TESTS)).replace("__DBG__", repr(debug)) + body
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=timeout)
    assert p.returncode == 0, (p.stdout[-3000:], p.stderr[-3000:])
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("RESULT ")]
    assert lines, p.stdout[-2000:]
    return lines[-1][7:]


def test_debug_build_clean_runs_match_the_oracle():
    assert _child(CLEAN, True) == "ok"


def test_debug_build_full_size_equals_the_release_build():
    dbg = json.loads(_child(FULL, True))
    rel = json.loads(_child(FULL, False))
    assert dbg["status"] == 0 and rel["status"] == 0
    assert dbg == rel


def test_debug_build_reports_a_failed_check_without_trapping():
    assert _child(HOOK, True) == "ok"
