"""A bounded device wait that runs out, on the GPU, without faulting or hanging it.

Every mbarrier wait of the tensor-core gradient kernels is bounded.  The test hook
lmce_test_stall_next_microstep makes the next micro-step's gradient launches start no
operand load and bounds their waits by 1 ms, so the real timeout path runs: the wait
records a timeout bit, the MMA warp waits for what it issued, tensor memory is released,
the kernel returns, and lmce_finalize reports LMCE_ERR_CUDA.  The context stays usable: a
fresh handle's next step is clean and matches the oracle.
"""

import pytest
import torch

from grad_lmce_microstep_gb300 import inputs as I
from grad_lmce_microstep_gb300 import lmce as M

from gpu_util import assert_parity, run_lib, run_oracle, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("path", ["tcgen05", "tcgen05_two_pass"])
def test_wait_that_runs_out_is_reported_and_the_context_survives(path):
    w = I.custom([300, 213], 256, 1000, "bf16", seed=17, ignore_frac=0.1)
    W, mbs = to_dev(w)
    gv = sum(w.valid_counts())
    dW = torch.empty(w.V, w.C, dtype=torch.float32, device="cuda")
    L = M.Lmce(w.C, w.V, 300, dW, "bf16", grad_accum_steps=2, path=path)
    try:
        assert L.test_stall_next_microstep(0) == M.ERR_ARG
        assert L.test_stall_next_microstep(1_000_000) == M.OK
        for h, y in mbs:
            dh = torch.empty_like(h)
            L.microstep(h, W, y, gv, dh)
        *_, st = L.finalize(check=False)
        assert st == M.ERR_CUDA, M.status_string(st)
        torch.cuda.synchronize()   # no sticky error: the kernels returned
        # the hook disarmed itself: the same handle's next step is clean
        for h, y in mbs:
            L.microstep(h, W, y, gv, torch.empty_like(h))
        *_, st = L.finalize(check=False)
        assert st == M.OK, M.status_string(st)
    finally:
        L.close()
    got = run_lib(w, path=path)   # a fresh handle
    assert got["status"] == M.OK
    assert_parity(got, run_oracle(w), "bf16")


def test_stall_hook_needs_the_tensor_core_path():
    w = I.tiny_char()
    dW = torch.empty(w.V, w.C, dtype=torch.float32, device="cuda")
    L = M.Lmce(w.C, w.V, 128, dW, "fp32", path="simt")
    try:
        assert L.test_stall_next_microstep(1_000_000) == M.ERR_STATE
    finally:
        L.close()
