"""Helpers for the GPU parity tests: run the library through its C-ABI binding and
compare with the float64 oracle on the same seeded inputs."""

import numpy as np
import torch

from grad_lmce_microstep_gb300 import lmce as M
from oracle import lmce_oracle as O

# Tolerances stated for the method: loss relative error <= 1e-3; dh and dW max absolute
# error <= 2e-2 * max|oracle| for bf16 inputs and <= 1e-5 * max|oracle| for fp32 inputs.
LOSS_REL = 1e-3
GRAD_REL = {"bf16": 2e-2, "fp32": 1e-5}


def to_dev(w, device="cuda"):
    W = w.W.to(device)
    mbs = [(h.to(device), y.to(device)) for h, y in w.micro]
    return W, mbs


def run_lib(w, path="auto", norm="global", row_loss=True, global_valid=None, compact=False):
    W, mbs = to_dev(w)
    dW, dhs, rls, res = M.run_step(W, mbs, w.dtype, norm=norm, path=path, row_loss=row_loss,
                                   global_valid=global_valid, compact=compact)
    torch.cuda.synchronize()
    return {
        "dW": dW.double().cpu().numpy(),
        "dh": [d.double().cpu().numpy() for d in dhs],
        "row_loss": [None if r is None else r.double().cpu().numpy() for r in rls],
        "loss_sum": res[0], "count": res[1], "loss_mean": res[2], "status": res[3],
    }


def run_oracle(w, norm="global"):
    return O.step([(h, y) for h, y in w.micro], w.W, norm=norm, ignore_id=w.ignore_id)


def max_rel_err(got, want):
    scale = float(np.abs(want).max())
    err = float(np.abs(got - want).max())
    return err / scale if scale > 0 else err


def assert_parity(got, ref, dtype):
    tol = GRAD_REL[dtype]
    assert got["count"] == ref.count
    assert abs(got["loss_sum"] - ref.loss_sum) <= LOSS_REL * abs(ref.loss_sum)
    assert abs(got["loss_mean"] - ref.objective) <= LOSS_REL * abs(ref.objective)
    e = max_rel_err(got["dW"], ref.dW)
    assert e <= tol, f"dW max err {e:.3e} > {tol:.1e} x max|oracle|"
    for k, m in enumerate(ref.micro):
        e = max_rel_err(got["dh"][k], m.dh)
        assert e <= tol, f"dh[{k}] max err {e:.3e} > {tol:.1e} x max|oracle|"
        if got["row_loss"][k] is not None:
            d = np.abs(got["row_loss"][k] - m.row_loss)
            assert float(d.max()) <= LOSS_REL * max(1.0, float(np.abs(m.row_loss).max()))
