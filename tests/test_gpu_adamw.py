"""The fused AdamW update on the tied matrix vs the float64 oracle, element by element.

The update runs in float32 on the GPU; the oracle takes the same float32 inputs to float64.
Per element the kernel rounds a handful of times, so p, m and v agree to a few float32 ulps:
the tolerances below are 1e-6 relative with an absolute floor of 1e-7 of the largest value.
W_out is the bf16 round-to-nearest-even of the kernel's own p, bit for bit, and within one
bf16 ulp of the oracle's p.
"""

import numpy as np
import pytest
import torch

from grad_lmce_microstep_gb300 import inputs as I
from grad_lmce_microstep_gb300 import lmce as M
from oracle import lmce_oracle as O

from gpu_util import to_dev

pytestmark = pytest.mark.gpu

RTOL = 1e-6
LR, BETAS, EPS, WD = 6e-4, (0.9, 0.95), 1e-8, 0.1


def _state(V, C, seed, gscale=1e-3):
    """Seeded master weights, moments of a few earlier steps and a gradient, all float32."""
    rng = np.random.default_rng(seed)
    p = (rng.standard_normal((V, C)) * 0.02).astype(np.float32)
    g = (rng.standard_normal((V, C)) * gscale).astype(np.float32)
    m = (rng.standard_normal((V, C)) * gscale * 0.5).astype(np.float32)
    v = ((rng.standard_normal((V, C)) * gscale) ** 2).astype(np.float32)
    g[0, :3] = 0.0
    return p, m, v, g


def _close(got, want, name):
    got = got.detach().double().cpu().numpy()
    np.testing.assert_allclose(got, want, rtol=RTOL, atol=1e-7 * np.abs(want).max(), err_msg=name)


def _check_wout(W_out, p_dev, p_ref):
    # bit-exact against torch's round-to-nearest-even of the kernel's p; one ulp of the oracle's
    assert torch.equal(W_out, p_dev.to(torch.bfloat16))
    w = W_out.double().cpu().numpy()
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(p_ref), 1e-30))) - 7)
    assert np.all(np.abs(w - p_ref) <= ulp)


def _dev(*xs, offset=0):
    """Copies on the GPU; offset=1 places each one float past a 16-byte boundary."""
    out = []
    for x in xs:
        buf = torch.empty(x.size + offset, dtype=torch.float32, device="cuda")
        t = buf[offset:].view(x.shape)
        t.copy_(torch.from_numpy(x))
        out.append(t)
    return out


@pytest.mark.parametrize("shape,offset", [((1000, 256), 0), ((301, 67), 0), ((301, 67), 1)])
def test_adamw_update_matches_oracle(shape, offset):
    # vector path, a ragged V*C (odd, not a multiple of four) and the unaligned scalar path
    V, C = shape
    p, m, v, g = _state(V, C, seed=21)
    dW, pd, md, vd = _dev(g, p, m, v, offset=offset)
    wb = torch.empty(V * C + offset, dtype=torch.bfloat16, device="cuda")
    W_out = wb[offset:].view(V, C)
    L = M.Lmce(C, V, 1, dW, "fp32" if C % 8 else "bf16")
    clip = O.clip_coef(O.dw_sumsq(g), 0.05)
    assert clip < 1.0
    L.adamw(pd, md, vd, 7, LR, W_out, BETAS, EPS, WD, clip)
    torch.cuda.synchronize()
    L.close()
    rp, rm, rv = O.adamw_step(p, m, v, g, 7, LR, BETAS, EPS, WD, clip)
    _close(pd, rp, "p")
    _close(md, rm, "m")
    _close(vd, rv, "v")
    _check_wout(W_out, pd, rp)
    assert float(dW.double().cpu().sub(torch.from_numpy(g).double()).abs().max()) == 0.0   # dW is read only


def test_adamw_first_step_from_zero_moments_no_wout():
    V, C = 512, 128
    p, _, _, g = _state(V, C, seed=22)
    z = np.zeros((V, C), np.float32)
    dW, pd, md, vd = _dev(g, p, z, z)
    L = M.Lmce(C, V, 1, dW, "bf16")
    L.adamw(pd, md, vd, 1, LR, None, BETAS, EPS, WD, 1.0)
    torch.cuda.synchronize()
    L.close()
    rp, rm, rv = O.adamw_step(p, z, z, g, 1, LR, BETAS, EPS, WD, 1.0)
    _close(pd, rp, "p")
    _close(md, rm, "m")
    _close(vd, rv, "v")


def test_adamw_three_steps_after_real_gradients():
    # three optimizer steps of the whole path: micro-steps, finalize, the clip norm, AdamW; each
    # step's update is compared with the oracle's update on the same float32 state and gradient
    w = I.custom([300, 173], 256, 1000, "bf16", seed=23, ignore_frac=0.1)
    W, mbs = to_dev(w)
    V, C = w.V, w.C
    dW = torch.empty(V, C, device="cuda")
    p = W.float().clone()
    m = torch.zeros_like(p)
    v = torch.zeros_like(p)
    W_cur = W.clone()
    L = M.Lmce(C, V, 300, dW, "bf16", grad_accum_steps=len(mbs))
    gv = sum(int(((y >= 0) & (y < V)).sum()) for _, y in mbs)
    for t in (1, 2, 3):
        for h, y in mbs:
            L.microstep(h, W_cur, y, gv, torch.empty_like(h))
        L.finalize()
        clip = O.clip_coef(L.dw_sumsq(), 1.0)
        before = [x.double().cpu().numpy() for x in (p, m, v, dW)]
        L.adamw(p, m, v, t, LR, W_cur, BETAS, EPS, WD, clip)
        torch.cuda.synchronize()
        rp, rm, rv = O.adamw_step(*before, t, LR, BETAS, EPS, WD, clip)
        _close(p, rp, f"p step {t}")
        _close(m, rm, f"m step {t}")
        _close(v, rv, f"v step {t}")
        _check_wout(W_cur, p, rp)
    L.close()


def test_adamw_argument_errors():
    V, C = 64, 64
    dW = torch.zeros(V, C, device="cuda")
    p, m, v = (torch.zeros(V, C, device="cuda") for _ in range(3))
    L = M.Lmce(C, V, 1, dW, "bf16")
    lib, hd = L.lib, L.handle
    P = [M._ptr(x) for x in (p, m, v)]
    st = M._stream(None)
    ok = (1, 1e-3, 0.9, 0.95, 1e-8, 0.1, 1.0)
    assert lib.lmce_adamw(hd, *P, None, *ok, st) == M.OK
    for i, bad in ((0, 0), (0, -1), (2, 1.0), (3, 1.0), (2, -0.1), (4, -1e-8), (4, float("nan")),
                   (1, float("inf")), (5, float("nan")), (6, float("inf"))):
        a = list(ok)
        a[i] = bad
        assert lib.lmce_adamw(hd, *P, None, *a, st) == M.ERR_ARG, (i, bad)
    assert lib.lmce_adamw(hd, None, P[1], P[2], None, *ok, st) == M.ERR_ARG
    torch.cuda.synchronize()
    L.close()
