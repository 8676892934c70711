"""ln_f in front of the head (lmce_microstep_ln) vs the float64 oracle's step_ln.

The head consumes h = ln_f(x) rounded to the input dtype, and the oracle rounds its float64 h the
same way (round to nearest-even), so both heads see the same operands up to the rare element whose
rounding differs between a float32 and a float64 normalisation.  Tolerances are the head's: loss
relative 1e-3, gradients (dx, dgamma, dbeta, dW) max-abs 2e-2 x max|oracle| for bf16 inputs and
1e-5 x max|oracle| for fp32 inputs."""

import numpy as np
import pytest
import torch

from grad_lmce_microstep_gb300 import inputs as I
from grad_lmce_microstep_gb300 import lmce as M
from oracle import lmce_oracle as O

from gpu_util import GRAD_REL, LOSS_REL, max_rel_err

pytestmark = pytest.mark.gpu

TDT = {"bf16": torch.bfloat16, "fp32": torch.float32}


def _params(C, kind, seed):
    g = torch.Generator().manual_seed(seed)
    gamma = 1 + 0.1 * torch.randn(C, generator=g)
    beta = 0.1 * torch.randn(C, generator=g) if kind == "layernorm" else None
    return gamma, beta


def _xs(w):
    # the residual stream in front of ln_f: shifted and scaled rows, in the input dtype
    return [((h.float() * 1.7 + 0.4).to(TDT[w.dtype]), y) for h, y in w.micro]


def _run(w, xs, gamma, beta, kind, eps, path="auto", steps=1, compact=False, count_on_device=False):
    C, V = w.C, w.V
    W = w.W.cuda()
    dW = torch.empty(V, C, device="cuda")
    dgamma = torch.full((C,), 7.0, device="cuda")
    dbeta = torch.full((C,), 7.0, device="cuda") if beta is not None else None
    g, b = gamma.cuda(), (beta.cuda() if beta is not None else None)
    max_N = max(int(y.numel()) for _, y in xs)
    L = M.Lmce(C, V, max_N, dW, w.dtype, grad_accum_steps=len(xs), path=path, final_norm=True, compact=compact)
    gv = sum(w.valid_counts())
    for _ in range(steps):   # a later step writes the parameter gradients afresh, as dW
        dxs, rls = [], []
        for x, y in xs:
            xd, yd = x.cuda(), y.cuda()
            dx = torch.full_like(xd, 5.0)
            rl = torch.empty(yd.numel(), device="cuda")
            nv = (-1 if count_on_device else int(((y >= 0) & (y < V)).sum())) if compact else None
            L.microstep_ln(xd, g, b, W, yd, gv, dx, dgamma, dbeta, kind, eps, rl, n_valid=nv)
            dxs.append(dx)
            rls.append(rl)
        res = L.finalize()
    L.close()
    torch.cuda.synchronize()
    return dW, dxs, rls, dgamma, dbeta, res


def _check(w, xs, gamma, beta, kind, eps, got):
    dW, dxs, rls, dgamma, dbeta, (ls, cnt, mean) = got
    rnd = None
    if w.dtype == "bf16":
        def rnd(h):
            return torch.from_numpy(h).to(torch.bfloat16).double().numpy()
    ref = O.step_ln(xs, gamma.double().numpy(), None if beta is None else beta.double().numpy(), w.W, kind, eps,
                    h_round=rnd)
    tol = GRAD_REL[w.dtype]
    assert cnt == ref.head.count
    assert abs(mean - ref.head.objective) <= LOSS_REL * abs(ref.head.objective)
    assert abs(ls - ref.head.loss_sum) <= LOSS_REL * abs(ref.head.loss_sum)
    assert max_rel_err(dW.double().cpu().numpy(), ref.head.dW) <= tol
    for k, m in enumerate(ref.head.micro):
        assert max_rel_err(dxs[k].double().cpu().numpy(), ref.dx[k]) <= tol, k
        d = np.abs(rls[k].double().cpu().numpy() - m.row_loss)
        assert float(d.max()) <= LOSS_REL * max(1.0, float(np.abs(m.row_loss).max()))
    assert max_rel_err(dgamma.double().cpu().numpy(), ref.dgamma) <= tol
    if beta is not None:
        assert max_rel_err(dbeta.double().cpu().numpy(), ref.dbeta) <= tol


@pytest.mark.parametrize("path", ["simt", "tcgen05", "tcgen05_two_pass"])
@pytest.mark.parametrize("kind", ["layernorm", "rmsnorm"])
def test_ln_bf16_matches_oracle(path, kind):
    # ragged micro-steps over several tiles, ignored targets; the second step checks that the
    # parameter gradients are written afresh after finalize
    w = I.custom([300, 173], 256, 1000, "bf16", seed=41, ignore_frac=0.1)
    xs = _xs(w)
    gamma, beta = _params(w.C, kind, 41)
    got = _run(w, xs, gamma, beta, kind, 1e-5, path=path, steps=2)
    _check(w, xs, gamma, beta, kind, 1e-5, got)


@pytest.mark.parametrize("kind", ["layernorm", "rmsnorm"])
def test_ln_fp32_char_level(kind):
    w = I.tiny_char()
    xs = _xs(w)
    gamma, beta = _params(w.C, kind, 42)
    _check(w, xs, gamma, beta, kind, 1e-6, _run(w, xs, gamma, beta, kind, 1e-6))


@pytest.mark.parametrize("C,dtype", [(67, "fp32"), (2048, "bf16"), (768, "bf16"), (1024, "bf16"), (520, "fp32")])
def test_ln_widths(C, dtype):
    # the register layout with 3 and 4 words per lane (768, 1024 bf16) and a partial last word
    # group (520 floats), and the row loop for rows that do not fit it: 67 floats (not a multiple
    # of 4), 2048 bf16 (wider than 6 words per lane)
    w = I.custom([96, 33], C, 301, dtype, seed=43, ignore_frac=0.1)
    xs = _xs(w)
    gamma, beta = _params(C, "layernorm", 43)
    _check(w, xs, gamma, beta, "layernorm", 1e-5, _run(w, xs, gamma, beta, "layernorm", 1e-5))


@pytest.mark.parametrize("path", ["simt", "tcgen05"])
@pytest.mark.parametrize("kind", ["layernorm", "rmsnorm"])
def test_ln_compact_masked_tails(path, kind):
    # ln_f over the valid rows only: masked sequence tails and scattered ignored targets; dx of an
    # ignored row is exactly zero, everything else matches the oracle's step_ln over all rows
    T = 128
    w = I.custom([3 * T] * 3, 256, 1000, "bf16", seed=45, ignore_frac=0.05)
    for k, tail in enumerate((0, T // 2, 3 * T // 4)):
        if tail:
            w.micro[k][1].view(3, T)[:, T - tail:] = I.IGNORE_ID
    xs = _xs(w)
    gamma, beta = _params(w.C, kind, 45)
    got = _run(w, xs, gamma, beta, kind, 1e-5, path=path, steps=2, compact=True)
    _check(w, xs, gamma, beta, kind, 1e-5, got)
    for (_, y), dx in zip(xs, got[1]):
        ign = ~((y >= 0) & (y < w.V))
        assert float(dx.cpu()[ign].abs().max()) == 0.0


@pytest.mark.parametrize("C,dtype", [(768, "bf16"), (1024, "bf16"), (520, "fp32"), (67, "fp32"), (2048, "bf16")])
def test_ln_compact_widths(C, dtype):
    # ln_f fused with the compaction for rows that fit its register layout (768 and 1024 bf16, 520
    # floats), the gather / separate ln_f / scatter sequence for rows that do not (67 floats, 2048
    # bf16); ragged micro-steps (N not a multiple of 32) with a whole 32-row block ignored
    w = I.custom([96, 45], C, 301, dtype, seed=47, ignore_frac=0.3)
    w.micro[0][1][32:64] = I.IGNORE_ID
    xs = _xs(w)
    gamma, beta = _params(C, "layernorm", 47)
    got = _run(w, xs, gamma, beta, "layernorm", 1e-5, steps=2, compact=True)
    _check(w, xs, gamma, beta, "layernorm", 1e-5, got)
    for (_, y), dx in zip(xs, got[1]):
        ign = ~((y >= 0) & (y < w.V))
        assert float(dx.cpu()[ign].abs().max()) == 0.0


@pytest.mark.parametrize("kind", ["layernorm", "rmsnorm"])
def test_ln_compact_count_on_device_and_empty_micro_step(kind):
    # n_valid = -1: the library reads the valid count back; the second micro-step has no valid
    # target at all (its dx is zero and it adds nothing to dgamma / dbeta)
    w = I.custom([200, 77], 256, 1000, "bf16", seed=48, ignore_frac=0.2)
    w.micro[1][1][:] = I.IGNORE_ID
    xs = _xs(w)
    gamma, beta = _params(w.C, kind, 48)
    got = _run(w, xs, gamma, beta, kind, 1e-5, steps=2, compact=True, count_on_device=True)
    _check(w, xs, gamma, beta, kind, 1e-5, got)
    assert float(got[1][1].abs().max()) == 0.0


def test_ln_compact_bitwise_reproducible():
    w = I.custom([300, 173], 768, 1000, "bf16", seed=49, ignore_frac=0.4)
    xs = _xs(w)
    gamma, beta = _params(w.C, "layernorm", 49)
    a = _run(w, xs, gamma, beta, "layernorm", 1e-5, path="tcgen05", compact=True)
    b = _run(w, xs, gamma, beta, "layernorm", 1e-5, path="tcgen05", compact=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])
    for x, y in zip(a[1], b[1]):
        assert torch.equal(x, y)
    for x, y in zip(a[2], b[2]):
        assert torch.equal(x, y)
    assert a[5] == b[5]


def test_ln_argument_errors_and_no_valid():
    w = I.custom([64], 256, 1000, "bf16", seed=44, ignore_frac=1.0)
    (x, y), = _xs(w)
    x, y, W = x.cuda(), y.cuda(), w.W.cuda()
    C = w.C
    gamma, beta = (t.cuda() for t in _params(C, "layernorm", 44))
    dW = torch.empty(w.V, C, device="cuda")
    dgamma = torch.full((C,), 3.0, device="cuda")
    L = M.Lmce(C, w.V, 64, dW, "bf16")
    assert L.microstep_ln(x, gamma, beta, W, y, 1, torch.empty_like(x), dgamma, None, check=False) == M.ERR_ARG
    L.close()
    L = M.Lmce(C, w.V, 64, dW, "bf16", final_norm=True)
    dx = torch.full_like(x, 2.0)
    assert L.microstep_ln(x, gamma, beta, W, y, 1, dx, dgamma, None, kind="rmsnorm", check=False) == M.ERR_ARG
    assert L.microstep_ln(x, gamma, beta, W, y, 1, dx, dgamma, None, eps=-1.0, check=False) == M.ERR_ARG
    # global normalisation with no valid target: refused, dx zeroed, dgamma untouched
    assert L.microstep_ln(x, gamma, beta, W, y, 0, dx, dgamma, None, check=False) == M.ERR_NO_VALID
    torch.cuda.synchronize()
    assert float(dx.abs().max()) == 0.0 and float(dgamma.min()) == 3.0
    L.close()


def test_ln_bitwise_reproducible():
    # the parameter-gradient partials are summed in a fixed order: two runs agree bit for bit
    w = I.custom([300, 173], 256, 1000, "bf16", seed=46, ignore_frac=0.1)
    xs = _xs(w)
    gamma, beta = _params(w.C, "layernorm", 46)
    a = _run(w, xs, gamma, beta, "layernorm", 1e-5, path="tcgen05")
    b = _run(w, xs, gamma, beta, "layernorm", 1e-5, path="tcgen05")
    assert torch.equal(a[0], b[0]) and torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])
    for x, y in zip(a[1], b[1]):
        assert torch.equal(x, y)
    assert a[5] == b[5]
