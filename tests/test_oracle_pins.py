"""Pins of the float64 oracle to facts fixed by the pages and by mathematics.

Each test names the plausible oracle mistake it would catch.  None of them
re-types the oracle's own formula: they use closed forms, printed worked
examples, finite differences, PyTorch's own cross-entropy under autograd, and
brute force in plain Python.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import lmce_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def _problem(Ns, C, V, ignore=(), bad=(), seed=0, wstd=0.5):
    rng = np.random.default_rng(seed)
    W = rng.normal(0, wstd, (V, C))
    mbs = []
    for k, N in enumerate(Ns):
        h = rng.normal(0, 1, (N, C))
        y = rng.integers(0, V, N)
        for (kk, n) in ignore:
            if kk == k:
                y[n] = O.IGNORE_ID
        for (kk, n, val) in bad:
            if kk == k:
                y[n] = val
        mbs.append((h, y))
    return W, mbs


# --- GPT-2 page, section 7: uniform logits give loss log V -------------------------------

def test_uniform_loss_matches_printed_value():
    g = json.load(open(os.path.join(GOLDEN, "uniform_loss.json")))
    V = g["V"]
    h = RNG.normal(0, 1, (3, 8))
    W = np.zeros((V, 8))
    y = np.array([0, 17, V - 1])
    r = O.step([(h, y)], W)
    assert abs(r.objective - g["loss_printed"]) < 0.5 * 10 ** -g["printed_decimals"]
    assert abs(r.objective - math.log(V)) < 1e-12


@pytest.mark.parametrize("V", [11, 65, 50304])
def test_uniform_loss_is_log_V_for_zero_hidden(V):
    # h = 0 makes every logit 0 whatever W is (catches a dropped max shift or a wrong log base)
    W = RNG.normal(0, 0.02, (V, 16))
    h = np.zeros((4, 16))
    y = np.array([0, 1, 2, 3])
    r = O.step([(h, y)], W)
    assert r.loss_sum == pytest.approx(4 * math.log(V), rel=1e-14)
    assert r.objective == pytest.approx(math.log(V), rel=1e-14)


def test_closed_form_zero_weight():
    # W = 0: softmax is uniform, so dW[v] = s * sum_n (1/V - [y_n = v]) h_n, dh = 0.
    N, C, V = 9, 5, 7
    h = RNG.normal(0, 1, (N, C))
    y = RNG.integers(0, V, N)
    y[3] = O.IGNORE_ID
    r = O.step([(h, y)], np.zeros((V, C)))
    s = 1.0 / (N - 1)
    expect = np.zeros((V, C))
    for n in range(N):
        if y[n] == O.IGNORE_ID:
            continue
        for v in range(V):
            expect[v] += s * ((1.0 / V) - (1.0 if v == y[n] else 0.0)) * h[n]
    assert np.abs(r.dW - expect).max() < 1e-15
    assert np.abs(r.micro[0].dh).max() == 0.0


def test_closed_form_zero_hidden():
    # h = 0: softmax is uniform, so dh_n = s * (mean_v W_v - W_{y_n}); dW = 0.
    N, C, V = 6, 4, 9
    W = RNG.normal(0, 1, (V, C))
    y = RNG.integers(0, V, N)
    r = O.step([(np.zeros((N, C)), y)], W)
    s = 1.0 / N
    for n in range(N):
        want = s * (W.sum(axis=0) / V - W[y[n]])
        assert np.abs(r.micro[0].dh[n] - want).max() < 1e-15
    assert np.abs(r.dW).max() == 0.0


# --- Gradients: finite differences and PyTorch autograd -----------------------------------

@pytest.mark.parametrize("norm", ["global", "micro_mean"])
def test_finite_differences(norm):
    # Catches a dropped one-hot term, a sign error, a transposed product or a missing scale.
    C, V = 8, 11
    W, mbs = _problem([5, 7], C, V, ignore=[(1, 2)], seed=3)
    r = O.step(mbs, W, norm=norm)

    def J(Wx, mbx):
        return O.step(mbx, Wx, norm=norm, want_dW=False).objective

    eps = 1e-6
    num_dW = np.zeros_like(W)
    for v in range(V):
        for c in range(C):
            Wp = W.copy(); Wp[v, c] += eps
            Wm = W.copy(); Wm[v, c] -= eps
            num_dW[v, c] = (J(Wp, mbs) - J(Wm, mbs)) / (2 * eps)
    assert np.abs(num_dW - r.dW).max() <= 1e-6 * max(1.0, np.abs(r.dW).max())
    for k, (h, y) in enumerate(mbs):
        num_dh = np.zeros_like(h)
        for n in range(h.shape[0]):
            for c in range(C):
                hp = h.copy(); hp[n, c] += eps
                hm = h.copy(); hm[n, c] -= eps
                mp = list(mbs); mp[k] = (hp, y)
                mm = list(mbs); mm[k] = (hm, y)
                num_dh[n, c] = (J(W, mp) - J(W, mm)) / (2 * eps)
        assert np.abs(num_dh - r.micro[k].dh).max() <= 1e-6 * max(1.0, np.abs(r.micro[k].dh).max())


@pytest.mark.parametrize("shape", [(64, 65, (64, 64)), (8, 11, (40, 24))])
@pytest.mark.parametrize("norm", ["global", "micro_mean"])
def test_torch_cross_entropy_autograd(shape, norm):
    # PyTorch's cross_entropy with ignore_index=-100 under float64 autograd is the library
    # special case of the same definition.
    C, V, Ns = shape
    W, mbs = _problem(list(Ns), C, V, ignore=[(0, 1), (1, 5)], seed=11, wstd=0.3)
    r = O.step(mbs, W, norm=norm)
    Wt = torch.tensor(W, requires_grad=True)
    counts = [int((y != O.IGNORE_ID).sum()) for _, y in mbs]
    G = len(mbs)
    total = 0.0
    hts = []
    for (h, y), c in zip(mbs, counts):
        ht = torch.tensor(h, requires_grad=True)
        hts.append(ht)
        ce = torch.nn.functional.cross_entropy(ht @ Wt.T, torch.tensor(y), ignore_index=-100,
                                               reduction="sum")
        s = 1.0 / sum(counts) if norm == "global" else 1.0 / (c * G)
        total = total + s * ce
    total.backward()
    assert abs(total.item() - r.objective) < 1e-12 * max(1, abs(r.objective))
    assert np.abs(Wt.grad.numpy() - r.dW).max() < 1e-12
    for ht, m in zip(hts, r.micro):
        assert np.abs(ht.grad.numpy() - m.dh).max() < 1e-12


def test_brute_force_tiny():
    # Plain-Python loops with math.exp / math.log on a 3 x 4 problem.
    h = [[0.5, -1.0], [2.0, 0.25], [-0.75, 1.5]]
    W = [[1.0, 0.0], [0.0, 1.0], [-1.0, 0.5], [0.3, -0.2]]
    y = [2, 0, -100]
    V = 4
    tot = 0.0
    for n in range(3):
        z = [sum(h[n][c] * W[v][c] for c in range(2)) for v in range(V)]
        if y[n] == -100:
            continue
        tot += math.log(sum(math.exp(zz) for zz in z)) - z[y[n]]
    r = O.step([(np.array(h), np.array(y))], np.array(W))
    assert r.loss_sum == pytest.approx(tot, rel=1e-14)
    assert r.count == 2
    assert r.objective == pytest.approx(tot / 2, rel=1e-14)


# --- Multi-GPU page: worked examples for micro-step and rank averaging ---------------------

def _two_class_rows(losses):
    """Rows of a V=2, C=1 problem whose cross-entropy losses are exactly ``losses``.

    With W = [[1], [0]], h_n = d_n and target 1, z_n = (d_n, 0) and the loss is
    log(1 + exp(d_n)); d_n = log(exp(L) - 1) gives loss L.
    """
    d = np.array([math.log(math.exp(L) - 1.0) for L in losses])
    return d[:, None], np.ones(len(losses), dtype=np.int64)


W2 = np.array([[1.0], [0.0]])


def test_p5_single_gpu_example():
    g = json.load(open(os.path.join(GOLDEN, "p5_worked_examples.json")))["single_gpu"]
    mbs = [_two_class_rows(l) for l in g["token_losses_per_micro_step"]]
    mm = O.step(mbs, W2, norm="micro_mean")
    for m, want in zip(mm.micro, g["micro_step_means"]):
        assert m.loss_sum / m.count == pytest.approx(want, rel=1e-12)
    assert mm.objective == pytest.approx(g["accumulated_objective"], rel=1e-12)
    whole = O.step([(np.concatenate([h for h, _ in mbs]), np.concatenate([y for _, y in mbs]))], W2)
    assert whole.objective == pytest.approx(g["whole_batch_mean"], rel=1e-12)
    # equal valid counts: the gradients of both objectives agree too
    assert np.abs(mm.dW - whole.dW).max() < 1e-14
    glob = O.step(mbs, W2, norm="global")
    assert np.abs(glob.dW - whole.dW).max() < 1e-14


def test_p5_two_gpu_example():
    g = json.load(open(os.path.join(GOLDEN, "p5_worked_examples.json")))["two_gpu"]
    ranks = [[_two_class_rows(l) for l in rk] for rk in g["rank_token_losses_per_micro_step"]]
    objs = [O.step(rk, W2, norm="micro_mean").objective for rk in ranks]
    assert objs == pytest.approx(g["rank_objectives"], rel=1e-12)
    assert sum(objs) / len(objs) == pytest.approx(g["ddp_average"], rel=1e-12)
    assert sum(objs) / len(objs) / 2 == pytest.approx(g["divided_by_world_size_again"], rel=1e-12)
    # token-weighted global normalisation with the count summed over ranks, reduced by SUM
    gv = sum(O.count_valid(y, 2) for rk in ranks for _, y in rk)
    summed = sum(O.step(rk, W2, norm="global", global_valid=gv).objective for rk in ranks)
    assert summed == pytest.approx(g["whole_batch_mean"], rel=1e-12)


# --- Accumulation: equal and unequal valid counts -----------------------------------------

def test_equal_split_matches_single_batch():
    C, V = 6, 13
    W, mbs = _problem([8, 8, 8], C, V, seed=5)
    whole = O.step([(np.concatenate([h for h, _ in mbs]), np.concatenate([y for _, y in mbs]))], W)
    for norm in ("global", "micro_mean"):
        r = O.step(mbs, W, norm=norm)
        assert r.objective == pytest.approx(whole.objective, rel=1e-13)
        assert np.abs(r.dW - whole.dW).max() < 1e-14
        dh = np.concatenate([m.dh for m in r.micro])
        assert np.abs(dh - whole.micro[0].dh).max() < 1e-15


def test_unequal_split_global_is_token_weighted():
    C, V = 6, 13
    W, mbs = _problem([8, 8], C, V, ignore=[(1, n) for n in range(5)], seed=6)
    whole = O.step([(np.concatenate([h for h, _ in mbs]), np.concatenate([y for _, y in mbs]))], W)
    g = O.step(mbs, W, norm="global")
    assert g.objective == pytest.approx(whole.objective, rel=1e-13)
    assert np.abs(g.dW - whole.dW).max() < 1e-14
    mm = O.step(mbs, W, norm="micro_mean")
    counts = [m.count for m in mm.micro]
    assert counts == [8, 3]
    # micro_mean weights micro-step k by total / (count_k * G) relative to the global mean
    for a, b, c in zip(mm.micro, g.micro, counts):
        assert np.abs(a.dW * (c * 2) - b.dW * sum(counts)).max() < 1e-13
    assert abs(mm.objective - g.objective) > 1e-3


# --- Invariants ---------------------------------------------------------------------------

def test_gradient_rows_sum_to_zero_and_shift_invariance():
    C, V = 7, 19
    W, mbs = _problem([10], C, V, ignore=[(0, 4)], seed=8)
    r = O.step(mbs, W)
    assert np.abs(r.dW.sum(axis=0)).max() < 1e-14
    u = RNG.normal(0, 3, C)
    r2 = O.step(mbs, W + u[None, :])
    assert r2.objective == pytest.approx(r.objective, rel=1e-12)
    assert np.abs(r2.micro[0].dh - r.micro[0].dh).max() < 1e-12
    assert np.abs(r2.dW - r.dW).max() < 1e-12


def test_large_logits_are_stable():
    # logits near 1000: exp without the max shift overflows (catches a dropped max).
    C, V = 5, 9
    W, mbs = _problem([6], C, V, seed=9)
    h, y = mbs[0]
    h2 = np.concatenate([h, np.ones((h.shape[0], 1))], axis=1)
    W2_ = np.concatenate([W, np.full((V, 1), 1000.0)], axis=1)
    r = O.step([(h, y)], W)
    r2 = O.step([(h2, y)], W2_)
    assert np.all(np.isfinite(r2.micro[0].lse))
    assert np.abs(r2.micro[0].lse - 1000.0 - r.micro[0].lse).max() < 1e-9
    assert r2.loss_sum == pytest.approx(r.loss_sum, rel=1e-9)
    assert np.abs(r2.dW[:, :C] - r.dW).max() < 1e-12


def test_ignored_rows_equal_removed_rows():
    C, V = 6, 10
    W, mbs = _problem([12], C, V, ignore=[(0, 0), (0, 5), (0, 11)], seed=10)
    h, y = mbs[0]
    keep = y != O.IGNORE_ID
    r = O.step([(h, y)], W)
    r2 = O.step([(h[keep], y[keep])], W)
    assert r.count == 9 and r.loss_sum == pytest.approx(r2.loss_sum, rel=1e-14)
    assert np.abs(r.dW - r2.dW).max() < 1e-15
    assert np.abs(r.micro[0].dh[~keep]).max() == 0.0
    assert np.all(r.micro[0].row_loss[~keep] == 0.0)


def test_bad_targets_are_ignored_and_counted():
    C, V = 4, 6
    W, mbs = _problem([5], C, V, bad=[(0, 1, V), (0, 3, -7)], seed=12)
    h, y = mbs[0]
    r = O.step([(h, y)], W)
    assert r.bad == 2 and r.count == 3
    keep = (y >= 0) & (y < V)
    r2 = O.step([(h[keep], y[keep])], W)
    assert np.abs(r.dW - r2.dW).max() < 1e-15


def test_no_valid_target():
    C, V = 4, 6
    W, mbs = _problem([3], C, V, ignore=[(0, 0), (0, 1), (0, 2)], seed=13)
    r = O.step(mbs, W)
    assert r.count == 0 and r.loss_sum == 0.0 and np.abs(r.dW).max() == 0.0


# --- Sampled-output helpers agree with the whole computation ------------------------------

def test_sampled_helpers_agree():
    C, V = 6, 23
    W, mbs = _problem([9, 7], C, V, ignore=[(1, 3)], seed=14)
    r = O.step(mbs, W)
    scales = [m.scale for m in r.micro]
    lses = [O.lse_all(h, W) for h, _ in mbs]
    vs = [0, 5, 22]
    got = O.dW_rows(mbs, W, lses, scales, vs)
    assert np.abs(got - r.dW[vs]).max() < 1e-15
    h, y = mbs[1]
    lse, rl, dh = O.row_outputs(h[[2, 3]], W, y[[2, 3]], scales[1])
    assert np.abs(dh - r.micro[1].dh[[2, 3]]).max() < 1e-15
    assert np.abs(rl - r.micro[1].row_loss[[2, 3]]).max() < 1e-15


def test_dw_sumsq_worked_examples():
    # 3-4-5 and 1-2-2 triangles, and the invariants a plain sum of squares must keep
    assert O.dw_sumsq(np.array([[3.0, 4.0]])) == 25.0
    assert O.dw_sumsq(np.array([[1.0], [2.0], [2.0]])) == 9.0
    rng = np.random.default_rng(5)
    x = rng.standard_normal((7, 5))
    assert abs(O.dw_sumsq(3.0 * x) - 9.0 * O.dw_sumsq(x)) <= 1e-12 * O.dw_sumsq(x) * 9.0
    assert abs(O.dw_sumsq(x) - (O.dw_sumsq(x[:3]) + O.dw_sumsq(x[3:]))) <= 1e-12 * O.dw_sumsq(x)
    assert O.dw_sumsq(np.zeros((4, 4))) == 0.0


def test_clip_coef_worked_examples_and_torch():
    # norm 2 > 1: scaled down to norm 1 (up to the 1e-6 guard); norm 0.5 < 1: untouched
    assert O.clip_coef(4.0, 1.0) == 1.0 / (2.0 + 1e-6)
    assert O.clip_coef(0.25, 1.0) == 1.0
    assert O.clip_coef(0.0, 1.0) == 1.0
    # torch's global-norm clip over two tensors scales each by the same coefficient
    rng = np.random.default_rng(11)
    a, b = rng.standard_normal((6, 4)), rng.standard_normal(9)
    ta, tb = torch.zeros(6, 4, dtype=torch.float64), torch.zeros(9, dtype=torch.float64)
    ta.grad, tb.grad = torch.tensor(a), torch.tensor(b)
    torch.nn.utils.clip_grad_norm_([ta, tb], 1.0, foreach=False)
    c = O.clip_coef(O.dw_sumsq(a) + O.dw_sumsq(b), 1.0)
    assert c < 1.0
    np.testing.assert_allclose(ta.grad.numpy(), c * a, rtol=1e-14, atol=0)
    np.testing.assert_allclose(tb.grad.numpy(), c * b, rtol=1e-14, atol=0)


def test_adamw_first_step_closed_form():
    # m = v = 0, t = 1: mhat = g and vhat = g^2, so the step is lr * g / (|g| + eps), plus the decay
    rng = np.random.default_rng(12)
    p = rng.standard_normal(50)
    g = rng.standard_normal(50)
    g[:3] = (0.0, 1e-9, -1e-9)
    lr, wd, eps = 6e-4, 0.1, 1e-8
    p1, m1, v1 = O.adamw_step(p, np.zeros(50), np.zeros(50), g, 1, lr, (0.9, 0.95), eps, wd)
    np.testing.assert_allclose(p1, p * (1 - lr * wd) - lr * g / (np.abs(g) + eps), rtol=1e-13, atol=1e-18)
    np.testing.assert_allclose(m1, 0.1 * g, rtol=1e-14)
    np.testing.assert_allclose(v1, 0.05 * g * g, rtol=1e-14)
    assert p1[0] == p[0] * (1 - lr * wd)   # a zero gradient leaves only the decay


def test_adamw_constant_gradient_geometric_series():
    # a constant gradient keeps mhat = g and vhat = g^2 at every step (the bias correction is
    # exact), so T steps sum a geometric series: p_T = p0 d^T - u (1 - d^T) / (1 - d)
    rng = np.random.default_rng(13)
    p0 = rng.standard_normal(20)
    g = rng.standard_normal(20) * 1e-2
    lr, wd, eps, T = 1e-3, 0.1, 1e-8, 25
    p, m, v = p0.copy(), np.zeros(20), np.zeros(20)
    for t in range(1, T + 1):
        p, m, v = O.adamw_step(p, m, v, g, t, lr, (0.9, 0.95), eps, wd)
    d = 1 - lr * wd
    u = lr * g / (np.abs(g) + eps)
    np.testing.assert_allclose(p, p0 * d ** T - u * (1 - d ** T) / (1 - d), rtol=1e-11, atol=1e-15)


@pytest.mark.parametrize("clip", [1.0, 0.37])
def test_adamw_matches_torch_optim(clip):
    # torch.optim.AdamW in float64 over several steps of varying gradients
    rng = np.random.default_rng(14)
    shape = (7, 9)
    p0 = rng.standard_normal(shape)
    w = torch.nn.Parameter(torch.tensor(p0))
    opt = torch.optim.AdamW([w], lr=6e-4, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1, foreach=False)
    p, m, v = p0.copy(), np.zeros(shape), np.zeros(shape)
    for t in range(1, 6):
        g = rng.standard_normal(shape) * (0.1 * t)
        w.grad = torch.tensor(clip * g)
        opt.step()
        p, m, v = O.adamw_step(p, m, v, g, t, 6e-4, (0.9, 0.95), 1e-8, 0.1, clip)
    st = opt.state[w]
    np.testing.assert_allclose(p, w.detach().numpy(), rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(m, st["exp_avg"].numpy(), rtol=1e-13, atol=1e-18)
    np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-13, atol=1e-20)


@pytest.mark.parametrize("kind", ["layernorm", "rmsnorm"])
def test_final_norm_matches_torch_autograd(kind):
    # PyTorch's float64 layer_norm / rms_norm and their autograd: h, dx, dgamma and dbeta
    rng = np.random.default_rng(21)
    N, C = 13, 24
    x = rng.standard_normal((N, C)) * 3 + 1.5
    gamma = 1 + 0.1 * rng.standard_normal(C)
    beta = 0.1 * rng.standard_normal(C) if kind == "layernorm" else None
    dh = rng.standard_normal((N, C))
    eps = 1e-5
    tx = torch.tensor(x, requires_grad=True)
    tg = torch.tensor(gamma, requires_grad=True)
    if kind == "layernorm":
        tb = torch.tensor(beta, requires_grad=True)
        th = torch.nn.functional.layer_norm(tx, (C,), tg, tb, eps)
    else:
        th = torch.nn.functional.rms_norm(tx, (C,), tg, eps)
    th.backward(torch.tensor(dh))
    h, _, _ = O.final_norm(x, gamma, beta, kind, eps)
    np.testing.assert_allclose(h, th.detach().numpy(), rtol=1e-12, atol=1e-12)
    dx, dg, db = O.final_norm_backward(dh, x, gamma, kind, eps)
    np.testing.assert_allclose(dx, tx.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dg, tg.grad.numpy(), rtol=1e-10, atol=1e-12)
    if kind == "layernorm":
        np.testing.assert_allclose(db, tb.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_final_norm_invariants():
    rng = np.random.default_rng(22)
    x = rng.standard_normal((9, 16)) * 2 - 0.7
    one, zero = np.ones(16), np.zeros(16)
    # LayerNorm with unit scale and no shift: every row has mean 0 and mean square var / (var + eps)
    eps = 1e-3
    h, mu, rstd = O.final_norm(x, one, zero, "layernorm", eps)
    var = x.var(axis=1)
    np.testing.assert_allclose(h.mean(axis=1), 0.0, atol=1e-14)
    np.testing.assert_allclose((h * h).mean(axis=1), var / (var + eps), rtol=1e-13)
    # with eps = 0: LayerNorm ignores a shift and a positive scale of the row, RMSNorm a scale
    a, b = 3.5, -2.25
    np.testing.assert_allclose(O.final_norm(a * x + b, one, None, "layernorm", 0.0)[0],
                               O.final_norm(x, one, None, "layernorm", 0.0)[0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(O.final_norm(a * x, one, None, "rmsnorm", 0.0)[0],
                               O.final_norm(x, one, None, "rmsnorm", 0.0)[0], rtol=1e-12, atol=1e-13)
    # LayerNorm's input gradient has zero row sums (the output does not move with a row shift)
    dh = rng.standard_normal(x.shape)
    dx, _, _ = O.final_norm_backward(dh, x, 1 + 0.2 * rng.standard_normal(16), "layernorm", 1e-5)
    np.testing.assert_allclose(dx.sum(axis=1), 0.0, atol=1e-12)


@pytest.mark.parametrize("kind", ["layernorm", "rmsnorm"])
def test_step_ln_finite_differences(kind):
    # the whole objective as a function of x, gamma and beta, through ln_f and the head
    C, V = 8, 11
    W, mbs = _problem([5, 7], C, V, ignore=[(1, 2)], seed=23)
    rng = np.random.default_rng(23)
    xs = [(h * 1.7 + 0.4, y) for h, y in mbs]
    gamma = 1 + 0.2 * rng.standard_normal(C)
    beta = 0.2 * rng.standard_normal(C) if kind == "layernorm" else None
    r = O.step_ln(xs, gamma, beta, W, kind, 1e-5)

    def J(xs_, g_, b_):
        return O.step_ln(xs_, g_, b_, W, kind, 1e-5).head.objective

    e = 1e-6
    num_g = np.array([(J(xs, gamma + e * np.eye(C)[c], beta) - J(xs, gamma - e * np.eye(C)[c], beta)) / (2 * e)
                      for c in range(C)])
    assert np.abs(num_g - r.dgamma).max() <= 1e-6 * max(1.0, np.abs(r.dgamma).max())
    if beta is not None:
        num_b = np.array([(J(xs, gamma, beta + e * np.eye(C)[c]) - J(xs, gamma, beta - e * np.eye(C)[c])) / (2 * e)
                          for c in range(C)])
        assert np.abs(num_b - r.dbeta).max() <= 1e-6 * max(1.0, np.abs(r.dbeta).max())
    for k, (x, y) in enumerate(xs):
        num = np.zeros_like(x)
        for n in range(x.shape[0]):
            for c in range(C):
                xp = x.copy(); xp[n, c] += e
                xm = x.copy(); xm[n, c] -= e
                mp = list(xs); mp[k] = (xp, y)
                mm = list(xs); mm[k] = (xm, y)
                num[n, c] = (J(mp, gamma, beta) - J(mm, gamma, beta)) / (2 * e)
        assert np.abs(num - r.dx[k]).max() <= 1e-6 * max(1.0, np.abs(r.dx[k]).max())


def test_optimizer_defaults_are_the_pages():
    # the printed hyperparameters (tests/golden/optimizer_hyperparameters.json, with citations)
    # are the defaults of the oracle's AdamW and clip and of the binding's adamw
    import inspect
    g = json.load(open(os.path.join(GOLDEN, "optimizer_hyperparameters.json")))
    sig = inspect.signature(O.adamw_step).parameters
    assert tuple(sig["betas"].default) == tuple(g["betas"])
    assert sig["eps"].default == g["eps"] and sig["weight_decay"].default == g["weight_decay"]
    assert inspect.signature(O.clip_coef).parameters["max_norm"].default == g["grad_norm_clip"]
    from grad_lmce_microstep_gb300 import lmce as M
    bs = inspect.signature(M.Lmce.adamw).parameters
    assert tuple(bs["betas"].default) == tuple(g["betas"])
    assert bs["eps"].default == g["eps"] and bs["weight_decay"].default == g["weight_decay"]
    assert inspect.signature(M.clip_coef).parameters["max_norm"].default == g["grad_norm_clip"]


def test_adamw_gradient_scale_invariance():
    # with eps = 0 and no decay, Adam's step does not change when every gradient is multiplied by
    # the same positive constant (m scales by c, sqrt(v) by c); a moment update that mixes the
    # two moments, or a bias correction applied to one side only, breaks this
    rng = np.random.default_rng(15)
    shape = (5, 6)
    p0 = rng.standard_normal(shape)
    gs = [rng.standard_normal(shape) for _ in range(4)]
    out = []
    for c in (1.0, 37.0, 1e-3):
        p, m, v = p0.copy(), np.zeros(shape), np.zeros(shape)
        for t, g in enumerate(gs, start=1):
            p, m, v = O.adamw_step(p, m, v, c * g, t, 1e-2, (0.9, 0.95), 0.0, 0.0)
        out.append(p)
    np.testing.assert_allclose(out[1], out[0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(out[2], out[0], rtol=1e-12, atol=1e-14)


def test_adamw_clip_equals_prescaled_gradient():
    # the clip coefficient multiplies the gradient before both moments
    rng = np.random.default_rng(16)
    p, m, v, g = (rng.standard_normal((4, 3)) for _ in range(4))
    v = np.abs(v)
    a = O.adamw_step(p, m, v, g, 3, 1e-3, clip=0.25)
    b = O.adamw_step(p, m, v, 0.25 * g, 3, 1e-3, clip=1.0)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-15, atol=0)


def test_head_invariants_property():
    # random small problems: shifting every vocabulary row of W by one vector u moves each row's
    # logits by a constant, so the loss and dh do not move; the vocabulary rows of dW add up to
    # the zero vector (softmax-minus-one-hot rows sum to zero); both normalisations
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    @hyp.settings(max_examples=25, deadline=None)
    @hyp.given(C=st.integers(1, 6), V=st.integers(2, 9), n1=st.integers(1, 7), n2=st.integers(0, 5),
               seed=st.integers(0, 10 ** 6), micro=st.booleans())
    def check(C, V, n1, n2, seed, micro):
        rng = np.random.default_rng(seed)
        W = rng.standard_normal((V, C))
        mbs = []
        for n in (n1, n2):
            h = rng.standard_normal((n, C))
            y = rng.integers(0, V, n)
            if n > 1:
                y[rng.integers(0, n)] = O.IGNORE_ID
            mbs.append((h, y))
        if all(O.count_valid(y, V) == 0 for _, y in mbs):
            return
        norm = "micro_mean" if micro else "global"
        r = O.step(mbs, W, norm=norm)
        u = rng.standard_normal(C)
        r2 = O.step(mbs, W + u, norm=norm)
        assert abs(r2.loss_sum - r.loss_sum) <= 1e-9 * max(1.0, abs(r.loss_sum))
        for a, b in zip(r.micro, r2.micro):
            np.testing.assert_allclose(b.dh, a.dh, rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(r.dW.sum(axis=0), 0.0, atol=1e-12)

    check()
