"""Parity at the full workload sizes, in the launch configuration bench.py times.

The float64 oracle cannot run these workloads whole in seconds, so each test compares
outputs it can compute one by one -- sampled rows of dh and of the per-row loss (each needs
only that row's logits), sampled rows of dW (given the oracle's logsumexp of every row) --
or uses special inputs with a closed form at full size (W = 0).  Tolerances are the
method's: loss relative error <= 1e-3; dh, dW max abs error <= 2e-2 x max|oracle| (bf16).
"""

import math

import numpy as np
import pytest
import torch

from grad_lmce_microstep_gb300 import inputs as I
from grad_lmce_microstep_gb300 import lmce as M
from oracle import lmce_oracle as O

import sched_util as S
from gpu_util import GRAD_REL, LOSS_REL

pytestmark = pytest.mark.gpu

ROWS_PER_MICRO = 48
DW_ROWS = 24


def _run(w, W=None, compact=False):
    """Whole optimizer step on the GPU, keeping outputs on the device."""
    Wd = (w.W if W is None else W).cuda()
    mbs = [(h.cuda(), y.cuda()) for h, y in w.micro]
    dW, dhs, rls, res = M.run_step(Wd, mbs, w.dtype, row_loss=True, compact=compact)
    torch.cuda.synchronize()
    return dW, dhs, rls, res


def _sample_rows(w, k, rng, extra=()):
    n = w.micro[k][1].numel()
    rows = set(rng.choice(n, size=min(ROWS_PER_MICRO, n), replace=False).tolist())
    rows.update(int(r) for r in extra if r < n)
    return np.array(sorted(rows))


def _check_rows(w, dhs, rls, scales, rng, extra=lambda k: ()):
    Wf = O.f64(w.W)
    for k, (h, y) in enumerate(w.micro):
        rows = _sample_rows(w, k, rng, extra(k))
        ti = torch.as_tensor(rows)
        lse, rl, dh = O.row_outputs(h[ti], Wf, y[ti], scales[k], w.ignore_id)
        got_dh = dhs[k][torch.as_tensor(rows, device="cuda")].double().cpu().numpy()
        got_rl = rls[k][torch.as_tensor(rows, device="cuda")].double().cpu().numpy()
        tol = GRAD_REL[w.dtype] * max(np.abs(dh).max(), 1e-30)
        assert np.abs(got_dh - dh).max() <= tol, (k, np.abs(got_dh - dh).max() / max(np.abs(dh).max(), 1e-30))
        assert np.abs(got_rl - rl).max() <= LOSS_REL * max(1.0, np.abs(rl).max())


def _check_dW_rows(w, dW, scales, rng, lses, extra=()):
    vs = sorted(set(rng.choice(w.V, size=DW_ROWS, replace=False).tolist()) | set(extra))
    want = O.dW_rows(w.micro, w.W, lses, scales, vs, w.ignore_id)
    got = dW[torch.as_tensor(vs, device="cuda")].double().cpu().numpy()
    tol = GRAD_REL[w.dtype] * np.abs(want).max()
    assert np.abs(got - want).max() <= tol, np.abs(got - want).max() / np.abs(want).max()


def _split_rows(w, compact=False):
    """Per micro-step, the token rows at the edges of the lse+dh pass's split tiles (in the
    input's row numbering), and the vocabulary rows at the edges of the dW pass's split tiles."""
    pairs = S.pairs_on_device()
    tok, voc = [], set()
    for h, y in w.micro:
        valid = np.nonzero(O.target_status(y, w.V, w.ignore_id)[0])[0]
        n = len(valid) if compact else y.numel()
        rows = S.split_tile_edge_rows(n, w.V, pairs)
        tok.append([int(valid[r]) for r in rows] if compact else rows)
        voc.update(S.split_tile_edge_rows(w.V, n, pairs))
    return tok, sorted(voc)


def _oracle_totals(w):
    lses = [O.lse_all(h, w.W) for h, _ in w.micro]
    loss = 0.0
    for (h, y), lse in zip(w.micro, lses):
        valid, _ = O.target_status(y, w.V, w.ignore_id)
        yy = O.i64(y)[valid]
        z_t = np.einsum("nc,nc->n", O.f64(h)[valid], O.f64(w.W)[yy])
        loss += float((lse[valid] - z_t).sum())
    return lses, loss


@pytest.mark.parametrize("name,compact", [("gpt2_124m_head", False), ("masked_unequal", False),
                                          ("masked_unequal", True), ("padded_docs", True)])
def test_full_size_head(name, compact):
    # compact: the valid-row path (lmce_microstep_compact) in the launch configuration that
    # bench.py --compact times
    w = I.make(name)
    rng = np.random.default_rng(7)
    dW, dhs, rls, (ls, cnt, mean, st) = _run(w, compact=compact)
    assert st == M.OK
    counts = w.valid_counts()
    assert cnt == sum(counts)
    scales = O.micro_scales(counts, "global", w.G)
    lses, loss = _oracle_totals(w)
    assert abs(ls - loss) <= LOSS_REL * abs(loss)
    assert abs(mean - loss / sum(counts)) <= LOSS_REL * abs(loss / sum(counts))
    # rows from each micro-step, incl. the masked tail of the masked workload, and the first and
    # last row of every split tile of the lse+dh pass
    tok, voc = _split_rows(w, compact)
    extra = (lambda k: [16383, 1023, 1024 * 16 - 1]) if name == "masked_unequal" else (lambda k: [0])
    if name == "padded_docs":   # the last token of a document and the first pad after it
        extra = lambda k: [r * 2048 + L + d for r, L in enumerate(w.meta["doc_lengths"][k][:3]) for d in (-1, 0)]
    _check_rows(w, dhs, rls, scales, rng, lambda k: list(extra(k)) + tok[k])
    # dW rows: random ones, the padded vocabulary tail, frequent targets and the edges of the dW
    # pass's split tiles
    ys = np.concatenate([O.i64(y) for _, y in w.micro])
    top = np.bincount(ys[ys >= 0], minlength=w.V).argsort()[-4:].tolist()
    _check_dW_rows(w, dW, scales, rng, lses, extra=top + [w.V - 1, 50257] + voc)


def test_full_batch_524k_sampled_and_closed_form():
    w = I.make("gpt2_124m_full_batch")
    rng = np.random.default_rng(8)
    dW, dhs, rls, (ls, cnt, mean, st) = _run(w)
    assert st == M.OK and cnt == 524288
    scales = O.micro_scales(w.valid_counts(), "global", w.G)
    tok, voc = _split_rows(w)
    _check_rows(w, dhs, rls, scales, rng, lambda k: tok[k])
    # the summed loss equals the sum of the per-row losses the library returned
    assert abs(ls - sum(float(r.double().sum()) for r in rls)) <= 1e-6 * abs(ls)
    del dhs, rls
    # W = 0 at the same shape: every softmax is uniform, so
    #   dW[v] = s * (sum_n h_n / V - sum_{n: y_n = v} h_n), dh = 0, loss = log V per row
    Wz = torch.zeros_like(w.W)
    dW0, dhs0, _, (ls0, cnt0, mean0, st0) = _run(w, Wz)
    assert st0 == M.OK
    assert abs(mean0 - math.log(w.V)) <= 1e-6 * math.log(w.V)
    assert all(float(d.abs().max()) == 0.0 for d in dhs0)
    s = 1.0 / 524288
    hsum = np.zeros(w.C)
    for h, _ in w.micro:
        hsum += h.double().sum(0).numpy()
    vs = np.array(sorted(set(rng.choice(w.V, 64, replace=False).tolist()) | set(voc)))
    want = np.tile(s * hsum / w.V, (len(vs), 1))
    for h, y in w.micro:
        yy = O.i64(y)
        for i, v in enumerate(vs):
            sel = np.nonzero(yy == v)[0]
            if len(sel):
                want[i] -= s * h[torch.as_tensor(sel)].double().sum(0).numpy()
    got = dW0[torch.as_tensor(vs, device="cuda")].double().cpu().numpy()
    assert np.abs(got - want).max() <= GRAD_REL["bf16"] * np.abs(want).max()


def test_full_logit_stress():
    w = I.make("logit_stress")
    rng = np.random.default_rng(9)
    dW, dhs, rls, (ls, cnt, mean, st) = _run(w)
    assert st == M.OK
    counts = w.valid_counts()
    scales = O.micro_scales(counts, "global", w.G)
    lses, loss = _oracle_totals(w)
    assert max(float(l.max()) for l in lses) > 60.0
    assert abs(ls - loss) <= LOSS_REL * abs(loss)
    # The x40 rows of every micro-step, ranked by how far a logit rises above the one-pass
    # kernel's reference (the maximum of the first block its segment processes): the eight
    # closest to the kernel's range guard (32 + 115 - ceil(log2 V) in base 2), and every row of
    # a tile that crosses it (flagged and recomputed by the exact repair).  Plus the edges of
    # every split tile of both gradient passes.
    pairs = S.pairs_on_device()
    guard = 32 + 115 - math.ceil(math.log2(w.V))
    near = []
    for h, y in w.micro:
        big = h.float().norm(dim=1).argsort(descending=True)[:w.meta["scaled_rows"]].numpy()
        z = O.f64(h[torch.as_tensor(big)]) @ O.f64(w.W).T
        ex = np.array([S.guard_excess(z[i], S.segment_blocks(h.shape[0], w.V, pairs, int(n) // S.XT))
                       for i, n in enumerate(big)])
        rows = big[np.argsort(-ex)[:8]].tolist()
        for n in big[ex > guard]:
            t0 = int(n) // S.XT * S.XT
            rows += list(range(t0, min(t0 + S.XT, h.shape[0])))
        near.append(rows)
    tok, voc = _split_rows(w)
    _check_rows(w, dhs, rls, scales, rng, extra=lambda k: near[k] + tok[k])
    _check_dW_rows(w, dW, scales, rng, lses, extra=voc)


@pytest.mark.parametrize("name", ["gpt2_124m_head", "logit_stress"])
def test_full_size_stored_exponentials_match_recompute(name):
    # Every element at full size, not a sample: the default path (dW from the stored exponentials,
    # with its per-segment copies of the scaled rows of h) against the path that recomputes the
    # logits for dW.  Both run the same one-pass logsumexp + dh kernel, so dh, the row losses and
    # the loss agree exactly; dW differs only by the rounding of p and f h against that of dz.
    w = I.make(name)
    Wd = w.W.cuda()
    mbs = [(h.cuda(), y.cuda()) for h, y in w.micro]
    a = M.run_step(Wd, mbs, w.dtype, row_loss=True, path="tcgen05")
    b = M.run_step(Wd, mbs, w.dtype, row_loss=True, path="tcgen05_recompute")
    torch.cuda.synchronize()
    assert a[3][3] == M.OK and b[3][3] == M.OK
    assert a[3][:3] == b[3][:3]
    for x, y in zip(a[1], b[1]):
        assert torch.equal(x, y)
    for x, y in zip(a[2], b[2]):
        assert torch.equal(x, y)
    d = float((a[0].double() - b[0].double()).abs().max())
    assert d <= GRAD_REL["bf16"] * float(b[0].double().abs().max()), d
