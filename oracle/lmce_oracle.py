"""Plain float64 CPU oracle for the fused LM-head + softmax cross-entropy micro-step.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The CUDA library never calls into it and shares no code with it.

What it computes, in the order the pages give it:

* "How I trained my own GPT-2 124M on FineWeb-Edu", section 4 (Implementing Loss
  Calculation): logits of shape (B, T, V) are flattened to (B*T, V) rows; for every
  row the logits go through a softmax, the probability of the target token is
  picked, its negative log is taken, and the result is averaged over positions.
  The output projection is bias-free and shares its weight with the token
  embedding (weight tying), so logits = h @ W.T with W of shape [V, C].
* Same page, section 8.1 (Gradient Accumulation): every micro-step's loss is
  divided by grad_accum_steps before backward, and backward adds into the
  parameter gradient, so the fp32 gradient buffer is a sum over micro-steps.
* "Multi-GPU calculation of gradients for accelerated training", sections
  "Gradient accumulation averages across micro-steps" and "DDP averages gradients
  across processes": the mean of micro-batch means equals the global token mean
  only when every micro-step has the same number of valid targets.  The default
  normalisation here is therefore the global token-weighted mean (scale
  s = 1 / global valid count); the pages' own loss/G rule is kept as
  ``norm="micro_mean"`` (s_k = 1 / (valid_k * G)).
* "How I trained my own GPT-2 124M", section 6, and "Reproduce GPT-2 124M", training
  configuration: after the accumulation the gradient is clipped to a global norm of
  1.0 and AdamW updates the weights (``dw_sumsq``, ``clip_coef``, ``adamw_step``).
* "How I trained my own GPT-2 124M", section 2.8, and "Reproduce GPT-2 124M", model
  definition: the final LayerNorm (or RMSNorm) that produces h, forward and backward
  (``final_norm``, ``final_norm_backward``, ``step_ln``).
* zerotofrontier "GPT", section "Document boundaries, packing and masking": a
  pad target is ignored by the loss.  Its id is -100 here (the default of the
  PyTorch cross-entropy function the multi-GPU page cites).

Readings taken where the pages are silent:
padded vocabulary columns take part in the softmax; a target outside [0, V)
that is not the ignore id is treated as ignored and flagged; dh is the
gradient of the scaled objective for this micro-step only (overwritten each
micro-step), dW is summed over micro-steps.

Every floating-point value is cast to float64 first (a bf16 -> float64 cast is
exact).  Rows are processed in blocks of ``block`` rows so that at most
block x V logits exist at a time; numpy's BLAS does the matrix products.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

IGNORE_ID = -100


def f64(x) -> np.ndarray:
    """Exact cast of a numpy array or a CPU torch tensor (any float dtype) to float64."""
    if hasattr(x, "detach"):  # torch tensor; .double() of bf16/fp32 is exact
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def i64(y) -> np.ndarray:
    if hasattr(y, "detach"):
        y = y.detach().to("cpu").numpy()
    return np.asarray(y, dtype=np.int64)


# ---------------------------------------------------------------------------
# Definition of the per-row quantities (section 4 of the GPT-2 124M page)
# ---------------------------------------------------------------------------

def logits(h: np.ndarray, W: np.ndarray) -> np.ndarray:
    """z[n, v] = sum_c h[n, c] * W[v, c]: the tied, bias-free output projection."""
    return f64(h) @ f64(W).T


def logsumexp_rows(z: np.ndarray) -> np.ndarray:
    """lse[n] = m[n] + log(sum_v exp(z[n, v] - m[n])) with m[n] = max_v z[n, v].

    Subtracting the row maximum keeps every exponent <= 0 so nothing overflows;
    the value is exactly log(sum_v exp(z[n, v])).
    """
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def target_status(y: np.ndarray, V: int, ignore_id: int = IGNORE_ID):
    """(valid, bad): valid targets lie in [0, V); bad ones are neither valid nor the ignore id."""
    y = i64(y)
    valid = (y >= 0) & (y < V)
    bad = (~valid) & (y != ignore_id)
    return valid, bad


def count_valid(y, V: int, ignore_id: int = IGNORE_ID) -> int:
    return int(target_status(y, V, ignore_id)[0].sum())


# ---------------------------------------------------------------------------
# One micro-step
# ---------------------------------------------------------------------------

@dataclass
class MicroResult:
    loss_sum: float          # sum over valid rows of (lse - z[target])
    count: int               # number of valid rows
    bad: int                 # number of out-of-range targets (treated as ignored)
    scale: float             # s used for the gradients of this micro-step
    row_loss: np.ndarray     # [N] per-row loss, 0 on ignored rows
    lse: np.ndarray          # [N] logsumexp of every row (ignored rows included)
    dh: np.ndarray           # [N, C] gradient of s * loss_sum w.r.t. h
    dW: np.ndarray           # [V, C] gradient of s * loss_sum w.r.t. W (this micro-step only)


def microstep(h, W, y, scale: float, ignore_id: int = IGNORE_ID, block: int = 64,
              want_dW: bool = True) -> MicroResult:
    """Loss and gradients of the objective  scale * sum_{valid n} (lse_n - z[n, y_n]).

    d/dz[n, v] of (lse_n - z[n, y_n]) is softmax(z_n)[v] - [v == y_n], so
    dz = scale * (softmax - onehot) on valid rows and 0 on ignored rows;
    dh = dz @ W and dW = dz.T @ h (chain rule through z = h @ W.T).
    """
    h = f64(h)
    W = f64(W)
    y = i64(y)
    N, C = h.shape
    V = W.shape[0]
    valid, bad = target_status(y, V, ignore_id)
    row_loss = np.zeros(N)
    lse_all = np.zeros(N)
    dh = np.zeros((N, C))
    dW = np.zeros((V, C)) if want_dW else None
    for r0 in range(0, N, block):
        r1 = min(N, r0 + block)
        z = h[r0:r1] @ W.T                       # [b, V]
        lse = logsumexp_rows(z)
        lse_all[r0:r1] = lse
        vb = valid[r0:r1]
        rows = np.nonzero(vb)[0]
        tz = z[rows, y[r0:r1][rows]]
        row_loss[r0 + rows] = lse[rows] - tz
        p = np.exp(z - lse[:, None])             # softmax
        p[rows, y[r0:r1][rows]] -= 1.0           # minus onehot
        p[~vb] = 0.0                             # ignored rows carry no gradient
        dz = scale * p
        dh[r0:r1] = dz @ W
        if want_dW:
            dW += dz.T @ h[r0:r1]
    return MicroResult(float(row_loss.sum()), int(valid.sum()), int(bad.sum()), float(scale),
                       row_loss, lse_all, dh, dW)


# ---------------------------------------------------------------------------
# Normalisation and a whole optimizer step (gradient accumulation)
# ---------------------------------------------------------------------------

def micro_scales(counts, norm: str, G: int, global_valid: int | None = None):
    """Gradient scale of every micro-step.

    norm == "global":     s_k = 1 / global_valid  (global token-weighted mean; global_valid
                          counts valid targets over all micro-steps and all ranks)
    norm == "micro_mean": s_k = 1 / (count_k * G)  (the pages' loss / grad_accum_steps applied
                          to each micro-batch mean; a micro-step without valid targets gets 0)
    """
    if norm == "global":
        gv = sum(counts) if global_valid is None else global_valid
        return [0.0 if gv == 0 else 1.0 / gv for _ in counts]
    if norm == "micro_mean":
        return [0.0 if c == 0 else 1.0 / (c * G) for c in counts]
    raise ValueError(norm)


@dataclass
class StepResult:
    loss_sum: float
    count: int
    bad: int
    objective: float          # sum_k s_k * loss_sum_k: the scalar whose gradient dW / dh are
    dW: np.ndarray            # summed over micro-steps
    micro: list = field(default_factory=list)


def step(micro_batches, W, norm: str = "global", G: int | None = None, global_valid: int | None = None,
         ignore_id: int = IGNORE_ID, block: int = 64, want_dW: bool = True) -> StepResult:
    """One optimizer step of G micro-steps: dW is the sum of every micro-step's dW.

    ``micro_batches`` is a list of (h_k, y_k).  ``global_valid`` defaults to the valid
    count over the micro-batches given (one rank); a data-parallel caller passes the
    count summed over ranks.
    """
    W = f64(W)
    V = W.shape[0]
    G = len(micro_batches) if G is None else G
    counts = [count_valid(y, V, ignore_id) for _, y in micro_batches]
    scales = micro_scales(counts, norm, G, global_valid)
    dW = np.zeros_like(W) if want_dW else None
    res = []
    loss_sum = 0.0
    objective = 0.0
    for (h, y), s in zip(micro_batches, scales):
        r = microstep(h, W, y, s, ignore_id, block, want_dW)
        res.append(r)
        loss_sum += r.loss_sum
        objective += s * r.loss_sum
        if want_dW:
            dW += r.dW
    return StepResult(loss_sum, sum(counts), sum(r.bad for r in res), objective, dW, res)


# ---------------------------------------------------------------------------
# The final normalisation in front of the head (ln_f)
# ---------------------------------------------------------------------------

def final_norm(x, gamma, beta=None, kind: str = "layernorm", eps: float = 1e-5):
    """h = ln_f(x) in float64, with the per-row mean (0 for RMSNorm) and 1/std.

    "How I trained my own GPT-2 124M", section 2.8: after the last block GPT-2 applies one
    LayerNorm, ln_f, whose output feeds the tied head; LayerNorm centres each row, divides by
    the square root of its (biased) variance plus eps, then scales by gamma and shifts by
    beta.  "Reproduce GPT-2 124M" (model definition) uses an RMSNorm there instead: no
    centring, the root mean square in place of the standard deviation, no shift.
    """
    x, g = f64(x), f64(gamma)
    if kind == "layernorm":
        mu = x.mean(axis=1)
        var = ((x - mu[:, None]) ** 2).mean(axis=1)
        rstd = 1.0 / np.sqrt(var + eps)
        h = (x - mu[:, None]) * rstd[:, None] * g
        if beta is not None:
            h = h + f64(beta)
    elif kind == "rmsnorm":
        mu = np.zeros(x.shape[0])
        rstd = 1.0 / np.sqrt((x * x).mean(axis=1) + eps)
        h = x * rstd[:, None] * g
    else:
        raise ValueError(kind)
    return h, mu, rstd


def final_norm_backward(dh, x, gamma, kind: str = "layernorm", eps: float = 1e-5):
    """(dx, dgamma, dbeta) of h = ln_f(x) for an upstream gradient dh, in float64.

    With xhat the normalised row and g = dh * gamma: dgamma = sum over rows of dh * xhat,
    dbeta = sum over rows of dh, and per row dx = rstd * (g - mean(g) - xhat * mean(g * xhat))
    for LayerNorm (the mean(g) term drops for RMSNorm, which does not centre).
    """
    dh, x, gm = f64(dh), f64(x), f64(gamma)
    _, mu, rstd = final_norm(x, np.ones_like(gm), None, kind, eps)
    xhat = (x - mu[:, None]) * rstd[:, None]
    g = dh * gm
    proj = (g * xhat).mean(axis=1, keepdims=True)
    if kind == "layernorm":
        dx = rstd[:, None] * (g - g.mean(axis=1, keepdims=True) - xhat * proj)
    else:
        dx = rstd[:, None] * (g - xhat * proj)
    return dx, (dh * xhat).sum(axis=0), dh.sum(axis=0)


@dataclass
class LnStepResult:
    head: StepResult           # the head's step on the normalised rows
    dx: list                   # per micro-step, float64 [N_k, C]
    dgamma: np.ndarray         # summed over micro-steps
    dbeta: np.ndarray


def step_ln(micro_batches, gamma, beta, W, kind: str = "layernorm", eps: float = 1e-5,
            h_round=None, **step_kw) -> LnStepResult:
    """A whole step with ln_f in front: micro_batches holds (x_k, y_k); h_k = ln_f(x_k),
    optionally rounded by ``h_round`` (the head's input dtype), goes through ``step``, and
    each micro-step's dh goes back through the normalisation."""
    hs, xs = [], []
    for x, y in micro_batches:
        h, _, _ = final_norm(x, gamma, beta, kind, eps)
        if h_round is not None:
            h = h_round(h)
        hs.append((h, y))
        xs.append(f64(x))
    head = step(hs, W, **step_kw)
    C = f64(gamma).shape[0]
    dgamma, dbeta, dxs = np.zeros(C), np.zeros(C), []
    for x, m in zip(xs, head.micro):
        dx, dg, db = final_norm_backward(m.dh, x, gamma, kind, eps)
        dxs.append(dx)
        dgamma += dg
        dbeta += db
    return LnStepResult(head, dxs, dgamma, dbeta)


# ---------------------------------------------------------------------------
# Sampled outputs for problems too large to run whole
# ---------------------------------------------------------------------------

def row_outputs(h_rows, W, y_rows, scale: float, ignore_id: int = IGNORE_ID):
    """lse, row loss and dh for a handful of rows (each costs V*C multiply-adds)."""
    r = microstep(h_rows, W, y_rows, scale, ignore_id, block=16, want_dW=False)
    return r.lse, r.row_loss, r.dh


def lse_all(h, W, block: int = 256) -> np.ndarray:
    """logsumexp of every row; the expensive half of a dW row sample."""
    h = f64(h)
    W = f64(W)
    out = np.empty(h.shape[0])
    for r0 in range(0, h.shape[0], block):
        out[r0:r0 + block] = logsumexp_rows(h[r0:r0 + block] @ W.T)
    return out


def dW_rows(micro_batches, W, lses, scales, vs, ignore_id: int = IGNORE_ID) -> np.ndarray:
    """Rows vs of the accumulated dW, given every row's logsumexp.

    dW[v] = sum_k s_k * sum_{valid n} (exp(z[n, v] - lse_n) - [y_n == v]) * h_n.
    """
    W = f64(W)
    V = W.shape[0]
    vs = np.asarray(vs, dtype=np.int64)
    Wv = W[vs]                                       # [S, C]
    out = np.zeros((len(vs), W.shape[1]))
    for (h, y), lse, s in zip(micro_batches, lses, scales):
        h = f64(h)
        y = i64(y)
        valid, _ = target_status(y, V, ignore_id)
        z = h @ Wv.T                                 # [N, S]
        dz = np.exp(z - lse[:, None])
        dz -= (y[:, None] == vs[None, :])
        dz[~valid] = 0.0
        out += s * (dz.T @ h)
    return out


def dw_sumsq(dW) -> float:
    """Sum over every element of dW of dW**2, in float64: the squared global norm that a
    gradient clip divides by ("Reproduce GPT-2 124M", training configuration: the global-norm
    clip grad_norm_clip = 1.0, applied with torch.nn.utils.clip_grad_norm_ after the
    accumulation and before the optimizer)."""
    x = f64(dW).ravel()
    return float(np.dot(x, x))


def clip_coef(sumsq: float, max_norm: float = 1.0) -> float:
    """The factor a global-norm clip multiplies every gradient by: max_norm / (norm + 1e-6),
    never above 1, with norm = sqrt(sum of squares over all gradients) (same training
    configuration; the 1e-6 guard is torch.nn.utils.clip_grad_norm_'s)."""
    return min(1.0, max_norm / (math.sqrt(sumsq) + 1e-6))


def adamw_step(p, m, v, g, step: int, lr: float, betas=(0.9, 0.95), eps: float = 1e-8,
               weight_decay: float = 0.1, clip: float = 1.0):
    """One AdamW update in float64, returning new (p, m, v).

    "How I trained my own GPT-2 124M", section 6 (Implementing the Optimizer): Adam with a
    decoupled weight decay that pulls every weight of a tensor with two or more dimensions
    toward zero, built as torch.optim.AdamW with betas (0.9, 0.95), eps 1e-8 and decay 0.1
    (training loop: learning rate 6e-4).  The update is that optimizer's: the decay
    multiplies the weight by 1 - lr * weight_decay, the moments are exponential averages of
    the gradient and of its square, each divided by 1 - beta^step to remove the bias of
    their zero start, and the step is lr * mhat / (sqrt(vhat) + eps).  The gradient is
    first multiplied by the clip coefficient.
    """
    b1, b2 = betas
    g = clip * f64(g)
    p, m, v = f64(p), f64(m), f64(v)
    m = b1 * m + (1.0 - b1) * g
    v = b2 * v + (1.0 - b2) * g * g
    mhat = m / (1.0 - b1 ** step)
    vhat = v / (1.0 - b2 ** step)
    p = p * (1.0 - lr * weight_decay) - lr * mhat / (np.sqrt(vhat) + eps)
    return p, m, v

