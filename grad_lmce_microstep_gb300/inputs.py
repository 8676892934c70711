"""Seeded synthetic inputs for the fused LM-head + cross-entropy micro-step.

Shared by the tests, the benchmark and the oracle's callers; it holds no part of
the loss or gradient arithmetic.  Every tensor comes from its own CPU
``torch.Generator`` whose seed is derived from (seed, tensor kind, micro-step), so
any one micro-batch can be regenerated alone.  Values are drawn in fp32 and, for
bf16 workloads, rounded to bf16 (round-to-nearest-even) once.

Distributions follow the GPT-2 124M pages: W ~ N(0, 0.02) (the GPT-2 initialisation,
"How I trained my own GPT-2 124M", section 7), h ~ N(0, 1) (the output of the final
LayerNorm), targets uniform over the 50,257 real tokens of the 50,304-entry padded
vocabulary (same page, section 8.3), ignore id -100.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

IGNORE_ID = -100
GPT2_REAL_VOCAB = 50257
GPT2_PADDED_VOCAB = 50304

_KIND = {"W": 1, "h": 101, "y": 201, "mask": 301, "stress": 401, "doclen": 501}


def _gen(seed: int, kind: str, k: int = 0) -> torch.Generator:
    return torch.Generator().manual_seed(seed * 1_000_003 + _KIND[kind] + k)


def _dt(dtype: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[dtype]


@dataclass
class Workload:
    name: str
    C: int
    V: int
    dtype: str                       # "bf16" or "fp32": dtype of h, W and dh
    W: torch.Tensor                  # [V, C]
    micro: list                      # [(h [N_k, C], y [N_k] int32)] one per micro-step
    ignore_id: int = IGNORE_ID
    meta: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return len(self.micro)

    @property
    def tokens(self) -> int:
        return sum(int(y.numel()) for _, y in self.micro)

    def valid_counts(self):
        return [int(((y >= 0) & (y < self.V)).sum()) for _, y in self.micro]


def draw_W(V: int, C: int, dtype: str, seed: int = 0, std: float = 0.02) -> torch.Tensor:
    return (torch.randn(V, C, generator=_gen(seed, "W")) * std).to(_dt(dtype))


def draw_h(N: int, C: int, dtype: str, seed: int, k: int) -> torch.Tensor:
    return torch.randn(N, C, generator=_gen(seed, "h", k)).to(_dt(dtype))


def draw_targets(N: int, hi: int, seed: int, k: int) -> torch.Tensor:
    return torch.randint(0, hi, (N,), generator=_gen(seed, "y", k), dtype=torch.int64).to(torch.int32)


def tail_mask(y: torch.Tensor, T: int, masked_tail: int, ignore_id: int = IGNORE_ID) -> torch.Tensor:
    """Set the last ``masked_tail`` targets of every length-T row to the ignore id."""
    y = y.clone().view(-1, T)
    if masked_tail > 0:
        y[:, T - masked_tail:] = ignore_id
    return y.view(-1)


def custom(Ns, C: int, V: int, dtype: str = "bf16", seed: int = 0, target_hi: int | None = None,
           ignore_frac: float = 0.0, name: str = "custom") -> Workload:
    """Micro-batches of sizes Ns; a seeded fraction ``ignore_frac`` of targets set to -100."""
    W = draw_W(V, C, dtype, seed)
    hi = V if target_hi is None else target_hi
    micro = []
    for k, N in enumerate(Ns):
        h = draw_h(N, C, dtype, seed, k)
        y = draw_targets(N, hi, seed, k)
        if ignore_frac > 0:
            m = torch.rand(N, generator=_gen(seed, "mask", k)) < ignore_frac
            y[m] = IGNORE_ID
        micro.append((h, y))
    return Workload(name, C, V, dtype, W, micro)


def tiny_char(seed: int = 0) -> Workload:
    """C=64, V=65 (64 characters + an end-of-text id), fp32, 2 micro-steps of B=2, T=64."""
    return custom([128, 128], 64, 65, "fp32", seed, name="tiny_char")


def gpt2_head(seed: int = 0, G: int = 4, B: int = 16, T: int = 1024, name: str = "gpt2_124m_head") -> Workload:
    """GPT-2 124M LM head: C=768, V=50304, bf16, G micro-steps of B*T tokens."""
    return custom([B * T] * G, 768, GPT2_PADDED_VOCAB, "bf16", seed, target_hi=GPT2_REAL_VOCAB, name=name)


def gpt2_full_batch(seed: int = 0) -> Workload:
    """524,288 tokens per optimizer step: 8 micro-steps of B=64, T=1024."""
    return gpt2_head(seed, G=8, B=64, T=1024, name="gpt2_124m_full_batch")


def masked_unequal(seed: int = 0, B: int = 16, T: int = 1024) -> Workload:
    """4 micro-steps whose valid fractions are 100/75/50/25 %: the tail of each row is -100."""
    w = gpt2_head(seed, G=4, B=B, T=T, name="masked_unequal")
    tails = [0, T // 4, T // 2, 3 * T // 4]
    w.micro = [(h, tail_mask(y, T, t)) for (h, y), t in zip(w.micro, tails)]
    w.meta["masked_tail"] = tails
    return w


def padded_docs(seed: int = 0, B: int = 8, T: int = 2048, G: int = 4, mean_len: int = 600,
                sd_len: int = 150) -> Workload:
    """One document per row, the rest of the row padded (pad targets = -100): zerotofrontier
    "GPT", section "Document boundaries, packing and masking", where ~600-token documents in
    T = 2048 windows waste about 70 % of every batch.  Document lengths are seeded draws from a
    normal(mean_len, sd_len) clipped to [16, T]; C = 768, V = 50304, bf16, G micro-steps of B rows."""
    w = gpt2_head(seed, G=G, B=B, T=T, name="padded_docs")
    lens = []
    micro = []
    for k, (h, y) in enumerate(w.micro):
        L = torch.randn(B, generator=_gen(seed, "doclen", k)) * sd_len + mean_len
        L = L.round().clamp(16, T).to(torch.int64)
        y = y.clone().view(B, T)
        pos = torch.arange(T).view(1, T)
        y[pos >= L.view(B, 1)] = IGNORE_ID
        micro.append((h, y.view(-1)))
        lens.append([int(v) for v in L])
    w.micro = micro
    w.meta["doc_lengths"] = lens
    return w


def logit_stress(seed: int = 0, B: int = 8, T: int = 2048, G: int = 2, C: int = 1024,
                 scale_frac: float = 0.01, scale: float = 40.0, argmax_frac: float = 0.02) -> Workload:
    """C=1024: 1 % of h rows multiplied by 40 (in fp32, before the bf16 rounding) and 2 % of
    targets replaced by the row's largest-logit index.

    Choosing those targets needs the row's logits.  They are computed here by a plain
    float64 matrix product of the bf16-rounded inputs (workload construction only; the
    lowest index wins a tie) so that the workload is fixed before either implementation
    sees it.
    """
    V = GPT2_PADDED_VOCAB
    N = B * T
    W = draw_W(V, C, "bf16", seed)
    Wd = W.double().numpy()
    micro = []
    n_scaled = int(round(scale_frac * N))
    n_argmax = int(round(argmax_frac * N))
    for k in range(G):
        g = _gen(seed, "stress", k)
        hf = torch.randn(N, C, generator=_gen(seed, "h", k))
        rows = torch.randperm(N, generator=g)[:n_scaled]
        hf[rows] *= scale
        h = hf.to(torch.bfloat16)
        y = draw_targets(N, GPT2_REAL_VOCAB, seed, k)
        am_rows = torch.randperm(N, generator=g)[:n_argmax]
        z = h[am_rows].double().numpy() @ Wd.T
        y[am_rows] = torch.from_numpy(np.argmax(z, axis=1).astype(np.int32))
        micro.append((h, y))
    return Workload("logit_stress", C, V, "bf16", W, micro,
                    meta={"scaled_rows": n_scaled, "argmax_targets": n_argmax, "scale": scale})


WORKLOADS = {
    "tiny_char": tiny_char,
    "gpt2_124m_head": gpt2_head,
    "gpt2_124m_full_batch": gpt2_full_batch,
    "masked_unequal": masked_unequal,
    "logit_stress": logit_stress,
    "padded_docs": padded_docs,
}


def make(name: str, seed: int = 0) -> Workload:
    return WORKLOADS[name](seed)
