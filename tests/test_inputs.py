"""The seeded input generator: reproducible, with the workload shapes and structure."""

import torch

from grad_lmce_microstep_gb300 import inputs as I


def test_reproducible_and_independent_streams():
    a = I.custom([5, 7], 16, 33, "bf16", seed=3)
    b = I.custom([5, 7], 16, 33, "bf16", seed=3)
    assert torch.equal(a.W, b.W)
    for (h1, y1), (h2, y2) in zip(a.micro, b.micro):
        assert torch.equal(h1, h2) and torch.equal(y1, y2)
    # regenerating one micro-batch alone gives the same bytes
    assert torch.equal(I.draw_h(7, 16, "bf16", 3, 1), a.micro[1][0])
    c = I.custom([5, 7], 16, 33, "bf16", seed=4)
    assert not torch.equal(a.W, c.W)


def test_tiny_char_shapes():
    w = I.tiny_char()
    assert (w.C, w.V, w.dtype, w.G, w.tokens) == (64, 65, "fp32", 2, 256)
    assert all(int(y.min()) >= 0 and int(y.max()) < 65 for _, y in w.micro)
    assert w.W.dtype == torch.float32


def test_masked_unequal_structure():
    w = I.masked_unequal(B=2, T=64)
    assert w.valid_counts() == [128, 96, 64, 32]
    for (_, y), tail in zip(w.micro, [0, 16, 32, 48]):
        rows = y.view(2, 64)
        if tail:
            assert bool((rows[:, 64 - tail:] == I.IGNORE_ID).all())
        assert bool((rows[:, :64 - tail] >= 0).all())
        assert int(rows[:, :64 - tail].max()) < I.GPT2_REAL_VOCAB


def test_logit_stress_structure():
    w = I.logit_stress(B=1, T=256, G=1, C=64)
    h, y = w.micro[0]
    norms = h.float().norm(dim=1)
    assert int((norms > 20 * norms.median()).sum()) == w.meta["scaled_rows"] == 3
    assert w.meta["argmax_targets"] == 5
    assert int(y.min()) >= 0 and int(y.max()) < I.GPT2_PADDED_VOCAB


def test_padded_docs_structure():
    # one document per row, then pad: every row's valid targets are a prefix of its T positions,
    # of the drawn length; about 70 % of the batch is padding, as the packing section says
    w = I.make("padded_docs")
    T = 2048
    assert w.C == 768 and w.V == 50304 and len(w.micro) == 4
    for (h, y), lens in zip(w.micro, w.meta["doc_lengths"]):
        assert h.shape == (8 * T, 768)
        rows = y.view(8, T)
        for r, L in enumerate(lens):
            assert 16 <= L <= T
            assert bool((rows[r, :L] >= 0).all()) and bool((rows[r, L:] == I.IGNORE_ID).all())
    frac = sum(w.valid_counts()) / w.tokens
    assert 0.2 < frac < 0.35
