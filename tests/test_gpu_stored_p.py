"""The dW pass from the stored exponentials (LMCE_PATH_TCGEN05) against the float64 oracle and
against the dW pass that recomputes the logits (LMCE_PATH_TCGEN05_RECOMPUTE).

The one-pass logsumexp + dh kernel stores its bf16 operand p = 2^(z log2 e - m) with m fixed per
row and per segment of the row's 128-token tile (the pairs of its schedule that share the tile);
the dW pass takes, for every (token tile, vocabulary block), the scaled copy of h of the segment
that covered it.  The shapes below make a tile's segments many (up to seven), put ragged tails
on both operands, and use every C-chunk layout, so a copy taken for the wrong segment or a
missing target correction shows up in whole dW rows."""

import numpy as np
import pytest
import torch

from grad_lmce_microstep_gb300 import inputs as I
from grad_lmce_microstep_gb300 import lmce as M

import sched_util as S
from gpu_util import GRAD_REL, assert_parity, max_rel_err, run_lib, run_oracle

pytestmark = pytest.mark.gpu

CASES = {
    # small N, full GPT-2 vocabulary: a token tile is shared by 5-7 pairs
    "many_segments_v50304": lambda: I.custom([2000, 1100], 256, 50304, "bf16", seed=71, ignore_frac=0.1),
    # C = 768 (three chunks), vocabulary tail of 185 rows, 20 % ignored
    "c768_ragged": lambda: I.custom([520, 130], 768, 3001, "bf16", seed=72, ignore_frac=0.2),
    # C = 1024: the dW pass runs over two ranges of C chunks, reading p twice
    "c1024": lambda: I.custom([300, 140], 1024, 900, "bf16", seed=73, ignore_frac=0.05),
    # token counts one past a 256-row block, one row, and a vocabulary smaller than one tile
    "one_row_and_tails": lambda: I.custom([257, 1, 129], 512, 100, "bf16", seed=74),
    # V = 257: the last 256-column block of p holds one valid column, the last 128-row dW tile
    # one valid row; 17 tokens in the second micro-step
    "v257": lambda: I.custom([300, 17], 256, 257, "bf16", seed=77, ignore_frac=0.1),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_stored_p_matches_oracle_and_recompute(case):
    w = CASES[case]()
    ref = run_oracle(w)
    got = run_lib(w, path="tcgen05")
    assert got["status"] == M.OK
    assert_parity(got, ref, "bf16")
    rec = run_lib(w, path="tcgen05_recompute")
    assert rec["status"] == M.OK
    assert_parity(rec, ref, "bf16")
    # the two dW passes differ only in rounding: p and f h each rounded once to bf16 against
    # dz rounded once
    assert max_rel_err(got["dW"], rec["dW"]) <= GRAD_REL["bf16"]
    for a, b in zip(got["dh"], rec["dh"]):
        assert np.array_equal(a, b)   # the same lse+dh pass


def test_many_segments_premise():
    # the first case above really splits its token tiles over many pairs on this device
    pairs = S.pairs_on_device()
    assert S.max_segments(2000, 50304, pairs) >= 5
    assert S.max_segments(2000, 50304, pairs) <= 8


@pytest.mark.parametrize("norm", ["global", "micro_mean"])
def test_stored_p_flagged_tiles(norm):
    # two flagged tiles (one token's logit far beyond the one-pass range): the repair rewrites
    # the tiles' rows of p with the normalised softmax and their references with lse log2 e
    w = I.custom([600, 260], 512, 3001, "bf16", seed=75, ignore_frac=0.1)
    for k, n, v in [(0, 3, 100), (0, 450, 2999), (1, 200, 7)]:
        w.W[v] = (0.5 * w.micro[k][0][n].float()).to(w.W.dtype)
        w.micro[k][1][n] = v
    got = run_lib(w, path="tcgen05", norm=norm)
    assert got["status"] == M.OK
    assert_parity(got, run_oracle(w, norm=norm), "bf16")


def test_selected_paths():
    W = torch.zeros(1000, 256, dtype=torch.float32, device="cuda")
    for path, want in (("auto", 2), ("tcgen05", 2), ("tcgen05_recompute", 4)):
        L = M.Lmce(256, 1000, 64, W, "bf16", path=path)
        assert L.path == M.PATH_NAMES[want], (path, L.path)
        L.close()


def test_far_segment_reference_is_repaired():
    # N = 300, V = 1000: every token tile is split over four pairs, one vocabulary block each, so
    # each pair's reference comes from its own block and no element passes the one-pass range
    # guard.  Token 5's logit at vocabulary row 700 (block 2) is ~128 nats above the rest, so
    # the references of the other three segments lie ~150 (base 2) below its lse: their scale
    # s 2^(m - lse log2 e) underflows and the target entry (token 5 targets block 0) would
    # overflow.  The stored path flags such a tile for the exact repair.
    pairs = S.pairs_on_device()
    assert len(S.segment_blocks(300, 1000, pairs, 0)) == 4
    w = I.custom([300, 173], 256, 1000, "bf16", seed=11)
    w.W[700] = (0.5 * w.micro[0][0][5].float()).to(w.W.dtype)
    assert int(w.micro[0][1][5]) < 256   # the target lies in the first block
    ref = run_oracle(w)
    assert ref.micro[0].lse[5] > 100.0
    got = run_lib(w, path="tcgen05")
    assert got["status"] == M.OK
    assert_parity(got, ref, "bf16")


def test_auto_falls_back_when_p_does_not_fit():
    # max_N = 4,000,000 rows: the stored exponentials would need ~400 GB (2 bytes x 50,432 per
    # row), more than the device has, while the rest of the scratch (~1 GB) fits.  LMCE_PATH_AUTO
    # then takes the recomputing dW pass; an explicit LMCE_PATH_TCGEN05 reports the failure.
    big = 4_000_000
    W0 = torch.zeros(50304, 768, dtype=torch.float32, device="cuda")
    with pytest.raises(M.LmceError) as e:
        M.Lmce(768, 50304, big, W0, "bf16", path="tcgen05")
    assert e.value.status == M.ERR_CUDA
    del W0
    w = I.custom([300, 173], 256, 50304, "bf16", seed=76, ignore_frac=0.1)
    W, mbs = (w.W.cuda(), [(h.cuda(), y.cuda()) for h, y in w.micro])
    dW = torch.empty(w.V, w.C, device="cuda")
    L = M.Lmce(w.C, w.V, big, dW, "bf16", grad_accum_steps=2, path="auto")
    assert L.path == "tcgen05_recompute"
    gv = sum(w.valid_counts())
    dhs = []
    for h, y in mbs:
        dh = torch.empty_like(h)
        L.microstep(h, W, y, gv, dh)
        dhs.append(dh)
    ls, cnt, mean = L.finalize()
    L.close()
    got = {"dW": dW.double().cpu().numpy(), "dh": [d.double().cpu().numpy() for d in dhs],
           "row_loss": [None, None], "loss_sum": ls, "count": cnt, "loss_mean": mean}
    assert_parity(got, run_oracle(w), "bf16")
