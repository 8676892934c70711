"""Rows that the tensor-core path's persistent schedule puts on its special paths.

The host splits (X tile, stream block) units evenly over the CTA pairs: units are t-major,
pair q takes [U q / P, U (q + 1) / P); a tile whose units two pairs share is a split tile,
summed from fp32 partials by the split-combine kernels.  X is the token rows in the
logsumexp + dh pass (stream: the vocabulary) and the vocabulary rows in the dW pass (stream:
the tokens).  These helpers restate that rule so that full-size parity tests check the first
and last row of every split tile on purpose, not by chance.
"""

import math

import numpy as np

XT = 128   # X rows per pair tile
YB = 256   # stream rows per block


def pairs_on_device() -> int:
    import torch

    return torch.cuda.get_device_properties(0).multi_processor_count // 2


def schedule(nX: int, nY: int, pairs: int):
    """(U, P, nblk) as the host computes them for one gradient launch."""
    nblk = (nY + YB - 1) // YB
    T = (nX + XT - 1) // XT
    U = T * nblk
    P = min(pairs, U * 6 // nblk, U)
    return U, max(P, 1), nblk


def split_tiles(nX: int, nY: int, pairs: int):
    U, P, nblk = schedule(nX, nY, pairs)
    out = []
    for q in range(1, P):
        u = U * q // P
        if u % nblk and (not out or out[-1] != u // nblk):
            out.append(u // nblk)
    return out


def split_tile_edge_rows(nX: int, nY: int, pairs: int):
    """First and last X row of every split tile (the last clipped to nX - 1)."""
    rows = []
    for t in split_tiles(nX, nY, pairs):
        rows += [t * XT, min(t * XT + XT - 1, nX - 1)]
    return rows


def rotation(nX: int, nY: int, pairs: int, t: int) -> int:
    """The vocabulary rotation of X tile t in the dh passes: the pair with the most units of the
    tile (the lowest on a tie) reaches block (tau mod nblk) at its tau-th unit."""
    U, P, nblk = schedule(nX, nY, pairs)
    best, tau, j = -1, 0, 0
    for q in range(P):
        a, b = max(U * q // P, t * nblk), min(U * (q + 1) // P, (t + 1) * nblk)
        if b - a > best:
            best, tau, j = b - a, a - U * q // P, a - t * nblk
    return (tau - j) % nblk


def segment_blocks(nX: int, nY: int, pairs: int, t: int):
    """For every segment covering X tile t in a dh pass: its vocabulary blocks in the order the
    pair processes them (the first one sets the one-pass reference)."""
    U, P, nblk = schedule(nX, nY, pairs)
    r = rotation(nX, nY, pairs, t)
    out = []
    for q in range(P):
        a, b = max(U * q // P, t * nblk), min(U * (q + 1) // P, (t + 1) * nblk)
        if a < b:
            out.append([(j - t * nblk + r) % nblk for j in range(a, b)])
    return out


def guard_excess(z_row: np.ndarray, segs):
    """Largest excess (base 2) of a token row's logits over the maximum of the first block its
    segment processes, over every segment of the row's tile."""
    zb = z_row / math.log(2.0)
    V = zb.shape[0]
    ex = -np.inf
    for blocks in segs:
        m = zb[blocks[0] * YB:min(V, blocks[0] * YB + YB)].max()
        for b in blocks:
            ex = max(ex, zb[b * YB:min(V, b * YB + YB)].max() - m)
    return ex


def max_segments(nX: int, nY: int, pairs: int) -> int:
    """Most pairs sharing one X tile: the copies of the scaled rows of h that the dW pass from
    the stored exponentials keeps, one per segment of a token tile."""
    return max(len(segment_blocks(nX, nY, pairs, t)) for t in range((nX + XT - 1) // XT))
