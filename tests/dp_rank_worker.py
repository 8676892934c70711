"""One data-parallel rank on the CPU, as launch.relaunch starts it (torchrun's environment).

Each rank takes its shard of every micro-batch's rows, runs the float64 oracle with the
globally reduced valid count, SUM-reduces dW and (loss_sum, count) through the library's
dp module over gloo, and rank 0 writes the reduced result to the JSON file named by argv[1].
"""

import json
import os
import sys

import numpy as np
import torch
import torch.distributed as dist

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from grad_lmce_microstep_gb300 import dp  # noqa: E402
from oracle import lmce_oracle as O  # noqa: E402


def problem(seed=31):
    rng = np.random.default_rng(seed)
    C, V = 5, 13
    W = rng.normal(0, 0.5, (V, C))
    mbs = []
    for k in range(3):
        h = rng.normal(0, 1, (11, C))
        y = rng.integers(0, V, 11)
        if k == 2:
            y[3:] = O.IGNORE_ID   # an uneven micro-step: 3 valid rows of 11
        mbs.append((h, y))
    return W, mbs


def main():
    rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
    assert int(os.environ["LOCAL_RANK"]) == rank
    dist.init_process_group("gloo")
    try:
        W, mbs = problem()
        local = []
        for h, y in mbs:
            a, b = dp.shard_rows(h.shape[0], rank, world)
            local.append((h[a:b], y[a:b]))
        gv = dp.global_valid_count(sum(O.count_valid(y, W.shape[0]) for _, y in local))
        r = O.step(local, W, norm="global", global_valid=gv)
        dW = torch.tensor(r.dW)
        ls, cnt = dp.reduce_step(dW, r.loss_sum, r.count)
        if rank == 0:
            with open(sys.argv[1], "w") as f:
                json.dump({"world": world, "global_valid": gv, "loss_sum": ls, "count": cnt,
                           "dW": dW.numpy().tolist()}, f)
    finally:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
