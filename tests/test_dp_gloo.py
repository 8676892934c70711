"""Data-parallel host logic on CPU ranks (gloo, world size 2 and 3).

Each rank runs the float64 oracle on its shard of rows with the globally reduced
valid count, then SUM-reduces dW and (loss_sum, count) through the library's dp
module.  The result must equal one process running every row, including with
unequal valid counts per rank, and must reproduce the two-GPU worked example.
"""

import json
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from grad_lmce_microstep_gb300 import dp
from oracle import lmce_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _problem(seed=21):
    rng = np.random.default_rng(seed)
    C, V = 6, 17
    W = rng.normal(0, 0.5, (V, C))
    mbs = []
    for k in range(2):
        h = rng.normal(0, 1, (10, C))
        y = rng.integers(0, V, 10)
        mbs.append((h, y))
    # unequal valid counts: rank 1's second micro-step loses 6 of its rows
    mbs[1][1][4:] = O.IGNORE_ID
    return W, mbs


def _ln_params(C, seed=22):
    rng = np.random.default_rng(seed)
    return 1 + 0.1 * rng.normal(size=C), 0.1 * rng.normal(size=C)


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        W, mbs = _problem()
        res = {}
        # each rank holds half of every micro-batch's rows
        local = []
        for h, y in mbs:
            a, b = dp.shard_rows(h.shape[0], rank, world)
            local.append((h[a:b], y[a:b]))
        lv = sum(O.count_valid(y, W.shape[0]) for _, y in local)
        gv = dp.global_valid_count(lv)
        r = O.step(local, W, norm="global", global_valid=gv)
        dW = torch.tensor(r.dW)
        ls, cnt = dp.reduce_step(dW, r.loss_sum, r.count)
        res["dW"] = dW.numpy()
        res["loss_sum"] = ls
        res["count"] = cnt
        res["objective"] = float(dp.reduce_step(torch.zeros(1, dtype=torch.float64), r.objective, 0)[0])
        # ln_f in front: the rows' x shard like h; dgamma and dbeta are reduced beside dW
        gamma, beta = _ln_params(W.shape[1])
        rl = O.step_ln([(h * 1.3 + 0.2, y) for h, y in local], gamma, beta, W, "layernorm", 1e-5, global_valid=gv)
        dW2, dg, db = torch.tensor(rl.head.dW), torch.tensor(rl.dgamma), torch.tensor(rl.dbeta)
        dp.reduce_step(dW2, rl.head.loss_sum, rl.head.count, extra=(dg, db))
        res["ln"] = (dW2.numpy(), dg.numpy(), db.numpy())
        if world == 2:
            # the two-GPU worked example: per-rank micro-mean objectives, averaged
            g = json.load(open(os.path.join(GOLDEN, "p5_worked_examples.json")))["two_gpu"]
            W2 = np.array([[1.0], [0.0]])
            rows = []
            for l in g["rank_token_losses_per_micro_step"][rank]:
                d = np.array([math.log(math.exp(L) - 1.0) for L in l])
                rows.append((d[:, None], np.ones(len(l), dtype=np.int64)))
            obj = O.step(rows, W2, norm="micro_mean").objective
            t = torch.tensor([obj], dtype=torch.float64)
            dist.all_reduce(t, op=dist.ReduceOp.SUM)
            res["p5_avg"] = t.item() / world
        out[rank] = res
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_sum_reduction_matches_single_process(world):
    # world 3 shards every 10-row micro-batch unevenly (4, 3, 3 rows)
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    W, mbs = _problem()
    whole = O.step(mbs, W, norm="global")
    g = json.load(open(os.path.join(GOLDEN, "p5_worked_examples.json")))["two_gpu"]
    for r in range(world):
        res = out[r]
        assert np.abs(res["dW"] - whole.dW).max() < 1e-14
        assert res["loss_sum"] == pytest.approx(whole.loss_sum, rel=1e-13)
        assert res["count"] == whole.count
        assert res["objective"] == pytest.approx(whole.objective, rel=1e-13)
        if world == 2:
            assert res["p5_avg"] == pytest.approx(g["ddp_average"], rel=1e-12)
        gamma, beta = _ln_params(W.shape[1])
        wl = O.step_ln([(h * 1.3 + 0.2, y) for h, y in mbs], gamma, beta, W, "layernorm", 1e-5)
        dW2, dg, db = res["ln"]
        assert np.abs(dW2 - wl.head.dW).max() < 1e-14
        assert np.abs(dg - wl.dgamma).max() < 1e-13 and np.abs(db - wl.dbeta).max() < 1e-13


def test_shard_rows_covers_everything():
    for n in (0, 1, 7, 16384):
        for w in (1, 2, 3, 8):
            spans = [dp.shard_rows(n, r, w) for r in range(w)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(spans[i][1] == spans[i + 1][0] for i in range(w - 1))
