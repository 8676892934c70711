"""The multi-rank launcher (launch.relaunch, which bench.py --gpus N uses) on CPU ranks.

Two gloo ranks started by the launcher each run the float64 oracle on their shard and
SUM-reduce through the dp module; the result must equal one process over every row.  The
benchmark's reference arm started with --gpus 2 runs under the same launcher and prints
exactly one JSON line (rank 0).
"""

import json
import os
import subprocess
import sys

import numpy as np

from grad_lmce_microstep_gb300 import launch
from oracle import lmce_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import dp_rank_worker  # noqa: E402


def test_launcher_runs_ranks_whose_sum_matches_one_process(tmp_path):
    out = tmp_path / "rank0.json"
    rc = launch.relaunch(os.path.join(ROOT, "tests", "dp_rank_worker.py"), [str(out)], 2)
    assert rc == 0
    got = json.load(open(out))
    W, mbs = dp_rank_worker.problem()
    whole = O.step(mbs, W, norm="global")
    assert got["world"] == 2
    assert got["count"] == whole.count == got["global_valid"]
    assert abs(got["loss_sum"] - whole.loss_sum) <= 1e-13 * abs(whole.loss_sum)
    assert np.abs(np.array(got["dW"]) - whole.dW).max() < 1e-14


def test_bench_gpus_flag_starts_the_ranks():
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0", "--workload", "tiny_char", "--cpu-sample-rows", "16"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    assert json.loads(lines[0])["impl"] == "reference"


def test_bench_refuses_more_gpus_than_it_sees():
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode != 0
    assert "visible GPUs" in r.stderr
