"""bench.py's own arm on the GPU: one JSON line with the keys the bench contract fixes, and the
figures that explain it (roofline of each heavy kernel, the recompute path, clocks, launches)."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3",
                        "--cpu-sample-rows", "16"], capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
              "gpu_launches", "clocks", "roofline_kernels", "recompute_path"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"] == "gpt2_124m_head" and d["config"]["path"] == "tcgen05"
    # eight launches per 16,384-token micro-step of the default path, four micro-steps per step
    assert d["gpu_launches"] == 3 * 4 * 8
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s" and 0 < rf["frac"] < 1.2
    assert set(d["roofline_kernels"]) >= {"lse_dh", "dW"}
    for v in d["roofline_kernels"].values():
        assert 0 < v["frac"] < 1.2
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    rc = d["recompute_path"]
    assert rc["path"] == "tcgen05_recompute" and rc["value"] > 0 and rc["executed_flop_per_token"] > 0
