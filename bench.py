"""Benchmark of the fused LM-head + cross-entropy micro-step library on GB300.

One step = one optimizer step of the GPT-2 124M LM-head workload: G micro-steps of
lmce_microstep (logits tiles -> online logsumexp and loss, dlogits -> dW and dh) and
one lmce_finalize, on synthetic seeded inputs already resident in device memory.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl lmce|reference]

Prints one JSON line (rank 0).  ``--impl reference`` times the float64 CPU oracle on
bounded samples of the same workload instead.  Under torchrun every rank runs its
own micro-steps (weak scaling); the valid count and dW are SUM-reduced over ranks.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s fused LM-head+CE fwd+bwd (1×GB300); % of dense BF16 tensor peak"
UNIT = "tokens/s"
FP32_LANES_PER_SM = 128
NOMINAL_BF16_TFLOPS = 2250.0   # GB300 dense bf16 datasheet figure, for context
N_SM = 152


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=40)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="lmce", choices=["lmce", "reference"])
    p.add_argument("--workload", default="gpt2_124m_head")
    p.add_argument("--path", default="auto", choices=["auto", "simt", "tcgen05", "tcgen05_two_pass", "tcgen05_recompute"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--final-norm", default=None, choices=["layernorm", "rmsnorm"],
                   help="ln_f in front of the head (lmce_microstep_ln); inputs become the rows x before it")
    p.add_argument("--compact", action="store_true",
                   help="micro-steps over the valid rows only (lmce_microstep_compact)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-sample-rows", type=int, default=2048)
    return p.parse_args()


def ncu_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the ncu summaries under profiles/, or None when the
    kernel source changed since the counters were taken."""
    import glob
    import hashlib
    import re

    src = os.path.join(ROOT, "grad_lmce_microstep_gb300", "csrc", "lmce_tc.cu")
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    for f in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        txt = open(f).read()
        m = re.search(r"traffic_bytes_per_launch:(.*)", txt)
        h = re.search(r"sha256\[:16\] = ([0-9a-f]{16})", txt)
        if not m or not h or h.group(1) != sha:
            continue
        for kv in m.group(1).split():
            k, v = kv.split("=")
            if k == kernel:
                return int(v)
    return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}, \
        "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(5)
        except Exception:
            self.proc.kill()
        self.t.join(2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_sample_rate(w, rows: int):
    """Float64 oracle tokens/s on one micro-step of ``rows`` rows (full C and V)."""
    from oracle import lmce_oracle as O

    h, y = w.micro[0]
    h = h[:rows]
    y = y[:rows]
    t0 = time.perf_counter()
    O.step([(h, y)], w.W)
    dt = time.perf_counter() - t0
    return rows / dt, dt


def run_reference(args, rank, world):
    from grad_lmce_microstep_gb300 import inputs as I

    if rank != 0:
        return
    w = I.make(args.workload)
    rows = args.cpu_sample_rows
    for _ in range(args.warmup):
        oracle_sample_rate(w, rows)
    rates = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        r, _ = oracle_sample_rate(w, rows)
        rates.append(r)
    wall = time.perf_counter() - t_all
    value = rows * args.steps / wall
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "C": w.C, "V": w.V,
                   "sample": f"one micro-step of {rows} rows of micro-batch 0 per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{rows} rows x full V x full C per step, float64 numpy/BLAS"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_lmce(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from grad_lmce_microstep_gb300 import dp
    from grad_lmce_microstep_gb300 import inputs as I
    from grad_lmce_microstep_gb300 import lmce as M

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = I.make(args.workload, seed=rank)
    if rank:   # every rank's own rows, one model: the tied matrix of seed 0 on all ranks
        w.W = I.draw_W(w.V, w.C, w.dtype, 0)
    if args.final_norm:   # the residual stream in front of ln_f: shifted, scaled rows
        w.micro = [((h.float() * 1.7 + 0.4).to(h.dtype), y) for h, y in w.micro]
    W = w.W.to(dev)
    mbs = [(h.to(dev), y.to(dev)) for h, y in w.micro]
    dhs = [torch.empty_like(h) for h, _ in mbs]
    dW = torch.empty(w.V, w.C, dtype=torch.float32, device=dev)
    max_N = max(int(y.numel()) for _, y in mbs)
    L = M.Lmce(w.C, w.V, max_N, dW, w.dtype, norm="global", grad_accum_steps=w.G, path=args.path,
               compact=args.compact, final_norm=bool(args.final_norm))
    if args.final_norm:
        gen = torch.Generator().manual_seed(rank)
        ln_gamma = (1 + 0.1 * torch.randn(w.C, generator=gen)).to(dev)
        ln_beta = (0.1 * torch.randn(w.C, generator=gen)).to(dev) if args.final_norm == "layernorm" else None
        ln_dgamma = torch.empty(w.C, device=dev)
        ln_dbeta = torch.empty(w.C, device=dev) if ln_beta is not None else None
    nvs = w.valid_counts()
    gv = dp.global_valid_count(sum(w.valid_counts()), device=dev if world > 1 else None)
    stream = torch.cuda.current_stream(dev)
    tokens_rank = w.tokens

    def micro(h, y, n_valid, dh):
        if args.final_norm:   # h is x and dh is dx here
            L.microstep_ln(h, ln_gamma, ln_beta, W, y, gv, dh, ln_dgamma, ln_dbeta, args.final_norm, 1e-5,
                           stream=stream, n_valid=n_valid if args.compact else None)
        elif args.compact:
            L.microstep_compact(h, W, y, n_valid, gv, dh, stream=stream)
        else:
            L.microstep(h, W, y, gv, dh, stream=stream)

    def step():
        for (h, y), dh, nv in zip(mbs, dhs, nvs):
            micro(h, y, nv, dh)
        res = L.finalize(stream=stream)
        if world > 1:
            dp.reduce_step(dW, res[0], res[1], extra=(ln_dgamma, ln_dbeta) if args.final_norm else ())
        return res

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        res = step()
    barrier()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    launches0 = L.launches
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier()
    ev0.record(stream)
    for _ in range(args.steps):
        res = step()
    ev1.record(stream)
    barrier()
    launches = L.launches - launches0
    clocks = sampler.stop() if sampler else None
    # per-kernel device times: a second timed pass of the same steps with the library's CUDA-event
    # records around every kernel (kept out of the pass above: the records sit between the
    # launches and cost 1-5 % of a step)
    L.profile(True)
    for _ in range(args.steps):
        step()
    barrier()
    L.profile(False)
    prof = L.profile_read()
    # host cost of one micro-step call through the binding (argument checks, cached tensor maps,
    # the launches), timed on the host with no event records; the GPU work runs behind it
    host_ns = []
    for _ in range(3):
        for (h, y), dh, nv in zip(mbs, dhs, nvs):
            t0 = time.perf_counter_ns()
            micro(h, y, nv, dh)
            host_ns.append(time.perf_counter_ns() - t0)
        L.finalize(stream=stream)
    host_us = statistics.median(host_ns) / 1e3
    ms = ev0.elapsed_time(ev1)
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_max = float(t.item())
    value = tokens_rank * world * args.steps / (ms_max / 1e3)

    # end to end through the public API: pinned host inputs copied every step, loss read back.
    # The copies run on their own stream into two alternating sets of device buffers (a data
    # loader's double buffering): micro-step k waits for its inputs' copy event, and the next
    # step's copies are issued while this step computes.  Every step's h2d bytes are copied
    # inside the timed region.
    e2e = None
    if not args.no_e2e:
        hs_host = [h.cpu().pin_memory() for h, _ in w.micro]
        ys_host = [y.cpu().pin_memory() for _, y in w.micro]
        h_dev = [[torch.empty_like(h) for h, _ in mbs] for _ in range(2)]
        y_dev = [[torch.empty_like(y) for _, y in mbs] for _ in range(2)]
        ready = [[torch.cuda.Event() for _ in mbs] for _ in range(2)]   # set b, micro-step k copied
        used = [[torch.cuda.Event() for _ in mbs] for _ in range(2)]    # set b, micro-step k computed
        copy_stream = torch.cuda.Stream(device=dev)

        def issue_copies(b):
            with torch.cuda.stream(copy_stream):
                for k in range(len(mbs)):
                    copy_stream.wait_event(used[b][k])   # the set's previous step has consumed it
                    h_dev[b][k].copy_(hs_host[k], non_blocking=True)
                    y_dev[b][k].copy_(ys_host[k], non_blocking=True)
                    ready[b][k].record(copy_stream)

        def step_e2e(b):
            for k, dh in enumerate(dhs):
                stream.wait_event(ready[b][k])
                micro(h_dev[b][k], y_dev[b][k], nvs[k], dh)
                used[b][k].record(stream)
                if k == 0:
                    issue_copies(1 - b)   # the next step's inputs stream in meanwhile
            res = L.finalize(stream=stream)
            if world > 1:   # the same exchange as the device-timed step
                dp.reduce_step(dW, res[0], res[1], extra=(ln_dgamma, ln_dbeta) if args.final_norm else ())
            return res

        issue_copies(0)
        for i in range(max(1, args.warmup)):
            step_e2e(i & 1)
        b0 = max(1, args.warmup) & 1
        barrier()
        t0 = time.perf_counter()
        for i in range(args.steps):
            step_e2e((b0 + i) & 1)
        copy_stream.synchronize()   # the copies issued for a step after the last one are timed too
        barrier()
        dt = time.perf_counter() - t0
        t = torch.tensor([dt], dtype=torch.float64, device=dev)
        if world > 1:
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
        h2d = sum(h.numel() * h.element_size() + y.numel() * y.element_size() for h, y in w.micro)
        e2e = {"value": tokens_rank * world * args.steps / float(t.item()), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": 48}

    # the squared dW norm a gradient clip needs (lmce_dw_sumsq): one read of the fp32 dW, timed by
    # the library's own event records around its two launches; after three untimed calls (the GPU
    # idles between the timed region and here), the best of five
    for _ in range(3):
        sq_value = L.dw_sumsq(stream=stream)
    sq_ms, sq_n = float("inf"), 0
    for _ in range(5):
        L.profile(True)
        sq_value = L.dw_sumsq(stream=stream)
        ms_r, n_r = L.profile_read().get("finish", (0.0, 0))
        if n_r and ms_r < sq_ms:
            sq_ms, sq_n = ms_r, n_r
    L.profile(False)
    if sq_n == 0:
        sq_ms = 0.0

    # the AdamW update of the tied matrix after the step (lmce_adamw): one pass over dW, the fp32
    # master weights and both moments, with the bf16 W for the next forward written beside them;
    # 30 bytes per element.  Timed like the norm: three untimed calls, then the best of five.
    p_master = W.float()
    m_st = torch.zeros_like(p_master)
    v_st = torch.zeros_like(p_master)
    W_next = torch.empty_like(W)
    clip = M.clip_coef(sq_value, 1.0)
    aw_ms, aw_n = float("inf"), 0
    for t in range(1, 9):
        if t > 3:
            L.profile(True)
        L.adamw(p_master, m_st, v_st, t, 6e-4, W_next if w.dtype == "bf16" else None, clip=clip, stream=stream)
        if t > 3:
            ms_r, n_r = L.profile_read().get("finish", (0.0, 0))
            if n_r and ms_r < aw_ms:
                aw_ms, aw_n = ms_r, n_r
    L.profile(False)
    if aw_n == 0:
        aw_ms = 0.0
    aw_bytes = p_master.numel() * (4 + 8 + 8 + 8 + (2 if w.dtype == "bf16" else 0))
    del p_master, m_st, v_st, W_next

    # the same steps on the path whose dW pass recomputes the logits (LMCE_PATH_TCGEN05_RECOMPUTE:
    # logits and dlogits never leave the chip, no N x V scratch), device-timed like the headline
    recompute = None
    if L.path == "tcgen05" and not args.compact and not args.final_norm and world == 1:
        dW_r = torch.empty_like(dW)
        L_r = M.Lmce(w.C, w.V, max_N, dW_r, w.dtype, norm="global", grad_accum_steps=w.G, path="tcgen05_recompute")

        def step_r():
            for (h, y), dh in zip(mbs, dhs):
                L_r.microstep(h, W, y, gv, dh, stream=stream)
            return L_r.finalize(stream=stream)

        for _ in range(max(3, args.warmup)):
            step_r()
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(args.steps):
            step_r()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        ms_r = ev0.elapsed_time(ev1) / args.steps
        v_r = tokens_rank / (ms_r / 1e3)
        recompute = {"path": "tcgen05_recompute", "value": v_r, "unit": UNIT, "ms_per_step": ms_r,
                     "frac_of_peak": v_r * sum(nvs) / tokens_rank * 6.0 * w.C * w.V / 1e12 / peaks()[0]["bf16_tflops"],
                     "executed_flop_per_token": 8.0 * w.C * w.V}
        L_r.close()
        del dW_r

    if rank != 0:
        return

    pk, pk_kind = peaks()
    dw_bytes = dW.numel() * dW.element_size()
    sq_gbs = dw_bytes / (sq_ms * 1e-3) / 1e9 if sq_ms > 0 else None
    dw_sumsq = {"ms": sq_ms, "launches": sq_n, "bytes": int(dw_bytes), "achieved_gbs": sq_gbs,
                "peak_gbs": pk["hbm_gbs"], "frac": sq_gbs / pk["hbm_gbs"] if sq_gbs else None,
                "bound": "hbm", "value": sq_value}
    aw_gbs = aw_bytes / (aw_ms * 1e-3) / 1e9 if aw_ms > 0 else None
    final_norm = None
    if args.final_norm and "ln" in prof and prof["ln"][1] > 0:
        # Per micro-step, plain: the forward reads x and writes h, the backward reads dh and x and
        # writes dx (5 row tensors over all rows).  Compacted (ln_f fused with the compaction):
        # the forward reads the valid rows of x and writes them normalised, the backward reads dh
        # and x of the valid rows and writes dx of every row (4 valid-row tensors + 1 full one),
        # and the compaction's count and scan read the targets; the compaction launches are
        # timed with ln_f's.  Both: the dgamma / dbeta partials (fp32, one row per backward block
        # of at most one per SM) written and read once.
        esz = 2 if w.dtype == "bf16" else 4
        nmicro = args.steps * w.G
        ln_ms = prof["ln"][0] / nmicro
        n_ln = prof["ln"][1]
        rows_all = tokens_rank // w.G
        rows_valid = sum(nvs) // w.G
        rows = rows_all
        rpb = -(-rows // N_SM)
        part_bytes = 2 * 2 * 4 * w.C * (-(-rows // rpb))
        if args.compact:
            ln_ms += prof.get("compact", (0.0, 0))[0] / nmicro
            n_ln += prof.get("compact", (0.0, 0))[1]
            ln_bytes = (4 * rows_valid + rows_all) * w.C * esz + 4 * rows_all + part_bytes
        else:
            ln_bytes = 5 * rows_all * w.C * esz + part_bytes
        ln_gbs = ln_bytes / (ln_ms * 1e-3) / 1e9
        final_norm = {"kind": args.final_norm, "ms_per_micro_step": ln_ms, "launches_per_micro_step":
                      n_ln / nmicro, "bytes_per_micro_step": int(ln_bytes), "achieved_gbs": ln_gbs,
                      "peak_gbs": pk["hbm_gbs"], "frac": ln_gbs / pk["hbm_gbs"], "bound": "hbm",
                      "with_compaction": bool(args.compact)}
    adamw = {"ms": aw_ms, "launches": aw_n, "bytes": int(aw_bytes), "achieved_gbs": aw_gbs,
             "peak_gbs": pk["hbm_gbs"], "frac": aw_gbs / pk["hbm_gbs"] if aw_gbs else None, "bound": "hbm",
             "hyper": {"lr": 6e-4, "betas": [0.9, 0.95], "eps": 1e-8, "weight_decay": 0.1, "clip": clip}}
    # algorithmic work: 6 C V flops per token for the whole path, 2 C V for each of the three
    # contractions (logits, dW, dh); the recomputed logits of the gradient passes are not counted
    # (the one-pass logsumexp + dh kernel does the logits and dh contractions: 4 C V).
    flop_tok = 6.0 * w.C * w.V
    kinds = {k: v for k, v in prof.items() if v[1] > 0}
    dom = max(kinds, key=lambda k: kinds[k][0])
    dom_ms, dom_n = kinds[dom]
    tok_per_launch = tokens_rank / w.G
    valid_rank = sum(nvs)
    # rows one heavy launch processes: every row, or the valid rows alone when compacted
    rows_per_launch = valid_rank / w.G if args.compact else tok_per_launch
    # a wide C runs each gradient pass once per range of C columns (two launches at C = 1024): the
    # micro-step's algorithmic work is shared between those launches
    runs = dom_n / (args.steps * w.G)
    alg_flop_launch = {"lse": 2.0, "dW": 2.0, "dh": 2.0, "lse_dh": 4.0}.get(dom, 0.0) * w.C * w.V * rows_per_launch \
        / max(runs, 1.0)
    achieved = alg_flop_launch / (dom_ms / dom_n / 1e3) / 1e12
    # the ncu traffic figures in profiles/ were taken on the 124M head on the default path
    traffic_of = (lambda k: ncu_traffic(k)) if (args.workload == "gpt2_124m_head" and L.path == "tcgen05" and
                                               not args.compact and not args.final_norm) else (lambda k: None)
    # the same figure for each heavy kernel (algorithmic flops per launch / its average launch time)
    per_kernel = {}
    for k in ("lse_dh", "dW", "dh", "lse"):
        if k in kinds and kinds[k][1] > 0:
            runs_k = kinds[k][1] / (args.steps * w.G)
            flop_k = {"lse": 2.0, "dW": 2.0, "dh": 2.0, "lse_dh": 4.0}[k] * w.C * w.V * rows_per_launch / max(runs_k, 1.0)
            per_kernel[k] = flop_k / (kinds[k][0] / kinds[k][1] / 1e3) / 1e12
    if L.path.startswith("tcgen05"):
        # the burst cuBLAS figure: the kernels run at the clocks of a short timed region (the
        # sustained figure was taken over seconds at a lower, power-capped clock)
        peak = pk["bf16_tflops"]
        bound = "tensor"
    else:
        clk = (clocks or {}).get("sm_max_mhz") or pk.get("sm_max_mhz", 2070.0)
        peak = N_SM * FP32_LANES_PER_SM * 2 * clk * 1e6 / 1e12
        bound = "alu"
    # useful work: 6 C V flop per VALID token (an ignored row's gradient is zero)
    valid_per_s = value * valid_rank / tokens_rank
    achieved_step = valid_per_s / world * flop_tok / 1e12   # TFLOP/s per GPU on 6 C V per valid token
    total_frac = achieved_step / pk["bf16_tflops"]
    sustained = pk.get("bf16_tflops_sustained")
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        rate, secs = oracle_sample_rate(w, args.cpu_sample_rows)
        cpu = {"value": rate, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"extrapolated from a sample: one micro-step of {args.cpu_sample_rows} rows "
                         f"(full C={w.C}, V={w.V}), float64 numpy/BLAS, {secs:.1f} s"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "fp32",
        "data": "synthetic",
        "config": {"workload": args.workload, "tokens_per_step": tokens_rank * world, "micro_steps": w.G,
                   "micro_batch_tokens": int(tok_per_launch), "valid_tokens": [int(n) for n in nvs],
                   "C": w.C, "V": w.V, "path": L.path, "compact": bool(args.compact),
                   "final_norm": args.final_norm,
                   "parallelism": f"dp{world}",
                   "l2": "no flush: inputs larger than L2 (per step %d distinct h buffers of %.0f MB, "
                         "W %.0f MB, fp32 dW %.0f MB)" % (w.G, mbs[0][0].numel() * 2 / 1e6,
                                                         W.numel() * W.element_size() / 1e6,
                                                         dW.numel() * 4 / 1e6)},
        "valid_tokens_per_s": valid_per_s,
        "frac_of_peak": {"value": total_frac, "achieved_tflops": achieved_step, "flop_per_token": flop_tok,
                         "tokens": "valid", "peak_tflops": pk["bf16_tflops"], "peak": f"bf16 burst, {pk_kind}",
                         "of_sustained": achieved_step / sustained if sustained else None,
                         "sustained_tflops": sustained, "of_nominal_dense": achieved_step / NOMINAL_BF16_TFLOPS,
                         "nominal_dense_tflops": NOMINAL_BF16_TFLOPS},
        "roofline": {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic_of(dom),
                     "frac_of_sustained": achieved / sustained if (sustained and bound == "tensor") else None,
                     "peak_source": ("bf16_tflops (burst) of " + pk_kind) if bound == "tensor"
                     else "fp32 FFMA: 152 SMs x 128 lanes x 2 flop x max SM clock"},
        "roofline_kernels": {k: {"achieved": v, "peak": peak, "unit": "TFLOP/s", "frac": v / peak,
                                 "traffic": traffic_of(k)}
                             for k, v in per_kernel.items()
                             if bound == "tensor" and kinds[k][0] / kinds[k][1] > 0.05},
        "kernels_ms": {k: {"total_ms": v[0], "launches": v[1], "avg_ms": v[0] / v[1]} for k, v in kinds.items()},
        "kernels_ms_source": "a second timed pass of the same steps with CUDA events around every kernel",
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "host_us_per_microstep": host_us,
        "dw_sumsq": dw_sumsq,
        "adamw": adamw,
        "final_norm": final_norm,
        "recompute_path": recompute,
        "clocks": clocks,
        "check": {"loss_mean": res[2], "valid": res[1]},
    }
    print(json.dumps(line), flush=True)
    L.close()


def main():
    args = parse()
    from grad_lmce_microstep_gb300 import launch

    if args.gpus > 1 and not launch.under_launcher():
        # started by hand: one rank per GPU, re-executed under torch.distributed.run
        if args.impl == "lmce":
            import torch

            have = torch.cuda.device_count()
            if have < args.gpus:
                print(f"bench.py: --gpus {args.gpus} needs {args.gpus} visible GPUs, found {have}", file=sys.stderr)
                sys.exit(2)
        sys.exit(launch.relaunch(os.path.abspath(__file__), sys.argv[1:], args.gpus))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "lmce" and world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but {world} ranks were started", file=sys.stderr)
        sys.exit(2)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_lmce(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
