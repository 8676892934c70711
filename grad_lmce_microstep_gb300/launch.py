"""One process per GPU for the data-parallel path.

The pages run data parallelism as one process per GPU started by torchrun
("Multi-GPU calculation of gradients for accelerated training", section "DDP
averages gradients across processes").  A script started by hand with ``--gpus N``
re-executes itself here under ``torch.distributed.run`` with N local ranks on
127.0.0.1; every rank then reads RANK / LOCAL_RANK / WORLD_SIZE / MASTER_* from
its environment as it would under torchrun.
"""

from __future__ import annotations

import os
import socket
import subprocess
import sys


def under_launcher() -> bool:
    """True inside a rank that torchrun (or this module) started."""
    return "WORLD_SIZE" in os.environ and "RANK" in os.environ and "LOCAL_RANK" in os.environ


def free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def relaunch(script: str, argv, nproc: int, env=None) -> int:
    """Run ``script argv`` as ``nproc`` local ranks; returns the launcher's exit code (non-zero
    when any rank failed)."""
    if nproc < 1:
        raise ValueError("nproc must be >= 1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={nproc}",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}", script, *argv]
    e = dict(os.environ if env is None else env)
    e.setdefault("OMP_NUM_THREADS", "1")
    return subprocess.call(cmd, env=e)
