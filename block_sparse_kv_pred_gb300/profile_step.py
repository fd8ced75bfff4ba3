"""Run a few decode steps of a workload, for profilers (ncu) on a small footprint.

    python -m block_sparse_kv_pred_gb300.profile_step --config qwen3_14b --pool-slots 65536 --steps 3

``--pool-slots`` (0: one slot per block) makes blocks share K/V pool slots so the device holds about
1.3 GB instead of 5.4 GB while every kernel keeps the launch configuration,
the digest size and the block counts of the full workload.  Outputs are not
checked (the aliased pool does not hold each block's own keys).
"""
from __future__ import annotations

import argparse

import torch

from . import workload as W
from .step import setup_step


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="qwen3_14b")
    ap.add_argument("--pool-slots", type=int, default=65536)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--serial", action="store_true", help="one stream, full grids")
    a = ap.parse_args()
    shape = W.CONFIGS[a.config]()
    wl, t, step = setup_step(shape, torch.device("cuda", 0), pool_slots=a.pool_slots or None, serial=a.serial)
    ev = torch.cuda.Event()
    ev.record()
    step.begin(ev)
    for _ in range(a.steps):
        step.issue()
    step.end(None)
    torch.cuda.synchronize()
    status = int(t["status"].item())
    print(f"profile_step {shape.name}: {a.steps} steps, pool slots {wl.n_slots}, status {status}")
    if status:
        raise SystemExit(1)


if __name__ == "__main__":
    main()
