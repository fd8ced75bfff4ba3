"""Run a few decode steps of a workload, for profilers (ncu) on a small footprint.

    python -m block_sparse_kv_pred_gb300.profile_step --config qwen3_14b --steps 3

By default the K/V pool holds only the GPU's share of the cache (the resident blocks and each
unit's tail block, 1.34 GB for the Qwen3-14B-shaped layer) and the whole cache, which the
digests are built from, is freed before the steps run, so the device holds about 1.8 GB and
every kernel reads exactly the bytes the benchmark's step reads.  ``--pool-slots N`` instead
makes all blocks share N pool slots (outputs then are not checked: an aliased pool does not hold
each block's own keys).
"""
from __future__ import annotations

import argparse

import torch

from . import workload as W
from .step import setup_step


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="qwen3_14b")
    ap.add_argument("--pool-slots", type=int, default=0)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--serial", action="store_true", help="one stream, full grids")
    a = ap.parse_args()
    shape = W.CONFIGS[a.config]()
    wl, t, step = setup_step(shape, torch.device("cuda", 0), pool_slots=a.pool_slots or None, serial=a.serial,
                             keep_all=False)
    ev = torch.cuda.Event()
    ev.record()
    step.begin(ev)
    for _ in range(a.steps):
        step.issue()
    step.end(None)
    torch.cuda.synchronize()
    status = int(t["status"].item())
    print(f"profile_step {shape.name}: {a.steps} steps, pool slots {t['n_slots']}, status {status}")
    if status:
        raise SystemExit(1)


if __name__ == "__main__":
    main()
