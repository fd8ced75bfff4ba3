"""Multi-step decode of one layer through the libscout C ABI: the residency sweep.

ScoutAttention (arXiv HTML), section 3.4 and Algorithm 1: a decode step appends one
token per sequence, selects the next blocks with the predicted query against the
previous step's CPU work list (so only the delta is new CPU work), and attends the
resident part of the selection on the GPU; every ``recall_every`` steps the selected
blocks that are not resident are brought in, taking the slots of unselected resident
blocks (lowest score first).

Readings taken where the pages leave it open (the same as the oracle's):
  * the GPU holds k blocks per (sequence, KV head) plus the block being written; the
    initial resident set is the top-k of the first decode step's true query (the
    blocks found important right after prefill) and each unit's tail block;
  * the true query walks by ``Workload.walk`` (step cosine ~0.96) and the predicted
    query sits at cosine 0.93 to it; selection uses the predicted query, GPU attention
    the true one;
  * a token that starts a new block gets a fresh page (copied from the host copy of
    the layer's KV, which stands for the page the model writes), and the block being
    written is never evicted by a recall.

Per step the sweep reports the CPU work-list size, its delta against the previous step,
the CPU ratio (CPU blocks over the budget) and, on recall steps, the bytes moved and
the host-to-device rate.  ``python -m block_sparse_kv_pred_gb300.sweep`` runs the
64-step sweep at batch 16 and 64K context and prints one line per step;
``--profile-layers L`` instead decodes L seeded layers without recalls and prints each
layer's recall interval (section 3.4, threshold ``--beta``).
"""
from __future__ import annotations

import argparse
import json
import time

import numpy as np
import torch

import block_sparse_kv_pred_gb300 as bs
from block_sparse_kv_pred_gb300 import workload as W
from block_sparse_kv_pred_gb300.workload import device as WD


def c4_shape(steps: int = 64) -> W.Shape:
    """Batch 16, 40/8 heads, 64K context (+ room for the appended tokens), 32-token pages,
    budget 2048 tokens (k = 64 blocks per KV head)."""
    T0 = 65536
    return W.Shape("sweep_b16_t64k", B=16, Hq=40, Hkv=8, T=T0 + steps, P=32, k=64, resident_frac=0.0,
                   seq_lens=(T0,) * 16, hidden=0)


def _bits(mask: np.ndarray) -> np.ndarray:
    """bool [units][nblk] -> uint32 [units][words]."""
    U, nb = mask.shape
    words = -(-nb // 32)
    padded = np.zeros((U, words * 32), dtype=np.uint64)
    padded[:, :nb] = mask
    w = padded.reshape(U, words, 32) << np.arange(32, dtype=np.uint64)
    return w.sum(axis=-1).astype(np.uint32)


class DecodeSweep:
    """The layer's state on the GPU and the host, and one method per decode step."""

    def __init__(self, shape: W.Shape, steps: int, recall_every: int = 16, device="cuda", host=None,
                 gather=True, pages=False, cpu_pool=None):
        """``recall_every`` 0: no recall (the profile from which recall intervals are read).
        ``host``: optional pair of pinned bf16 host tensors of at least [units][nblk][P][D]
        elements each, reused for the host copy of the layer's K/V (a multi-layer sweep keeps
        one pair).  ``gather``: recalls move their pages with the gather kernel reading mapped
        host memory (scout_recall_gather_async); False: one cudaMemcpyAsync per run of pages.
        ``pages``: residency per page, a page being one block of a sequence for all its KV heads
        (the 128 KB transfer unit of section 2.3, Figure 3): the initial resident pages are the k
        most important of each sequence (importance: the largest of its heads' scores, ties to the
        lower block) plus the page being written, and each recall follows scout_plan_recall_pages
        with the page being written counted as selected by every head; otherwise per block.
        ``cpu_pool``: a ``CpuPool``; each step then also computes the CPU side (section 3.2: the
        CPU list attended with Q_pred on the host copy of the K/V) on the pool's threads and
        reports its time beside the GPU time of the step's kernels."""
        self.gather = gather
        self.pages = pages
        self.cpu_pool = cpu_pool
        self.s = s = shape
        self.steps, self.recall_every = steps, recall_every
        dev = self.dev = torch.device(device)
        self.wl = wl = W.Workload(s)
        self.qs, self.ps = wl.walk(steps)
        U, nb, P, D = s.units, s.nblk, s.P, s.D
        full = WD.materialize(wl, device=dev, with_gemm=False)
        # every block in logical order [U][nblk][P][D]; its host copy (pinned) is the CPU-resident
        # KV that recalls read
        order = full["page_table"].reshape(-1).long()
        logical = {}
        for i, n in enumerate(("K", "V")):
            logical[n] = full[n + "_pool"][order]
            if host is None:
                hbuf = torch.empty((U, nb, P, D), dtype=torch.bfloat16, pin_memory=True)
            else:
                hbuf = host[i].view(-1)[: U * nb * P * D].view(U, nb, P, D)
            hbuf.copy_(logical[n].reshape(U, nb, P, D))
            setattr(self, "h" + n, hbuf)
        # prefill: digests over every valid block (the whole context was on the GPU)
        self.seq = wl.seq_len.astype(np.int32).copy()
        self.d_seq = WD.to_dev(self.seq, dev)
        self.digest = torch.empty((s.B, s.Hkv, nb, 2, D), dtype=torch.bfloat16, device=dev)
        bs.build_digest("minmax", full["K_pool"], full["page_table"], self.d_seq, s.B, s.Hkv, P, self.digest)
        # initial residency: the top-k of the first step's true query, plus the tail block
        self.ws = bs.score_topk_workspace(s.B, s.Hkv, nb, device=dev)
        none = torch.zeros((s.B, s.Hkv, s.words), dtype=torch.int32, device=dev)
        sc0 = torch.empty((s.B, s.Hkv, nb), dtype=torch.float32, device=dev)
        first = bs.score_topk("minmax", WD.to_dev(self.qs[0], dev), self.digest, self.d_seq, none, s.B, s.Hq, s.Hkv,
                              P, nb, s.k, self.ws, scores=sc0)
        topk = first["topk"].cpu().numpy().reshape(U, -1)
        tc = first["topk_count"].cpu().numpy().reshape(-1)
        res = np.zeros((U, nb), dtype=bool)
        if pages:
            imp = sc0.cpu().numpy().max(axis=1)  # [B][nblk], -inf past the valid blocks
            for b in range(s.B):
                nv = -(-int(self.seq[b]) // P)
                order = sorted(range(nv), key=lambda j: (-float(imp[b, j]), j))[: s.k]
                res[b * s.Hkv:(b + 1) * s.Hkv, order] = True
                res[b * s.Hkv:(b + 1) * s.Hkv, nv - 1] = True
        else:
            for u in range(U):
                res[u, topk[u, :tc[u]]] = True
                res[u, (int(self.seq[u // s.Hkv]) - 1) // P] = True
        del sc0
        # the pool: k + 1 resident blocks per unit and room for the blocks the decode starts
        spare_per_unit = -(-steps // P) + 1
        self.n_slots = int(res.sum()) + spare_per_unit * U
        table = np.full((U, nb), -1, dtype=np.int32)
        table[res] = np.arange(int(res.sum()), dtype=np.int32)
        self.spare = list(range(int(res.sum()), self.n_slots))
        src = torch.from_numpy(np.flatnonzero(res.reshape(-1)).astype(np.int64)).to(dev)
        self.K_pool = torch.zeros((self.n_slots, P, D), dtype=torch.bfloat16, device=dev)
        self.V_pool = torch.zeros((self.n_slots, P, D), dtype=torch.bfloat16, device=dev)
        self.K_pool[: src.numel()] = logical["K"][src]
        self.V_pool[: src.numel()] = logical["V"][src]
        del full, order, src, logical
        torch.cuda.empty_cache()
        self.res, self.table = res, table
        self.d_table = WD.to_dev(table.reshape(s.B, s.Hkv, nb), dev)
        self.d_bits = WD.to_dev(_bits(res).reshape(s.B, s.Hkv, -1).view(np.int32), dev)
        self.wa = bs.sparse_attn_workspace(s.B, s.Hq, s.Hkv, P, device=dev)
        self.scores = torch.empty((s.B, s.Hkv, nb), dtype=torch.float32, device=dev)
        self.side = torch.cuda.Stream(dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.prev = None
        self.t = 0

    def _move_in(self, ops) -> tuple[int, float]:
        """Copy the ops' blocks from the host into their slots on the side stream, then commit
        the page table and residency bits after the copy.  Returns (bytes, seconds)."""
        s = self.s
        d_ops = WD.to_dev(np.asarray(ops, dtype=np.int32).reshape(-1, 4), self.dev)
        self.side.wait_stream(torch.cuda.current_stream(self.dev))  # d_ops is on the device
        t0, done = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(self.side)
        if self.gather:
            bs.recall_gather_async(d_ops, self.hK, self.hV, self.K_pool, self.V_pool, s.B, s.Hkv, s.P, s.nblk, self.side,
                                   status=self.status)
        else:
            bs.recall_async([tuple(int(x) for x in r) for r in ops], self.hK, self.hV, self.K_pool, self.V_pool, s.B,
                            s.Hkv, s.P, s.nblk, self.side)
        done.record(self.side)
        bs.commit_residency(d_ops, self.d_table, self.d_bits, self.n_slots, s.B, s.Hkv, wait_event=done)
        done.synchronize()
        return len(ops) * 2 * s.P * s.D * 2, t0.elapsed_time(done) / 1e3

    def step(self) -> dict:
        """One decode step.  Returns host copies of its outputs and the state it ran on."""
        s, t = self.s, self.t
        U, P = s.units, s.P
        # one token per sequence; a block that starts gets a fresh page
        self.seq += 1
        fresh = []
        for u in range(U):
            j = (int(self.seq[u // s.Hkv]) - 1) // P
            if not self.res[u, j]:
                slot = self.spare.pop()
                fresh.append((u, j, slot, -1))
                self.res[u, j], self.table[u, j] = True, slot
        if fresh:
            self._move_in(fresh)
        self.d_seq = WD.to_dev(self.seq, self.dev)
        tail = WD.to_dev(np.array([[u, (int(self.seq[u // s.Hkv]) - 1) // P] for u in range(U)], np.int32), self.dev)
        qp, q = WD.to_dev(self.ps[t], self.dev), WD.to_dev(self.qs[t], self.dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        if self.cpu_pool is not None and hasattr(torch.cuda, "_sleep"):
            # the GPU spins ~1 ms first (PyTorch's test helper), so that the three launches below are
            # queued before it reaches them and the events time the kernels back to back, not the
            # host's launch gaps (without it the gaps are counted)
            torch.cuda._sleep(2_000_000)
        ev[0].record()  # the step's kernels: digest append, selection, attention
        bs.build_digest("minmax", self.K_pool, self.d_table, self.d_seq, s.B, s.Hkv, P, self.digest, block_list=tail)
        resident_before = self.res.copy()
        out = bs.score_topk("minmax", qp, self.digest, self.d_seq, self.d_bits, s.B, s.Hq, s.Hkv, P, s.nblk, s.k,
                            self.ws, prev_cpu=self.prev, scores=self.scores, status=self.status)
        O, lse = bs.sparse_attn(q, self.K_pool, self.V_pool, self.d_table, self.d_seq, out["res"], out["res_count"],
                                s.B, s.Hq, s.Hkv, P, s.k, s.scale, self.wa, status=self.status)
        ev[1].record()
        torch.cuda.synchronize(self.dev)
        if int(self.status.item()) != 0:
            raise RuntimeError(f"device status {int(self.status.item())} at step {t}")
        rec = {"t": t, "seq": self.seq.copy(), "resident": resident_before, "O": O.cpu().numpy(),
               "lse": lse.cpu().numpy(), "prev_cpu": None}
        if self.prev is not None:
            rec["prev_cpu"] = (self.prev[0].cpu().numpy().reshape(U, -1), self.prev[1].cpu().numpy().reshape(-1))
        for n in ("topk", "res", "cpu", "delta"):
            rec[n] = out[n].cpu().numpy().reshape(U, -1)
            rec[n + "_count"] = out[n + "_count"].cpu().numpy().reshape(-1)
        self.prev = (out["cpu"].clone(), out["cpu_count"].clone())
        n_cpu, n_delta = int(rec["cpu_count"].sum()), int(rec["delta_count"].sum())
        stats = {"step": t, "cpu_blocks": n_cpu, "delta_blocks": n_delta, "cpu_ratio": n_cpu / (s.k * U),
                 "recall_blocks": 0, "recall_bytes": 0, "recall_h2d_gbs": None, "gpu_ms": ev[0].elapsed_time(ev[1])}
        if self.cpu_pool is not None:
            # the CPU side of this step's selection (the next layer's partial, one layer ahead)
            h_q = torch.from_numpy(np.ascontiguousarray(self.ps[t]).view(np.int16)).view(torch.bfloat16)
            o_cpu = torch.empty((s.B, s.Hq, s.D), dtype=torch.float32)
            l_cpu = torch.empty((s.B, s.Hq), dtype=torch.float32)
            c0 = time.perf_counter()
            self.cpu_pool.submit(h_q, self.hK, self.hV, torch.from_numpy(self.seq.copy()),
                                 torch.from_numpy(rec["cpu"].reshape(s.B, s.Hkv, s.k).copy()),
                                 torch.from_numpy(rec["cpu_count"].reshape(s.B, s.Hkv).copy()), s.B, s.Hq, s.Hkv, P,
                                 s.k, s.scale, o_cpu, l_cpu)
            if not self.cpu_pool.wait(60.0):
                raise TimeoutError(f"the CPU side of step {t} took over 60 s")
            cpu_s = time.perf_counter() - c0
            rec["O_cpu"], rec["lse_cpu"] = o_cpu.numpy(), l_cpu.numpy()
            stats["cpu_ms"] = cpu_s * 1e3
            stats["cpu_gbs"] = n_cpu * 2 * P * s.D * 2 / cpu_s / 1e9
            # with the CPU partial of layer i+1 made while the GPU runs layer i (Algorithm 1), the GPU
            # waits for whatever of the CPU time its own step does not cover
            stats["gpu_idle_frac"] = max(0.0, cpu_s * 1e3 - stats["gpu_ms"]) / max(cpu_s * 1e3, stats["gpu_ms"])
        if self.recall_every > 0 and t % self.recall_every == self.recall_every - 1:
            # the block being written stays on the GPU: the planner sees it as the most important
            # resident block, so it is evicted last, and never (at least k + 1 blocks are resident,
            # at most k come in)
            sc = self.scores.cpu().numpy().reshape(U, s.nblk).copy()
            for u in range(U):
                sc[u, (int(self.seq[u // s.Hkv]) - 1) // P] = np.inf
            rec.update(scores=sc, res_before=self.res.copy(), table_before=self.table.copy())
            if self.pages:
                # the page being written is never evicted: it joins every head's selection (more
                # than k + 1 pages may come in with pages, so its infinite score is not enough)
                tails = np.array([(int(self.seq[u // s.Hkv]) - 1) // P for u in range(U)], np.int32)
                ti = np.concatenate([rec["topk"], tails[:, None]], axis=1)
                tc = rec["topk_count"].copy()
                for u in range(U):
                    if tails[u] in ti[u, :tc[u]]:
                        ti[u, tc[u]:] = -1
                    else:
                        ti[u, tc[u]], ti[u, tc[u] + 1:] = tails[u], -1
                        tc[u] += 1
                ops = bs.plan_recall_pages(sc, ti, tc, _bits(self.res), self.table, s.B, s.Hkv, s.k + 1)
            else:
                ops = bs.plan_recall(sc, rec["topk"], rec["topk_count"], _bits(self.res), self.table, s.k)
            if len(ops):
                nbytes, secs = self._move_in(ops)
                for u, j, slot, ev in ops:
                    if ev >= 0:
                        self.res[u, ev], self.table[u, ev] = False, -1
                    self.res[u, j], self.table[u, j] = True, slot
                stats.update(recall_blocks=len(ops), recall_bytes=nbytes, recall_h2d_gbs=nbytes / secs / 1e9)
            rec["ops"] = ops
        rec["stats"] = stats
        self.t += 1
        return rec


def profile_recall_intervals(layers: int, steps: int, beta: float = 0.12, shape: W.Shape | None = None):
    """Offline profile of section 3.4: each layer (its own seeded workload) decodes ``steps``
    steps without recalls; its CPU compute ratio trace gives its recall interval, the largest
    number of steps that keeps the ratio below ``beta``.  Returns (traces [layers][steps],
    intervals [layers])."""
    import dataclasses

    base = shape or c4_shape(steps)
    traces = np.zeros((layers, steps), dtype=np.float32)
    for layer in range(layers):
        sw = DecodeSweep(dataclasses.replace(base, seed=base.seed + layer), steps, recall_every=0)
        for t in range(steps):
            traces[layer, t] = sw.step()["stats"]["cpu_ratio"]
        del sw
        torch.cuda.empty_cache()
    return traces, bs.recall_intervals(traces, beta)


def run_layers(layers: int, steps: int, recall_every=16, beta: float = 0.12, shape: W.Shape | None = None,
               gather: bool = True, pages: bool = False, cpu_pool=None):
    """The decode sweep over ``layers`` layers, one after another (each its own seeded workload,
    freed before the next, the pinned host copy of its K/V reused): yields (layer, sweep, record)
    for every decode step.  ``recall_every``: a step count, or a sequence of per-layer intervals
    (e.g. the recall intervals profiled by :func:`profile_recall_intervals`, section 3.4)."""
    import dataclasses

    base = shape or c4_shape(steps)
    U, nb, P, D = base.units, base.nblk, base.P, base.D
    host = [torch.empty(U * nb * P * D, dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    every = [int(recall_every)] * layers if np.isscalar(recall_every) else [int(x) for x in recall_every]
    if len(every) != layers:
        raise ValueError("one recall interval per layer")
    for layer in range(layers):
        sw = DecodeSweep(dataclasses.replace(base, seed=base.seed + layer), steps, recall_every=every[layer],
                         host=host, gather=gather, pages=pages, cpu_pool=cpu_pool)
        for _ in range(steps):
            yield layer, sw, sw.step()
        del sw
        torch.cuda.empty_cache()


def probe_recall_bandwidth(total_mib: int = 256, device="cuda", seed: int = 0) -> list[dict]:
    """Host-to-device rate of recall transfers by granularity (the pages compare ~800 MB/s for
    4 KB per-token transfers with ~15 GB/s for 128 KB pages over PCIe 4.0; section 2.3, Figure 3).
    Pages of P tokens (P x 128 bf16 = P * 256 bytes for K, the same for V) move from pinned host
    memory into randomly chosen pool slots; 4 KB = P 16 and 8 KB = P 32 scattered, 128 KB = runs of
    16 consecutive 8 KB pages into consecutive slots.  Both movers: one cudaMemcpyAsync per run of
    pages (scout_recall_async) and the gather kernel (scout_recall_gather_async)."""
    dev = torch.device(device)
    rng = np.random.default_rng(seed)
    out = []
    side = torch.cuda.Stream(dev)
    for gran, P, run in ((4096, 16, 1), (8192, 32, 1), (131072, 32, 16)):
        page = P * 128 * 2
        n_ops = (total_mib << 20) // (2 * page)  # K and V
        nb = n_ops  # one unit holding every block: block i of the host copy
        hK = torch.empty((nb, P, 128), dtype=torch.bfloat16, pin_memory=True)
        hV = torch.empty_like(hK, pin_memory=True)
        hK.view(torch.int16).copy_(torch.from_numpy(rng.integers(-2 ** 15, 2 ** 15, size=hK.shape, dtype=np.int16)))
        hV.copy_(hK)
        runs = n_ops // run
        slot0 = rng.permutation(runs) * run  # each run lands on `run` consecutive slots, runs scattered
        ops = np.array([(0, r * run + i, slot0[r] + i, -1) for r in range(runs) for i in range(run)], np.int32)
        Kp = torch.empty((n_ops, P, 128), dtype=torch.bfloat16, device=dev)
        Vp = torch.empty_like(Kp)
        d_ops = WD.to_dev(ops, dev)
        h_ops = (bs.RecallOp * n_ops)(*[bs.RecallOp(*(int(x) for x in o)) for o in ops])  # built before timing
        row = {"granularity_bytes": gran, "transfers": int(2 * runs), "bytes": int(2 * n_ops * page)}
        for name in ("copies", "gather"):
            best = None
            for _ in range(3):
                torch.cuda.synchronize(dev)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(side)
                if name == "copies":
                    rc = bs.lib().scout_recall_async(h_ops, n_ops, hK.data_ptr(), hV.data_ptr(), Kp.data_ptr(),
                                                     Vp.data_ptr(), n_ops, 1, 1, 128, P, nb, None, None,
                                                     side.cuda_stream, None)
                    if rc:
                        raise bs.ScoutError(f"scout_recall_async: {rc}")
                else:
                    bs.recall_gather_async(d_ops, hK, hV, Kp, Vp, 1, 1, P, nb, side)
                b.record(side)
                b.synchronize()
                ms = a.elapsed_time(b)
                best = ms if best is None else min(best, ms)
            row[name + "_GB_s"] = row["bytes"] / (best / 1e3) / 1e9
        # both movers put every page where the ops say
        assert torch.equal(Kp.view(torch.int16)[torch.from_numpy(ops[:, 2]).long().to(dev)].cpu(),
                           hK.view(torch.int16)[torch.from_numpy(ops[:, 1]).long()])
        out.append(row)
        del hK, hV, Kp, Vp
    return out


def main():
    ap = argparse.ArgumentParser(description="Residency sweep: one layer, many decode steps, per-step report")
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--recall-every", type=int, default=16, help="0: no recall")
    ap.add_argument("--profile-layers", type=int, default=0,
                    help="instead: profile this many layers without recalls and print their recall intervals")
    ap.add_argument("--beta", type=float, default=0.12, help="CPU compute ratio threshold of the profile")
    ap.add_argument("--layers", type=int, default=0,
                    help="instead: the sweep over this many seeded layers, one JSON row per (layer, step); with "
                         "--recall-every 0 ... no recall, with --profiled the per-layer intervals of a profile")
    ap.add_argument("--profiled", action="store_true",
                    help="with --layers: recall at each layer's interval profiled without recalls first (--beta)")
    ap.add_argument("--copies", action="store_true", help="recall with cudaMemcpyAsync calls, not the gather kernel")
    ap.add_argument("--pages", action="store_true",
                    help="residency per page (a block of a sequence for all its KV heads), not per block")
    ap.add_argument("--cpu-side", action="store_true",
                    help="also compute every step's CPU side on a worker pool of the host's cores and report its "
                         "time, GB/s and the GPU-idle fraction of the layer-ahead overlap")
    ap.add_argument("--probe-recall", action="store_true",
                    help="instead: host-to-device recall rate at 4 KB, 8 KB and 128 KB granularity")
    a = ap.parse_args()
    pool = None
    if a.cpu_side:
        import os

        pool = bs.CpuPool(len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else 0)
    if a.probe_recall:
        for row in probe_recall_bandwidth():
            print(json.dumps(row), flush=True)
        return
    if a.layers > 0:
        every = a.recall_every
        if a.profiled:
            traces, iv = profile_recall_intervals(a.layers, a.steps, a.beta)
            print(json.dumps({"profile_beta": a.beta, "intervals": [int(x) for x in iv],
                              "mean_interval": float(iv.mean())}), flush=True)
            every = iv
        for layer, sw, rec in run_layers(a.layers, a.steps, every, gather=not a.copies, pages=a.pages, cpu_pool=pool):
            print(json.dumps({"layer": layer, **rec["stats"]}), flush=True)
        return
    if a.profile_layers > 0:
        traces, iv = profile_recall_intervals(a.profile_layers, a.steps, a.beta)
        for layer in range(a.profile_layers):
            print(json.dumps({"layer": layer, "interval": int(iv[layer]),
                              "ratio": [round(float(x), 4) for x in traces[layer]]}), flush=True)
        print(json.dumps({"beta": a.beta, "mean_interval": float(iv.mean())}), flush=True)
        return
    sw = DecodeSweep(c4_shape(a.steps), a.steps, a.recall_every, gather=not a.copies, pages=a.pages, cpu_pool=pool)
    for _ in range(a.steps):
        print(json.dumps(sw.step()["stats"]), flush=True)


if __name__ == "__main__":
    main()
