#!/usr/bin/env python
"""Decode-step benchmark of libscout on the Qwen3-14B-shaped layer.

One step = the whole GPU hot path of one layer's decode step (ScoutAttention
Algorithm 1, layer-ahead prediction), issued on four streams with the persistent
kernels capped to share the SMs:
  GEMM stream: predict_q (next layer's Q_pred = X W_Q^T, 40 x 5120 x 5120), after the
    previous step's attention (its output is this step's layer input);
  selection stream: score_topk (digest scores with Q_pred, top-64 of 1024 blocks,
    residency split), after this step's GEMM;
  attention stream: sparse_attn_merge (true query over the resident blocks the
    previous step selected, merged with the CPU partial);
  append stream: build_digest (append: the tail block of every (sequence, KV head)).
Metric: decode-attention query-heads per second (B * Hq per step, summed over ranks).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config qwen3_14b] [--impl scout|reference]
                  [--serial] [--split GEMM,SEL,ATTN]

--impl reference times the fp64 oracle (the plain CPU implementation) on this
machine's host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 << 20  # GB300 L2
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--config", default="qwen3_14b")
    ap.add_argument("--impl", default="scout", choices=["scout", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--no-cpu-side", action="store_true", help="skip timing scout_cpu_attend on the host cores")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target oracle time for cpu_baseline")
    ap.add_argument("--serial", action="store_true", help="one stream, full grids (no overlap)")
    ap.add_argument("--split", default=None,
                    help="CTAs of the GEMM,selection,attention kernels (default 80,0,72, 0 = one per SM; two "
                         "values: GEMM and selection share the first)")
    ap.add_argument("--early", default=None,
                    help="kernels that start early after the kernel they wait for, comma-separated among "
                         "predict_q,score_topk,sparse_attn_merge ('none' for none; default: the step's)")
    a = ap.parse_args()
    a.warmup = max(a.warmup, 3)
    return a


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


GRAPH_STEPS = 20  # steps per captured CUDA graph (even: the list sets alternate)


def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (x itself on one rank)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    m = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(m, op=dist.ReduceOp.MAX)
    return float(m.item())


# ---------------------------------------------------------------------------
# libscout arm
# ---------------------------------------------------------------------------
from block_sparse_kv_pred_gb300.step import EARLY, KERNELS, SPLIT, STREAM_OF, algorithmic_bytes, setup_step  # noqa: E402


def run_scout(args, rank, world, local):
    import torch
    import torch.distributed as dist

    from block_sparse_kv_pred_gb300 import workload as W

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    shape = W.CONFIGS[args.config]()
    split = tuple(int(x) for x in args.split.split(",")) if args.split else SPLIT
    early = EARLY if args.early is None else tuple(x for x in args.early.split(",") if x and x != "none")
    wl, t, step = setup_step(shape, device, serial=args.serial, split=split, early=early)
    s = shape

    def barrier():
        if world > 1:
            dist.barrier()

    cur = torch.cuda.current_stream()
    ev0 = torch.cuda.Event()
    ev0.record(cur)
    step.begin(ev0)
    for i in range(args.warmup):
        step.issue()
    step.end(None)
    torch.cuda.synchronize()
    if int(t["status"].item()) != 0:
        raise RuntimeError(f"device status {int(t['status'].item())} after warm-up")

    # the timed steps replay CUDA graphs of GRAPH_STEPS steps (plus one graph of the remainder),
    # captured from the same calls; every replay waits for the previous one to finish
    T = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    gstep = step.fresh()
    n_full, rest = divmod(args.steps, GRAPH_STEPS)
    g_full = gstep.capture(GRAPH_STEPS, device) if n_full else None
    g_rest = gstep.capture(rest, device) if rest else None
    for _ in range(max(1, args.warmup // GRAPH_STEPS)):
        (g_full or g_rest).replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    e_start, e_end = T(), T()
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    e_start.record(cur)
    for _ in range(n_full):
        g_full.replay()
    if g_rest is not None:
        g_rest.replay()
    e_end.record(cur)
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    if int(t["status"].item()) != 0:
        raise RuntimeError(f"device status {int(t['status'].item())} in the timed steps")
    ms = e_start.elapsed_time(e_end) / args.steps

    # per-kernel durations from a second pass, issued on the streams with events around every
    # launch (not the timed pass: the events sit between the selection stream's two kernels)
    step = step.fresh()
    n_prof = max(50, args.steps // 4)
    ev = [{name: (T(), T()) for name in KERNELS} for _ in range(n_prof)]
    e0, e1 = T(), T()
    e0.record(cur)
    step.begin(e0)
    for i in range(n_prof):
        step.issue(timing=ev[i])
    step.end(e1)
    torch.cuda.synchronize()
    kern_ms = {name: statistics.mean(e[name][0].elapsed_time(e[name][1]) for e in ev) for name in KERNELS}
    ms = max_over_ranks(ms, device)
    value = world * s.B * s.Hq / (ms / 1e3)

    e2e = run_e2e(args, t, step, s, world, device)
    return s, wl, t, dict(ms=ms, value=value, kern_ms=kern_ms, clocks=clocks, wall=wall, e2e=e2e,
                          launches=step.launches_per_step * args.steps, split=None if args.serial else split,
                          early=() if args.serial else early, step=step)


def isolated(t, step, nbytes, peak, reps=20):
    """Each kernel on its own: full grids (one CTA per SM), the L2 flushed before every launch by
    reading a 256 MB buffer (a read leaves no dirty lines whose write-back would fall inside the
    next launch).  Device time only: a CUDA graph of ``reps`` (flush, launch) pairs is timed
    against a graph of the flushes alone, so no host enqueue gap is counted.  The selection and
    the attention together are the pair the roofline target names; their serialised durations
    sum to the pair's time."""
    import torch

    dev = t["Qp0"].device
    flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    saved = {}
    for key in ("gemm", "score", "attn"):
        for par in (0, 1):
            lp = t.get(f"_launch_{key}{par}")
            if lp:
                saved[(key, par)] = lp.contents.max_ctas
                lp.contents.max_ctas = 0

    def graph_ms(stream, call):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                flush.sum()
                if call is not None:
                    call()
        best = None
        for _ in range(4):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):  # a graph replays on the current stream
                a.record(stream)
                g.replay()
                b.record(stream)
            b.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        return best

    try:
        out = {}
        calls = step.calls[0]
        for name in KERNELS:
            stream = step.streams[0 if step.serial else STREAM_OF[name]]
            torch.cuda.synchronize()
            m = (graph_ms(stream, calls[name]) - graph_ms(stream, None)) / reps
            gbs = nbytes[name] / (m / 1e3) / 1e9
            out[name] = {"us": m * 1e3, "GB_s": gbs, "frac_of_hbm_peak": gbs / peak}
        pair_us = out["score_topk"]["us"] + out["sparse_attn_merge"]["us"]
        pair_b = nbytes["score_topk"] + nbytes["sparse_attn_merge"]
        out["score_topk+sparse_attn_merge"] = {"us": pair_us, "bytes": pair_b,
                                               "GB_s": pair_b / (pair_us / 1e6) / 1e9,
                                               "frac_of_hbm_peak": pair_b / (pair_us / 1e6) / 1e9 / peak}
        out["note"] = (f"one kernel at a time, one CTA per SM, L2 flushed before each launch; graph of {reps} "
                       f"(flush, launch) pairs minus a graph of the flushes, best of 4")
        torch.cuda.synchronize()
        if int(t["status"].item()) != 0:
            return {"unavailable": f"device status {int(t['status'].item())}"}
        return out
    finally:
        for (key, par), v in saved.items():
            t[f"_launch_{key}{par}"].contents.max_ctas = v


def run_e2e(args, t, step, s, world, device):
    """Same metric through the public calls with every step's inputs (X, q, the CPU partial)
    copied from pinned host memory and its results (output, LSE, the CPU work list) read back,
    one copy each way (each set is one buffer).  Inputs and outputs alternate between two
    device buffers, as Q_pred and the lists do: step i's inputs are copied on one copy stream
    once the step two back has read that buffer, and step i's kernels wait for them; its
    results are read back on another once its kernels are done, and the kernels two steps
    later, which write those buffers again, wait for that.  So the copies overlap the kernels
    as the steps do.  Like the timed loop, the steps replay CUDA graphs captured from those
    calls."""
    import torch
    import torch.distributed as dist

    h_in = torch.empty_like(t["in0"], device="cpu").pin_memory()
    h_in.copy_(t["in0"])
    h_out = torch.empty_like(t["out0"], device="cpu").pin_memory()
    h2d, d2h = h_in.numel(), h_out.numel()
    gstep = step.fresh()
    sA, sB, sC, sD = (gstep.streams * 4)[:4] if gstep.serial else gstep.streams
    sE = sA if gstep.serial else torch.cuda.Stream(device)  # host-to-device copies
    sF = sA if gstep.serial else torch.cuda.Stream(device)  # device-to-host copies
    read = [torch.cuda.Event(), torch.cuda.Event()]  # step i's results are read back (per parity)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream(device)):
        cur = torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(cur)
        gstep.begin(start)
        sE.wait_event(start)
        sF.wait_event(start)
        for j in range(GRAPH_STEPS):
            par = gstep.i % 2
            if j >= 2 and not gstep.serial:
                # buffers par were last read two steps back: the inputs by that step's GEMM and
                # attention, the outputs by that step's read-back
                sE.wait_event(gstep.gemm_done[par])
                sE.wait_event(gstep.attn_done[par])
                sA.wait_event(read[par])
                sB.wait_event(read[par])
            with torch.cuda.stream(sE):
                t[f"in{par}"].copy_(h_in, non_blocking=True)
            landed = torch.cuda.Event()
            landed.record(sE)
            sD.wait_event(landed)
            sB.wait_event(landed)
            gstep.issue(after_begin=(j == 0))
            if not gstep.serial:
                sF.wait_event(gstep.sel_done[par])
                sF.wait_event(gstep.attn_done[par])
            with torch.cuda.stream(sF):
                h_out.copy_(t[f"out{par}"], non_blocking=True)
            read[par].record(sF)
        gstep.end(None)
        for side in (sE, sF):
            done = torch.cuda.Event()
            done.record(side)
            cur.wait_event(done)
    for _ in range(3):
        g.replay()
    reps = max(3, args.steps // (4 * GRAPH_STEPS))
    cur = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    a.record(cur)
    for _ in range(reps):
        g.replay()
    b.record(cur)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b) / (reps * GRAPH_STEPS), device)
    return {"value": world * s.B * s.Hq / (ms / 1e3), "unit": "query-heads/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": reps * GRAPH_STEPS}


def cpu_side(s, t, seconds=1.0, max_seqs=None):
    """The CPU side of the collaborative attention (scout_cpu_attend) on this host's cores:
    attention over the CPU work list of the last timed step with its Q_pred, for the first
    ``max_seqs`` sequences (all by default; their K/V gathered into logical block order on the
    host).  Reported beside the GPU numbers, never part of them; a failure is reported, not
    raised, so that it cannot cost the GPU measurement."""
    import numpy as np

    import block_sparse_kv_pred_gb300 as bs

    try:
        Bs = s.B if max_seqs is None else min(s.B, max_seqs)
        # the whole cache (the step's compact pool holds only the GPU's share of it)
        slots = t.get("page_table_all", t["page_table"])[:Bs].reshape(-1).long()
        if int(slots.min()) < 0:
            return {"unavailable": "a block of the sample has no pool slot"}
        kv = {n: t.get(n + "_all", t[n + "_pool"]).index_select(0, slots).view(Bs, s.Hkv, s.nblk, s.P, s.D).cpu()
              for n in "KV"}
        q = t["Qp1"][:Bs].reshape(Bs, s.Hq, s.D).cpu()
        lst, cnt, seq = (t[n][:Bs].cpu().contiguous() for n in ("cpu1", "cpu_count1", "seq_len"))
        listed = np.arange(s.k)[None, None, :] < cnt.numpy()[:, :, None]
        toks = np.clip(seq.numpy().astype(np.int64)[:, None, None] - lst.numpy().astype(np.int64) * s.P, 0, s.P)
        nbytes = int((toks * listed).sum()) * s.D * 2 * 2  # K and V of the listed blocks' tokens
        # the cores this process may run on (the machine may have more)
        threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)

        def call():
            bs.cpu_attend(q, kv["K"], kv["V"], seq, lst, cnt, Bs, s.Hq, s.Hkv, s.P, s.k, s.scale, n_threads=threads)

        call()
        n, t0 = 0, time.perf_counter()
        while True:
            call()
            n += 1
            el = time.perf_counter() - t0
            if el >= seconds or n >= 50:
                break
        per = el / n
        return {"value": nbytes / per / 1e9, "unit": "GB/s", "kind": "scout_cpu_attend", "threads": threads,
                "ms_per_call": per * 1e3, "query_heads_per_s": Bs * s.Hq / per, "kv_bytes_per_call": nbytes,
                "full_batch_ms_estimate": per * 1e3 * s.B / Bs,
                "sample": f"{Bs} of {s.B} sequences of {s.name}: the CPU work list of the last timed step with "
                          f"its Q_pred, {n} calls"}
    except Exception as e:  # noqa: BLE001
        return {"unavailable": f"{type(e).__name__}: {e}"[:300]}


def layer_ahead(s, t, step, gpu_ms, steps=24, warm=4, limit_s=60.0):
    """Algorithm 1's pipeline with the CPU side computed for real (``pipeline.LayerAhead``):
    after step i's selection its CPU work list and Q_pred go down to the host, where the
    worker pool computes the next layer's CPU partial on the host cores while the GPU goes on;
    the partial goes up before step i+1's attention, which waits for it.  Host wall time per
    step against the GPU-only step (graph replay) gives the fraction of the time the GPU would
    idle.  Every wait is bounded and a failure is reported, not raised, so that it cannot cost
    the GPU measurement."""
    import torch

    from block_sparse_kv_pred_gb300.pipeline import LayerAhead

    if step.serial:
        return {"unavailable": "serial step"}
    dev = t["Qp0"].device
    try:
        with LayerAhead(s, t, step, timeout_s=limit_s) as la:
            r = la.run(steps, warm)
        ms = r["ms_per_step"]
        return {"ms_per_step": ms, "value": s.B * s.Hq / (ms / 1e3), "unit": "query-heads/s",
                "cpu_ms_per_layer": r["cpu_ms_per_layer"], "host_wait_ms_per_step": r["host_wait_ms"],
                "gpu_step_ms": gpu_ms, "gpu_idle_frac": max(0.0, 1.0 - gpu_ms / ms), "threads": r["threads"],
                "steps": steps,
                "note": "the step issued on its streams (not graph-replayed), the CPU partial of every step "
                        "computed by the worker pool (scout_cpu_pool) from the previous step's work list; "
                        "gpu_idle_frac compares the graph-replayed GPU-only step with this wall time"}
    except Exception as e:  # noqa: BLE001
        return {"unavailable": f"{type(e).__name__}: {e}"[:300]}
    finally:
        try:
            torch.cuda.synchronize(dev)
        except Exception:  # noqa: BLE001  (already reported above)
            pass


# ---------------------------------------------------------------------------
# oracle timing (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------
class OracleSample:
    """The fp64 oracle's version of one step, on a few (sequence, KV head) units."""

    STAGES = ("build_digest", "predict_q", "score_topk", "sparse_attn", "merge")

    def __init__(self, shape, n_units=8, seed=1):
        import numpy as np

        import oracle as O
        from block_sparse_kv_pred_gb300 import workload as W

        self.O, self.np = O, np
        s = self.s = shape
        wl = self.wl = W.Workload(s)
        rng = np.random.default_rng(seed)
        self.units = sorted(int(u) for u in rng.choice(s.units, size=min(n_units, s.units), replace=False))
        X = wl.gemm_x()
        o_cpu, l_cpu = wl.cpu_partial()
        self.data = []
        for u in self.units:  # inputs resident in host memory, as the GPU's are in HBM
            b, kvh = divmod(u, s.Hkv)
            L = int(wl.seq_len[b])
            K, V = wl.unit_kv(u), wl.unit_kv(u, "V")
            mn, mx = O.digest_minmax(K, L, s.P)
            rows = slice(kvh * s.G * s.D, (kvh + 1) * s.G * s.D)
            self.data.append(dict(u=u, b=b, kvh=kvh, L=L, K=K, Kf=O.bf16_to_f64(K), Vf=O.bf16_to_f64(V), mn=mn,
                                  mx=mx, X=X[b:b + 1], Wr=wl.gemm_w(rows), q=wl.q[b, kvh * s.G:(kvh + 1) * s.G],
                                  ocpu=o_cpu[b, kvh * s.G:(kvh + 1) * s.G], lcpu=l_cpu[b, kvh * s.G:(kvh + 1) * s.G],
                                  prev=[]))
        self.i = 0

    def step(self, timer=None):
        """One unit: tail digest, Q_pred rows, scores, top-k, split, GPU-side attention, merge.
        ``timer``: optional dict stage -> seconds, to which each stage's time is added."""
        O, s = self.O, self.s
        d = self.data[self.i % len(self.data)]
        self.i += 1
        t0 = time.perf_counter()
        j = -(-d["L"] // s.P) - 1
        tmn, tmx = O.digest_minmax(d["K"][j * s.P:], d["L"] - j * s.P, s.P)
        d["mn"][j], d["mx"][j] = tmn[0], tmx[0]
        t1 = time.perf_counter()
        qp = O.f64_to_bf16(O.predict_q(d["X"], d["Wr"])).reshape(s.G, s.D)
        t2 = time.perf_counter()
        U = O.pool_group(O.scores_minmax(O.bf16_to_f64(qp), d["mn"], d["mx"]))
        S = O.select_topk(U, s.k)
        res, cpu = O.split_residency(S, self.wl.resident[d["u"]])
        O.delta_list(cpu, d["prev"])
        d["prev"] = cpu
        t3 = time.perf_counter()
        toks = O.block_tokens(res, s.P, d["L"])
        qa = O.bf16_to_f64(d["q"])
        parts = [O.attention_partial(qa[h], d["Kf"][toks], d["Vf"][toks], s.scale) for h in range(s.G)]
        t4 = time.perf_counter()
        for h, (o, l) in enumerate(parts):
            O.merge(o, l, d["ocpu"][h].astype("float64"), float(d["lcpu"][h]))
        t5 = time.perf_counter()
        if timer is not None:
            for name, dt in zip(self.STAGES, (t1 - t0, t2 - t1, t3 - t2, t4 - t3, t5 - t4)):
                timer[name] = timer.get(name, 0.0) + dt
        return s.G  # query heads processed


def _oracle_worker(job):
    """One process of the all-cores oracle timing: its own units, its own timing loop."""
    shape, seed, seconds = job
    smp = OracleSample(shape, n_units=2, seed=seed)
    smp.step()
    heads, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        heads += smp.step()
    return heads, time.perf_counter() - t0


def cpu_baseline(shape, seconds, all_cores=True):
    """The oracle on the host cores: one thread with each stage timed, then (``all_cores``) one
    process per core over different sampled units at once (started with spawn: this process
    has used the GPU).  The value is the single-thread rate; the all-cores rate sits beside it."""
    smp = OracleSample(shape)
    smp.step()
    heads, timer, t0 = 0, {}, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        heads += smp.step(timer)
    el = time.perf_counter() - t0
    n = smp.i - 1
    out = {"value": heads / el, "unit": "query-heads/s", "cores": 1, "kind": "oracle",
           "sample": f"{len(smp.units)} of {shape.units} (sequence, KV head) units of {shape.name}, "
                     f"{n} unit-steps in {el:.1f} s, single thread (BLAS/OpenMP pinned to 1)",
           "stages_ms_per_unit_step": {k: v / n * 1e3 for k, v in timer.items()}}
    if all_cores:
        import multiprocessing as mp

        cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
        try:
            with mp.get_context("spawn").Pool(cores) as pool:
                res = pool.map(_oracle_worker, [(shape, 100 + i, seconds / 2) for i in range(cores)])
            out["all_cores"] = {"value": sum(h / e for h, e in res), "unit": "query-heads/s", "cores": cores,
                                "processes": cores,
                                "sample": f"one process per core, each on 2 sampled units of {shape.name} for "
                                          f"{seconds / 2:.1f} s (rates summed)"}
        except Exception as e:  # noqa: BLE001
            out["all_cores"] = {"unavailable": f"{type(e).__name__}: {e}"[:300]}
    return out


def run_reference(args, rank, world):
    from block_sparse_kv_pred_gb300 import workload as W

    if rank != 0:
        return None
    shape = W.CONFIGS[args.config]()
    smp = OracleSample(shape)
    for _ in range(args.warmup):
        smp.step()
    t0 = time.perf_counter()
    heads = 0
    for _ in range(args.steps):
        heads += smp.step()
    el = time.perf_counter() - t0
    value = heads / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "query-heads/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": DATA,
            "config": config_of(shape, world, SPLIT, EARLY),
            "cpu_baseline": {"value": value, "unit": "query-heads/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step is one of {len(smp.units)} sampled (sequence, KV head) units "
                                       f"of {shape.name}; single thread"},
            "e2e": {"value": value, "unit": "query-heads/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    return line


# ---------------------------------------------------------------------------
METRIC = "sparse-decode query-heads/s and achieved HBM GB/s vs ~8 TB/s (1xGB300)"
DATA = "synthetic: seeded Qwen3-14B-shaped K/V/q/X/W_Q (stand-in for LongBench prompts and trained weights)"


def streams_of(split):
    if not split:
        return "one stream"
    g, sel, att = split if len(split) == 3 else (split[0], split[0], split[1])
    n = lambda c: f"{c} CTAs" if c else "one CTA per SM"  # noqa: E731
    nsel = f"{sel} CTAs" if sel else "its default grid: ceil(units / ceil(units / SMs)) CTAs, whole units dealt"
    return (f"GEMM ({n(g)}) after the previous attention || selection ({nsel}) after the GEMM || "
            f"attention ({n(att)}) after the previous selection || digest append")


def config_of(s, world, split=None, early=(), n_slots=None):
    pool = None
    if n_slots is not None:
        pool = (f"{n_slots} slots of {s.P}-token K and V pages ({2 * n_slots * s.P * s.D * 2 / 1e9:.2f} GB): the "
                f"resident blocks and each unit's tail block, in a seeded slot order")
    return {"workload": s.name, "kv_pool": pool, "batch": s.B, "q_heads": s.Hq, "kv_heads": s.Hkv, "head_dim": s.D,
            "context": s.T, "page": s.P, "budget_tokens": s.k * s.P, "resident_frac": s.resident_frac,
            "digest": s.kind, "gemm_mnk": [s.B, s.Hq * s.D, s.hidden],
            "l2": "not flushed: one step reads inputs larger than L2 (see step_input_bytes), in an order "
                  "that evicts each input before its next use",
            "streams": streams_of(split),
            "early_start": list(early),
            "parallelism": f"independent replicas x{world} (one batch of sequences per GPU)"}


def attention_path(s, nbytes, kern_ms, peak):
    """The selection and attention kernels on their own: B * Hq over the sum of their durations
    (the merge runs inside the attention kernel), with the bytes they move over that time."""
    ms = kern_ms["score_topk"] + kern_ms["sparse_attn_merge"]
    nb = nbytes["score_topk"] + nbytes["sparse_attn_merge"]
    gbs = nb / (ms / 1e3) / 1e9
    return {"value": s.B * s.Hq / (ms / 1e3), "unit": "query-heads/s", "ms": ms, "bytes": nb, "GB_s": gbs,
            "frac_of_hbm_peak": gbs / peak,
            "note": "score_topk + sparse_attn_merge concurrent durations summed (they overlap inside the step)"}


def traffic_of(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this workload and
    the kernel source is unchanged since."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "dram_traffic_per_launch_qwen3_14b_b40_t32k.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec or not rec.get("workload", "").startswith(workload):
        return None
    h = hashlib.sha256()
    for src in rec.get("sources", []):
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return rec["dram_bytes_per_launch"] if h.hexdigest() == rec.get("sources_sha256") else None


def main():
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(v, "1")
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        if world > 1:
            import torch.distributed as dist

            dist.init_process_group("gloo")
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    import torch

    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    s, wl, t, r = run_scout(args, rank, world, local)
    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    nbytes = algorithmic_bytes(s, wl, t)
    kernels = {}
    for name in KERNELS:
        ms = r["kern_ms"][name]
        gbs = nbytes[name] / (ms / 1e3) / 1e9
        kernels[name] = {"ms": ms, "bytes": nbytes[name], "GB_s": gbs, "frac_of_hbm_peak": gbs / peak}
    dom = max(KERNELS, key=lambda k: nbytes[k])  # the kernel that moves the most bytes
    ach = kernels[dom]["GB_s"]
    src = f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback 6.8 TB/s"
    roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
            "peak_source": src, "traffic": traffic_of(dom, s.name), "algorithmic_bytes_per_launch": nbytes[dom],
            "note": "launch duration measured while the other stream's kernels share the GPU"
            if r["split"] else "serial step"}
    step_bytes = sum(nbytes[k] for k in KERNELS)
    step_gbs = step_bytes / (r["ms"] / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": r["value"], "unit": "query-heads/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": DATA, "config": config_of(s, world, r["split"], r["early"], t["n_slots"]),
        "roofline": roof,
        "step_roofline": {"bound": "hbm", "achieved": step_gbs, "peak": peak, "unit": "GB/s",
                          "frac": step_gbs / peak, "algorithmic_bytes_per_step": step_bytes,
                          "note": "all four kernels' algorithmic bytes / device time of a step"},
        "e2e": {k: v for k, v in r["e2e"].items() if k in ("value", "unit", "h2d_bytes_per_step",
                                                          "d2h_bytes_per_step", "ms_per_step")},
        "gpu_launches": r["launches"], "clocks": r["clocks"], "kernels": kernels,
        "kv_tokens_per_s": nbytes["_res_blocks"] * s.P / (r["kern_ms"]["sparse_attn_merge"] / 1e3),
        "attention_path": attention_path(s, nbytes, r["kern_ms"], peak),
        "kernels_isolated": isolated(t, r["step"], nbytes, peak),
        "wall_s_timed": r["wall"],
    }
    if world == 1 and not args.no_cpu_side:
        line["cpu_side"] = cpu_side(s, t)
        line["layer_ahead"] = layer_ahead(s, t, r["step"], r["ms"])
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(s, args.cpu_seconds)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
