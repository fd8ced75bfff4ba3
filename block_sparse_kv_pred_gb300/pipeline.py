"""The layer-ahead pipeline with the CPU side computed on the host cores.

ScoutAttention (arXiv HTML), section 3.3 and Algorithm 1: once layer i has predicted layer
i+1's query and chosen its blocks, the CPU starts layer i+1's attention over the blocks that
are not on the GPU (CPUAttn, with the predicted query) while the GPU goes on with layer i;
layer i+1's attention on the GPU then merges that partial with its own over the resident
blocks.

Here step i of ``step.Step`` stands for layer i's attention and layer i+1's selection.  Per
step, on the host:

1. the step's GEMM, selection and digest append are issued;
2. the CPU partial of this step, started one step earlier, is waited for (bounded: a partial
   later than ``timeout_s`` is an error, never an endless wait) and copied up on the copy
   stream; the attention stream waits for that copy, and the attention is issued;
3. the copy stream waits for the selection and brings its CPU work list and Q_pred down;
   the host waits for that copy (bounded) and hands the next step's CPU partial to the
   worker pool (``scout_cpu_pool``), which computes it while the GPU runs this step's
   attention and the next step's GEMM and selection.

Buffers alternate by step parity as the step's own do.  A host buffer is rewritten only after
what read it has finished: the partial buffer of parity p is copied up in step i+1's stage 2
and rewritten by the job of step i+2, submitted after that step's download, which the copy
stream orders after the upload; a work-list buffer is rewritten by the download of step i+2,
after the job that read it was waited for in step i+1.

The single synthetic layer stands for every layer, as in the step.
"""
from __future__ import annotations

import os
import time

import torch

import block_sparse_kv_pred_gb300 as bs


def host_threads() -> int:
    """The cores this process may run on (the machine may have more)."""
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


class LayerAhead:
    """Drives a prepared ``Step`` (four streams, not graph-captured) with the CPU partial of
    every step computed by the worker pool from the previous step's work list."""

    def __init__(self, s, t, step, n_threads: int = 0, timeout_s: float = 10.0):
        if step.serial:
            raise ValueError("the layer-ahead pipeline runs on the four-stream step")
        self.s, self.t, self.timeout_s = s, t, timeout_s
        self.dev = dev = t["Qp0"].device
        slots = t.get("page_table_all", t["page_table"]).reshape(-1).long()
        if int(slots.min()) < 0:
            raise ValueError("a block of the layer has no pool slot: the host copy needs every block")
        # the layer's K/V in logical block order on the host: the copy the CPU side attends
        self.hkv = {n: t.get(n + "_all", t[n + "_pool"]).index_select(0, slots)
                    .view(s.B, s.Hkv, s.nblk, s.P, s.D).cpu() for n in "KV"}
        self.seq = t["seq_len"].cpu().contiguous()
        self.pool = bs.CpuPool(n_threads or host_threads())
        self.step = step.fresh()
        self.sH = torch.cuda.Stream(dev)  # the pipeline's host<->device copies, in issue order

        def pin(x):
            return torch.empty_like(x, device="cpu").pin_memory()

        self.h_q = [pin(t[f"Qp{p}"]) for p in (0, 1)]
        self.h_list = [pin(t[f"cpu{p}"]) for p in (0, 1)]
        self.h_cnt = [pin(t[f"cpu_count{p}"]) for p in (0, 1)]
        self.h_O = [pin(t["O_cpu0"]) for _ in (0, 1)]
        self.h_L = [pin(t["lse_cpu0"]) for _ in (0, 1)]
        self.down = [torch.cuda.Event(), torch.cuda.Event()]
        self.up = [torch.cuda.Event(), torch.cuda.Event()]
        self.wait_s = []  # host time spent waiting for a CPU partial, per step
        self.job_s = []  # submit-to-done time of a job whose end the host had to wait for

    def _submit(self, par):
        """The CPU partial of the step after the one that wrote work-list set ``par``."""
        s = self.s
        self.pool.submit(self.h_q[par].view(s.B, s.Hq, s.D), self.hkv["K"], self.hkv["V"], self.seq,
                         self.h_list[par], self.h_cnt[par], s.B, s.Hq, s.Hkv, s.P, s.k, s.scale,
                         self.h_O[1 - par], self.h_L[1 - par])
        self._t_submit = time.perf_counter()

    def _download(self, par, first=False):
        """Work-list set ``par`` and its Q_pred to the host, after the selection that wrote it."""
        t = self.t
        if not first:
            self.sH.wait_event(self.step.sel_done[par])
        with torch.cuda.stream(self.sH):
            self.h_q[par].copy_(t[f"Qp{par}"], non_blocking=True)
            self.h_list[par].copy_(t[f"cpu{par}"], non_blocking=True)
            self.h_cnt[par].copy_(t[f"cpu_count{par}"], non_blocking=True)
        self.down[par].record(self.sH)
        deadline = time.perf_counter() + self.timeout_s
        while not self.down[par].query():
            if time.perf_counter() > deadline:
                raise TimeoutError("the CPU work list did not reach the host in time")
            time.sleep(2e-5)

    def _bring_partial(self, par, attn_stream):
        """Stage 2: wait for the CPU partial of this step and copy it up before the attention."""
        t0 = time.perf_counter()
        if not self.pool.wait(self.timeout_s):
            raise TimeoutError(f"the CPU partial was not ready within {self.timeout_s} s (a late CPU partial)")
        t1 = time.perf_counter()
        self.wait_s.append(t1 - t0)
        if t1 - t0 > 1e-4:
            self.job_s.append(t1 - self._t_submit)
        if self.step.i >= 2:
            self.sH.wait_event(self.step.attn_done[par])  # the attention two steps back read this buffer
        t = self.t
        with torch.cuda.stream(self.sH):
            t[f"O_cpu{par}"].copy_(self.h_O[par], non_blocking=True)
            t[f"lse_cpu{par}"].copy_(self.h_L[par], non_blocking=True)
        self.up[par].record(self.sH)
        attn_stream.wait_event(self.up[par])

    def run(self, steps: int, warm: int = 0) -> dict:
        """``warm`` + ``steps`` pipelined steps; returns the host wall time per timed step and the
        time the host waited for CPU partials.  Raises on a late partial or a device error."""
        st, dev = self.step, self.dev
        ev0 = torch.cuda.Event()
        ev0.record(torch.cuda.current_stream(dev))
        self.sH.wait_event(ev0)
        # the list set the first step's attention reads was written before the pipeline started
        first = 1 - st.i % 2
        self._download(first, first=True)
        self._submit(first)
        st.begin(ev0)
        t0 = time.perf_counter()
        for i in range(warm + steps):
            if i == warm:
                t0 = time.perf_counter()
                self.wait_s.clear()
                self.job_s.clear()
            par = st.i % 2
            st.issue(after_begin=(i == 0), before_attention=self._bring_partial)
            self._download(par)
            self._submit(par)
        ok = self.pool.wait(self.timeout_s)  # the job started by the last step feeds no attention
        st.end(None)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        if not ok:
            raise TimeoutError("the last CPU partial was not ready in time")
        status = int(self.t["status"].item())
        if status != 0:
            raise RuntimeError(f"device status {status}")
        n = max(1, steps)
        return {"ms_per_step": wall / n * 1e3, "host_wait_ms": sum(self.wait_s) / n * 1e3,
                "cpu_ms_per_layer": (sum(self.job_s) / len(self.job_s) * 1e3) if self.job_s else None,
                "threads": self.pool.threads, "steps": steps}

    def close(self):
        self.pool.close()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
