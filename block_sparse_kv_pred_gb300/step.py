"""One decode step of one layer through the libscout C ABI.

ScoutAttention (arXiv HTML), Algorithm 1 (layer-ahead prediction): while layer i
attends with the block set chosen one layer earlier, the next layer's query is
predicted and its top-k chosen.  Step i here is layer i's attention together with
layer i+1's selection, issued on four CUDA streams, the persistent kernels capped to
share the SMs (``scout_launch.max_ctas``):

* GEMM stream: Q_pred = X W_Q^T (``scout_predict_q``) into Q_pred buffer ``i % 2``;
* selection stream: scoring and top-k over the next layer's digests
  (``scout_score_topk``) with that Q_pred, into list set ``i % 2``;
* attention stream: attention over the resident blocks of list set ``(i + 1) % 2``
  merged with the CPU partial (``scout_sparse_attn_merge``);
* append stream: the digest append for the token just written (``scout_build_digest``
  on this layer's tail blocks).  Nothing in the step reads it (the next step's selection
  of this layer does), so its few small CTAs run beside the persistent kernels.

The layer input X of step i is the output of step i-1's attention (through the merge and
the MLP), so step i's GEMM waits for step i-1's attention and nothing else; its
selection waits for its GEMM (and, being on one stream, for step i-1's selection); step
i's attention waits for step i-1's selection, whose lists it reads.  The GEMM of a step
therefore runs beside the previous step's selection, on the SMs the attention has just
left, and the period is bounded by (attention + GEMM + selection) / 2 rather than by
GEMM + selection.  Q_pred alternates between two buffers, as the lists do: a GEMM
overwrites the buffer the selection two steps earlier read, and that selection finished
before the attention the GEMM waits for began.  The single layer of the synthetic
workload stands for both layers: ``digest_next`` (scored) and ``digest_cur`` (appended
to) are separate buffers, as the two layers' are.

``serial=True`` issues the same four calls on one stream with full grids.
``algorithmic_bytes`` gives the bytes each kernel must move per launch, the
numerator of the roofline.
"""
from __future__ import annotations

import math

KERNELS = ("build_digest", "predict_q", "score_topk", "sparse_attn_merge")
# stream of each kernel: 0 = selection, 1 = attention, 2 = digest append, 3 = GEMM
STREAM_OF = {"build_digest": 2, "predict_q": 3, "score_topk": 0, "sparse_attn_merge": 1}
# CTAs of the GEMM, selection and attention kernels when overlapped (0: one per SM).  The
# selection deals whole units to its CTAs as they start, so it takes every SM the others
# leave; measured on GB300 (graph replay): 80/0/72 60.6 us per step, 80/72/72 62.9 us,
# 80/0/56 62.7 us, 80/0/88 61.2 us, 120/0/72 61.4 us.
SPLIT = (80, 0, 72)
# kernels that may start before the kernel they wait for has finished (programmatic dependent
# launch: the kernel waited for records a programmatic event; the early starter does its
# independent part at once and waits for that kernel only before reading its output).  None by
# default: an early starter holds its SMs while it waits, and in this step every SM is in use.
# Measured on GB300 (graph replay, 80/0/72): none 59.7 us per step, the GEMM early 59.6, the
# attention early 62.1, all three 64.3, the selection early 72.8 (its CTAs take the SMs the
# same step's attention needs, then wait for the GEMM).
EARLY_OF = {"predict_q": "sparse_attn_merge", "score_topk": "predict_q", "sparse_attn_merge": "score_topk"}
EARLY = ()
_LAUNCH_KEY = {"predict_q": "gemm", "score_topk": "score", "sparse_attn_merge": "attn"}


class Step:
    """The prepared calls, streams and events of a step; ``issue()`` launches the next step."""

    def __init__(self, t, calls, streams, serial):
        import torch

        self.t = t
        self.calls = calls  # name -> Prepared
        self.streams = streams
        self.serial = serial
        self.gemm_done = [torch.cuda.Event(), torch.cuda.Event()]
        self.sel_done = [torch.cuda.Event(), torch.cuda.Event()]
        self.attn_done = [torch.cuda.Event(), torch.cuda.Event()]
        # early starters: kernel -> the two programmatic events (by parity) it waits for, which
        # the kernel it waits for records; a record creates each now (timing disabled, as a
        # programmatic event must be), outside any capture
        self.early = {}
        for k in t.get("_early_kernels", ()):
            evs = [torch.cuda.Event(), torch.cuda.Event()]
            for e in evs:
                e.record(torch.cuda.current_stream())
            self.early[k] = evs
        self.i = 0

    @property
    def launches_per_step(self) -> int:
        return len(KERNELS)

    def fresh(self):
        """The same calls and streams with their own events (for a separate issue sequence,
        e.g. one captured in a CUDA graph, whose events may not be waited on outside it)."""
        twin = Step(self.t, self.calls, self.streams, self.serial)
        twin.i = self.i
        return twin

    def capture(self, n_steps, device):
        """A CUDA graph of n_steps steps (its first step ordered by the graph launch itself)."""
        import torch

        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device)
        with torch.cuda.graph(g, stream=side):
            cur = torch.cuda.current_stream()
            ev = torch.cuda.Event()
            ev.record(cur)
            self.begin(ev)
            for j in range(n_steps):
                self.issue(after_begin=(j == 0))
            self.end(None)
        return g

    def begin(self, event):
        """Make every stream wait for ``event`` (recorded on the current stream)."""
        for s in self.streams:
            s.wait_event(event)

    def end(self, event):
        """Join every stream into the current stream and record ``event`` there."""
        import torch

        cur = torch.cuda.current_stream()
        for s in self.streams:
            ev = torch.cuda.Event()
            ev.record(s)
            cur.wait_event(ev)
        if event is not None:
            event.record(cur)

    def issue(self, timing=None, after_begin=False, before_attention=None):
        """Launch the next step.  ``timing``: optional name -> (start, end) timing events.
        ``after_begin``: the step directly follows ``begin`` (e.g. the first step of a CUDA
        graph), whose event already orders it after everything before, so it waits for no
        earlier step's events (a graph capture may not wait on events recorded outside it).
        ``before_attention``: optional callable, given the step's parity and the attention
        stream, called after the GEMM, selection and digest append are issued and before the
        attention is (the layer-ahead pipeline brings the CPU partial in there)."""
        par = self.i % 2
        cross = not self.serial and not after_begin
        sA, sB, sC, sD = (self.streams * 4)[:4] if self.serial else self.streams
        c = self.calls[par]

        def run(name, stream):
            if timing is not None:
                timing[name][0].record(stream)
            c[name]()
            if timing is not None:
                timing[name][1].record(stream)

        early = self.early
        for k, evs in early.items():  # the kernel k waits for records this step's event
            self.t[f"_launch_{_LAUNCH_KEY[EARLY_OF[k]]}{par}"].contents.early_event = evs[par].cuda_event
        if cross:
            # X of this layer: the previous attention's output
            sD.wait_event((early.get("predict_q") or self.attn_done)[1 - par])
        run("predict_q", sD)  # Q_pred buffer i % 2
        if not self.serial:
            self.gemm_done[par].record(sD)
            sA.wait_event((early.get("score_topk") or self.gemm_done)[par])
        run("score_topk", sA)  # list set i % 2
        self.sel_done[par].record(sA)
        run("build_digest", sC)
        if cross:
            # step i-1's selection wrote list set (i+1) % 2
            sB.wait_event((early.get("sparse_attn_merge") or self.sel_done)[1 - par])
        if before_attention is not None:
            before_attention(par, sB)
        run("sparse_attn_merge", sB)
        self.attn_done[par].record(sB)
        self.i += 1


def packed(specs, device):
    """One byte buffer holding tensors of the given (name, shape, dtype), each at a 256-byte
    aligned offset, and the tensors as views of it (one copy moves them all)."""
    import torch

    layout, off = [], 0
    for name, shape, dtype in specs:
        n = int(math.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        layout.append((name, tuple(shape), dtype, off, n))
        off += (n + 255) // 256 * 256
    buf = torch.empty(off, dtype=torch.uint8, device=device)
    return buf, {name: buf[o:o + n].view(dtype).view(shape) for name, shape, dtype, o, n in layout}


def setup_step(shape, device, pool_slots=None, serial=False, split=SPLIT, early=EARLY, pdl=False, compact=True,
               keep_all=True):
    """Device inputs, prefill digests, both list sets and the prepared calls of a step.
    ``compact``: the K/V pool the step reads holds only the resident blocks and each unit's
    tail block (the one being written), as the GPU's share of the cache (25% of the blocks in
    the Qwen3-14B-shaped layer: 1.34 GB instead of 5.4 GB); the prefill digests are built from
    the whole cache first, which stays on the device as ``K_all`` / ``V_all`` (with
    ``page_table_all``) only for the CPU-side legs of the benchmark, which read every block
    (``keep_all=False`` frees it).
    ``early``: the kernels (of ``EARLY_OF``) that start early after the kernel they wait for.
    ``pdl`` (serial only): the three persistent kernels start early after the kernel before
    them on the one stream (the selection after the GEMM, the attention after the digest
    append, which itself waits for the selection, the GEMM after the attention)."""
    if pdl and not serial:
        raise ValueError("pdl applies to the serial step: on four streams the kernel before a selection on its "
                         "stream is the previous selection, whose CPU list it reads before it waits")
    if any(k not in EARLY_OF for k in early):
        raise ValueError(f"early starters must be among {sorted(EARLY_OF)}")
    import torch

    import block_sparse_kv_pred_gb300 as bs
    from block_sparse_kv_pred_gb300 import workload as W
    from block_sparse_kv_pred_gb300.workload import device as WD

    s = shape
    if pool_slots is not None:
        compact = False  # the aliased profiling pool is its own layout
    wl = W.Workload(s, pool_slots=pool_slots)
    d = WD.materialize(wl, device=device)
    U, nb, D = s.units, s.nblk, s.D
    t = {k: v for k, v in d.items()}
    t["digest_next"] = torch.empty((s.B, s.Hkv, nb, 2, D), dtype=torch.bfloat16, device=device)
    bs.build_digest("minmax", d["K_pool"], d["page_table"], d["seq_len"], s.B, s.Hkv, s.P, t["digest_next"])
    t["digest_cur"] = t["digest_next"].clone()
    tail = [[u, int(wl.nvalid[u // s.Hkv]) - 1] for u in range(U)]
    t["tail"] = torch.tensor(tail, dtype=torch.int32, device=device)
    n_slots = wl.n_slots
    if compact:
        keep = wl.resident.astype(bool)
        for u, j in tail:
            if j >= 0:
                keep[u, j] = True
        t["K_all"], t["V_all"], t["page_table_all"] = t["K_pool"], t["V_pool"], t["page_table"]
        t["K_pool"], t["V_pool"], t["page_table"], n_slots = WD.materialize_pool(wl, keep, device)
        if not keep_all:
            for n in ("K_all", "V_all", "page_table_all"):
                del t[n]
            del d
            torch.cuda.synchronize(device)
            torch.cuda.empty_cache()
    t["n_slots"] = n_slots
    i32, f32, bf16 = torch.int32, torch.float32, torch.bfloat16
    for par in (0, 1):
        t[f"Qp{par}"] = torch.empty((s.B, s.Hq * D), dtype=bf16, device=device)
        # the step's inputs (layer input X, query, CPU partial) alternate between two buffers too,
        # so that a copy of step i+1's inputs may land while step i still reads its own; each set
        # is one buffer, so that one copy brings it in
        t[f"in{par}"], views = packed([(n, t[n].shape, t[n].dtype) for n in ("X", "q", "O_cpu", "lse_cpu")], device)
        for n, v in views.items():
            t[f"{n}{par}"] = v
            v.copy_(t[n])
        # the outputs alternate too, so a step's may be read back while the next is written; the
        # ones read back every step (O, LSE, the CPU work list) are one buffer
        t[f"out{par}"], views = packed([("O", (s.B, s.Hq, D), bf16), ("lse", (s.B, s.Hq), f32),
                                        ("cpu", (s.B, s.Hkv, s.k), i32), ("cpu_count", (s.B, s.Hkv), i32)], device)
        for n, v in views.items():
            t[f"{n}{par}"] = v
        for name in ("topk", "res", "delta"):
            t[f"{name}{par}"] = torch.empty((s.B, s.Hkv, s.k), dtype=i32, device=device)
            t[f"{name}_count{par}"] = torch.empty((s.B, s.Hkv), dtype=i32, device=device)
        for name in ("topk", "res", "cpu", "delta"):
            t[f"{name}{par}"].fill_(-1)
            t[f"{name}_count{par}"].zero_()
    t["ws_t"] = bs.score_topk_workspace(s.B, s.Hkv, nb, device=device)
    t["ws_a"] = bs.sparse_attn_workspace(s.B, s.Hq, s.Hkv, s.P, device=device)
    t["status"] = torch.zeros(1, dtype=torch.int32, device=device)

    if serial:
        streams = [torch.cuda.Stream(device)]  # not the legacy default stream: it can be captured
        cap_gemm = cap_sel = cap_attn = None
    else:
        streams = [torch.cuda.Stream(device) for _ in range(4)]
        cap_gemm, cap_sel, cap_attn = split if len(split) == 3 else (split[0], split[0], split[1])
    early = () if serial else tuple(early)
    # launch options per kernel and parity; a Step writes the programmatic event of each kernel
    # that an early starter waits for into its options before the launch
    t["_early_kernels"] = early
    for par in (0, 1):
        for key, cap in (("gemm", cap_gemm), ("score", cap_sel), ("attn", cap_attn)):
            t[f"_launch_{key}{par}"] = bs._launch(cap if cap is not None or not early else 0, pdl=pdl)
    sA, sB, sC, sD = ((streams * 4)[:4] if serial else streams)
    sA, sB, sC, sD = sA.cuda_stream, sB.cuda_stream, sC.cuda_stream, sD.cuda_stream
    p = lambda name: t[name].data_ptr()  # noqa: E731
    append = bs.Prepared("scout_build_digest", bs.MINMAX, p("K_pool"), n_slots, p("page_table"), p("seq_len"),
                         s.B, s.Hkv, D, s.P, nb, p("tail"), U, p("digest_cur"), p("status"), sC)
    calls = []
    for par in (0, 1):
        new, old = str(par), str(1 - par)
        calls.append({
            "build_digest": append,
            "predict_q": bs.Prepared("scout_predict_q", p("X" + new), p("W"), p("Qp" + new), s.B, s.Hq * D,
                                     s.hidden, p("status"), t["_launch_gemm" + new], sD),
            # the previous step's CPU list is the prev list, so delta = newly offloaded blocks
            "score_topk": bs.Prepared(
                "scout_score_topk", bs.MINMAX, p("Qp" + new), p("digest_next"), p("seq_len"), p("resident_bits"),
                p("cpu" + old), p("cpu_count" + old), s.B, s.Hq, s.Hkv, D, s.P, nb, s.k, None, p("topk" + new),
                p("topk_count" + new), p("res" + new), p("res_count" + new), p("cpu" + new), p("cpu_count" + new),
                p("delta" + new), p("delta_count" + new), p("ws_t"), t["ws_t"].numel(), p("status"),
                t["_launch_score" + new], sA),
            "sparse_attn_merge": bs.Prepared(
                "scout_sparse_attn_merge", p("q" + new), p("K_pool"), p("V_pool"), n_slots, p("page_table"),
                p("seq_len"), p("res" + old), p("res_count" + old), s.B, s.Hq, s.Hkv, D, s.P, nb, s.k, s.scale,
                p("O_cpu" + new), p("lse_cpu" + new), p("O" + new), p("lse" + new), p("ws_a"), t["ws_a"].numel(),
                p("status"), t["_launch_attn" + new], sB),
        })
    # list set 1 holds a selection before step 0 (the one the prefill step would have made)
    calls[1]["predict_q"]()
    torch.cuda.synchronize(device)  # the two calls sit on different streams
    calls[1]["score_topk"]()
    torch.cuda.synchronize(device)
    return wl, t, Step(t, calls, streams, serial)


def algorithmic_bytes(s, wl, t):
    """Bytes each kernel must move per launch (inputs read once, outputs written once)."""
    U, D, P, k = s.units, s.D, s.P, s.k
    nvalid = int(sum(int(wl.nvalid[u // s.Hkv]) for u in range(U)))
    res_total = int(t["res_count1"].sum().item())
    cpu_total = int(t["cpu_count1"].sum().item())
    q_bytes = s.B * s.Hq * D * 2
    cpu_part = s.B * s.Hq * (D * 4 + 4)
    out = s.B * s.Hq * (D * 2 + 4)
    return {
        "build_digest": U * (P * D * 2 + 2 * D * 2 + 8) + s.B * 4,
        "predict_q": s.Hq * D * s.hidden * 2 + s.B * s.hidden * 2 + s.B * s.Hq * D * 2,
        "score_topk": nvalid * 2 * D * 2 + q_bytes + U * s.words * 4 + s.B * 4 + cpu_total * 4 + U * 4
        + 4 * (U * k * 4 + U * 4),
        "sparse_attn_merge": res_total * (2 * P * D * 2 + 8) + q_bytes + cpu_part + out + U * 4 + s.B * 4,
        "_res_blocks": res_total,
    }
