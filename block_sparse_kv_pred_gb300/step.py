"""One decode step of one layer through the libscout C ABI.

``setup_step`` materialises a seeded workload on the device, builds the prefill
digests and prepares the five calls of a step (digest append, Q_pred, score and
select, sparse attention, merge) with their arguments converted once, so that a
step costs five foreign calls of host work.  ``algorithmic_bytes`` gives the
bytes each kernel must move per launch, the numerator of the roofline.
"""
from __future__ import annotations

KERNELS = ("build_digest", "predict_q", "score_topk", "sparse_attn", "merge")


def setup_step(shape, device, pool_slots=None):
    """Device inputs, prefill digests and the five prepared C-ABI calls of one step."""
    import torch

    import block_sparse_kv_pred_gb300 as bs
    from block_sparse_kv_pred_gb300 import workload as W
    from block_sparse_kv_pred_gb300.workload import device as WD

    s = shape
    wl = W.Workload(s, pool_slots=pool_slots)
    d = WD.materialize(wl, device=device)
    U, nb, D = s.units, s.nblk, s.D
    t = {k: v for k, v in d.items()}
    t["digest"] = torch.empty((s.B, s.Hkv, nb, 2, D), dtype=torch.bfloat16, device=device)
    bs.build_digest("minmax", d["K_pool"], d["page_table"], d["seq_len"], s.B, s.Hkv, s.P, t["digest"])
    tail = [[u, int(wl.nvalid[u // s.Hkv]) - 1] for u in range(U)]
    t["tail"] = torch.tensor(tail, dtype=torch.int32, device=device)
    t["Qp"] = torch.empty((s.B, s.Hq * D), dtype=torch.bfloat16, device=device)
    t["ws_t"] = bs.score_topk_workspace(s.B, s.Hkv, nb, device=device)
    for name in ("topk", "res", "cpu", "delta"):
        t[name] = torch.full((s.B, s.Hkv, s.k), -1, dtype=torch.int32, device=device)
        t[name + "_count"] = torch.zeros((s.B, s.Hkv), dtype=torch.int32, device=device)
    t["ws_a"] = bs.sparse_attn_workspace(s.B, s.Hq, s.Hkv, s.P, device=device)
    t["O_gpu"] = torch.empty((s.B, s.Hq, D), dtype=torch.float32, device=device)
    t["lse_gpu"] = torch.empty((s.B, s.Hq), dtype=torch.float32, device=device)
    t["O"] = torch.empty((s.B, s.Hq, D), dtype=torch.bfloat16, device=device)
    t["lse"] = torch.empty((s.B, s.Hq), dtype=torch.float32, device=device)
    t["status"] = torch.zeros(1, dtype=torch.int32, device=device)
    st = torch.cuda.current_stream(device).cuda_stream
    p = lambda name: t[name].data_ptr()  # noqa: E731
    calls = [
        bs.Prepared("scout_build_digest", bs.MINMAX, p("K_pool"), wl.n_slots, p("page_table"), p("seq_len"), s.B,
                    s.Hkv, D, s.P, nb, p("tail"), U, p("digest"), p("status"), st),
        bs.Prepared("scout_predict_q", p("X"), p("W"), p("Qp"), s.B, s.Hq * D, s.hidden, p("status"), st),
        # the previous step's CPU list is this step's prev list (in place), so delta = newly offloaded blocks
        bs.Prepared("scout_score_topk", bs.MINMAX, p("Qp"), p("digest"), p("seq_len"), p("resident_bits"), p("cpu"),
                    p("cpu_count"), s.B, s.Hq, s.Hkv, D, s.P, nb, s.k, None, p("topk"), p("topk_count"), p("res"),
                    p("res_count"), p("cpu"), p("cpu_count"), p("delta"), p("delta_count"), p("ws_t"),
                    t["ws_t"].numel(), st),
        bs.Prepared("scout_sparse_attn", p("q"), p("K_pool"), p("V_pool"), wl.n_slots, p("page_table"),
                    p("seq_len"), p("res"), p("res_count"), s.B, s.Hq, s.Hkv, D, s.P, nb, s.k, s.scale, p("O_gpu"),
                    p("lse_gpu"), p("ws_a"), t["ws_a"].numel(), p("status"), st),
        bs.Prepared("scout_merge", p("O_gpu"), p("lse_gpu"), p("O_cpu"), p("lse_cpu"), s.B * s.Hq, D, p("O"),
                    p("lse"), st),
    ]
    return wl, t, calls


def algorithmic_bytes(s, wl, t):
    """Bytes each kernel must move per launch (inputs read once, outputs written once)."""
    U, D, P, k = s.units, s.D, s.P, s.k
    nvalid = int(sum(int(wl.nvalid[u // s.Hkv]) for u in range(U)))
    res_total = int(t["res_count"].sum().item())
    cpu_total = int(t["cpu_count"].sum().item())
    q_bytes = s.B * s.Hq * D * 2
    part = s.B * s.Hq * (D * 4 + 4)
    return {
        "build_digest": U * (P * D * 2 + 2 * D * 2 + 8) + s.B * 4,
        "predict_q": s.Hq * D * s.hidden * 2 + s.B * s.hidden * 2 + s.B * s.Hq * D * 2,
        "score_topk": nvalid * 2 * D * 2 + q_bytes + U * s.words * 4 + s.B * 4 + cpu_total * 4 + U * 4
        + 4 * (U * k * 4 + U * 4),
        "sparse_attn": res_total * (2 * P * D * 2 + 8) + q_bytes + part + U * 4 + s.B * 4,
        "merge": 2 * part + s.B * s.Hq * (D * 2 + 4),
        "_res_blocks": res_total,
    }
