"""Multi-step decode sweep (scaled down): the true query walks, Q_pred sits at cosine 0.93,
one token is appended per step (digest append of the tail block, a fresh page when a
block starts), the CPU work list's delta is taken against the previous step, and every
8 steps a recall brings the selected blocks in.  Each step is checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import block_sparse_kv_pred_gb300 as bs
from block_sparse_kv_pred_gb300 import workload as W
from block_sparse_kv_pred_gb300.workload import device as WD
from _parity import bits_from_mask, check_attention, check_list_algebra, check_selection, ensure_built, to_dev

pytestmark = pytest.mark.gpu

STEPS, RECALL_EVERY = 24, 8


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _host_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()


def test_decode_sweep_with_walk_append_delta_and_recall():
    s = W.Shape("sweep", B=2, Hq=8, Hkv=2, T=4096, P=32, k=16, resident_frac=0.25, seq_lens=(4096 - 40, 4096 - 70))
    wl = W.Workload(s)
    U, nb, P, D = s.units, s.nblk, s.P, s.D
    qs, ps = wl.walk(STEPS)
    hostK = np.stack([wl.unit_kv(u).reshape(nb, P, D) for u in range(U)])
    hostV = np.stack([wl.unit_kv(u, "V").reshape(nb, P, D) for u in range(U)])
    hK, hV = _host_bf16(hostK), _host_bf16(hostV)

    # prefill digests over every block (the whole context was on the GPU at prefill)
    full = WD.materialize(wl, with_gemm=False)
    dg = torch.empty((s.B, s.Hkv, nb, 2, D), dtype=torch.bfloat16, device="cuda")
    bs.build_digest("minmax", full["K_pool"], full["page_table"], full["seq_len"], s.B, s.Hkv, P, dg)
    torch.cuda.synchronize()
    del full

    # a pool of the resident blocks plus spare pages for the blocks the decode starts
    res = wl.resident.astype(bool).copy()
    table = np.full((U, nb), -1, np.int32)
    n_res = int(res.sum())
    n_slots = n_res + 4 * U
    it = iter(np.random.default_rng(3).permutation(n_res))
    for u in range(U):
        for j in np.flatnonzero(res[u]):
            table[u, j] = next(it)
    spare = list(range(n_res, n_slots))
    Kp = np.zeros((n_slots, P, D), np.uint16)
    Vp = np.zeros((n_slots, P, D), np.uint16)
    for u in range(U):
        for j in np.flatnonzero(res[u]):
            Kp[table[u, j]], Vp[table[u, j]] = hostK[u, j], hostV[u, j]
    K_pool, V_pool = to_dev(Kp), to_dev(Vp)
    d_table = to_dev(table.reshape(s.B, s.Hkv, nb))
    d_bits = to_dev(bits_from_mask(res).reshape(s.B, s.Hkv, -1).view(np.int32))
    side = torch.cuda.Stream()

    seq = wl.seq_len.astype(np.int32).copy()
    ws = bs.score_topk_workspace(s.B, s.Hkv, nb)
    wa = bs.sparse_attn_workspace(s.B, s.Hq, s.Hkv, P)
    scores = torch.empty((s.B, s.Hkv, nb), dtype=torch.float32, device="cuda")
    prev = None
    cpu_sizes, delta_sizes = [], []

    def move_in(ops):
        """Copy ops' blocks into their slots on the side stream, commit after the copy event."""
        done = torch.cuda.Event()
        bs.recall_async([tuple(int(x) for x in r) for r in ops], hK, hV, K_pool, V_pool, s.B, s.Hkv, P, nb, side,
                        done_event=done)
        bs.commit_residency(to_dev(np.array(ops, np.int32).reshape(-1, 4)), d_table, d_bits, n_slots, s.B, s.Hkv,
                            wait_event=done)

    for t in range(STEPS):
        # one token per sequence; a block that starts gets a fresh page
        seq += 1
        fresh = []
        for u in range(U):
            j = int(seq[u // s.Hkv] - 1) // P
            if not res[u, j]:
                slot = spare.pop()
                fresh.append((u, j, slot, -1))
                res[u, j], table[u, j] = True, slot
        if fresh:
            move_in(fresh)
        d_seq = to_dev(seq)
        tail = to_dev(np.array([[u, int(seq[u // s.Hkv] - 1) // P] for u in range(U)], np.int32))
        bs.build_digest("minmax", K_pool, d_table, d_seq, s.B, s.Hkv, P, dg, block_list=tail)
        q, qp = to_dev(qs[t]), to_dev(ps[t])
        out = bs.score_topk("minmax", qp, dg, d_seq, d_bits, s.B, s.Hq, s.Hkv, P, nb, s.k, ws, prev_cpu=prev,
                            scores=scores)
        Og, Lg = bs.sparse_attn(q, K_pool, V_pool, d_table, d_seq, out["res"], out["res_count"], s.B, s.Hq, s.Hkv, P,
                                s.k, s.scale, wa)
        torch.cuda.synchronize()
        g = {n: out[n].cpu().numpy().reshape(U, -1) for n in ("topk", "res", "cpu", "delta")}
        c = {n: out[n + "_count"].cpu().numpy().reshape(-1) for n in ("topk", "res", "cpu", "delta")}
        pc = None if prev is None else (prev[0].cpu().numpy().reshape(U, -1), prev[1].cpu().numpy().reshape(-1))
        Og, Lg = Og.cpu().numpy(), Lg.cpu().numpy()
        for u in range(U):
            b, kvh = divmod(u, s.Hkv)
            L = int(seq[b])
            mn, mx = O.digest_minmax(hostK[u].reshape(nb * P, D), L, P)
            Uref = O.pool_group(O.scores_minmax(O.bf16_to_f64(ps[t][b, kvh * s.G:(kvh + 1) * s.G]), mn, mx))
            S = g["topk"][u, :c["topk"][u]]
            exact = check_selection(Uref, s.k, S, what=(t, u))
            # the split and delta of the GPU's own set are unique: checked at near-ties too
            r_gpu, c_gpu = O.split_residency(S, res[u])
            assert list(g["res"][u, :c["res"][u]]) == list(r_gpu) and list(g["cpu"][u, :c["cpu"][u]]) == list(c_gpu)
            d_ref = O.delta_list(c_gpu, [] if pc is None else pc[0][u, :pc[1][u]])
            assert list(g["delta"][u, :c["delta"][u]]) == list(d_ref), (t, u)
            if not exact:
                continue  # the output over a resident part the oracle did not select is not checked
            r_ref, _ = O.split_residency(O.select_topk(Uref, s.k), res[u])
            K, V = O.bf16_to_f64(hostK[u].reshape(nb * P, D)), O.bf16_to_f64(hostV[u].reshape(nb * P, D))
            toks = O.block_tokens(r_ref, P, L)
            for h in range(s.G):
                hq = kvh * s.G + h
                o, l = O.attention_partial(O.bf16_to_f64(qs[t][b, hq]), K[toks], V[toks], s.scale)
                check_attention(Og[b, hq], Lg[b, hq], o, l, what=(t, u, h))
        cpu_sizes.append(int(c["cpu"].sum()))
        delta_sizes.append(int(c["delta"].sum()))
        prev = (out["cpu"].clone(), out["cpu_count"].clone())

        if t % RECALL_EVERY == RECALL_EVERY - 1:
            sc = scores.cpu().numpy().reshape(U, nb)
            ops = bs.plan_recall(sc, g["topk"], c["topk"], bits_from_mask(res).reshape(U, -1), table, s.k)
            if len(ops):
                move_in(ops)
                torch.cuda.synchronize()
                for u in range(U):
                    mine = [(int(b_), int(sl), int(e)) for uu, b_, sl, e in ops if uu == u]
                    table[u], res[u] = O.apply_recall(table[u], res[u], mine)
                assert np.array_equal(d_table.cpu().numpy().reshape(U, nb), table)
                # the recall brings the selected set in: right after it, nothing selected is off-GPU
                assert all(res[u, j] for u in range(U) for j in g["topk"][u, :c["topk"][u]])
    # the sweep's report: CPU work-list sizes and deltas per step (blocks over all units)
    print("cpu list sizes", cpu_sizes)
    print("delta sizes", delta_sizes)
    assert delta_sizes[0] == cpu_sizes[0] and all(dz <= cz for dz, cz in zip(delta_sizes, cpu_sizes))


def test_page_granular_residency_sweep():
    """The variant of residency per page (one block of a sequence for all its KV heads, the
    transfer unit of section 2.3, Figure 3) through the decode sweep: the residency of a
    sequence's heads stays identical, every step's lists, split and attention match the oracle,
    every recall is the oracle's page plan (recall_plan_pages, the page being written counted as
    selected) applied to each head, and the page being written stays resident."""
    from block_sparse_kv_pred_gb300.sweep import DecodeSweep

    steps, every = 20, 6
    s = W.Shape("sweep_pages", B=2, Hq=8, Hkv=2, T=4096, P=32, k=16, resident_frac=0.0, seq_lens=(4000, 3950),
                hidden=0)
    sw = DecodeSweep(s, steps, recall_every=every, pages=True)
    U, nb, P, D = s.units, s.nblk, s.P, s.D
    hK = {u: sw.hK[u].view(torch.int16).numpy().view(np.uint16).reshape(nb * P, D) for u in range(U)}
    hV = {u: sw.hV[u].view(torch.int16).numpy().view(np.uint16).reshape(nb * P, D) for u in range(U)}
    n_recalls = 0
    for t in range(steps):
        rec = sw.step()
        check_list_algebra(s, rec, nb)
        res = rec["resident"].reshape(s.B, s.Hkv, nb)
        assert np.all(res == res[:, :1, :]), t  # one residency per page
        for u in range(U):
            b, kvh = divmod(u, s.Hkv)
            L = int(rec["seq"][b])
            mn, mx = O.digest_minmax(hK[u], L, P)
            Uref = O.pool_group(O.scores_minmax(O.bf16_to_f64(sw.ps[t][b, kvh * s.G:(kvh + 1) * s.G]), mn, mx))
            S = rec["topk"][u, :rec["topk_count"][u]]
            if not check_selection(Uref, s.k, S, what=(t, u)):
                continue  # a near-tie: the GPU's resident part differs from the oracle's, so does its output
            r_ref, _ = O.split_residency(O.select_topk(Uref, s.k), rec["resident"][u])
            toks = O.block_tokens(r_ref, P, L)
            K, V = O.bf16_to_f64(hK[u]), O.bf16_to_f64(hV[u])
            for h in range(s.G):
                hq = kvh * s.G + h
                o, l = O.attention_partial(O.bf16_to_f64(sw.qs[t][b, hq]), K[toks], V[toks], s.scale)
                check_attention(rec["O"][b, hq], rec["lse"][b, hq], o, l, what=(t, u, h))
        if "ops" in rec:
            n_recalls += 1
            ops = np.asarray(rec["ops"]).reshape(-1, 4)
            for b in range(s.B):
                us = range(b * s.Hkv, (b + 1) * s.Hkv)
                tail = (int(rec["seq"][b]) - 1) // P  # the page being written counts as selected
                want = O.recall_plan_pages([rec["scores"][u].astype(np.float64) for u in us],
                                           [list(rec["topk"][u, :rec["topk_count"][u]]) + [tail] for u in us],
                                           rec["res_before"][b * s.Hkv], [rec["table_before"][u] for u in us])
                for h, u in enumerate(us):
                    got = [(int(j), int(sl), int(e)) for uu, j, sl, e in ops if uu == u]
                    assert got == want[h], (t, u)
            # the pool holds each recalled block's own K/V at its new slot
            Kp = sw.K_pool.view(torch.int16).cpu().numpy().view(np.uint16)
            for u, j, sl, _ in ops[:: max(1, len(ops) // 8)]:
                assert np.array_equal(Kp[sl], hK[int(u)][int(j) * P:(int(j) + 1) * P]), (t, u, j)
        tails = (rec["seq"].astype(np.int64) - 1) // P
        assert all(sw.res[u, tails[u // s.Hkv]] for u in range(U)), t  # the page being written stays
    assert n_recalls == steps // every


def test_sweep_cpu_side_matches_oracle_and_reports_idle():
    """The sweep's CPU side (the worker pool over each step's CPU list with Q_pred on the host copy
    of the K/V) against the oracle's attention over the same blocks, and its report fields."""
    from block_sparse_kv_pred_gb300.sweep import DecodeSweep

    s = W.Shape("sweep_cpu", B=2, Hq=8, Hkv=2, T=4096, P=32, k=16, resident_frac=0.0, seq_lens=(4000, 3950),
                hidden=0)
    with bs.CpuPool(4) as pool:
        sw = DecodeSweep(s, 3, recall_every=0, cpu_pool=pool)
        nb, P, D = s.nblk, s.P, s.D
        for t in range(3):
            rec = sw.step()
            st = rec["stats"]
            assert st["cpu_ms"] > 0 and st["gpu_ms"] > 0 and 0.0 <= st["gpu_idle_frac"] <= 1.0
            for u in range(s.units):
                b, kvh = divmod(u, s.Hkv)
                K = O.bf16_to_f64(sw.hK[u].view(torch.int16).numpy().view(np.uint16).reshape(nb * P, D))
                V = O.bf16_to_f64(sw.hV[u].view(torch.int16).numpy().view(np.uint16).reshape(nb * P, D))
                toks = O.block_tokens(rec["cpu"][u, :rec["cpu_count"][u]], P, int(rec["seq"][b]))
                for h in range(s.G):
                    hq = kvh * s.G + h
                    o, l = O.attention_partial(O.bf16_to_f64(sw.ps[t][b, hq]), K[toks], V[toks], s.scale)
                    check_attention(rec["O_cpu"][b, hq], rec["lse_cpu"][b, hq], o, l, what=(t, u, h))
