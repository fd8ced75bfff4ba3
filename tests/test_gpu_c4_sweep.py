"""The residency sweep at its full shape (batch 16, 40/8 heads, 64K context, 32-token pages,
budget 2048 = 64 blocks per KV head, the GPU holding k blocks per head): 33 decode steps of
the query walk with one token appended per step, the CPU work list's delta against the
previous step, and recalls after steps 16 and 32.  Every step is checked against the fp64
oracle on sampled units: selection with Q_pred, residency split and delta, attention with
the true query over the resident part; every recall against the oracle's plan."""
import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_kv_pred_gb300.sweep import DecodeSweep, c4_shape
from _parity import check_attention, check_selection, ensure_built

pytestmark = pytest.mark.gpu

STEPS, RECALL_EVERY = 33, 16
SAMPLE = (0, 45, 127)


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_c4_sweep_full_shape():
    sw = DecodeSweep(c4_shape(STEPS), STEPS, RECALL_EVERY)
    s = sw.s
    nb, P, D, G = s.nblk, s.P, s.D, s.G
    hK = sw.hK.view(torch.int16).numpy().view(np.uint16)  # [U][nblk][P][D] bf16 bits
    hV = sw.hV.view(torch.int16).numpy().view(np.uint16)
    KV = {u: (O.bf16_to_f64(hK[u].reshape(nb * P, D)), O.bf16_to_f64(hV[u].reshape(nb * P, D))) for u in SAMPLE}
    stats = []
    for t in range(STEPS):
        rec = sw.step()
        stats.append(rec["stats"])
        for u in SAMPLE:
            b, kvh = divmod(u, s.Hkv)
            L = int(rec["seq"][b])
            mn, mx = O.digest_minmax(hK[u].reshape(nb * P, D), L, P)
            Uref = O.pool_group(O.scores_minmax(O.bf16_to_f64(sw.ps[t][b, kvh * G:(kvh + 1) * G]), mn, mx))
            S = rec["topk"][u, :rec["topk_count"][u]]
            exact = check_selection(Uref, s.k, S, what=(t, u))
            # the split and delta of the GPU's own set are unique: checked at near-ties too
            r_gpu, c_gpu = O.split_residency(S, rec["resident"][u])
            assert list(rec["res"][u, :rec["res_count"][u]]) == list(r_gpu), (t, u)
            assert list(rec["cpu"][u, :rec["cpu_count"][u]]) == list(c_gpu), (t, u)
            prev = [] if rec["prev_cpu"] is None else rec["prev_cpu"][0][u, :rec["prev_cpu"][1][u]]
            assert list(rec["delta"][u, :rec["delta_count"][u]]) == list(O.delta_list(c_gpu, prev)), (t, u)
            if not exact:
                continue  # the output over a resident part the oracle did not select is not checked
            r_ref, _ = O.split_residency(O.select_topk(Uref, s.k), rec["resident"][u])
            K, V = KV[u]
            toks = O.block_tokens(r_ref, P, L)
            for h in range(G):
                hq = kvh * G + h
                o, l = O.attention_partial(O.bf16_to_f64(sw.qs[t][b, hq]), K[toks], V[toks], s.scale)
                check_attention(rec["O"][b, hq], rec["lse"][b, hq], o, l, what=(t, u, h))
        if "ops" in rec:
            ops = np.asarray(rec["ops"]).reshape(-1, 4)
            for u in SAMPLE:
                want = O.recall_plan(rec["scores"][u].astype(np.float64), rec["topk"][u, :rec["topk_count"][u]],
                                     rec["res_before"][u], rec["table_before"][u])
                got = [(int(j), int(sl), int(e)) for uu, j, sl, e in ops if uu == u]
                assert got == want, (t, u)
                table, res = O.apply_recall(rec["table_before"][u], rec["res_before"][u], want)
                assert np.array_equal(sw.table[u], table) and np.array_equal(sw.res[u], res)
            # the selected blocks are resident afterwards (the resident set keeps its size)
            assert all(sw.res[u, j] for u in range(s.units) for j in rec["topk"][u, :rec["topk_count"][u]])
    print("per-step", [(st["step"], st["cpu_blocks"], st["delta_blocks"], round(st["cpu_ratio"], 3))
                       for st in stats])
    print("recalls", [(st["step"], st["recall_blocks"], st["recall_h2d_gbs"]) for st in stats if st["recall_blocks"]])
    assert stats[0]["delta_blocks"] == stats[0]["cpu_blocks"]
    assert all(st["delta_blocks"] <= st["cpu_blocks"] for st in stats)
    # right after a recall the whole selection is resident, so the CPU list only holds what
    # the next selection adds
    assert stats[RECALL_EVERY]["cpu_blocks"] < stats[RECALL_EVERY - 1]["cpu_blocks"]
