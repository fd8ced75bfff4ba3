"""The 40-layer decode sweep at its full scope: batch 16, 40/8 heads, 64K context, 32-token
pages, budget 2048 (k = 64 blocks held per KV head), 40 seeded layers x 64 decode steps, one
token appended per step, the query walk (step cosine ~0.96, Q_pred at cosine 0.93), a recall
every 16 steps (section 3.4).

Every (layer, step): the list algebra of every unit (top-k count and order, the residency
split, the delta against the previous step's CPU list).  A seeded unit per layer, on the first
and last step and on the steps either side of each recall: the selection against the oracle's
fp64 scores over its digests (kept up to date block by block as tokens are appended), the
attention over the resident part against the oracle's, and each recall against the oracle's
plan."""
import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_kv_pred_gb300.sweep import c4_shape, run_layers
from _parity import check_attention, check_list_algebra, check_selection, ensure_built

pytestmark = pytest.mark.gpu

LAYERS, STEPS, EVERY = 40, 64, 16
CHECKED = sorted({0, 1, STEPS - 1} | {r + d for r in range(EVERY - 1, STEPS - 1, EVERY) for d in (0, 1, 2)})


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_forty_layers_sixty_four_steps():
    s0 = c4_shape(STEPS)
    nb, P, D, G = s0.nblk, s0.P, s0.D, s0.G
    rng = np.random.default_rng(40)
    units = rng.integers(0, s0.units, size=LAYERS)
    per_layer = {}
    state = {}
    for layer, sw, rec in run_layers(LAYERS, STEPS, EVERY):
        s, t = sw.s, rec["t"]
        check_list_algebra(s, rec, nb)
        u = int(units[layer])
        b, kvh = divmod(u, s.Hkv)
        L = int(rec["seq"][b])
        if t == 0:  # the sampled unit's K/V (host copy = the pool's pages) and its digests
            hK = sw.hK[u].view(torch.int16).numpy().view(np.uint16).reshape(nb * P, D)
            hV = sw.hV[u].view(torch.int16).numpy().view(np.uint16).reshape(nb * P, D)
            mn, mx = np.zeros((nb, D)), np.zeros((nb, D))  # rows past the valid blocks are never read
            v = -(-L // P)
            mn[:v], mx[:v] = O.digest_minmax(hK, L, P)
            state = dict(K=O.bf16_to_f64(hK), V=O.bf16_to_f64(hV), Kbits=hK, mn=mn, mx=mx)
        else:  # the appended token changes the tail block's digest only (it may start a new block)
            j = (L - 1) // P
            tmn, tmx = O.digest_minmax(state["Kbits"][j * P:(j + 1) * P], L - j * P, P)
            state["mn"][j], state["mx"][j] = tmn[0], tmx[0]
        per_layer.setdefault(layer, []).append(rec["stats"])
        if t in CHECKED:
            v = -(-L // P)
            Uref = O.pool_group(O.scores_minmax(O.bf16_to_f64(sw.ps[t][b, kvh * G:(kvh + 1) * G]), state["mn"][:v],
                                                state["mx"][:v]))
            S = rec["topk"][u, :rec["topk_count"][u]]
            # at a near-tie the GPU's resident part differs from the oracle's, and so does its output
            if check_selection(Uref, s.k, S, what=(layer, t, u)):
                r_ref, _ = O.split_residency(O.select_topk(Uref, s.k), rec["resident"][u])
                toks = O.block_tokens(r_ref, P, L)
                for h in range(G):
                    hq = kvh * G + h
                    o, l = O.attention_partial(O.bf16_to_f64(sw.qs[t][b, hq]), state["K"][toks], state["V"][toks],
                                               s.scale)
                    check_attention(rec["O"][b, hq], rec["lse"][b, hq], o, l, what=(layer, t, u, h))
        if "ops" in rec:
            ops = np.asarray(rec["ops"]).reshape(-1, 4)
            want = O.recall_plan(rec["scores"][u].astype(np.float64), rec["topk"][u, :rec["topk_count"][u]],
                                 rec["res_before"][u], rec["table_before"][u])
            assert [(int(j), int(sl), int(e)) for uu, j, sl, e in ops if uu == u] == want, (layer, t)
            assert all(sw.res[uu, j] for uu in range(s.units) for j in rec["topk"][uu, :rec["topk_count"][uu]])
    assert sorted(per_layer) == list(range(LAYERS)) and all(len(v) == STEPS for v in per_layer.values())
    for layer, stats in per_layer.items():
        assert stats[0]["delta_blocks"] == stats[0]["cpu_blocks"]
        assert all(st["delta_blocks"] <= st["cpu_blocks"] for st in stats)
        recalls = [st for st in stats if st["recall_blocks"]]
        # a recall at the end of steps 15, 31, 47 and 63
        assert [st["step"] for st in recalls] == list(range(EVERY - 1, STEPS, EVERY))
        assert all(st["recall_h2d_gbs"] > 0 for st in recalls)
        # right after a recall the whole selection was resident: the CPU list holds only what changed
        for r in range(EVERY, STEPS, EVERY):
            assert stats[r]["cpu_blocks"] < stats[r - 1]["cpu_blocks"], (layer, r)
