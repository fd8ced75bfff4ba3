"""The library's host-side recall planner (scout_plan_recall) against the oracle's
reading of section 3.4, on many seeded units with ties (no GPU needed)."""
import os

import numpy as np
import pytest

import oracle as O
import block_sparse_kv_pred_gb300 as bs
from block_sparse_kv_pred_gb300 import build as B


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not os.path.exists(bs.lib_path()):
        B.build()


def _case(seed, units=6, nblk=70, k=12):
    rng = np.random.default_rng(seed)
    scores = np.round(rng.standard_normal((units, nblk)), 1).astype(np.float32)  # coarse: many ties
    nvalid = rng.integers(1, nblk + 1, size=units)
    topk = np.full((units, k), -1, np.int32)
    cnt = np.zeros(units, np.int32)
    res = np.zeros((units, nblk), bool)
    table = np.full((units, nblk), -1, np.int32)
    slots = rng.permutation(units * nblk).astype(np.int32)
    for u in range(units):
        scores[u, nvalid[u]:] = -np.inf
        S = O.select_topk(scores[u, : nvalid[u]].astype(np.float64), k)
        topk[u, : len(S)] = S
        cnt[u] = len(S)
        res[u, : nvalid[u]] = rng.random(nvalid[u]) < rng.uniform(0.1, 0.9)
        table[u, res[u]] = slots[u * nblk: u * nblk + res[u].sum()]
    bits = np.zeros((units, (nblk + 31) // 32), np.uint32)
    for u in range(units):
        for j in np.flatnonzero(res[u]):
            bits[u, j >> 5] |= np.uint32(1 << (j & 31))
    return scores, topk, cnt, bits, table, res, k


@pytest.mark.parametrize("seed", range(12))
def test_plan_recall_matches_oracle(seed):
    scores, topk, cnt, bits, table, res, k = _case(seed)
    got = bs.plan_recall(scores, topk, cnt, bits, table, k)
    want = []
    for u in range(scores.shape[0]):
        for b, slot, e in O.recall_plan(scores[u].astype(np.float64), topk[u, : cnt[u]], res[u], table[u]):
            want.append((u, b, slot, e))
    assert [tuple(int(x) for x in r) for r in got] == want


def test_plan_recall_rejects_bad_input():
    scores, topk, cnt, bits, table, res, k = _case(0, units=2)
    bad = topk.copy()
    bad[0, 0] = 10_000
    with pytest.raises(bs.ScoutError):
        bs.plan_recall(scores, bad, cnt, bits, table, k)
    lost = table.copy()
    lost[res] = -1  # resident blocks without a slot
    if any(len(O.recall_plan(scores[u].astype(np.float64), topk[u, : cnt[u]], res[u], table[u])) for u in range(2)):
        with pytest.raises(bs.ScoutError):
            bs.plan_recall(scores, topk, cnt, bits, lost, k)


def test_planner_shapes_are_checked_before_the_foreign_call():
    """Arrays whose shapes do not match (units, nblk_cap, k) are refused by the binding before the
    C planner could read past them."""
    scores, topk, cnt, bits, table, _, k = _case(5)
    for bad in (dict(topk=topk[:-1]), dict(topk=topk[:, :-1]), dict(cnt=cnt[:-1]), dict(bits=bits[:, :1]),
                dict(table=table[:, :-3]), dict(table=table[:-1])):
        a = dict(scores=scores, topk=topk, cnt=cnt, bits=bits, table=table)
        a.update(bad)
        with pytest.raises(bs.ScoutError):
            bs.plan_recall(a["scores"], a["topk"], a["cnt"], a["bits"], a["table"], k)
    with pytest.raises(bs.ScoutError):
        bs.plan_recall_pages(scores, topk, cnt[:-1], bits, table, 3, 2, k)
