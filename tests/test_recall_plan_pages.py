"""Recall with residency per page: one block of a sequence for all its KV heads, the 128 KB
transfer unit the pages compare with per-token PCIe transfers (recall of section 3.4).  The
oracle's reading is pinned by a hand-worked example and by the properties that fix a plan;
scout_plan_recall_pages is checked against it on seeded sequences.  Parity unpinned as a
reading: the pages do not say how per-head selections map to shared pages (here: a page is
needed when any head selects it, and ranked by the largest of its heads' scores).  Host only."""
import ctypes

import numpy as np
import pytest

import oracle as O
import block_sparse_kv_pred_gb300 as bs
from _parity import bits_from_mask, ensure_built


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_hand_worked_example():
    U = [[5, 1, 4, 9, 0, 7, 2, 3], [0, 6, 8, 2, 1, 1, 3, 3]]  # importance (max): 5 6 8 9 1 7 3 3
    sel = [[0, 3, 5], [2, 3]]                                  # chosen pages {0, 2, 3, 5}
    slots = [[100 * h + j for j in range(8)] for h in range(2)]
    res = np.zeros(8, bool)
    res[[0, 1, 4, 6]] = True
    # need 3 (9), 2 (8), 5 (7); free 4 (1), 6 (3), 1 (6); pairs (3,4) (2,6) (5,1)
    want = [[(2, 6, 6), (3, 4, 4), (5, 1, 1)], [(2, 106, 6), (3, 104, 4), (5, 101, 1)]]
    assert O.recall_plan_pages(U, sel, res, slots) == want
    res[:] = False
    res[[0, 4]] = True  # one free page: only the most important needed page comes in
    assert O.recall_plan_pages(U, sel, res, slots) == [[(3, 4, 4)], [(3, 104, 4)]]


def _random_case(rng, B, Hkv, nb, k):
    U = rng.standard_normal((B * Hkv, nb)).astype(np.float32)
    U[rng.random(U.shape) < 0.05] = 0.5  # ties
    topk = np.full((B * Hkv, k), -1, np.int32)
    cnt = np.zeros(B * Hkv, np.int32)
    for u in range(B * Hkv):
        c = int(rng.integers(0, k + 1))
        topk[u, :c] = np.sort(rng.choice(nb, size=c, replace=False))
        cnt[u] = c
    pages = rng.random((B, nb)) < 0.3
    res = np.repeat(pages, Hkv, axis=0)  # identical bits for the heads of a sequence
    table = np.full((B * Hkv, nb), -1, np.int32)
    table[res] = rng.permutation(int(res.sum())).astype(np.int32)
    return U, topk, cnt, res, table


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_library_matches_oracle_and_the_plan_properties(seed):
    rng = np.random.default_rng(seed)
    B, Hkv, nb, k = 3, 4, 70, 9
    U, topk, cnt, res, table = _random_case(rng, B, Hkv, nb, k)
    ops = bs.plan_recall_pages(U, topk, cnt, bits_from_mask(res), table, B, Hkv, k)
    for b in range(B):
        us = range(b * Hkv, (b + 1) * Hkv)
        want = O.recall_plan_pages([U[u] for u in us], [topk[u, :cnt[u]] for u in us], res[b * Hkv],
                                   [table[u] for u in us])
        for h, u in enumerate(us):
            got = [(int(j), int(sl), int(e)) for uu, j, sl, e in ops if uu == u]
            assert got == want[h], (b, h)
        # properties: every head moves the same pages; in pages chosen by some head and not
        # resident, out pages resident and chosen by none; the sequence keeps its page count;
        # the plan is full on one side
        chosen = set().union(*[set(topk[u, :cnt[u]].tolist()) for u in us])
        pairs = [(j, e) for j, _, e in want[0]]
        assert all(want[h] and [(j, e) for j, _, e in want[h]] == pairs or not want[h] and not pairs
                   for h in range(Hkv))
        assert all(j in chosen and not res[b * Hkv, j] for j, _ in pairs)
        assert all(e not in chosen and res[b * Hkv, e] for _, e in pairs)
        need = sum(1 for j in chosen if not res[b * Hkv, j])
        free = sum(1 for j in range(nb) if res[b * Hkv, j] and j not in chosen)
        assert len(pairs) == min(need, free)
        after = res[b * Hkv].copy()
        for j, e in pairs:
            after[e], after[j] = False, True
        assert after.sum() == res[b * Hkv].sum()
    assert [tuple(o[:2]) for o in ops] == sorted(tuple(o[:2]) for o in ops)  # by unit, then block in


def test_bad_arguments_are_rejected():
    rng = np.random.default_rng(9)
    B, Hkv, nb, k = 2, 2, 40, 6
    U, topk, cnt, res, table = _random_case(rng, B, Hkv, nb, k)
    bits = bits_from_mask(res)
    L = bs.lib()
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    ops = (bs.RecallOp * 64)()
    n = ctypes.c_int(-5)

    def call(bits_=bits, table_=table, cap=64):
        return L.scout_plan_recall_pages(p(U), p(topk), p(cnt), p(bits_), p(table_), B, Hkv, nb, k, ops, cap,
                                         ctypes.byref(n))

    odd = bits.copy()
    odd[1, 0] ^= 1  # head 1 of sequence 0 disagrees with head 0
    assert call(bits_=odd) == 1
    topk[0, 0] = nb
    cnt[0] = max(cnt[0], 1)
    assert call() == 1  # a listed block outside the table
    topk[0, 0] = 0
    assert call() == 0 and n.value >= 0
    if n.value:
        assert call(cap=n.value - 1) == 3  # too little room for the ops
        u, evicted = ops[0].unit, ops[0].evict_block
        other = (u // Hkv) * Hkv + (1 - u % Hkv)  # the other head of the same sequence
        bad = table.copy()
        bad[other, evicted] = -1  # the evicted page has no slot in that head
        assert call(table_=bad) == 1
