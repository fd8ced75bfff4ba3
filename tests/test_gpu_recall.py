"""GPU recall path (section 3.4): host plan -> side-stream copies -> commit after the
copy event -> attention over the new residency, checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import block_sparse_kv_pred_gb300 as bs
from block_sparse_kv_pred_gb300 import workload as W
from block_sparse_kv_pred_gb300.workload import device as WD
from _parity import bits_from_mask, check_attention, ensure_built, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _host_bf16(a):
    """uint16 bit patterns -> pinned bf16 host tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()


def _setup():
    """A small pool holding the resident blocks, the selection over the full cache, and the plan."""
    s = W.Shape("recall_g4", B=2, Hq=8, Hkv=2, T=3000, P=32, k=12, resident_frac=0.3, seq_lens=(3000, 2050))
    wl = W.Workload(s)
    d = WD.materialize(wl, with_gemm=False)
    U, nb, P, D = s.units, s.nblk, s.P, s.D
    # scores and the selection over every block (the full pool holds every block)
    dg = torch.empty((s.B, s.Hkv, nb, 2, D), dtype=torch.bfloat16, device="cuda")
    bs.build_digest("minmax", d["K_pool"], d["page_table"], d["seq_len"], s.B, s.Hkv, P, dg)
    scores = torch.empty((s.B, s.Hkv, nb), dtype=torch.float32, device="cuda")
    ws = bs.score_topk_workspace(s.B, s.Hkv, nb)
    sel = bs.score_topk("minmax", d["q"], dg, d["seq_len"], d["resident_bits"], s.B, s.Hq, s.Hkv, P, nb, s.k, ws,
                        scores=scores)
    torch.cuda.synchronize()

    # a small pool that holds only the resident blocks, filled from the host copy of the cache
    hostK = np.stack([wl.unit_kv(u).reshape(nb, P, D) for u in range(U)])  # [U][nb][P][D] bits
    hostV = np.stack([wl.unit_kv(u, "V").reshape(nb, P, D) for u in range(U)])
    res = wl.resident.astype(bool).copy()
    table = np.full((U, nb), -1, np.int32)
    n_slots = int(res.sum())
    order = np.random.default_rng(7).permutation(n_slots)
    it = iter(order)
    for u in range(U):
        for j in np.flatnonzero(res[u]):
            table[u, j] = next(it)
    Kp = np.zeros((n_slots, P, D), np.uint16)
    Vp = np.zeros((n_slots, P, D), np.uint16)
    for u in range(U):
        for j in np.flatnonzero(res[u]):
            Kp[table[u, j]], Vp[table[u, j]] = hostK[u, j], hostV[u, j]
    K_pool, V_pool = to_dev(Kp), to_dev(Vp)
    d_table = to_dev(table.reshape(s.B, s.Hkv, nb))
    d_bits = to_dev(bits_from_mask(res).reshape(s.B, s.Hkv, -1).view(np.int32))

    sc = scores.cpu().numpy().reshape(U, nb)
    topk = sel["topk"].cpu().numpy().reshape(U, s.k)
    cnt = sel["topk_count"].cpu().numpy().reshape(U)
    ops = bs.plan_recall(sc, topk, cnt, bits_from_mask(res).reshape(U, -1), table, s.k)
    want = [(u, b, sl, e) for u in range(U)
            for b, sl, e in O.recall_plan(sc[u].astype(np.float64), topk[u, :cnt[u]], res[u], table[u])]
    assert [tuple(int(x) for x in r) for r in ops] == want and len(ops) > 0
    return dict(s=s, wl=wl, d=d, hostK=hostK, hostV=hostV, res=res, table=table, n_slots=n_slots, K_pool=K_pool,
                V_pool=V_pool, d_table=d_table, d_bits=d_bits, topk=topk, cnt=cnt, ops=ops, want=want)


def _snapshot(st):
    return [t.clone() for t in (st["K_pool"], st["V_pool"], st["d_table"], st["d_bits"])]


@pytest.mark.parametrize("mode", ["copies", "gather"])
def test_recall_then_attention_over_the_new_residency(mode):
    st = _setup()
    s, wl, d, hostK, hostV, res, table, n_slots = (st[k] for k in ("s", "wl", "d", "hostK", "hostV", "res", "table",
                                                                    "n_slots"))
    K_pool, V_pool, d_table, d_bits, topk, cnt, ops, want = (st[k] for k in ("K_pool", "V_pool", "d_table", "d_bits",
                                                                             "topk", "cnt", "ops", "want"))
    U, nb, P = s.units, s.nblk, s.P
    side = torch.cuda.Stream()
    done = torch.cuda.Event()
    hK, hV = _host_bf16(hostK), _host_bf16(hostV)
    d_ops = to_dev(ops)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if mode == "copies":
        bs.recall_async([tuple(int(x) for x in r) for r in ops], hK, hV, K_pool, V_pool, s.B, s.Hkv, P, nb, side,
                        done_event=done)
    else:
        bs.recall_gather_async(d_ops, hK, hV, K_pool, V_pool, s.B, s.Hkv, P, nb, side, done_event=done,
                               status=status)
    bs.commit_residency(d_ops, d_table, d_bits, n_slots, s.B, s.Hkv, wait_event=done)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    # the tables are the oracle's, and every recalled slot holds its block's keys and values
    table2, res2 = table.copy(), res.copy()
    for u in range(U):
        mine = [(b, sl, e) for uu, b, sl, e in want if uu == u]
        table2[u], res2[u] = O.apply_recall(table[u], res[u], mine)
    assert np.array_equal(d_table.cpu().numpy().reshape(U, nb), table2)
    assert np.array_equal(d_bits.cpu().numpy().view(np.uint32).reshape(U, -1), bits_from_mask(res2).reshape(U, -1))
    Kg = K_pool.cpu().view(torch.int16).numpy().view(np.uint16)
    Vg = V_pool.cpu().view(torch.int16).numpy().view(np.uint16)
    for u, b, sl, _ in want:
        assert np.array_equal(Kg[sl], hostK[u, b]) and np.array_equal(Vg[sl], hostV[u, b])

    # attention over the selected blocks that are now resident equals the oracle's over S & R'
    res_list = np.full((U, s.k), -1, np.int32)
    res_cnt = np.zeros(U, np.int32)
    for u in range(U):
        r = [int(j) for j in topk[u, :cnt[u]] if res2[u, j]]
        res_list[u, :len(r)] = r
        res_cnt[u] = len(r)
    wa = bs.sparse_attn_workspace(s.B, s.Hq, s.Hkv, P)
    Og, Lg = bs.sparse_attn(d["q"], K_pool, V_pool, d_table, d["seq_len"], to_dev(res_list.reshape(s.B, s.Hkv, s.k)),
                            to_dev(res_cnt.reshape(s.B, s.Hkv)), s.B, s.Hq, s.Hkv, P, s.k, s.scale, wa)
    torch.cuda.synchronize()
    Og, Lg = Og.cpu().numpy(), Lg.cpu().numpy()
    for u in range(U):
        b, kvh = divmod(u, s.Hkv)
        K, V = O.bf16_to_f64(wl.unit_kv(u)), O.bf16_to_f64(wl.unit_kv(u, "V"))
        toks = O.block_tokens(res_list[u, :res_cnt[u]], P, int(wl.seq_len[b]))
        for h in range(s.G):
            hq = kvh * s.G + h
            o, l = O.attention_partial(O.bf16_to_f64(wl.q[b, hq]), K[toks], V[toks], s.scale)
            check_attention(Og[b, hq], Lg[b, hq], o, l, what=(u, h))


def test_rejected_recall_leaves_pool_and_tables_unchanged():
    """A recall the host rejects (a slot outside the pool) enqueues nothing: the caller never
    commits, and the pool and tables still describe the old residency."""
    B_, Hkv, P, D, nb = 1, 1, 32, 128, 4
    Kp = torch.zeros((2, P, D), dtype=torch.bfloat16, device="cuda")
    Vp = torch.zeros_like(Kp)
    hostK = torch.ones((B_, Hkv, nb, P, D), dtype=torch.bfloat16).pin_memory()
    hostV = torch.ones_like(hostK).pin_memory()
    side = torch.cuda.Stream()
    with pytest.raises(bs.ScoutError):
        bs.recall_async([(0, 1, 0, -1), (0, 2, 5, -1)], hostK, hostV, Kp, Vp, B_, Hkv, P, nb, side)
    torch.cuda.synchronize()
    assert int(Kp.abs().sum().item()) == 0 and int(Vp.abs().sum().item()) == 0


def test_recall_copy_refused_midway_leaves_tables_and_evictions_recover():
    """A copy the runtime refuses midway (an error code injected in place of cudaMemcpyAsync's):
    the call reports SCOUT_ERR_CUDA, the tables still describe the old residency (nothing is
    committed), and committing the evictions alone, as the header asks, leaves no block whose
    slot may have been overwritten looking resident."""
    st = _setup()
    s, ops = st["s"], st["ops"]
    runs = 1 + sum(1 for a, b in zip(ops, ops[1:]) if not (a[0] == b[0] and b[1] == a[1] + 1 and b[2] == a[2] + 1))
    assert runs >= 2  # the injected refusal hits the second run
    before = _snapshot(st)
    side = torch.cuda.Stream()
    hK, hV = _host_bf16(st["hostK"]), _host_bf16(st["hostV"])
    with pytest.raises(bs.ScoutError, match="SCOUT_ERR_CUDA"):
        bs.recall_async([tuple(int(x) for x in r) for r in ops], hK, hV, st["K_pool"], st["V_pool"], s.B, s.Hkv, s.P,
                        s.nblk, side, inject=bs.INJECT_COPY_FAIL)
    torch.cuda.synchronize()
    assert torch.equal(st["d_table"], before[2]) and torch.equal(st["d_bits"], before[3])
    evict_only = np.array([(u, -1, sl, e) for u, _, sl, e in ops], np.int32)
    bs.commit_residency(to_dev(evict_only), st["d_table"], st["d_bits"], st["n_slots"], s.B, s.Hkv)
    torch.cuda.synchronize()
    U, nb = s.units, s.nblk
    table = st["table"].copy()
    res = st["res"].copy()
    for u, _, _, e in ops:
        table[u, e], res[u, e] = -1, False
    assert np.array_equal(st["d_table"].cpu().numpy().reshape(U, nb), table)
    assert np.array_equal(st["d_bits"].cpu().numpy().view(np.uint32).reshape(U, -1), bits_from_mask(res).reshape(U, -1))


def test_recall_gather_refused_enqueues_nothing():
    """The gather recall is one launch: refused (injected), it leaves the pool and the tables bit for
    bit as they were; the same recall then succeeds."""
    st = _setup()
    s, ops = st["s"], st["ops"]
    before = _snapshot(st)
    side = torch.cuda.Stream()
    hK, hV = _host_bf16(st["hostK"]), _host_bf16(st["hostV"])
    d_ops = to_dev(ops)
    with pytest.raises(bs.ScoutError, match="SCOUT_ERR_CUDA"):
        bs.recall_gather_async(d_ops, hK, hV, st["K_pool"], st["V_pool"], s.B, s.Hkv, s.P, s.nblk, side,
                               inject=bs.INJECT_COPY_FAIL)
    torch.cuda.synchronize()
    for a, b in zip(_snapshot(st), before):
        assert torch.equal(a, b)
    done = torch.cuda.Event()
    bs.recall_gather_async(d_ops, hK, hV, st["K_pool"], st["V_pool"], s.B, s.Hkv, s.P, s.nblk, side, done_event=done)
    bs.commit_residency(d_ops, st["d_table"], st["d_bits"], st["n_slots"], s.B, s.Hkv, wait_event=done)
    torch.cuda.synchronize()
    Kg = st["K_pool"].cpu().view(torch.int16).numpy().view(np.uint16)
    for u, b, sl, _ in st["want"]:
        assert np.array_equal(Kg[sl], st["hostK"][u, b])


def test_recall_gather_needs_mapped_host_memory():
    """Pageable host memory is not pinned and mapped: the gather recall refuses it before any launch,
    whether or not the device could reach it through the host's page tables."""
    B_, Hkv, P, D, nb = 1, 1, 32, 128, 4
    Kp = torch.zeros((2, P, D), dtype=torch.bfloat16, device="cuda")
    hostK = torch.ones((B_, Hkv, nb, P, D), dtype=torch.bfloat16)  # not pinned
    L = bs.lib()
    rc = L.scout_recall_gather_async(to_dev(np.array([[0, 1, 0, -1]], np.int32)).data_ptr(), 1, hostK.data_ptr(),
                                     hostK.data_ptr(), Kp.data_ptr(), Kp.data_ptr(), 2, B_, Hkv, D, P, nb, None, None,
                                     None, torch.cuda.current_stream().cuda_stream, None)
    torch.cuda.synchronize()
    assert rc == 2 and int(Kp.abs().sum().item()) == 0
