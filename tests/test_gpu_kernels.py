"""GPU parity of every libscout kernel against the fp64 oracle, on seeded inputs
small enough for the oracle to finish in seconds but spanning several tiles and
ragged tails (sequence lengths that end inside a block, units with no block)."""
import numpy as np
import pytest
import torch

import oracle as O
import block_sparse_kv_pred_gb300 as bs
from block_sparse_kv_pred_gb300 import workload as W
from block_sparse_kv_pred_gb300.workload import device as WD
from _parity import (bf16_bits, bits_from_mask, check_attention, check_selection, check_topk_property,
                     ensure_built, nvalid, pools_from_units, to_dev, SCORE_REL)

pytestmark = pytest.mark.gpu

SHAPES = {
    "tiny": W.tiny(),
    "ragged_g5_p32": W.Shape("ragged_g5_p32", B=3, Hq=10, Hkv=2, T=5000, P=32, k=8, resident_frac=0.25,
                             seq_lens=(5000, 4097, 33)),
    "mean_p16": W.Shape("mean_p16", B=2, Hq=8, Hkv=2, T=4100, P=16, k=20, resident_frac=0.25, kind="mean",
                        seq_lens=(4100, 2049)),
    "p64_g4": W.Shape("p64_g4", B=2, Hq=16, Hkv=4, T=9000, P=64, k=10, resident_frac=0.5, seq_lens=(9000, 6401)),
    "g1": W.Shape("g1", B=2, Hq=4, Hkv=4, T=640, P=32, k=5, resident_frac=0.5),
    "g8_mean": W.Shape("g8_mean", B=1, Hq=16, Hkv=2, T=2048, P=32, k=12, resident_frac=0.25, kind="mean"),
}
_CACHE = {}


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def get(name):
    if name not in _CACHE:
        wl = W.Workload(SHAPES[name])
        _CACHE[name] = (wl, WD.materialize(wl, with_gemm=False))
    return _CACHE[name]


def kind_id(kind):
    return bs.MINMAX if kind == "minmax" else bs.MEAN


def make_digest(s, d, kind, sentinel=True):
    if kind == "minmax":
        dg = torch.empty((s.B, s.Hkv, s.nblk, 2, s.D), dtype=torch.bfloat16, device="cuda")
    else:
        dg = torch.empty((s.B, s.Hkv, s.nblk, s.D), dtype=torch.float32, device="cuda")
    if sentinel:
        dg.fill_(4096.0)  # exactly representable in bf16 and fp32
    bs.build_digest(kind, d["K_pool"], d["page_table"], d["seq_len"], s.B, s.Hkv, s.P, dg)
    return dg


def unit_q(wl, u):
    s = wl.s
    b, kvh = divmod(u, s.Hkv)
    return wl.q[b, kvh * s.G:(kvh + 1) * s.G]


# ---------------------------------------------------------------------------
def test_device_generator_matches_host():
    wl, d = get("ragged_g5_p32")
    s = wl.s
    for u in (0, s.units - 1):
        slots = torch.as_tensor(wl.page_table[u], device="cuda").long()
        for which, pool in (("K", d["K_pool"]), ("V", d["V_pool"])):
            host = wl.unit_kv(u, which).reshape(s.nblk, s.P, s.D)
            assert np.array_equal(bf16_bits(pool[slots]), host)
    assert np.array_equal(bf16_bits(d["q"]), wl.q)
    t = torch.empty(3000, dtype=torch.bfloat16, device="cuda")
    WD.fill_normal(t, 0, W.STREAM_W, 0.02, offset=777)
    assert np.array_equal(bf16_bits(t), W.normal_bf16(0, W.STREAM_W, (3000,), 0.02, offset=777))


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("kind", ["minmax", "mean"])
def test_digest_parity(name, kind):
    wl, d = get(name)
    s = wl.s
    dg = make_digest(s, d, kind)
    torch.cuda.synchronize()
    host = dg.cpu().view(s.units, s.nblk, -1)
    for u in range(s.units):
        L = int(wl.seq_len[u // s.Hkv])
        nv = nvalid(L, s.P)
        K = wl.unit_kv(u)
        if kind == "minmax":
            mn, mx = O.digest_minmax(K, L, s.P)
            got = bf16_bits(host[u, :nv]).reshape(nv, 2, s.D)
            assert np.array_equal(got[:, 0], O.f64_to_bf16(mn)) and np.array_equal(got[:, 1], O.f64_to_bf16(mx))
        else:
            ref = O.digest_mean(K, L, s.P)
            got = host[u, :nv].double().numpy()
            scale = np.abs(O.bf16_to_f64(K[:L])).mean()
            assert np.all(np.abs(got - ref) <= 1e-6 * np.abs(ref) + 1e-6 * scale)
        # blocks past the sequence are left untouched
        if nv < s.nblk:
            assert torch.all(host[u, nv:].float() == 4096.0)


def test_digest_block_list_rebuilds_only_listed_blocks():
    wl, d = get("tiny")
    s = wl.s
    dg = torch.full((s.B, s.Hkv, s.nblk, 2, s.D), 7.0, dtype=torch.bfloat16, device="cuda")
    pairs = np.array([[0, 5], [1, 127], [1, 0]], dtype=np.int32)
    bs.build_digest("minmax", d["K_pool"], d["page_table"], d["seq_len"], s.B, s.Hkv, s.P, dg,
                    block_list=to_dev(pairs))
    host = dg.cpu().view(s.units, s.nblk, 2, s.D)
    listed = {(int(u), int(j)) for u, j in pairs}
    for u in range(s.units):
        mn, mx = O.digest_minmax(wl.unit_kv(u), s.T, s.P)
        for j in range(s.nblk):
            if (u, j) in listed:
                assert np.array_equal(bf16_bits(host[u, j, 0]), O.f64_to_bf16(mn[j]))
                assert np.array_equal(bf16_bits(host[u, j, 1]), O.f64_to_bf16(mx[j]))
            else:
                assert torch.all(host[u, j].float() == 7.0)


def prev_lists(s, rng):
    """Seeded previous-step CPU lists (ascending, -1 padded) for the delta output."""
    pl = np.full((s.units, s.k), -1, dtype=np.int32)
    pc = np.zeros(s.units, dtype=np.int32)
    for u in range(s.units):
        nv = nvalid(s.lens()[u // s.Hkv], s.P)
        n = int(rng.integers(0, min(s.k, nv) + 1))
        sel = np.sort(rng.choice(nv, size=n, replace=False))
        pl[u, :n] = sel
        pc[u] = n
    return pl, pc


@pytest.mark.parametrize("name", list(SHAPES))
def test_score_topk_parity(name):
    wl, d = get(name)
    s = wl.s
    kind = s.kind
    dg = make_digest(s, d, kind)
    ws = bs.score_topk_workspace(s.B, s.Hkv, s.nblk)
    scores = torch.empty((s.B, s.Hkv, s.nblk), dtype=torch.float32, device="cuda")
    pl, pc = prev_lists(s, np.random.default_rng(5))
    prev = (to_dev(pl.reshape(s.B, s.Hkv, s.k)), to_dev(pc.reshape(s.B, s.Hkv)))
    res = None
    for rep in range(2):  # the second call checks that the workspace counters reset
        out = bs.score_topk(kind, d["q"], dg, d["seq_len"], d["resident_bits"], s.B, s.Hq, s.Hkv, s.P, s.nblk,
                            s.k, ws, prev_cpu=prev, scores=scores)
        torch.cuda.synchronize()
        cur = {kk: v.cpu().numpy().reshape(s.units, -1) for kk, v in out.items()}
        if res is not None:
            for kk in cur:
                assert np.array_equal(cur[kk], res[kk]), kk
        res = cur
    assert torch.all(ws[: 4 * s.units] == 0)
    exact = 0
    for u in range(s.units):
        L = int(wl.seq_len[u // s.Hkv])
        nv = nvalid(L, s.P)
        qg = unit_q(wl, u)
        r = O.unit_step(qg, qg, wl.unit_kv(u), wl.unit_kv(u, "V"), L, s.P, s.k, kind, wl.resident[u].astype(bool),
                        s.scale, prev_cpu=pl[u, :pc[u]])
        g = res["scores"][u]
        if nv:
            big = np.abs(r["scores"]).max()
            assert np.all(np.abs(g[:nv] - r["scores"]) <= SCORE_REL * big), u
        assert np.all(np.isneginf(g[nv:]))
        keff = min(s.k, nv)
        S = res["topk"][u][: res["topk_count"][u][0]]
        assert res["topk_count"][u][0] == keff and np.all(res["topk"][u][keff:] == -1)
        check_topk_property(g[:nv], S, s.k, nv, what=(name, u))
        if check_selection(r["scores"], s.k, S, what=(name, u)):
            exact += 1
            for key in ("res", "cpu", "delta"):
                n = res[key + "_count"][u][0]
                assert n == len(r[key]) and list(res[key][u][:n]) == list(r[key]), (key, u)
                assert np.all(res[key][u][n:] == -1)
        else:  # near-tie: the GPU lists must still split its own selection, and the delta follow
            Rm = wl.resident[u].astype(bool)
            rr = list(res["res"][u][: res["res_count"][u][0]])
            cc = list(res["cpu"][u][: res["cpu_count"][u][0]])
            assert sorted(rr + cc) == list(S) and rr == sorted(rr) and cc == sorted(cc)
            assert all(Rm[j] for j in rr) and not any(Rm[j] for j in cc)
            dd = list(res["delta"][u][: res["delta_count"][u][0]])
            assert dd == [int(j) for j in O.delta_list(cc, pl[u, :pc[u]])], u
            for key in ("res", "cpu", "delta"):
                assert np.all(res[key][u][res[key + "_count"][u][0]:] == -1), (key, u)
    assert exact >= s.units - 1


def _integer_case(kind, seed=0, k_range=(-3, 4), q_range=(-2, 3), nblk=301, k=37):
    """Small-integer K and q: every fp32 score is exact, so GPU and fp64 scores agree bit for bit and
    the many ties exercise the lowest-index rule."""
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, P, T = 2, 10, 2, 32, (nblk - 1) * 32 + 8
    G, D = Hq // Hkv, 128
    nb = -(-T // P)
    seq = np.array([T, 130 * 32 + 1], dtype=np.int32)
    Ku = W.f32_to_bf16(rng.integers(*k_range, size=(B * Hkv, nb * P, D)).astype(np.float32))
    Vu = W.f32_to_bf16(rng.standard_normal((B * Hkv, nb * P, D)).astype(np.float32))
    q = W.f32_to_bf16(rng.integers(*q_range, size=(B, Hq, D)).astype(np.float32))
    Kp, Vp, table = pools_from_units(Ku, Vu, P, rng)
    resident = rng.random((B * Hkv, nb)) < 0.3
    dev = dict(K_pool=to_dev(Kp), V_pool=to_dev(Vp), page_table=to_dev(table.reshape(B, Hkv, nb)),
               seq_len=to_dev(seq), q=to_dev(q), resident_bits=to_dev(bits_from_mask(resident).reshape(B, Hkv, -1)))
    return dict(B=B, Hq=Hq, Hkv=Hkv, G=G, P=P, T=T, k=k, nb=nb, seq=seq, Ku=Ku, Vu=Vu, q=q, resident=resident,
                dev=dev)


def _check_integer_case(c, kind, max_ctas=None, min_ties=0):
    B, Hkv, nb, k, P = c["B"], c["Hkv"], c["nb"], c["k"], c["P"]
    d = c["dev"]
    dg = (torch.empty((B, Hkv, nb, 2, 128), dtype=torch.bfloat16, device="cuda") if kind == "minmax"
          else torch.empty((B, Hkv, nb, 128), dtype=torch.float32, device="cuda"))
    bs.build_digest(kind, d["K_pool"], d["page_table"], d["seq_len"], B, Hkv, P, dg)
    ws = bs.score_topk_workspace(B, Hkv, nb)
    scores = torch.empty((B, Hkv, nb), dtype=torch.float32, device="cuda")
    out = bs.score_topk(kind, d["q"], dg, d["seq_len"], d["resident_bits"], B, c["Hq"], Hkv, P, nb, k, ws,
                        scores=scores, max_ctas=max_ctas)
    torch.cuda.synchronize()
    res = {kk: v.cpu().numpy().reshape(B * Hkv, -1) for kk, v in out.items()}
    ties = 0
    for u in range(B * Hkv):
        b, kvh = divmod(u, Hkv)
        L = int(c["seq"][b])
        qg = c["q"][b, kvh * c["G"]:(kvh + 1) * c["G"]]
        r = O.unit_step(qg, qg, c["Ku"][u], c["Vu"][u], L, P, k, kind, c["resident"][u], 0.1)
        nv = nvalid(L, P)
        assert np.array_equal(res["scores"][u][:nv].astype(np.float64), r["scores"])
        ties += len(r["scores"]) - len(np.unique(r["scores"]))
        for key in ("topk", "res", "cpu", "delta"):
            n = res[key + "_count"][u][0]
            assert n == len(r[key]) and list(res[key][u][:n]) == list(r[key]), (key, u, max_ctas)
            assert np.all(res[key][u][n:] == -1)
    assert ties > min_ties


@pytest.mark.parametrize("max_ctas", [None, 1, 2, 3])
@pytest.mark.parametrize("kind", ["minmax", "mean"])
def test_score_topk_bit_exact_on_exact_scores(kind, max_ctas):
    """Whole units are dealt to the CTAs from a ticket counter: one CTA per unit (uncapped) and
    grids of 1 to 3 CTAs that each take many units give the oracle's lists."""
    _check_integer_case(_integer_case(kind), kind, max_ctas, min_ties=100)


@pytest.mark.parametrize("max_ctas", [None, 1, 2])
@pytest.mark.parametrize("k_range", [(0, 1), (0, 2)])
def test_score_topk_ties_beyond_the_candidate_limit(k_range, max_ctas):
    """K = 0 everywhere (every score equal) or K in {0, 1} (almost every block maximal): far more
    than 64 candidates share the k-th key, and the lowest-index ones are taken."""
    c = _integer_case("minmax", seed=3, k_range=k_range, q_range=(1, 2))
    _check_integer_case(c, "minmax", max_ctas, min_ties=200)


@pytest.mark.parametrize("kind,k_range,k", [("minmax", (-3, 4), 37), ("mean", (-3, 4), 200), ("minmax", (0, 2), 64)])
def test_score_topk_bit_exact_over_several_key_groups(kind, k_range, k):
    """2,101 blocks per unit: the selection takes the keys 1,024 at a time (three groups, the last
    ragged) in every counting round; tie-heavy integer scores keep the lists bit-exact."""
    c = _integer_case(kind, seed=7, k_range=k_range, q_range=(1, 2) if k_range == (0, 2) else (-2, 3),
                      nblk=2101, k=k)
    _check_integer_case(c, kind, None, min_ties=500)


def _attn_lists(s, rng, force_split=False):
    """Seeded resident lists chosen by the test: empty, single-block, full-k and random units."""
    lists = np.full((s.units, s.k), -1, dtype=np.int32)
    counts = np.zeros(s.units, dtype=np.int32)
    for u in range(s.units):
        nv = nvalid(s.lens()[u // s.Hkv], s.P)
        choice = u % 4 if not force_split else 2
        n = [0, 1, min(s.k, nv), int(rng.integers(0, min(s.k, nv) + 1))][choice]
        n = min(n, nv)
        sel = rng.choice(nv, size=n, replace=False)
        if n and nv > 1 and u % 3 == 0:
            sel[0] = nv - 1  # include the (possibly partial) tail block
            sel = np.unique(sel)
            n = len(sel)
        lists[u, :n] = np.sort(sel)
        counts[u] = n
    return lists, counts


@pytest.mark.parametrize("name", list(SHAPES))
def test_sparse_attn_parity(name):
    wl, d = get(name)
    s = wl.s
    rng = np.random.default_rng(11)
    lists, counts = _attn_lists(s, rng)
    ws = bs.sparse_attn_workspace(s.B, s.Hq, s.Hkv, s.P)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for rep in range(2):
        Og, Lg = bs.sparse_attn(d["q"], d["K_pool"], d["V_pool"], d["page_table"], d["seq_len"],
                                to_dev(lists.reshape(s.B, s.Hkv, s.k)), to_dev(counts.reshape(s.B, s.Hkv)), s.B, s.Hq,
                                s.Hkv, s.P, s.k, s.scale, ws, status=status)
        torch.cuda.synchronize()
    assert int(status.item()) == 0 and torch.all(ws[: 4 * s.units] == 0)
    Og, Lg = Og.cpu().numpy(), Lg.cpu().numpy()
    for u in range(s.units):
        b, kvh = divmod(u, s.Hkv)
        L = int(wl.seq_len[b])
        K, V = O.bf16_to_f64(wl.unit_kv(u)), O.bf16_to_f64(wl.unit_kv(u, "V"))
        toks = O.block_tokens(lists[u, :counts[u]], s.P, L)
        for h in range(s.G):
            hq = kvh * s.G + h
            o, l = O.attention_partial(O.bf16_to_f64(wl.q[b, hq]), K[toks], V[toks], s.scale)
            check_attention(Og[b, hq], Lg[b, hq], o, l, what=(name, u, h))


def test_sparse_attn_units_split_over_many_ctas():
    """Few blocks per unit but many units' worth of CTAs: every unit is cut into several CTA ranges."""
    wl, d = get("p64_g4")
    s = wl.s
    lists, counts = _attn_lists(s, np.random.default_rng(3), force_split=True)
    ws = bs.sparse_attn_workspace(s.B, s.Hq, s.Hkv, s.P)
    Og, Lg = bs.sparse_attn(d["q"], d["K_pool"], d["V_pool"], d["page_table"], d["seq_len"],
                            to_dev(lists.reshape(s.B, s.Hkv, s.k)), to_dev(counts.reshape(s.B, s.Hkv)), s.B, s.Hq,
                            s.Hkv, s.P, s.k, s.scale, ws)
    torch.cuda.synchronize()
    Og, Lg = Og.cpu().numpy(), Lg.cpu().numpy()
    for u in range(s.units):
        b, kvh = divmod(u, s.Hkv)
        K, V = O.bf16_to_f64(wl.unit_kv(u)), O.bf16_to_f64(wl.unit_kv(u, "V"))
        toks = O.block_tokens(lists[u, :counts[u]], s.P, int(wl.seq_len[b]))
        for h in range(s.G):
            hq = kvh * s.G + h
            o, l = O.attention_partial(O.bf16_to_f64(wl.q[b, hq]), K[toks], V[toks], s.scale)
            check_attention(Og[b, hq], Lg[b, hq], o, l, what=(u, h))


def test_bad_page_table_entry_is_skipped_and_reported():
    wl, d = get("tiny")
    s = wl.s
    table = d["page_table"].clone()
    table[0, 0, 3] = -1
    table[0, 1, 4] = wl.n_slots + 5
    lists = np.full((s.units, s.k), -1, dtype=np.int32)
    lists[0, :3] = [1, 3, 9]
    lists[1, :2] = [4, 6]
    counts = np.array([3, 2], dtype=np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = bs.sparse_attn_workspace(s.B, s.Hq, s.Hkv, s.P)
    Og, Lg = bs.sparse_attn(d["q"], d["K_pool"], d["V_pool"], table, d["seq_len"],
                            to_dev(lists.reshape(s.B, s.Hkv, s.k)), to_dev(counts.reshape(s.B, s.Hkv)), s.B, s.Hq,
                            s.Hkv, s.P, s.k, s.scale, ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 1
    Og, Lg = Og.cpu().numpy(), Lg.cpu().numpy()
    for u, good in ((0, [1, 9]), (1, [6])):
        K, V = O.bf16_to_f64(wl.unit_kv(u)), O.bf16_to_f64(wl.unit_kv(u, "V"))
        toks = O.block_tokens(good, s.P, s.T)
        for h in range(s.G):
            hq = u * s.G + h
            o, l = O.attention_partial(O.bf16_to_f64(wl.q[0, hq]), K[toks], V[toks], s.scale)
            check_attention(Og[0, hq], Lg[0, hq], o, l)


def test_merge_parity_including_empty_partials():
    rng = np.random.default_rng(21)
    rows = 300
    Oa = rng.standard_normal((rows, 128)).astype(np.float32)
    Ob = rng.standard_normal((rows, 128)).astype(np.float32) * 3
    La = (rng.standard_normal(rows) * 4).astype(np.float32)
    Lb = (rng.standard_normal(rows) * 4).astype(np.float32)
    La[::7] = -np.inf
    Lb[::5] = -np.inf
    Lb[3] = La[3] = 50.0  # equal weights
    Oa[La == -np.inf] = 0
    Ob[Lb == -np.inf] = 0
    Og, Lg = bs.merge(to_dev(Oa), to_dev(La), to_dev(Ob), to_dev(Lb))
    torch.cuda.synchronize()
    Og = Og.float().cpu().numpy()
    Lg = Lg.cpu().numpy()
    for r in range(rows):
        o, l = O.merge(Oa[r].astype(np.float64), float(La[r]), Ob[r].astype(np.float64), float(Lb[r]))
        check_attention(Og[r], Lg[r], o, l, what=r)


@pytest.mark.parametrize("M,N,K", [(1, 1024, 1024), (8, 256, 512), (40, 640, 5120), (130, 384, 192), (256, 256, 128),
                                   (40, 5120, 5120), (8, 4096, 4096)])
def test_predict_q_parity(M, N, K):
    X = W.normal_bf16(1, W.STREAM_X, (M, K))
    Wq = W.normal_bf16(1, W.STREAM_W, (N, K), sigma=0.02)
    Q = bs.predict_q(to_dev(X), to_dev(Wq))
    torch.cuda.synchronize()
    ref = O.predict_q(X, Wq)
    got = O.bf16_to_f64(bf16_bits(Q))
    assert np.linalg.norm(got - ref) <= 1e-2 * np.linalg.norm(ref)
    # stronger than the acceptance bound: each entry within bf16 rounding of the fp32 sum
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-3 * np.abs(ref).max())


@pytest.mark.parametrize("max_ctas", [10, 20, 30, 110])
def test_predict_q_split_k_reduction(max_ctas):
    """M = 130 pads to 144 batch columns (18 groups of 8); 10 W tiles under caps of 10, 20, 30 and
    110 CTAs give split-K clusters of 1, 2, 3 and 8 CTAs, over which the groups are dealt: every
    group is reduced by its owner CTA, whatever the cluster size."""
    X = W.normal_bf16(3, W.STREAM_X, (130, 2048))
    Wq = W.normal_bf16(3, W.STREAM_W, (1280, 2048), sigma=0.02)
    Q = bs.predict_q(to_dev(X), to_dev(Wq), max_ctas=max_ctas)
    torch.cuda.synchronize()
    ref = O.predict_q(X, Wq)
    got = O.bf16_to_f64(bf16_bits(Q))
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-3 * np.abs(ref).max())


@pytest.mark.parametrize("name", ["tiny", "ragged_g5_p32", "mean_p16"])
def test_end_to_end_step_matches_topk_attention(name):
    """digest -> select -> GPU partial -> merge with the CPU partial over B_cpu equals attention over B_pred."""
    wl, d = get(name)
    s = wl.s
    dg = make_digest(s, d, s.kind)
    ws = bs.score_topk_workspace(s.B, s.Hkv, s.nblk)
    out = bs.score_topk(s.kind, d["q"], dg, d["seq_len"], d["resident_bits"], s.B, s.Hq, s.Hkv, s.P, s.nblk, s.k, ws)
    wa = bs.sparse_attn_workspace(s.B, s.Hq, s.Hkv, s.P)
    Og, Lg = bs.sparse_attn(d["q"], d["K_pool"], d["V_pool"], d["page_table"], d["seq_len"], out["res"],
                            out["res_count"], s.B, s.Hq, s.Hkv, s.P, s.k, s.scale, wa)
    torch.cuda.synchronize()
    # CPU partial over the oracle's own B_cpu, computed by the oracle (stands in for the CPU worker)
    Oc = np.zeros((s.B, s.Hq, s.D), np.float32)
    Lc = np.full((s.B, s.Hq), -np.inf, np.float32)
    refs = {}
    for u in range(s.units):
        b, kvh = divmod(u, s.Hkv)
        L = int(wl.seq_len[b])
        qg = unit_q(wl, u)
        r = O.unit_step(qg, qg, wl.unit_kv(u), wl.unit_kv(u, "V"), L, s.P, s.k, s.kind,
                        wl.resident[u].astype(bool), s.scale)
        K, V = O.bf16_to_f64(wl.unit_kv(u)), O.bf16_to_f64(wl.unit_kv(u, "V"))
        tc, ts = O.block_tokens(r["cpu"], s.P, L), O.block_tokens(r["topk"], s.P, L)
        for h in range(s.G):
            hq = kvh * s.G + h
            qh = O.bf16_to_f64(wl.q[b, hq])
            Oc[b, hq], Lc[b, hq] = O.attention_partial(qh, K[tc], V[tc], s.scale)
            refs[(b, hq)] = O.attention_partial(qh, K[ts], V[ts], s.scale)
        got = out["topk"].cpu().numpy().reshape(s.units, -1)[u]
        assert list(got[: len(r["topk"])]) == list(r["topk"]), "selection differs (near-tie): pick another seed"
    Of, Lf = bs.merge(Og, Lg, to_dev(Oc), to_dev(Lc))
    torch.cuda.synchronize()
    Of, Lf = Of.float().cpu().numpy(), Lf.cpu().numpy()
    for (b, hq), (o, l) in refs.items():
        check_attention(Of[b, hq], Lf[b, hq], o, l, what=(b, hq))


def test_dense_edge_case_equals_full_attention():
    """top-k = all blocks and every block resident: the merged output is full softmax attention."""
    s = W.Shape("dense", B=2, Hq=40, Hkv=8, T=8192 - 5, P=32, k=256, resident_frac=1.0)
    wl = W.Workload(s)
    d = WD.materialize(wl, with_gemm=False)
    dg = make_digest(s, d, "minmax")
    ws = bs.score_topk_workspace(s.B, s.Hkv, s.nblk)
    out = bs.score_topk("minmax", d["q"], dg, d["seq_len"], d["resident_bits"], s.B, s.Hq, s.Hkv, s.P, s.nblk, s.k,
                        ws)
    wa = bs.sparse_attn_workspace(s.B, s.Hq, s.Hkv, s.P)
    Og, Lg = bs.sparse_attn(d["q"], d["K_pool"], d["V_pool"], d["page_table"], d["seq_len"], out["res"],
                            out["res_count"], s.B, s.Hq, s.Hkv, s.P, s.k, s.scale, wa)
    empty_O = torch.zeros_like(Og)
    empty_L = torch.full_like(Lg, float("-inf"))
    Of, Lf = bs.merge(Og, Lg, empty_O, empty_L)
    torch.cuda.synchronize()
    assert torch.all(out["res_count"] == s.nblk) and torch.all(out["cpu_count"] == 0)
    Of, Lf = Of.float().cpu().numpy(), Lf.cpu().numpy()
    for u in (0, 5, 13):
        b, kvh = divmod(u, s.Hkv)
        K, V = O.bf16_to_f64(wl.unit_kv(u))[: s.T], O.bf16_to_f64(wl.unit_kv(u, "V"))[: s.T]
        for h in range(s.G):
            hq = kvh * s.G + h
            o, l = O.attention_partial(O.bf16_to_f64(wl.q[b, hq]), K, V, s.scale)
            check_attention(Of[b, hq], Lf[b, hq], o, l, what=(u, h))
