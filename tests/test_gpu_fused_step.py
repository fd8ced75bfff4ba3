"""GPU parity of the fused attention + merge entry point, of the launch options
(CTA caps) of the persistent kernels, and of the multi-stream decode step, against
the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import block_sparse_kv_pred_gb300 as bs
from block_sparse_kv_pred_gb300 import workload as W
from block_sparse_kv_pred_gb300.step import setup_step
from block_sparse_kv_pred_gb300.workload import device as WD
from _parity import bf16_bits, check_attention, check_qpred, check_selection, ensure_built, nvalid, oracle_qpred, to_dev

pytestmark = pytest.mark.gpu

SHAPES = {
    "ragged_g5_p32": W.Shape("ragged_g5_p32", B=3, Hq=10, Hkv=2, T=5000, P=32, k=8, resident_frac=0.25,
                             seq_lens=(5000, 4097, 33)),
    "p16_g4": W.Shape("p16_g4", B=2, Hq=16, Hkv=4, T=4100, P=16, k=20, resident_frac=0.5, seq_lens=(4100, 2049)),
    "p64_g8": W.Shape("p64_g8", B=2, Hq=16, Hkv=2, T=9000, P=64, k=10, resident_frac=0.5, seq_lens=(9000, 6401)),
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


def _lists(s, rng):
    """Seeded resident lists: empty, single-block, full and random units."""
    lists = np.full((s.units, s.k), -1, dtype=np.int32)
    counts = np.zeros(s.units, dtype=np.int32)
    for u in range(s.units):
        nv = nvalid(s.lens()[u // s.Hkv], s.P)
        n = min(nv, [0, 1, s.k, int(rng.integers(0, s.k + 1))][u % 4])
        lists[u, :n] = np.sort(rng.choice(nv, size=n, replace=False))
        counts[u] = n
    return lists, counts


def _cpu_partial(s, rng):
    """A CPU partial with empty rows (lse = -inf), equal-weight rows and ordinary rows."""
    Oc = rng.standard_normal((s.B, s.Hq, s.D)).astype(np.float32)
    Lc = (rng.standard_normal((s.B, s.Hq)) * 3).astype(np.float32)
    Lc.reshape(-1)[::3] = -np.inf
    Oc[Lc == -np.inf] = 0
    return Oc, Lc


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("max_ctas", [None, 1, 3, 7])
def test_sparse_attn_merge_parity(name, max_ctas):
    """O = MERGE(A_gpu over the resident list, A_cpu) in one launch, for full and capped grids."""
    wl, d = get(name)
    s = wl.s
    rng = np.random.default_rng(5)
    lists, counts = _lists(s, rng)
    Oc, Lc = _cpu_partial(s, rng)
    ws = bs.sparse_attn_workspace(s.B, s.Hq, s.Hkv, s.P)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):  # the second call checks that the workspace counters were left at zero
        Om, Lm = bs.sparse_attn_merge(d["q"], d["K_pool"], d["V_pool"], d["page_table"], d["seq_len"],
                                      to_dev(lists.reshape(s.B, s.Hkv, s.k)), to_dev(counts.reshape(s.B, s.Hkv)),
                                      s.B, s.Hq, s.Hkv, s.P, s.k, s.scale, ws, to_dev(Oc), to_dev(Lc),
                                      status=status, max_ctas=max_ctas)
        torch.cuda.synchronize()
    assert int(status.item()) == 0 and torch.all(ws[: 4 * s.units] == 0)
    Om, Lm = Om.float().cpu().numpy(), Lm.cpu().numpy()
    for u in range(s.units):
        b, kvh = divmod(u, s.Hkv)
        K, V = O.bf16_to_f64(wl.unit_kv(u)), O.bf16_to_f64(wl.unit_kv(u, "V"))
        toks = O.block_tokens(lists[u, :counts[u]], s.P, int(wl.seq_len[b]))
        for h in range(s.G):
            hq = kvh * s.G + h
            og, lg = O.attention_partial(O.bf16_to_f64(wl.q[b, hq]), K[toks], V[toks], s.scale)
            o, l = O.merge(og, lg, Oc[b, hq].astype(np.float64), float(Lc[b, hq]))
            # bf16 output: its rounding (2^-9 relative) lies well inside the attention tolerance
            check_attention(Om[b, hq], Lm[b, hq], o, l, what=(name, max_ctas, u, h))


@pytest.mark.parametrize("max_ctas", [1, 2, 5])
def test_score_topk_lists_do_not_depend_on_the_cta_cap(max_ctas):
    """Scores and selection are per unit, so any grid gives bit-identical lists."""
    wl, d = get("p16_g4")
    s = wl.s
    dg = torch.empty((s.B, s.Hkv, s.nblk, 2, s.D), dtype=torch.bfloat16, device="cuda")
    bs.build_digest("minmax", d["K_pool"], d["page_table"], d["seq_len"], s.B, s.Hkv, s.P, dg)
    ws = bs.score_topk_workspace(s.B, s.Hkv, s.nblk)
    ref = bs.score_topk("minmax", d["q"], dg, d["seq_len"], d["resident_bits"], s.B, s.Hq, s.Hkv, s.P, s.nblk, s.k,
                        ws)
    got = bs.score_topk("minmax", d["q"], dg, d["seq_len"], d["resident_bits"], s.B, s.Hq, s.Hkv, s.P, s.nblk, s.k,
                        ws, max_ctas=max_ctas)
    torch.cuda.synchronize()
    for key in ("topk", "topk_count", "res", "res_count", "cpu", "cpu_count"):
        assert torch.equal(ref[key], got[key]), key


@pytest.mark.parametrize("max_ctas", [1, 4, 41, 110])
def test_predict_q_with_cta_cap(max_ctas):
    X = W.normal_bf16(1, W.STREAM_X, (40, 5120))
    Wq = W.normal_bf16(1, W.STREAM_W, (1280, 5120), sigma=0.02)
    Q = bs.predict_q(to_dev(X), to_dev(Wq), max_ctas=max_ctas)
    torch.cuda.synchronize()
    ref = O.predict_q(X, Wq)
    got = O.bf16_to_f64(bf16_bits(Q))
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-3 * np.abs(ref).max())


@pytest.mark.parametrize("serial", [False, True])
def test_two_stream_step_matches_oracle(serial):
    """Three steps of the multi-stream step: the lists step i selects with Q_pred are the
    oracle's, and step i+1's output is attention over those resident blocks merged with
    the CPU partial."""
    s = W.Shape("step_g4", B=2, Hq=8, Hkv=2, T=4100, P=32, k=16, resident_frac=0.5, hidden=1024,
                seq_lens=(4100, 3001))
    wl, t, step = setup_step(s, torch.device("cuda", 0), serial=serial, split=(3, 2))
    ev = torch.cuda.Event()
    ev.record()
    step.begin(ev)
    for _ in range(3):
        step.issue()
    step.end(None)
    torch.cuda.synchronize()
    assert int(t["status"].item()) == 0
    last = (step.i - 1) % 2  # set written by the last step; the last attention read the other set
    assert np.array_equal(bf16_bits(t["Qp0"]), bf16_bits(t["Qp1"]))  # same X and W_Q every step
    qp_ref = oracle_qpred(s)  # the oracle's own Q_pred, which the GPU's must match first
    check_qpred(bf16_bits(t["Qp0"]), qp_ref)
    qp_bits = O.f64_to_bf16(qp_ref)  # rounded as the step stores it
    lists = {par: (t[f"topk{par}"].cpu().numpy().reshape(s.units, -1),
                   t[f"res{par}"].cpu().numpy().reshape(s.units, -1),
                   t[f"res_count{par}"].cpu().numpy().reshape(-1)) for par in (0, 1)}
    Of, Lf = t[f"O{last}"].float().cpu().numpy(), t[f"lse{last}"].cpu().numpy()
    o_cpu, l_cpu = wl.cpu_partial()
    for u in range(s.units):
        b, kvh = divmod(u, s.Hkv)
        L = int(wl.seq_len[b])
        qg = qp_bits[b, kvh * s.G * s.D:(kvh + 1) * s.G * s.D].reshape(s.G, s.D)
        r = O.unit_step(qg, wl.q[b, kvh * s.G:(kvh + 1) * s.G], wl.unit_kv(u), wl.unit_kv(u, "V"), L, s.P, s.k,
                        "minmax", wl.resident[u].astype(bool), s.scale)
        exact = True
        for par in (0, 1):  # both sets hold the same selection (same Q_pred and digests)
            topk, res, rc = lists[par]
            exact &= check_selection(r["scores"], s.k, topk[u][: len(r["topk"])], what=(serial, u))
            if exact:
                assert list(topk[u][: len(r["topk"])]) == list(r["topk"])
                assert list(res[u][: rc[u]]) == list(r["res"])
        if not exact:
            continue  # a near-tie: the resident part differs from the oracle's, so does the output
        assert lists[1 - last][2][u] == len(r["res"])
        for h in range(s.G):
            hq = kvh * s.G + h
            o, l = O.merge(r["O"][h], r["L"][h], o_cpu[b, hq].astype(np.float64), float(l_cpu[b, hq]))
            check_attention(Of[b, hq], Lf[b, hq], o, l, what=(serial, u, h))


def test_stale_nan_rows_past_the_sequence_end_do_not_leak():
    """Rows of a sequence's last page past its end may hold anything (a reused page, fresh
    memory): fill them with NaN and infinities; the output must still equal the oracle's."""
    wl, d = get("ragged_g5_p32")
    s = wl.s
    Kp, Vp = d["K_pool"].clone(), d["V_pool"].clone()
    table = d["page_table"].cpu().numpy().reshape(s.units, -1)
    lists = np.full((s.units, s.k), -1, np.int32)
    counts = np.zeros(s.units, np.int32)
    for u in range(s.units):
        L = int(wl.seq_len[u // s.Hkv])
        j, v = (L - 1) // s.P, L % s.P
        if v:
            slot = int(table[u, j])
            Kp.view(torch.int16)[slot, v:] = 0x7FC0  # NaN
            Vp.view(torch.int16)[slot, v:] = 0x7F80  # +inf
        nv = -(-L // s.P)
        sel = sorted(set([nv - 1] + list(range(min(s.k - 1, nv - 1)))))
        lists[u, :len(sel)] = sel
        counts[u] = len(sel)
    ws = bs.sparse_attn_workspace(s.B, s.Hq, s.Hkv, s.P)
    Og, Lg = bs.sparse_attn(d["q"], Kp, Vp, d["page_table"], d["seq_len"], to_dev(lists.reshape(s.B, s.Hkv, s.k)),
                            to_dev(counts.reshape(s.B, s.Hkv)), s.B, s.Hq, s.Hkv, s.P, s.k, s.scale, ws)
    torch.cuda.synchronize()
    Og, Lg = Og.cpu().numpy(), Lg.cpu().numpy()
    assert np.all(np.isfinite(Og)) and np.all(np.isfinite(Lg))
    for u in range(s.units):
        b, kvh = divmod(u, s.Hkv)
        K, V = O.bf16_to_f64(wl.unit_kv(u)), O.bf16_to_f64(wl.unit_kv(u, "V"))
        toks = O.block_tokens(lists[u, :counts[u]], s.P, int(wl.seq_len[b]))
        for h in range(s.G):
            hq = kvh * s.G + h
            o, l = O.attention_partial(O.bf16_to_f64(wl.q[b, hq]), K[toks], V[toks], s.scale)
            check_attention(Og[b, hq], Lg[b, hq], o, l, what=(u, h))


def test_maximum_unit_count_selection_and_merged_attention():
    """B * Hkv = 4,096 units, the most one attention launch takes: its unit prefix (16 KB of shared
    memory) leaves no room for the six-warp ring's combine state at G = 5, so the launch takes four
    consumer warps with the whole ring.  Ragged lengths; the selection over every unit and the
    merged attention over its resident lists are checked against the oracle on sampled units."""
    B = 512
    s = W.Shape("max_units", B=B, Hq=40, Hkv=8, T=320, P=32, k=4, resident_frac=0.5,
                seq_lens=tuple(320 - (7 * b) % 250 for b in range(B)))
    assert s.units == 4096
    wl = W.Workload(s)
    d = WD.materialize(wl, with_gemm=False)
    dg = torch.empty((s.B, s.Hkv, s.nblk, 2, s.D), dtype=torch.bfloat16, device="cuda")
    bs.build_digest("minmax", d["K_pool"], d["page_table"], d["seq_len"], s.B, s.Hkv, s.P, dg)
    out = bs.score_topk("minmax", d["q"], dg, d["seq_len"], d["resident_bits"], s.B, s.Hq, s.Hkv, s.P, s.nblk,
                        s.k, bs.score_topk_workspace(s.B, s.Hkv, s.nblk))
    Oc, Lc = _cpu_partial(s, np.random.default_rng(11))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Om, Lm = bs.sparse_attn_merge(d["q"], d["K_pool"], d["V_pool"], d["page_table"], d["seq_len"], out["res"],
                                  out["res_count"], s.B, s.Hq, s.Hkv, s.P, s.k, s.scale,
                                  bs.sparse_attn_workspace(s.B, s.Hq, s.Hkv, s.P), to_dev(Oc), to_dev(Lc),
                                  status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    Om, Lm = Om.float().cpu().numpy(), Lm.cpu().numpy()
    lists = {n: out[n].cpu().numpy().reshape(s.units, -1) for n in ("topk", "res", "res_count", "topk_count")}
    exact = 0
    sample = sorted(set(range(0, s.units, 61)) | {1, s.units - 1})
    for u in sample:
        b, kvh = divmod(u, s.Hkv)
        qg = wl.q[b, kvh * s.G:(kvh + 1) * s.G]
        r = O.unit_step(qg, qg, wl.unit_kv(u), wl.unit_kv(u, "V"), int(wl.seq_len[b]), s.P, s.k, "minmax",
                        wl.resident[u].astype(bool), s.scale)
        if not check_selection(r["scores"], s.k, lists["topk"][u][: lists["topk_count"][u][0]], what=u):
            continue  # a near-tie: the resident part differs from the oracle's, so does the output
        exact += 1
        assert list(lists["res"][u][: lists["res_count"][u][0]]) == list(r["res"]), u
        for h in range(s.G):
            hq = kvh * s.G + h
            o, l = O.merge(r["O"][h], r["L"][h], Oc[b, hq].astype(np.float64), float(Lc[b, hq]))
            check_attention(Om[b, hq], Lm[b, hq], o, l, what=(u, h))
    assert exact >= len(sample) - 2
