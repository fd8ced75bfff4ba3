"""The variants of the method's open readings on the GPU, against the oracle's variants:
  * sum pooling of a GQA group's block scores (scout_score_topk with SCOUT_POOL_SUM);
  * the GPU attending every resident block rather than the selected ones among them
    (scout_resident_list feeding scout_sparse_attn), whose merge with the CPU partial over
    S minus R is attention over R union S."""
import numpy as np
import pytest
import torch

import oracle as O
import block_sparse_kv_pred_gb300 as bs
from block_sparse_kv_pred_gb300 import workload as W
from block_sparse_kv_pred_gb300.workload import device as WD
from _parity import SCORE_REL, check_attention, check_selection, check_topk_property, ensure_built, nvalid, to_dev

pytestmark = pytest.mark.gpu

SHAPES = {
    "ragged_g5_p32": W.Shape("v_ragged_g5_p32", B=3, Hq=10, Hkv=2, T=5000, P=32, k=8, resident_frac=0.25,
                             seq_lens=(5000, 4097, 33)),
    "mean_g8_p16": W.Shape("v_mean_g8_p16", B=2, Hq=16, Hkv=2, T=4100, P=16, k=20, resident_frac=0.25, kind="mean",
                           seq_lens=(4100, 2049)),
    "g3_p64": W.Shape("v_g3_p64", B=2, Hq=6, Hkv=2, T=9000, P=64, k=10, resident_frac=0.5, seq_lens=(9000, 6401)),
    "qwen3_8b": W.qwen3_8b(),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _digest(s, d):
    if s.kind == "minmax":
        dg = torch.empty((s.B, s.Hkv, s.nblk, 2, s.D), dtype=torch.bfloat16, device="cuda")
    else:
        dg = torch.empty((s.B, s.Hkv, s.nblk, s.D), dtype=torch.float32, device="cuda")
    bs.build_digest(s.kind, d["K_pool"], d["page_table"], d["seq_len"], s.B, s.Hkv, s.P, dg)
    return dg


def _units(s):
    return range(s.units) if s.units <= 16 else sorted({0, 1, s.units // 2, s.units - 1})


@pytest.mark.parametrize("name", list(SHAPES))
def test_sum_pooled_selection(name):
    s = SHAPES[name]
    wl = W.Workload(s)
    d = WD.materialize(wl, with_gemm=False)
    dg = _digest(s, d)
    ws = bs.score_topk_workspace(s.B, s.Hkv, s.nblk)
    scores = torch.empty((s.B, s.Hkv, s.nblk), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = bs.score_topk(s.kind, d["q"], dg, d["seq_len"], d["resident_bits"], s.B, s.Hq, s.Hkv, s.P, s.nblk, s.k, ws,
                        scores=scores, status=status, pool="sum")
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    g = scores.cpu().numpy().reshape(s.units, -1)
    res = {n: out[n].cpu().numpy().reshape(s.units, -1) for n in out if n != "scores"}
    for u in _units(s):
        b, kvh = divmod(u, s.Hkv)
        L = int(wl.seq_len[b])
        nv = nvalid(L, s.P)
        r = O.unit_step(wl.q[b, kvh * s.G:(kvh + 1) * s.G], wl.q[b, kvh * s.G:(kvh + 1) * s.G], wl.unit_kv(u),
                        wl.unit_kv(u, "V"), L, s.P, s.k, s.kind, wl.resident[u].astype(bool), s.scale, pool="sum")
        if nv:  # the scores within the score bar of the oracle's sums
            big = np.abs(r["scores"]).max()
            assert np.all(np.abs(g[u, :nv] - r["scores"]) <= SCORE_REL * big), u
        assert np.all(np.isneginf(g[u, nv:]))
        S = res["topk"][u][: res["topk_count"][u][0]]
        check_topk_property(g[u, :nv], S, s.k, nv, what=u)  # exact against the GPU's own sums
        assert list(S) == list(O.select_topk(g[u, :nv].astype(np.float64), s.k)), u
        check_selection(r["scores"], s.k, S, what=u)  # and the fp64 selection, up to near-ties
        rr, cc = O.split_residency(S, wl.resident[u].astype(bool))
        assert list(res["res"][u][: res["res_count"][u][0]]) == list(rr)
        assert list(res["cpu"][u][: res["cpu_count"][u][0]]) == list(cc)


@pytest.mark.parametrize("name", ["ragged_g5_p32", "mean_g8_p16", "g3_p64"])
@pytest.mark.parametrize("pool", ["max", "sum"])
def test_gpu_attends_every_resident_block(name, pool):
    s = SHAPES[name]
    wl = W.Workload(s)
    d = WD.materialize(wl, with_gemm=False)
    dg = _digest(s, d)
    ws = bs.score_topk_workspace(s.B, s.Hkv, s.nblk)
    out = bs.score_topk(s.kind, d["q"], dg, d["seq_len"], d["resident_bits"], s.B, s.Hq, s.Hkv, s.P, s.nblk, s.k, ws,
                        pool=pool)
    cap = s.nblk
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lst, cnt = bs.resident_list(d["resident_bits"], d["seq_len"], s.B, s.Hkv, s.P, s.nblk, cap, status=status)
    # the CPU partial over S minus R, from the oracle (the CPU side's output), merged in the epilogue
    o_cpu = np.zeros((s.B, s.Hq, s.D), np.float32)
    l_cpu = np.full((s.B, s.Hq), -np.inf, np.float32)
    torch.cuda.synchronize()
    topk = out["topk"].cpu().numpy().reshape(s.units, -1)
    tc = out["topk_count"].cpu().numpy().reshape(-1)
    cpu = out["cpu"].cpu().numpy().reshape(s.units, -1)
    cc = out["cpu_count"].cpu().numpy().reshape(-1)
    refs = {}
    for u in range(s.units):
        b, kvh = divmod(u, s.Hkv)
        L = int(wl.seq_len[b])
        qg = wl.q[b, kvh * s.G:(kvh + 1) * s.G]
        r = O.unit_step(qg, qg, wl.unit_kv(u), wl.unit_kv(u, "V"), L, s.P, s.k, s.kind, wl.resident[u].astype(bool),
                        s.scale, pool=pool, gpu_blocks="resident")
        refs[u] = r
        K, V = O.bf16_to_f64(wl.unit_kv(u)), O.bf16_to_f64(wl.unit_kv(u, "V"))
        toks = O.block_tokens(cpu[u, :cc[u]], s.P, L)
        for h in range(s.G):
            o, l = O.attention_partial(O.bf16_to_f64(qg[h]), K[toks], V[toks], s.scale)
            o_cpu[b, kvh * s.G + h], l_cpu[b, kvh * s.G + h] = o, l
    wa = bs.sparse_attn_workspace(s.B, s.Hq, s.Hkv, s.P)
    Og, Lg = bs.sparse_attn(d["q"], d["K_pool"], d["V_pool"], d["page_table"], d["seq_len"], lst, cnt, s.B, s.Hq,
                            s.Hkv, s.P, cap, s.scale, wa, status=status)
    Om, Lm = bs.sparse_attn_merge(d["q"], d["K_pool"], d["V_pool"], d["page_table"], d["seq_len"], lst, cnt, s.B,
                                  s.Hq, s.Hkv, s.P, cap, s.scale, wa, to_dev(o_cpu), to_dev(l_cpu), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    lst, cnt = lst.cpu().numpy().reshape(s.units, -1), cnt.cpu().numpy().reshape(-1)
    Og, Lg, Om, Lm = Og.cpu().numpy(), Lg.cpu().numpy(), Om.float().cpu().numpy(), Lm.cpu().numpy()
    for u in range(s.units):
        b, kvh = divmod(u, s.Hkv)
        r = refs[u]
        assert list(lst[u, :cnt[u]]) == list(r["gpu"]) and np.all(lst[u, cnt[u]:] == -1), u  # bit-exact list
        if not check_selection(r["scores"], s.k, topk[u, :tc[u]], what=u):
            continue  # a near-tie: the CPU list differs from the oracle's, so does the merge
        L = int(wl.seq_len[b])
        K, V = O.bf16_to_f64(wl.unit_kv(u)), O.bf16_to_f64(wl.unit_kv(u, "V"))
        union = O.block_tokens(sorted(set(r["gpu"].tolist()) | set(int(j) for j in r["topk"])), s.P, L)
        for h in range(s.G):
            hq = kvh * s.G + h
            check_attention(Og[b, hq], Lg[b, hq], r["O"][h], r["L"][h], what=(u, h))
            # the merged output is attention over R union S
            o, l = O.attention_partial(O.bf16_to_f64(wl.q[b, hq]), K[union], V[union], s.scale)
            check_attention(Om[b, hq], Lm[b, hq], o, l, what=(u, h, "merged"))


def test_resident_list_caps_and_reports_overflow():
    s = SHAPES["g3_p64"]
    wl = W.Workload(s)
    bits = to_dev(wl.resident_bits().view(np.int32))
    seq = to_dev(wl.seq_len.astype(np.int32))
    full = [np.flatnonzero(wl.resident[u][: nvalid(int(wl.seq_len[u // s.Hkv]), s.P)]) for u in range(s.units)]
    cap = min(len(f) for f in full) - 1
    assert cap >= 1
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lst, cnt = bs.resident_list(bits, seq, s.B, s.Hkv, s.P, s.nblk, cap, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 4  # SCOUT_DEV_OVERFLOW
    lst, cnt = lst.cpu().numpy().reshape(s.units, -1), cnt.cpu().numpy().reshape(-1)
    for u in range(s.units):
        assert cnt[u] == cap and list(lst[u]) == list(full[u][:cap])
