"""Failures made on purpose, without faulting or hanging the GPU: a bounded wait of the
selection kernel that expires (scout_launch.inject = SCOUT_INJECT_ABANDON) must be reported
in the status word, must leave the workspace counter at zero, and must not change what the
next ordinary call on the same workspace computes."""
import numpy as np
import pytest
import torch

import oracle as O
import block_sparse_kv_pred_gb300 as bs
from block_sparse_kv_pred_gb300 import workload as W
from block_sparse_kv_pred_gb300.workload import device as WD
from _parity import check_selection, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _outputs(s, fill):
    o = {}
    for name in ("topk", "res", "cpu", "delta"):
        o[name] = torch.full((s.B, s.Hkv, s.k), fill, dtype=torch.int32, device="cuda")
        o[name + "_count"] = torch.full((s.B, s.Hkv), fill, dtype=torch.int32, device="cuda")
    return o


def test_expired_wait_is_reported_and_the_next_call_is_exact():
    # 64 units over 8 CTAs: every CTA abandons after its first unit, so 56 units are skipped
    s = W.Shape("failure_c2", B=8, Hq=32, Hkv=8, T=16384, P=32, k=64, resident_frac=0.25)
    wl = W.Workload(s)
    d = WD.materialize(wl, with_gemm=False)
    dg = torch.empty((s.B, s.Hkv, s.nblk, 2, s.D), dtype=torch.bfloat16, device="cuda")
    bs.build_digest("minmax", d["K_pool"], d["page_table"], d["seq_len"], s.B, s.Hkv, s.P, dg)
    ws = bs.score_topk_workspace(s.B, s.Hkv, s.nblk)
    args = ("minmax", d["q"], dg, d["seq_len"], d["resident_bits"], s.B, s.Hq, s.Hkv, s.P, s.nblk, s.k, ws)

    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = _outputs(s, -7)
    bs.score_topk(*args, out=bad, status=status, max_ctas=8, inject=bs.INJECT_ABANDON)
    torch.cuda.synchronize()
    assert int(status.item()) & 2, "the expired wait must set SCOUT_DEV_TIMEOUT"
    assert int(ws[:4].view(torch.int32).item()) == 0, "the unit ticket counter must be back at zero"
    # each CTA that got a unit finished that one only: the skipped units kept their stale lists
    untouched = int((bad["topk_count"] == -7).sum().item())
    assert s.units - 8 <= untouched < s.units, untouched

    # the next ordinary call on the same workspace, and one on a fresh workspace, agree bit for bit
    status.zero_()
    got = _outputs(s, -9)
    scores = torch.empty((s.B, s.Hkv, s.nblk), dtype=torch.float32, device="cuda")
    bs.score_topk(*args, out=got, status=status, scores=scores, max_ctas=8)
    ref = _outputs(s, -11)
    bs.score_topk(*args[:-1], bs.score_topk_workspace(s.B, s.Hkv, s.nblk), out=ref, max_ctas=8)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for key in ref:  # the lists and counts (got also holds the scores it was asked for)
        assert torch.equal(got[key], ref[key]), key
    # and the oracle: re-selection from the GPU's fp32 scores is bit-exact, the fp64 scores agree
    sc = scores.cpu().numpy().reshape(s.units, s.nblk)
    topk = got["topk"].cpu().numpy().reshape(s.units, s.k)
    cnt = got["topk_count"].cpu().numpy().reshape(-1)
    for u in (0, 13, s.units - 1):
        b, kvh = divmod(u, s.Hkv)
        L = int(wl.seq_len[b])
        mn, mx = O.digest_minmax(wl.unit_kv(u), L, s.P)
        Uref = O.pool_group(O.scores_minmax(O.bf16_to_f64(wl.q[b, kvh * s.G:(kvh + 1) * s.G]), mn, mx))
        check_selection(Uref, s.k, topk[u, :cnt[u]], what=u)
        nv = -(-L // s.P)
        assert list(topk[u, :cnt[u]]) == list(O.select_topk(sc[u, :nv].astype(np.float64), s.k)), u


def test_inject_value_checked_on_the_host():
    """An injection the selection does not know is refused before any launch."""
    s = W.tiny()
    ws = bs.score_topk_workspace(s.B, s.Hkv, s.nblk)
    q = torch.zeros((s.B, s.Hq, s.D), dtype=torch.bfloat16, device="cuda")
    dg = torch.zeros((s.B, s.Hkv, s.nblk, 2, s.D), dtype=torch.bfloat16, device="cuda")
    seq = torch.full((s.B,), s.T, dtype=torch.int32, device="cuda")
    bits = torch.zeros((s.B, s.Hkv, s.words), dtype=torch.int32, device="cuda")
    with pytest.raises(bs.ScoutError, match="INVALID_ARG"):
        bs.score_topk("minmax", q, dg, seq, bits, s.B, s.Hq, s.Hkv, s.P, s.nblk, s.k, ws, inject=bs.INJECT_COPY_FAIL)
