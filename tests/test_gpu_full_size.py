"""Full-size workloads on sampled units: the Qwen3-14B-shaped layer in the launch
configuration bench.py times (four streams, capped grids), the Qwen3-8B-shaped layer,
and the stress shapes (page 16/32/64, budgets 512/2048/8192, min/max and mean digests,
128K context, plus the dense edge case), each checked against the fp64 oracle on a
handful of (sequence, KV head) units the oracle finishes in seconds."""
import functools

import numpy as np
import pytest
import torch

import oracle as O
import block_sparse_kv_pred_gb300 as bs
from block_sparse_kv_pred_gb300 import workload as W
from block_sparse_kv_pred_gb300.step import EARLY_OF, SPLIT, setup_step
from block_sparse_kv_pred_gb300.workload import device as WD
from _parity import bf16_bits, check_attention, check_qpred, check_selection, ensure_built, oracle_qpred

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _sample(U, extra=0):
    """Units checked against the oracle: the ends and thirds, plus `extra` seeded others."""
    base = {0, 1, U // 3, U // 2, U - 1}
    if extra:
        base |= set(int(x) for x in np.random.default_rng(U).choice(U, size=min(extra, U), replace=False))
    return sorted(base)


def _check_all_lists(s, wl, topk, tc, res, rc, cpu, cc):
    """Every unit's lists, without the oracle: k_eff entries of top-k, each list ascending and
    padded with -1, and res / cpu the resident / non-resident parts of top-k."""
    nvalid = -(-wl.seq_len.astype(np.int64) // s.P)
    for u in range(s.units):
        keff = min(s.k, int(nvalid[u // s.Hkv]))
        S, R, C = topk[u, :tc[u]], res[u, :rc[u]], cpu[u, :cc[u]]
        assert tc[u] == keff and rc[u] + cc[u] == keff, u
        for lst, n in ((topk[u], tc[u]), (res[u], rc[u]), (cpu[u], cc[u])):
            assert np.all(np.diff(lst[:n]) > 0) and np.all(lst[n:] == -1), u
        mask = wl.resident[u].astype(bool)
        assert list(R) == [j for j in S if mask[j]] and list(C) == [j for j in S if not mask[j]], u


@functools.lru_cache(maxsize=None)
def _oracle_q(cfg):
    """The oracle's Q_pred of a config's layer (fp64), computed once per module."""
    return oracle_qpred(W.CONFIGS[cfg]())


def _check_unit(wl, u, q_sel_bits, kind, topk, tc, res, rc, cpu, cc, O_out, L_out, o_cpu, l_cpu):
    """Selection of unit u against the oracle's (with the oracle's own selection query), then,
    when the sets agree, the output (merged with the CPU partial) against the oracle's attention
    over its resident list; at a near-tie only the split of the GPU's own set is checked."""
    s = wl.s
    b, kvh = divmod(u, s.Hkv)
    L = int(wl.seq_len[b])
    Kb = wl.unit_kv(u)
    qs = O.bf16_to_f64(q_sel_bits)
    if kind == "minmax":
        mn, mx = O.digest_minmax(Kb, L, s.P)
        Uref = O.pool_group(O.scores_minmax(qs, mn, mx))
    else:
        Uref = O.pool_group(O.scores_mean(qs, O.digest_mean(Kb, L, s.P)))
    S_gpu = topk[u, :tc[u]]
    assert all(t == -1 for t in topk[u, tc[u]:]) and all(t == -1 for t in res[u, rc[u]:])
    if not check_selection(Uref, s.k, S_gpu, what=u):  # a near-tie: the split of the GPU's own set is exact
        r_gpu, _ = O.split_residency(S_gpu, wl.resident[u].astype(bool))
        assert list(res[u, :rc[u]]) == list(r_gpu), u
        return
    r_ref, c_ref = O.split_residency(O.select_topk(Uref, s.k), wl.resident[u].astype(bool))
    assert list(res[u, :rc[u]]) == list(r_ref) and list(cpu[u, :cc[u]]) == list(c_ref), u
    K, V = O.bf16_to_f64(Kb), O.bf16_to_f64(wl.unit_kv(u, "V"))
    toks = O.block_tokens(r_ref, s.P, L)
    for h in range(s.G):
        hq = kvh * s.G + h
        og, lg = O.attention_partial(O.bf16_to_f64(wl.q[b, hq]), K[toks], V[toks], s.scale)
        o, l = O.merge(og, lg, o_cpu[b, hq].astype(np.float64), float(l_cpu[b, hq]))
        check_attention(O_out[b, hq], L_out[b, hq], o, l, what=(u, h))


@pytest.mark.parametrize("cfg,mode,early", [("qwen3_14b", "streams", ()), ("qwen3_14b", "graph", ()),
                                            ("qwen3_14b", "streams", tuple(EARLY_OF)),
                                            ("qwen3_14b", "graph", tuple(EARLY_OF)), ("qwen3_8b", "serial", ())])
def test_full_size_step_sampled(cfg, mode, early):
    """Three steps of the decode step at full size (or, as bench.py times it, a captured CUDA
    graph of two steps replayed twice), with and without early starts; selection with Q_pred,
    attention with q.  Every unit's lists are checked for consistency; sampled units (32 in the
    configuration bench.py times) against the oracle."""
    shape = W.CONFIGS[cfg]()
    wl, t, step = setup_step(shape, torch.device("cuda", 0), serial=(mode == "serial"), split=SPLIT, early=early)
    if mode == "graph":
        g = step.capture(2, torch.device("cuda", 0))
        for _ in range(2):
            g.replay()
    else:
        ev = torch.cuda.Event()
        ev.record()
        step.begin(ev)
        for _ in range(3):
            step.issue()
        step.end(None)
    torch.cuda.synchronize()
    assert int(t["status"].item()) == 0
    s = shape
    par = 1 - (step.i - 1) % 2  # the list set the last attention read
    grab = lambda n: t[f"{n}{par}"].cpu().numpy().reshape(s.units, -1)  # noqa: E731
    topk, res, cpu = grab("topk"), grab("res"), grab("cpu")
    tc, rc, cc = (t[f"{n}_count{par}"].cpu().numpy().reshape(-1) for n in ("topk", "res", "cpu"))
    assert np.array_equal(bf16_bits(t["Qp0"]), bf16_bits(t["Qp1"]))  # same X and W_Q every step
    q_ref = _oracle_q(cfg)
    check_qpred(bf16_bits(t["Qp0"]), q_ref)
    qp = O.f64_to_bf16(q_ref).reshape(s.B, s.Hq, s.D)  # the oracle selects with its own Q_pred
    last = (step.i - 1) % 2  # output buffer of the last step
    O_out, L_out = t[f"O{last}"].float().cpu().numpy(), t[f"lse{last}"].cpu().numpy()
    o_cpu, l_cpu = wl.cpu_partial()
    _check_all_lists(s, wl, topk, tc, res, rc, cpu, cc)
    # the configuration bench.py times is checked on more units against the oracle
    for u in _sample(s.units, extra=27 if mode == "graph" and not early else 0):
        b, kvh = divmod(u, s.Hkv)
        _check_unit(wl, u, qp[b, kvh * s.G:(kvh + 1) * s.G], "minmax", topk, tc, res, rc, cpu, cc, O_out, L_out,
                    o_cpu, l_cpu)


def _run_steps(early, graph, n=3, serial=False, pdl=False):
    """n steps of the Qwen3-14B-shaped layer; every output buffer of both parities, on the host."""
    dev = torch.device("cuda", 0)
    wl, t, step = setup_step(W.CONFIGS["qwen3_14b"](), dev, serial=serial, split=SPLIT, early=early, pdl=pdl)
    if graph:
        step.capture(n, dev).replay()
    else:
        ev = torch.cuda.Event()
        ev.record()
        step.begin(ev)
        for _ in range(n):
            step.issue()
        step.end(None)
    torch.cuda.synchronize()
    assert int(t["status"].item()) == 0
    names = ["Qp", "O", "lse"] + [f"{n}{c}" for n in ("topk", "res", "cpu", "delta") for c in ("", "_count")]
    out = {f"{n}{par}": t[f"{n}{par}"].view(torch.int16 if t[f"{n}{par}"].dtype == torch.bfloat16 else
                                            (torch.int32 if t[f"{n}{par}"].dtype == torch.float32 else
                                             t[f"{n}{par}"].dtype)).cpu().numpy()
           for n in names for par in (0, 1)}
    del wl, t, step
    torch.cuda.empty_cache()
    return out


def test_early_start_changes_no_bit():
    """The step with every kernel starting early after the one it waits for (programmatic
    dependent launch, graph-captured as bench.py times it) leaves every output buffer bit for bit
    as the step without early starts does: each kernel waits before it reads what the other wrote,
    and writes only after that wait."""
    plain = _run_steps((), graph=False)
    early = _run_steps(tuple(EARLY_OF), graph=True)
    for k in plain:
        assert np.array_equal(plain[k], early[k]), k


@pytest.mark.parametrize("graph", [False, True])
def test_same_stream_early_start_changes_no_bit(graph):
    """The serial step with its three persistent kernels started early after the kernel before
    them on the one stream (scout_launch.pdl) leaves every output buffer as the plain serial step
    does, issued on the stream and captured in a CUDA graph."""
    plain = _run_steps((), graph=False, serial=True)
    early = _run_steps((), graph=graph, serial=True, pdl=True)
    for k in plain:
        assert np.array_equal(plain[k], early[k]), k


# every point of the stress sweep: page 16/32/64 x budget 512/2048/8192 tokens x min/max and mean
STRESS = [(P, budget, kind) for P in (16, 32, 64) for budget in (512, 2048, 8192) for kind in ("minmax", "mean")]


@pytest.mark.parametrize("P,budget,kind", STRESS)
def test_stress_shapes_sampled(P, budget, kind):
    """B=4 at 128K context: k from 8 to 512 blocks, nblk from 2048 to 8192, both digest kinds;
    three units checked against the oracle, and the list algebra of every unit."""
    s = W.stress(P, budget, kind)
    wl = W.Workload(s)
    d = WD.materialize(wl, with_gemm=False)
    nb = s.nblk
    if kind == "minmax":
        dg = torch.empty((s.B, s.Hkv, nb, 2, s.D), dtype=torch.bfloat16, device="cuda")
    else:
        dg = torch.empty((s.B, s.Hkv, nb, s.D), dtype=torch.float32, device="cuda")
    bs.build_digest(kind, d["K_pool"], d["page_table"], d["seq_len"], s.B, s.Hkv, P, dg)
    ws = bs.score_topk_workspace(s.B, s.Hkv, nb)
    out = bs.score_topk(kind, d["q"], dg, d["seq_len"], d["resident_bits"], s.B, s.Hq, s.Hkv, P, nb, s.k, ws)
    wa = bs.sparse_attn_workspace(s.B, s.Hq, s.Hkv, P)
    O_out, L_out = bs.sparse_attn_merge(d["q"], d["K_pool"], d["V_pool"], d["page_table"], d["seq_len"], out["res"],
                                        out["res_count"], s.B, s.Hq, s.Hkv, P, s.k, s.scale, wa, d["O_cpu"],
                                        d["lse_cpu"])
    torch.cuda.synchronize()
    grab = lambda n: out[n].cpu().numpy().reshape(s.units, -1)  # noqa: E731
    cnt = lambda n: out[n].cpu().numpy().reshape(-1)  # noqa: E731
    o_cpu, l_cpu = wl.cpu_partial()
    _check_list_algebra(s, wl, grab, cnt)
    for u in (0, s.units // 2 + 1, s.units - 1):
        b, kvh = divmod(u, s.Hkv)
        _check_unit(wl, u, wl.q[b, kvh * s.G:(kvh + 1) * s.G], kind, grab("topk"), cnt("topk_count"), grab("res"),
                    cnt("res_count"), grab("cpu"), cnt("cpu_count"), O_out.float().cpu().numpy(),
                    L_out.cpu().numpy(), o_cpu, l_cpu)


def _check_list_algebra(s, wl, grab, cnt):
    """Every unit, without the oracle: k_eff entries in ascending order, res and cpu partition the
    selection by the residency bits, the delta (no previous list) is the cpu list, -1 past the counts."""
    topk, tc, res, rc, cpu, cc, dl, dc = (grab("topk"), cnt("topk_count"), grab("res"), cnt("res_count"), grab("cpu"),
                                          cnt("cpu_count"), grab("delta"), cnt("delta_count"))
    for u in range(s.units):
        nv = int(wl.nvalid[u // s.Hkv])
        S = topk[u, :tc[u]]
        assert tc[u] == min(s.k, nv) and np.all(np.diff(S) > 0) and np.all(topk[u, tc[u]:] == -1), u
        r, c = res[u, :rc[u]], cpu[u, :cc[u]]
        assert rc[u] + cc[u] == tc[u] and np.array_equal(np.union1d(r, c), S), u
        assert np.all(wl.resident[u, r] == 1) and np.all(wl.resident[u, c] == 0), u
        assert dc[u] == cc[u] and np.array_equal(dl[u, :dc[u]], c), u
        assert np.all(res[u, rc[u]:] == -1) and np.all(cpu[u, cc[u]:] == -1) and np.all(dl[u, dc[u]:] == -1), u


def test_dense_edge_case_at_128k():
    """top-k = every block and everything resident: the output is full softmax attention."""
    s = W.Shape("dense_128k", B=2, Hq=40, Hkv=8, T=131072 - 7, P=32, k=4096, resident_frac=1.0)
    wl = W.Workload(s)
    d = WD.materialize(wl, with_gemm=False)
    dg = torch.empty((s.B, s.Hkv, s.nblk, 2, s.D), dtype=torch.bfloat16, device="cuda")
    bs.build_digest("minmax", d["K_pool"], d["page_table"], d["seq_len"], s.B, s.Hkv, s.P, dg)
    ws = bs.score_topk_workspace(s.B, s.Hkv, s.nblk)
    out = bs.score_topk("minmax", d["q"], dg, d["seq_len"], d["resident_bits"], s.B, s.Hq, s.Hkv, s.P, s.nblk, s.k,
                        ws)
    wa = bs.sparse_attn_workspace(s.B, s.Hq, s.Hkv, s.P)
    Og, Lg = bs.sparse_attn(d["q"], d["K_pool"], d["V_pool"], d["page_table"], d["seq_len"], out["res"],
                            out["res_count"], s.B, s.Hq, s.Hkv, s.P, s.k, s.scale, wa)
    torch.cuda.synchronize()
    assert torch.all(out["res_count"] == s.nblk) and torch.all(out["cpu_count"] == 0)
    Og, Lg = Og.cpu().numpy(), Lg.cpu().numpy()
    for u in (3, s.units - 1):
        b, kvh = divmod(u, s.Hkv)
        L = int(wl.seq_len[b])
        K, V = O.bf16_to_f64(wl.unit_kv(u))[:L], O.bf16_to_f64(wl.unit_kv(u, "V"))[:L]
        for h in (0, s.G - 1):
            hq = kvh * s.G + h
            o, l = O.attention_partial(O.bf16_to_f64(wl.q[b, hq]), K, V, s.scale)
            check_attention(Og[b, hq], Lg[b, hq], o, l, what=(u, h))
