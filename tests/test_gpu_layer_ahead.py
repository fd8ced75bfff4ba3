"""The layer-ahead pipeline on the GPU against the oracle (ScoutAttention (arXiv HTML), section
3.3 and Algorithm 1): every step's CPU partial is computed on the host cores by the worker pool
from the previous step's CPU work list and Q_pred, copied up, and merged by the attention with
its own partial over the resident blocks (true query).  The output of the last step must be the
oracle's merge of attention over R (true query) and attention over C (predicted query), R and C
being the oracle's split of the oracle's top-k under the predicted query (the oracle's own
Q_pred from the seeded X and W_Q, which the GPU's must match within the Q_pred bar first)."""
import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_kv_pred_gb300 import workload as W
from block_sparse_kv_pred_gb300.pipeline import LayerAhead
from block_sparse_kv_pred_gb300.step import setup_step
from _parity import bf16_bits, check_attention, check_qpred, check_selection, ensure_built, oracle_qpred

pytestmark = pytest.mark.gpu

SHAPES = {
    "g4_p32": W.Shape("la_g4_p32", B=2, Hq=8, Hkv=2, T=4100, P=32, k=16, resident_frac=0.5, hidden=1024,
                      seq_lens=(4100, 3001)),
    "qwen3_8b": W.qwen3_8b(),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


@pytest.mark.parametrize("name", list(SHAPES))
def test_layer_ahead_merged_output_matches_oracle(name):
    s = SHAPES[name]
    wl, t, step = setup_step(s, torch.device("cuda", 0))
    with LayerAhead(s, t, step, timeout_s=60.0) as la:
        r = la.run(steps=4, warm=1)
        last = (la.step.i - 1) % 2
    assert r["ms_per_step"] > 0 and int(t["status"].item()) == 0
    assert np.array_equal(bf16_bits(t["Qp0"]), bf16_bits(t["Qp1"]))  # the same X and W_Q every step
    qp_ref = oracle_qpred(s)
    check_qpred(bf16_bits(t["Qp0"]), qp_ref)
    qp_bits = O.f64_to_bf16(qp_ref)  # the oracle's Q_pred, rounded as the step stores it
    Of, Lf = t[f"O{last}"].float().cpu().numpy(), t[f"lse{last}"].cpu().numpy()
    sets = {par: {n: t[f"{n}{par}"].cpu().numpy().reshape(s.units, -1) for n in ("topk", "res", "cpu")}
            for par in (0, 1)}
    counts = {par: {n: t[f"{n}_count{par}"].cpu().numpy().reshape(-1) for n in ("topk", "res", "cpu")}
              for par in (0, 1)}
    units = range(s.units) if s.units <= 16 else sorted({0, 1, s.units // 2, s.units - 1, 17, 42})
    for u in units:
        b, kvh = divmod(u, s.Hkv)
        L = int(wl.seq_len[b])
        qp = qp_bits[b, kvh * s.G * s.D:(kvh + 1) * s.G * s.D].reshape(s.G, s.D)
        qt = wl.q[b, kvh * s.G:(kvh + 1) * s.G]
        ref = O.unit_step(qp, qt, wl.unit_kv(u), wl.unit_kv(u, "V"), L, s.P, s.k, "minmax",
                          wl.resident[u].astype(bool), s.scale)
        exact = [check_selection(ref["scores"], s.k, sets[par]["topk"][u, :counts[par]["topk"][u]], what=(name, u))
                 for par in (0, 1)]  # both sets hold the same selection
        if not all(exact):
            continue  # a near-tie: the split differs from the oracle's, so does the output
        res = sets[1 - last]["res"][u, :counts[1 - last]["res"][u]]
        cpu = sets[1 - last]["cpu"][u, :counts[1 - last]["cpu"][u]]
        assert list(res) == list(ref["res"]) and list(cpu) == list(ref["cpu"]), (name, u)
        K, V = O.bf16_to_f64(wl.unit_kv(u)), O.bf16_to_f64(wl.unit_kv(u, "V"))
        toks = O.block_tokens(ref["cpu"], s.P, L)
        for h in range(s.G):
            hq = kvh * s.G + h
            oc, lc = O.attention_partial(O.bf16_to_f64(qp[h]), K[toks], V[toks], s.scale)
            o, l = O.merge(ref["O"][h], ref["L"][h], oc, lc)
            check_attention(Of[b, hq], Lf[b, hq], o, l, what=(name, u, h))


def test_a_late_cpu_partial_is_an_error_not_a_hang():
    """The pool's bounded wait reports the partial late (a fake of the wait that times out): the
    pipeline raises TimeoutError before issuing the attention that would read it, and the device
    is left usable, every kernel it issued having run."""
    s = SHAPES["g4_p32"]
    wl, t, step = setup_step(s, torch.device("cuda", 0))
    with LayerAhead(s, t, step, timeout_s=60.0) as la:
        real = la.pool.wait
        la.pool.wait = lambda timeout_s: False
        with pytest.raises(TimeoutError, match="late CPU partial"):
            la.run(steps=3)
        la.pool.wait = real
        assert la.pool.wait(60.0)
    torch.cuda.synchronize()
    assert int(t["status"].item()) == 0
