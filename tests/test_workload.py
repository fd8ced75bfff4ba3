"""Host generator: exactness, determinism, statistics and structure."""
import numpy as np

from block_sparse_kv_pred_gb300 import workload as W


def test_irwin_hall_exact_in_fp32_and_deterministic():
    idx = np.arange(0, 50000, dtype=np.uint64)
    z = W.irwin_hall(0, W.STREAM_K, idx)
    # every value is an integer multiple of 2^-16 in [-6, 6)
    scaled = (z.astype(np.float64) + 6.0) * 65536.0
    assert np.all(scaled == np.round(scaled)) and z.min() >= -6 and z.max() < 6
    assert np.array_equal(z, W.irwin_hall(0, W.STREAM_K, idx))
    # random access: any slice equals the matching part of the full draw
    assert np.array_equal(z[1234:1300], W.irwin_hall(0, W.STREAM_K, idx[1234:1300]))
    # streams and seeds differ
    assert not np.array_equal(z[:100], W.irwin_hall(0, W.STREAM_V, idx[:100]))
    assert not np.array_equal(z[:100], W.irwin_hall(1, W.STREAM_K, idx[:100]))


def test_irwin_hall_moments():
    z = W.irwin_hall(3, W.STREAM_Q, np.arange(400000, dtype=np.uint64)).astype(np.float64)
    assert abs(z.mean()) < 0.01
    assert abs(z.var() - 1.0) < 0.01


def test_workload_structure():
    s = W.Shape("t", B=2, Hq=8, Hkv=2, T=1000, P=32, k=8, resident_frac=0.25, seq_lens=(1000, 777))
    wl = W.Workload(s)
    nb = s.nblk
    assert sorted(wl.page_table.ravel().tolist()) == list(range(s.units * nb))
    for u in range(s.units):
        nv = int(wl.nvalid[u // s.Hkv])
        assert wl.resident[u].sum() == round(0.25 * nv)
        assert wl.heavy[u].sum() == round(0.05 * nv)
        assert wl.resident[u, nv:].sum() == 0 and wl.heavy[u, nv:].sum() == 0
    bits = wl.resident_bits().reshape(s.units, s.words)
    for u in range(s.units):
        for j in range(nb):
            assert ((int(bits[u, j // 32]) >> (j % 32)) & 1) == wl.resident[u, j]
    K = wl.unit_kv(1)
    assert K.shape == (nb * s.P, s.D) and K.dtype == np.uint16
    # outlier channels carry about outlier_scale times the spread
    Kf = W.bf16_to_f32(K).astype(np.float64)
    non_heavy = ~np.repeat(wl.heavy[1].astype(bool), s.P)
    sd = Kf[non_heavy].std(axis=0)
    assert np.all(sd[wl.outliers] > 6.0) and np.median(sd) < 1.2


def test_query_walk_cosines_and_norms():
    """The walk keeps ||q|| = sqrt(D), steps at cosine ~0.96, and Q_pred sits at cosine 0.93
    (the smallest value of the pages' Table 1) from the true query."""
    wl = W.Workload(W.tiny())
    q, p = wl.walk(6)
    f = lambda a: W.bf16_to_f32(a).astype(np.float64)  # noqa: E731
    cos = lambda a, b: (a * b).sum(-1) / np.linalg.norm(a, axis=-1) / np.linalg.norm(b, axis=-1)  # noqa: E731
    assert np.array_equal(q[0], wl.q)
    for t in range(1, 6):
        assert abs(cos(f(q[t]), f(q[t - 1])).mean() - 1 / np.sqrt(1.09)) < 0.02
        assert np.allclose(cos(f(q[t]), f(p[t])), 0.93, atol=3e-3)
        assert np.allclose(np.linalg.norm(f(q[t]), axis=-1), np.sqrt(128), rtol=5e-3)
    q2, p2 = wl.walk(6)
    assert np.array_equal(q, q2) and np.array_equal(p, p2)


def _table1():
    """Model -> cosine between predicted and true query, from the golden file (the pages'
    section 3.3, Table 1)."""
    import os

    path = os.path.join(os.path.dirname(__file__), "golden", "table1_query_cosine.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    return {name: float(v) for name, v in rows}


def test_walk_draws_qpred_at_the_table_cosines():
    """The walk's default predicted-query cosine is the smallest of Table 1's, and for every
    model's value the predicted queries it draws sit at that cosine to the true ones (up to the
    bf16 rounding of both)."""
    import inspect

    table = _table1()
    assert len(table) == 5 and all(0.9 < v < 1.0 for v in table.values())
    assert inspect.signature(W.Workload.walk).parameters["cosine"].default == min(table.values())
    s = W.Shape("walk", B=2, Hq=8, Hkv=2, T=256, P=32, k=4, resident_frac=0.25, seq_lens=(256, 200))
    wl = W.Workload(s)
    for name, c in sorted(table.items()):
        qs, ps = wl.walk(3, cosine=c)
        q = W.bf16_to_f32(qs).astype(np.float64)
        p = W.bf16_to_f32(ps).astype(np.float64)
        cos = (q * p).sum(-1) / np.linalg.norm(q, axis=-1) / np.linalg.norm(p, axis=-1)
        assert np.all(np.abs(cos - c) < 3e-3), (name, float(np.abs(cos - c).max()))
        assert abs(cos.mean() - c) < 5e-4, name
