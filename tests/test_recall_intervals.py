"""Per-layer recall intervals (ScoutAttention, section 3.4: for each layer, the largest number
of decoding steps that keeps the measured CPU compute ratio below the threshold beta, read from
an offline profile).  The oracle's rule is pinned by closed forms and boundary cases; the
library's scout_recall_intervals is checked against it on seeded traces.  Host code only."""
import ctypes

import numpy as np
import pytest

import oracle as O
import block_sparse_kv_pred_gb300 as bs
from _parity import ensure_built


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_oracle_rule_closed_forms_and_boundaries():
    # a linear drift a * (s + 1) with a = 1/64 (exact in fp32): below 0.12 while s + 1 <= 7
    a = 1.0 / 64
    assert O.recall_intervals([[a * (s + 1) for s in range(20)]], 0.12) == [7]
    # ... and in general floor-then-adjust: the count of n >= 1 with a n < beta
    for beta in (0.05, 0.08, 0.12, 0.2):
        n = int(np.ceil(beta / a)) - 1
        assert O.recall_intervals([[a * (s + 1) for s in range(40)]], beta) == [n]
    assert O.recall_intervals([[0.01, 0.02, 0.03, 0.12, 0.05]], 0.12) == [3]  # strictly below beta
    assert O.recall_intervals([[0.2, 0.01, 0.01]], 0.12) == [1]               # first step already above
    assert O.recall_intervals([[0.01] * 9], 0.12) == [9]                      # never reaches beta
    assert O.recall_intervals([[0.01, 0.02, float("nan"), 0.01]], 0.12) == [2]  # NaN is not below
    # a ratio that dips back below beta after crossing it does not extend the interval
    assert O.recall_intervals([[0.05, 0.13, 0.05, 0.05]], 0.12) == [1]
    # layers are independent
    assert O.recall_intervals([[0.2], [0.01]], 0.12) == [1, 1]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_library_matches_oracle_on_seeded_traces(seed):
    rng = np.random.default_rng(seed)
    layers, steps = 40, 64
    # drifting ratios like the profile of a decode without recalls: a per-layer slope plus noise
    slope = rng.uniform(0.002, 0.05, size=(layers, 1))
    trace = (slope * np.arange(1, steps + 1)[None, :] + rng.normal(0, 0.01, size=(layers, steps))).astype(np.float32)
    trace[3, 10] = np.nan
    trace[5, :] = 0.0                      # a layer that never drifts
    trace[7, 0] = 0.5                      # one that starts above
    trace[9, 4] = np.float32(0.12)         # exactly at beta
    for beta in (0.08, 0.12, 0.2):
        got = bs.recall_intervals(trace, beta)
        ref = O.recall_intervals(trace.tolist(), np.float32(beta))
        assert list(got) == ref, beta
    assert bs.recall_intervals(trace)[5] == steps and bs.recall_intervals(trace)[7] == 1


def test_bad_arguments_are_rejected():
    L = bs.lib()
    r = np.zeros((2, 3), np.float32)
    out = np.full(2, -7, np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    f = ctypes.c_float
    assert L.scout_recall_intervals(None, 2, 3, f(0.12), p(out)) == 1
    assert L.scout_recall_intervals(p(r), 0, 3, f(0.12), p(out)) == 1
    assert L.scout_recall_intervals(p(r), 2, 0, f(0.12), p(out)) == 1
    assert L.scout_recall_intervals(p(r), 2, 3, f(0.0), p(out)) == 1
    assert L.scout_recall_intervals(p(r), 2, 3, f(float("inf")), p(out)) == 1
    assert L.scout_recall_intervals(p(r), 2, 3, f(float("nan")), p(out)) == 1
    assert np.all(out == -7)
    assert L.scout_recall_intervals(p(r), 2, 3, f(0.12), p(out)) == 0 and list(out) == [3, 3]


def test_profile_assembles_one_seeded_trace_per_layer(monkeypatch):
    """sweep.profile_recall_intervals without a GPU: a scripted stand-in for the decode sweep
    checks that every layer gets its own seed, decodes without recalls, and that the traces are
    assembled in step order and turned into intervals by the rule."""
    torch = pytest.importorskip("torch")
    import block_sparse_kv_pred_gb300.sweep as S
    from block_sparse_kv_pred_gb300 import workload as W

    seen = []

    class Scripted:
        def __init__(self, shape, steps, recall_every=16, device="cuda"):
            assert recall_every == 0
            seen.append(shape.seed)
            self.slope, self.t = 0.01 * (shape.seed + 1), 0

        def step(self):
            self.t += 1
            return {"stats": {"cpu_ratio": self.slope * self.t}}

    monkeypatch.setattr(S, "DecodeSweep", Scripted)
    monkeypatch.setattr(torch.cuda, "empty_cache", lambda: None)
    base = W.Shape("p", B=1, Hq=8, Hkv=2, T=256, P=32, k=4, resident_frac=0.0, seed=3)
    traces, iv = S.profile_recall_intervals(3, 10, 0.12, shape=base)
    assert seen == [3, 4, 5]
    want = np.array([[0.01 * (sd + 1) * (t + 1) for t in range(10)] for sd in (3, 4, 5)], dtype=np.float32)
    assert np.allclose(traces, want)
    assert list(iv) == O.recall_intervals(traces.tolist(), np.float32(0.12))
