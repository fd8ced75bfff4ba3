"""Pins for the fp64 oracle: closed forms, brute force, invariants and library routines.

None of these re-types an oracle formula; each checks the oracle against
something it does not compute itself, so that a dropped term, a wrong sign,
a wrong index or a transposed operand fails at least one test.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle as O
from block_sparse_kv_pred_gb300 import workload as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split()
            out[k] = float(v)
    return out


def bits(x):
    """bf16 bits of values that are exactly representable."""
    x = np.asarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not exactly bf16"
    return (b >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# bf16 helpers
# ---------------------------------------------------------------------------
def test_bf16_round_half_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties to the even mantissa (1.0)
    assert O.f64_to_bf16(1.0 + 2.0**-8) == 0x3F80
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert O.f64_to_bf16(1.0 + 3 * 2.0**-8) == 0x3F82
    assert O.f64_to_bf16(-2.0) == 0xC000
    assert O.f64_to_bf16(0.0) == 0x0000
    # just above a tie rounds up
    assert O.f64_to_bf16(1.0 + 2.0**-8 + 2.0**-30) == 0x3F81


def test_bf16_decode_exact_and_agrees_with_integer_rounding():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(20000).astype(np.float32) * 37.0
    # two independent roundings: frexp/rint in fp64 and the integer carry trick in fp32
    assert np.array_equal(O.f64_to_bf16(x.astype(np.float64)), W.f32_to_bf16(x))
    b = W.f32_to_bf16(x)
    assert np.array_equal(O.bf16_to_f64(b), W.bf16_to_f32(b).astype(np.float64))


# ---------------------------------------------------------------------------
# Q_pred = W_Q X  (section 3.3)
# ---------------------------------------------------------------------------
def test_predict_q_hand_example():
    # X rows are inputs, W rows are output features: Q[m][n] = sum_k X[m][k] W[n][k]
    X = bits([[1.0, 2.0], [3.0, 4.0]])
    Wq = bits([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    Q = O.predict_q(X, Wq)
    assert np.array_equal(Q, np.array([[1.0, 2.0, 3.0], [3.0, 4.0, 7.0]]))


def test_predict_q_identity_and_permutation():
    rng = np.random.default_rng(2)
    X = bits(rng.integers(-8, 8, size=(3, 5)).astype(np.float32))
    eye = bits(np.eye(5, dtype=np.float32))
    assert np.array_equal(O.predict_q(X, eye), O.bf16_to_f64(X))
    perm = [3, 0, 4, 1, 2]
    Pm = np.zeros((5, 5), dtype=np.float32)
    for n, kk in enumerate(perm):
        Pm[n, kk] = 1.0
    out = O.predict_q(X, bits(Pm))
    assert np.array_equal(out, O.bf16_to_f64(X)[:, perm])


def test_predict_q_brute_force_tiny():
    rng = np.random.default_rng(3)
    X = bits(rng.integers(-6, 7, size=(2, 4)).astype(np.float32))
    Wq = bits(rng.integers(-6, 7, size=(3, 4)).astype(np.float32))
    Xi = O.bf16_to_f64(X).astype(int)
    Wi = O.bf16_to_f64(Wq).astype(int)
    Q = O.predict_q(X, Wq)
    for m in range(2):
        for n in range(3):
            acc = 0
            for kk in range(4):
                acc += int(Xi[m][kk]) * int(Wi[n][kk])
            assert Q[m][n] == acc


# ---------------------------------------------------------------------------
# digests (section 2.2: Quest min/max, MoBA mean)
# ---------------------------------------------------------------------------
def _ramp_keys(T, D):
    # K[t][c] = t (c + 1) - 5 c : increasing in t for every channel
    t = np.arange(T, dtype=np.float32)[:, None]
    c = np.arange(D, dtype=np.float32)[None, :]
    return bits(t * (c + 1) - 5 * c)


def test_digest_minmax_closed_form_with_ragged_tail():
    P, D, seq_len = 4, 3, 10  # blocks [0..3], [4..7], [8, 9]
    K = _ramp_keys(12, D)
    mn, mx = O.digest_minmax(K, seq_len, P)
    assert mn.shape == (3, D)
    for j in range(3):
        first, last = j * P, min((j + 1) * P, seq_len) - 1
        for c in range(D):
            assert mn[j, c] == first * (c + 1) - 5 * c
            assert mx[j, c] == last * (c + 1) - 5 * c


def test_digest_mean_closed_form_with_ragged_tail():
    P, D, seq_len = 4, 3, 10
    K = _ramp_keys(12, D)
    mean = O.digest_mean(K, seq_len, P)
    for j in range(3):
        toks = list(range(j * P, min((j + 1) * P, seq_len)))
        tbar = sum(toks) / len(toks)
        for c in range(D):
            assert mean[j, c] == pytest.approx(tbar * (c + 1) - 5 * c, abs=0)


def test_digest_invariants_random():
    rng = np.random.default_rng(4)
    P, D, seq_len = 8, 16, 45
    K = W.f32_to_bf16(rng.standard_normal((48, D)).astype(np.float32))
    mn, mx = O.digest_minmax(K, seq_len, P)
    Kf = O.bf16_to_f64(K)
    for j in range(mn.shape[0]):
        rows = Kf[j * P: min((j + 1) * P, seq_len)]
        assert np.all(mn[j] <= rows) and np.all(rows <= mx[j])
        # attained: every bound is one of the block's values in that channel
        for c in range(D):
            assert mn[j, c] in rows[:, c] and mx[j, c] in rows[:, c]
    # tokens past seq_len do not enter the digest
    K2 = K.copy()
    K2[seq_len:] = W.f32_to_bf16(np.full((48 - seq_len, D), 1e4, dtype=np.float32))
    mn2, mx2 = O.digest_minmax(K2, seq_len, P)
    assert np.array_equal(mn, mn2) and np.array_equal(mx, mx2)
    assert np.array_equal(O.digest_mean(K, seq_len, P), O.digest_mean(K2, seq_len, P))


# ---------------------------------------------------------------------------
# scores (section 3.2: query . digest)
# ---------------------------------------------------------------------------
def test_minmax_score_is_max_of_linear_form_over_the_box():
    # max over v in the box [mn, mx] of q.v is attained at a corner: enumerate all 2^D corners
    rng = np.random.default_rng(5)
    D = 5
    for _ in range(50):
        a = rng.standard_normal(D)
        b = rng.standard_normal(D)
        mn, mx = np.minimum(a, b), np.maximum(a, b)
        q = rng.standard_normal((3, D))
        u = O.scores_minmax(q, mn[None], mx[None])[:, 0]
        for h in range(3):
            best = max(float(q[h] @ np.where(np.array(sel), mx, mn)) for sel in itertools.product([0, 1], repeat=D))
            assert u[h] == pytest.approx(best, rel=1e-13, abs=1e-13)


def test_minmax_score_bounds_true_block_max_and_is_tight_for_one_token():
    rng = np.random.default_rng(6)
    P, D, seq_len = 8, 32, 41  # last block holds one token
    K = W.f32_to_bf16(rng.standard_normal((48, D)).astype(np.float32))
    q = rng.standard_normal((4, D))
    mn, mx = O.digest_minmax(K, seq_len, P)
    u = O.scores_minmax(q, mn, mx)
    Kf = O.bf16_to_f64(K)
    for j in range(mn.shape[0]):
        rows = Kf[j * P: min((j + 1) * P, seq_len)]
        true_max = (rows @ q.T).max(axis=0)
        assert np.all(u[:, j] >= true_max - 1e-12)
    last = mn.shape[0] - 1
    assert np.allclose(u[:, last], q @ Kf[seq_len - 1], rtol=0, atol=1e-12)


def test_mean_score_is_average_token_score():
    rng = np.random.default_rng(7)
    P, D, seq_len = 8, 16, 30
    K = W.f32_to_bf16(rng.standard_normal((32, D)).astype(np.float32))
    q = rng.standard_normal((2, D))
    u = O.scores_mean(q, O.digest_mean(K, seq_len, P))
    Kf = O.bf16_to_f64(K)
    for j in range(u.shape[1]):
        rows = Kf[j * P: min((j + 1) * P, seq_len)]
        for h in range(2):
            assert u[h, j] == pytest.approx(sum(float(q[h] @ r) for r in rows) / len(rows), rel=1e-12)


def test_pool_group_takes_max_over_heads():
    u = np.array([[1.0, 5.0, -2.0], [3.0, 4.0, -1.0]])
    assert np.array_equal(O.pool_group(u), np.array([3.0, 5.0, -1.0]))


def test_sum_pooling_is_the_summed_query_against_the_digest():
    """Sum pooling (a variant): for the mean digest, linearity makes it the group's summed query
    dotted with each block's mean key; for one-token blocks the min/max bound is tight, so it is
    the summed query's logit exactly; with one head it equals max pooling."""
    rng = np.random.default_rng(21)
    G, D, P, T = 3, 8, 4, 22
    K = W.f32_to_bf16(rng.integers(-4, 5, size=(T, D)).astype(np.float32))
    q = W.f32_to_bf16(rng.integers(-3, 4, size=(G, D)).astype(np.float32))
    Kf, qf = O.bf16_to_f64(K), O.bf16_to_f64(q)
    mean = O.digest_mean(K, T, P)
    U = O.pool_group_sum(O.scores_mean(qf, mean))
    for j in range(len(U)):
        rows = Kf[j * P:min(T, (j + 1) * P)]
        assert U[j] == pytest.approx(float(qf.sum(axis=0) @ rows.mean(axis=0)), abs=1e-12)
    mn, mx = O.digest_minmax(K, T, 1)  # one token per block
    assert np.array_equal(O.pool_group_sum(O.scores_minmax(qf, mn, mx)), Kf @ qf.sum(axis=0))
    one = O.scores_minmax(qf[:1], mn, mx)
    assert np.array_equal(O.pool_group_sum(one), O.pool_group(one))
    # and the bound: the summed logit of every token of a block is at most the block's sum-pooled score
    mn, mx = O.digest_minmax(K, T, P)
    Us = O.pool_group_sum(O.scores_minmax(qf, mn, mx))
    for t in range(T):
        assert float(Kf[t] @ qf.sum(axis=0)) <= Us[t // P] + 1e-12


# ---------------------------------------------------------------------------
# top-k (Algorithm 1: B_pred = TopK(...)), ties to the lower block index
# ---------------------------------------------------------------------------
def _dominates(U, a, b):
    return U[a] > U[b] or (U[a] == U[b] and a < b)


@pytest.mark.parametrize("n", [1, 2, 5, 7, 9])
def test_topk_matches_exhaustive_subset_search(n):
    rng = np.random.default_rng(100 + n)
    for _ in range(30):
        U = rng.integers(-2, 3, size=n).astype(np.float64)  # many ties
        for k in range(0, n + 2):
            keff = min(k, n)
            winners = []
            for sub in itertools.combinations(range(n), keff):
                rest = [j for j in range(n) if j not in sub]
                if all(_dominates(U, a, b) for a in sub for b in rest):
                    winners.append(sub)
            assert len(winners) == 1
            assert list(O.select_topk(U, k)) == list(winners[0])


def test_topk_hand_example_with_ties():
    U = np.array([2.0, 7.0, 7.0, -1.0, 7.0, 3.0])
    assert list(O.select_topk(U, 2)) == [1, 2]
    assert list(O.select_topk(U, 4)) == [1, 2, 4, 5]
    assert list(O.select_topk(U, 10)) == [0, 1, 2, 3, 4, 5]
    assert list(O.select_topk(U, 0)) == []


def test_split_and_delta_set_algebra():
    rng = np.random.default_rng(8)
    for _ in range(200):
        n = int(rng.integers(1, 40))
        U = rng.standard_normal(n)
        k = int(rng.integers(0, n + 3))
        R = rng.random(n) < 0.3
        S = O.select_topk(U, k)
        res, cpu = O.split_residency(S, R)
        assert set(res) | set(cpu) == set(S.tolist())
        assert not (set(res) & set(cpu))
        assert all(R[j] for j in res) and not any(R[j] for j in cpu)
        assert list(res) == sorted(res) and list(cpu) == sorted(cpu)
        prev = rng.choice(n, size=int(rng.integers(0, n + 1)), replace=False)
        d = O.delta_list(cpu, np.sort(prev))
        assert set(d) == set(cpu) - set(prev.tolist()) and list(d) == sorted(d)


# ---------------------------------------------------------------------------
# attention partials and merge (section 3.2: FlashAttention / online-softmax merge)
# ---------------------------------------------------------------------------
def test_attention_special_cases():
    rng = np.random.default_rng(9)
    D, scale = 8, 0.3
    q = rng.standard_normal(D)
    K = rng.standard_normal((1, D))
    V = rng.standard_normal((1, D))
    o, l = O.attention_partial(q, K, V, scale)
    assert np.allclose(o, V[0]) and l == pytest.approx(scale * float(K[0] @ q))
    # two tokens with equal scores: plain average, lse + ln 2
    K2 = np.vstack([K, K])
    V2 = rng.standard_normal((2, D))
    o, l = O.attention_partial(q, K2, V2, scale)
    assert np.allclose(o, V2.mean(axis=0)) and l == pytest.approx(scale * float(K[0] @ q) + math.log(2))
    # zero query: uniform weights
    Kn = rng.standard_normal((5, D))
    Vn = rng.standard_normal((5, D))
    o, l = O.attention_partial(np.zeros(D), Kn, Vn, scale)
    assert np.allclose(o, Vn.mean(axis=0)) and l == pytest.approx(math.log(5))
    # empty set
    o, l = O.attention_partial(q, np.zeros((0, D)), np.zeros((0, D)), scale)
    assert np.all(o == 0) and l == -math.inf


def test_attention_matches_scipy_softmax():
    rng = np.random.default_rng(10)
    D, n, scale = 16, 37, 1 / 4
    q = rng.standard_normal(D) * 3
    K = rng.standard_normal((n, D))
    V = rng.standard_normal((n, D))
    o, l = O.attention_partial(q, K, V, scale)
    logits = scale * np.einsum("nd,d->n", K, q)
    assert np.allclose(o, scipy.special.softmax(logits) @ V, rtol=1e-12, atol=1e-12)
    assert l == pytest.approx(float(scipy.special.logsumexp(logits)), rel=1e-13)


def test_merge_identity_commutative_associative():
    rng = np.random.default_rng(11)
    a = (rng.standard_normal(6), 1.5)
    b = (rng.standard_normal(6), -0.25)
    c = (rng.standard_normal(6), 4.0)
    e = (np.zeros(6), -math.inf)
    o, l = O.merge(*a, *e)
    assert np.allclose(o, a[0]) and l == a[1]
    o, l = O.merge(*e, *e)
    assert np.all(o == 0) and l == -math.inf
    ab = O.merge(*a, *b)
    ba = O.merge(*b, *a)
    assert np.allclose(ab[0], ba[0]) and ab[1] == pytest.approx(ba[1])
    left = O.merge(*O.merge(*a, *b), *c)
    right = O.merge(*a, *O.merge(*b, *c))
    assert np.allclose(left[0], right[0], atol=1e-14) and left[1] == pytest.approx(right[1])
    # equal weights: average, lse + ln 2
    o, l = O.merge(a[0], 2.0, b[0], 2.0)
    assert np.allclose(o, (a[0] + b[0]) / 2) and l == pytest.approx(2.0 + math.log(2))


def test_any_partition_merged_equals_unsplit():
    rng = np.random.default_rng(12)
    D, n, scale = 16, 50, 0.25
    q = rng.standard_normal(D) * 2
    K = rng.standard_normal((n, D)) * 2
    V = rng.standard_normal((n, D))
    whole = O.attention_partial(q, K, V, scale)
    for _ in range(20):
        mask = rng.random(n) < rng.random()
        p1 = O.attention_partial(q, K[mask], V[mask], scale)
        p2 = O.attention_partial(q, K[~mask], V[~mask], scale)
        o, l = O.merge(*p1, *p2)
        assert np.allclose(o, whole[0], atol=1e-12) and l == pytest.approx(whole[1], abs=1e-12)


# ---------------------------------------------------------------------------
# whole unit step: dense edge case equals full attention
# ---------------------------------------------------------------------------
def test_dense_edge_case_equals_full_attention():
    rng = np.random.default_rng(13)
    G, D, P, T, seq_len = 3, 16, 8, 64, 61
    K = W.f32_to_bf16(rng.standard_normal((T, D)).astype(np.float32))
    V = W.f32_to_bf16(rng.standard_normal((T, D)).astype(np.float32))
    q = W.f32_to_bf16(rng.standard_normal((G, D)).astype(np.float32))
    nb = T // P
    for kind in ("minmax", "mean"):
        r = O.unit_step(q, q, K, V, seq_len, P, nb, kind, np.ones(nb, bool), 0.25)
        assert list(r["topk"]) == list(range(nb)) and list(r["res"]) == list(range(nb)) and len(r["cpu"]) == 0
        Kf, Vf, qf = O.bf16_to_f64(K)[:seq_len], O.bf16_to_f64(V)[:seq_len], O.bf16_to_f64(q)
        for h in range(G):
            logits = 0.25 * (Kf @ qf[h])
            assert np.allclose(r["O"][h], scipy.special.softmax(logits) @ Vf, atol=1e-12)
            assert r["L"][h] == pytest.approx(float(scipy.special.logsumexp(logits)), rel=1e-13)


def test_gpu_plus_cpu_partials_merge_to_attention_over_topk():
    rng = np.random.default_rng(14)
    G, D, P, T = 2, 16, 4, 64
    K = W.f32_to_bf16(rng.standard_normal((T, D)).astype(np.float32))
    V = W.f32_to_bf16(rng.standard_normal((T, D)).astype(np.float32))
    q = W.f32_to_bf16(rng.standard_normal((G, D)).astype(np.float32))
    R = rng.random(T // P) < 0.5
    r = O.unit_step(q, q, K, V, T, P, 6, "minmax", R, 0.25)
    Kf, Vf, qf = O.bf16_to_f64(K), O.bf16_to_f64(V), O.bf16_to_f64(q)
    tc = O.block_tokens(r["cpu"], P, T)
    ts = O.block_tokens(r["topk"], P, T)
    for h in range(G):
        cpu = O.attention_partial(qf[h], Kf[tc], Vf[tc], 0.25)
        o, l = O.merge(r["O"][h], r["L"][h], *cpu)
        logits = 0.25 * (Kf[ts] @ qf[h])
        assert np.allclose(o, scipy.special.softmax(logits) @ Vf[ts], atol=1e-12)
        assert l == pytest.approx(float(scipy.special.logsumexp(logits)), abs=1e-12)


def test_all_resident_variant_merges_to_attention_over_resident_and_selected():
    """The variant where the GPU attends every resident block: its partial merged with the CPU
    partial over S minus R is softmax attention over R union S (computed here directly); with
    R inside S it is the main reading's result; sum pooling picks the blocks of the summed query."""
    rng = np.random.default_rng(15)
    G, D, P, T, k = 2, 16, 4, 62, 5
    K = W.f32_to_bf16(rng.standard_normal((T, D)).astype(np.float32))
    V = W.f32_to_bf16(rng.standard_normal((T, D)).astype(np.float32))
    q = W.f32_to_bf16(rng.standard_normal((G, D)).astype(np.float32))
    Kf, Vf, qf = O.bf16_to_f64(K), O.bf16_to_f64(V), O.bf16_to_f64(q)
    nb = -(-T // P)
    R = rng.random(nb) < 0.4
    for pool in ("max", "sum"):
        r = O.unit_step(q, q, K, V, T, P, k, "minmax", R, 0.25, pool=pool, gpu_blocks="resident")
        assert list(r["gpu"]) == list(np.flatnonzero(R))
        union = sorted(set(np.flatnonzero(R)) | set(int(j) for j in r["topk"]))
        tu, tc = O.block_tokens(union, P, T), O.block_tokens(r["cpu"], P, T)
        for h in range(G):
            o, l = O.merge(r["O"][h], r["L"][h], *O.attention_partial(qf[h], Kf[tc], Vf[tc], 0.25))
            logits = 0.25 * (Kf[tu] @ qf[h])
            assert np.allclose(o, scipy.special.softmax(logits) @ Vf[tu], atol=1e-12)
            assert l == pytest.approx(float(scipy.special.logsumexp(logits)), abs=1e-12)
        mn, mx = O.digest_minmax(K, T, P)
        sc = O.scores_minmax(qf, mn, mx)
        want = sc.max(axis=0) if pool == "max" else sc.sum(axis=0)
        assert list(r["topk"]) == sorted(np.argsort(-want, kind="stable")[:k])
    # R inside S: both readings attend the same blocks
    r0 = O.unit_step(q, q, K, V, T, P, k, "minmax", np.zeros(nb, bool), 0.25)
    Rin = np.zeros(nb, bool)
    Rin[r0["topk"][:2]] = True
    a = O.unit_step(q, q, K, V, T, P, k, "minmax", Rin, 0.25)
    b = O.unit_step(q, q, K, V, T, P, k, "minmax", Rin, 0.25, gpu_blocks="resident")
    assert np.array_equal(a["O"], b["O"]) and np.array_equal(a["L"], b["L"])


# ---------------------------------------------------------------------------
# layout constant from the pages
# ---------------------------------------------------------------------------
def test_layout_constant_matches_the_pages():
    g = read_golden("layout_constant.txt")
    s = W.qwen3_14b()
    per_token = s.Hkv * s.D * 2 * 2
    assert per_token == g["bytes_per_token_per_layer"] == g["kv_heads"] * g["head_dim"] * g["tensors"] * g["bytes_per_element"]
    assert per_token * s.P == g["page_bytes"] and s.P == g["page_tokens"]
    ev = read_golden("evaluation_setup.txt")
    assert s.k * s.P == ev["budget_tokens"] and s.P == ev["block_size"]


# ---------------------------------------------------------------------------
# recall (section 3.4): properties any correct plan has, and a hand example
# ---------------------------------------------------------------------------
def test_recall_plan_hand_example_with_ties():
    # blocks 0..7; resident {0, 1, 2, 5}; selected {1, 3, 4, 6}
    U = [0.5, 9.0, 0.5, 7.0, 8.0, 0.1, 7.0, 3.0]
    res = np.array([1, 1, 1, 0, 0, 1, 0, 0], dtype=bool)
    slot = np.array([10, 11, 12, -1, -1, 15, -1, -1])
    ops = O.recall_plan(U, [1, 3, 4, 6], res, slot)
    # incoming by importance: 4 (8.0), 3 (7.0, lower index), 6 (7.0); evict by least importance:
    # 5 (0.1), 0 (0.5, lower index), 2 (0.5)
    assert ops == [(3, 10, 0), (4, 15, 5), (6, 12, 2)]
    slot2, res2 = O.apply_recall(slot, res, ops)
    assert list(np.flatnonzero(res2)) == [1, 3, 4, 6]
    assert sorted(slot2[res2]) == [10, 11, 12, 15]


@pytest.mark.parametrize("seed", range(20))
def test_recall_plan_properties_random(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 40))
    U = np.round(rng.standard_normal(n), 1)  # coarse values: many ties
    res = rng.random(n) < rng.random()
    slot = np.where(res, rng.permutation(1000)[:n], -1)
    sel = O.select_topk(U, int(rng.integers(1, n + 1)))
    ops = O.recall_plan(U, sel, res, slot)
    incoming = [j for j in sel if not res[j]]
    evictable = [j for j in range(n) if res[j] and j not in set(sel)]
    assert len(ops) == min(len(incoming), len(evictable))
    brought = [b for b, _, _ in ops]
    evicted = [e for _, _, e in ops]
    assert brought == sorted(brought) and set(brought) <= set(incoming) and set(evicted) <= set(evictable)
    key_in = lambda j: (-U[j], j)  # noqa: E731  (importance order of the pages' reading)
    key_ev = lambda j: (U[j], j)  # noqa: E731
    for j in set(incoming) - set(brought):  # every block left out is less important than every one brought
        assert all(key_in(b) < key_in(j) for b in brought)
    for j in set(evictable) - set(evicted):  # every kept block is more important than every evicted one
        assert all(key_ev(e) < key_ev(j) for e in evicted)
    slot2, res2 = O.apply_recall(slot, res, ops)
    assert res2.sum() == res.sum()  # the pool keeps its size
    assert sorted(slot2[res2]) == sorted(slot[res])  # the same slots, reassigned
    if len(evictable) >= len(incoming):
        assert all(res2[j] for j in sel)
