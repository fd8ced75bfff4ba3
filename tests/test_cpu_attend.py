"""scout_cpu_attend, the CPU side of the collaborative attention (ScoutAttention, section 3.2
and Algorithm 1, CPUAttn of the non-resident selected blocks), against the fp64 oracle on
seeded workloads.  Host code only: these tests need no GPU.

The work lists are the oracle's own (selection from the digests, then the residency split),
so they have the shapes scout_score_topk gives: ragged counts, ascending block indices, blocks
at the ragged tail of a sequence.  Tolerance: the attention bar of the GPU kernels (2e-3
absolute / 1e-2 relative), and a tighter fp32 bar (check_fp32): both sides read the same bf16
inputs, so they differ only by fp32 rounding in 128-term dot products, exp and log, and sums of
at most a few thousand terms (measured: at most 4e-6 on O and 7e-7 on the LSE here)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import block_sparse_kv_pred_gb300 as bs
from block_sparse_kv_pred_gb300 import workload as W
from _parity import check_attention, ensure_built


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


SHAPES = {
    "g5_p32": W.Shape("g5_p32", B=2, Hq=10, Hkv=2, T=3000, P=32, k=24, resident_frac=0.25, seq_lens=(3000, 1777)),
    "g8_p16": W.Shape("g8_p16", B=2, Hq=16, Hkv=2, T=2100, P=16, k=40, resident_frac=0.25, seq_lens=(2100, 1000)),
    "g4_p64": W.Shape("g4_p64", B=3, Hq=8, Hkv=2, T=5000, P=64, k=12, resident_frac=0.5,
                      seq_lens=(5000, 4097, 3000)),
}


def check_fp32(o, l, o_ref, l_ref, what=""):
    """fp32 bar: 1e-4 absolute + 1e-4 relative on O, 1e-5 + 1e-5 relative on the LSE."""
    check_attention(o, l, o_ref, l_ref, what)
    if l_ref == -np.inf:
        return
    assert abs(l - l_ref) <= 1e-5 * (1 + abs(l_ref)), (what, l, l_ref)
    assert np.all(np.abs(o - o_ref) <= 1e-4 * (1 + np.abs(o_ref))), (what, float(np.max(np.abs(o - o_ref))))


def _bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _setup(s):
    """Host K/V in logical block order, the query, and the oracle's CPU work lists."""
    wl = W.Workload(s)
    U, nb = s.units, s.nblk
    Kb = np.stack([wl.unit_kv(u) for u in range(U)]).reshape(s.B, s.Hkv, nb, s.P, s.D)
    Vb = np.stack([wl.unit_kv(u, "V") for u in range(U)]).reshape(s.B, s.Hkv, nb, s.P, s.D)
    cpu = np.full((U, s.k), -1, dtype=np.int32)
    cnt = np.zeros(U, dtype=np.int32)
    res_lists = []
    for u in range(U):
        b, kvh = divmod(u, s.Hkv)
        L = int(wl.seq_len[b])
        mn, mx = O.digest_minmax(Kb.reshape(U, nb * s.P, s.D)[u], L, s.P)
        qg = O.bf16_to_f64(wl.q[b, kvh * s.G:(kvh + 1) * s.G])
        S = O.select_topk(O.pool_group(O.scores_minmax(qg, mn, mx)), s.k)
        r, c = O.split_residency(S, wl.resident[u].astype(bool))
        cpu[u, :len(c)] = c
        cnt[u] = len(c)
        res_lists.append(np.asarray(r))
    return wl, Kb, Vb, cpu, cnt, res_lists


def _run(s, wl, Kb, Vb, cpu, cnt, n_threads=3):
    return bs.cpu_attend(_bf16(wl.q), _bf16(Kb), _bf16(Vb), torch.from_numpy(wl.seq_len.astype(np.int32)),
                         torch.from_numpy(cpu.reshape(s.B, s.Hkv, s.k)), torch.from_numpy(cnt.reshape(s.B, s.Hkv)),
                         s.B, s.Hq, s.Hkv, s.P, s.k, s.scale, n_threads=n_threads)


def _ref(s, wl, Kb, Vb, u, blocks):
    """The oracle's partial over the listed blocks, for each query head of unit u."""
    b, kvh = divmod(u, s.Hkv)
    L = int(wl.seq_len[b])
    K = O.bf16_to_f64(Kb[b, kvh].reshape(-1, s.D))
    V = O.bf16_to_f64(Vb[b, kvh].reshape(-1, s.D))
    toks = O.block_tokens(blocks, s.P, L)
    return [O.attention_partial(O.bf16_to_f64(wl.q[b, kvh * s.G + h]), K[toks], V[toks], s.scale)
            for h in range(s.G)]


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_cpu_partial_matches_oracle(name):
    s = SHAPES[name]
    wl, Kb, Vb, cpu, cnt, _ = _setup(s)
    O_cpu, L_cpu = _run(s, wl, Kb, Vb, cpu, cnt)
    O_cpu, L_cpu = O_cpu.numpy(), L_cpu.numpy()
    assert cnt.min() >= 0 and cnt.max() > 0
    for u in range(s.units):
        b, kvh = divmod(u, s.Hkv)
        for h, (o, l) in enumerate(_ref(s, wl, Kb, Vb, u, cpu[u, :cnt[u]])):
            check_fp32(O_cpu[b, kvh * s.G + h], L_cpu[b, kvh * s.G + h], o, l, what=(name, u, h))


@pytest.mark.parametrize("G", range(1, 9))
def test_tiled_and_scalar_forms_agree_within_the_fp32_bar(G):
    """The register-tiled form (the default) against the plain scalar loops, for every group
    size (each is its own tile shape, three tokens per tile with five or six heads, so the tile
    does not divide the page) and the three page sizes; both against the oracle as well."""
    P = (16, 32, 64)[G % 3]
    s = W.Shape(f"g{G}_p{P}", B=2, Hq=2 * G, Hkv=2, T=2500, P=P, k=2048 // P, resident_frac=0.25,
                seq_lens=(2500, 1111))
    wl, Kb, Vb, cpu, cnt, _ = _setup(s)
    args = (_bf16(wl.q), _bf16(Kb), _bf16(Vb), torch.from_numpy(wl.seq_len.astype(np.int32)),
            torch.from_numpy(cpu.reshape(s.B, s.Hkv, s.k)), torch.from_numpy(cnt.reshape(s.B, s.Hkv)),
            s.B, s.Hq, s.Hkv, s.P, s.k, s.scale)
    Ot, Lt = (x.numpy() for x in bs.cpu_attend(*args, n_threads=2))
    Os, Ls = (x.numpy() for x in bs.cpu_attend(*args, n_threads=2, scalar=True))
    assert cnt.max() > 0
    for u in range(s.units):
        b, kvh = divmod(u, s.Hkv)
        for h, (o, l) in enumerate(_ref(s, wl, Kb, Vb, u, cpu[u, :cnt[u]])):
            hq = kvh * s.G + h
            check_fp32(Ot[b, hq], Lt[b, hq], o, l, what=("tiled", u, h))
            check_fp32(Os[b, hq], Ls[b, hq], o, l, what=("scalar", u, h))
            check_fp32(Ot[b, hq], Lt[b, hq], Os[b, hq].astype(np.float64), float(Ls[b, hq]), what=("pair", u, h))


def test_split_merged_with_the_resident_partial_is_the_selection():
    """The CPU partial over S minus R, merged by LSE with the partial over S and R, equals
    attention over the whole selected set S (the merge of section 3.2)."""
    s = SHAPES["g5_p32"]
    wl, Kb, Vb, cpu, cnt, res_lists = _setup(s)
    O_cpu, L_cpu = (x.numpy() for x in _run(s, wl, Kb, Vb, cpu, cnt))
    for u in range(s.units):
        b, kvh = divmod(u, s.Hkv)
        whole = np.sort(np.concatenate([res_lists[u], cpu[u, :cnt[u]]]))
        for h, ((o_r, l_r), (o_s, l_s)) in enumerate(zip(_ref(s, wl, Kb, Vb, u, res_lists[u]),
                                                         _ref(s, wl, Kb, Vb, u, whole))):
            hq = kvh * s.G + h
            o, l = O.merge(O_cpu[b, hq].astype(np.float64), float(L_cpu[b, hq]), o_r, l_r)
            check_attention(o, l, o_s, l_s, what=(u, h))


def test_every_block_listed_is_dense_attention():
    """k = every block, all of them on the CPU: plain softmax attention over the sequence."""
    s = W.Shape("dense", B=1, Hq=8, Hkv=2, T=1000, P=32, k=32, resident_frac=0.0, seq_lens=(1000,))
    wl = W.Workload(s)
    Kb = np.stack([wl.unit_kv(u) for u in range(s.units)]).reshape(s.B, s.Hkv, s.nblk, s.P, s.D)
    Vb = np.stack([wl.unit_kv(u, "V") for u in range(s.units)]).reshape(s.B, s.Hkv, s.nblk, s.P, s.D)
    cpu = np.tile(np.arange(s.nblk, dtype=np.int32), (s.units, 1))
    cnt = np.full(s.units, s.nblk, dtype=np.int32)
    O_cpu, L_cpu = (x.numpy() for x in _run(s, wl, Kb, Vb, cpu, cnt))
    for u in range(s.units):
        kvh = u % s.Hkv
        K = O.bf16_to_f64(Kb[0, kvh].reshape(-1, s.D))[:1000]
        V = O.bf16_to_f64(Vb[0, kvh].reshape(-1, s.D))[:1000]
        for h in range(s.G):
            q = O.bf16_to_f64(wl.q[0, kvh * s.G + h])
            sc = s.scale * (K @ q)
            w = np.exp(sc - sc.max())
            check_fp32(O_cpu[0, kvh * s.G + h], L_cpu[0, kvh * s.G + h], (w @ V) / w.sum(),
                       sc.max() + np.log(w.sum()), what=h)


def test_empty_lists_blocks_past_the_end_and_thread_counts():
    """An empty list gives (0, -inf); a listed block with no token yet is skipped; the result
    does not depend on the number of threads (each unit is one thread's, in list order)."""
    s = SHAPES["g4_p64"]
    wl, Kb, Vb, cpu, cnt, _ = _setup(s)
    cnt[1] = 0
    u = 2 * s.Hkv  # a unit of the shortest sequence: add its last (empty) block to the list
    past = s.nblk - 1
    assert past * s.P >= wl.seq_len[2] and cnt[u] < s.k
    cpu[u, cnt[u]] = past
    cnt[u] += 1
    runs = [tuple(x.numpy() for x in _run(s, wl, Kb, Vb, cpu, cnt, n_threads=n)) for n in (1, 0, 7)]
    for o, l in runs[1:]:
        assert np.array_equal(o, runs[0][0]) and np.array_equal(l, runs[0][1])
    O_cpu, L_cpu = runs[0]
    b1, kvh1 = divmod(1, s.Hkv)
    assert np.all(L_cpu[b1, kvh1 * s.G:(kvh1 + 1) * s.G] == -np.inf)
    assert np.all(O_cpu[b1, kvh1 * s.G:(kvh1 + 1) * s.G] == 0)
    b, kvh = divmod(u, s.Hkv)
    for h, (o, l) in enumerate(_ref(s, wl, Kb, Vb, u, cpu[u, :cnt[u] - 1])):
        check_fp32(O_cpu[b, kvh * s.G + h], L_cpu[b, kvh * s.G + h], o, l, what=h)


def test_bad_arguments_are_rejected_before_anything_is_written():
    L = bs.lib()
    B, Hq, Hkv, D, P, nb, k = 1, 4, 2, 128, 32, 4, 2
    q = np.zeros((B, Hq, D), np.uint16)
    K = np.zeros((B, Hkv, nb, P, D), np.uint16)
    seq = np.array([100], np.int32)
    lst = np.zeros((B, Hkv, k), np.int32)
    cnt = np.ones((B, Hkv), np.int32)
    Oc = np.full((B, Hq, D), 7.0, np.float32)
    Lc = np.full((B, Hq), 7.0, np.float32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731

    def call(**kw):
        a = dict(q=p(q), K=p(K), V=p(K), seq=p(seq), lst=p(lst), cnt=p(cnt), B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, nb=nb,
                 k=k, scale=0.1, O=p(Oc), L=p(Lc), nt=2)
        a.update(kw)
        return L.scout_cpu_attend(a["q"], a["K"], a["V"], a["seq"], a["lst"], a["cnt"], a["B"], a["Hq"], a["Hkv"],
                                  a["D"], a["P"], a["nb"], a["k"], ctypes.c_float(a["scale"]), a["O"], a["L"], a["nt"])

    assert call(q=None) == 1
    assert call(Hq=5) == 1          # not a multiple of Hkv
    assert call(Hq=18) == 1         # 9 query heads per KV head
    assert call(scale=0.0) == 1
    assert call(D=64) == 2
    assert call(P=8) == 2
    cnt[0, 1] = k + 1
    assert call() == 1              # a count above k
    cnt[0, 1] = 1
    lst[0, 0, 0] = nb
    assert call() == 1              # a block outside the table
    assert np.all(Oc == 7.0) and np.all(Lc == 7.0)
    lst[0, 0, 0] = 0
    assert call() == 0
    assert np.all(np.isfinite(Lc))


def _random_job(B=4, Hq=40, Hkv=8, nb=96, P=32, k=64, seed=3):
    """Host inputs of a larger job (no oracle: the pool is compared with the synchronous call)."""
    rng = np.random.default_rng(seed)
    bf = lambda a: _bf16((a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16))  # noqa: E731
    q = bf(rng.standard_normal((B, Hq, 128)))
    K = bf(rng.standard_normal((B, Hkv, nb, P, 128)))
    V = bf(rng.standard_normal((B, Hkv, nb, P, 128)))
    seq = torch.full((B,), nb * P - 5, dtype=torch.int32)
    lists = np.sort(np.stack([rng.choice(nb, size=k, replace=False) for _ in range(B * Hkv)]), axis=-1)
    cnt = torch.from_numpy(rng.integers(k // 2, k + 1, size=(B, Hkv)).astype(np.int32))
    return q, K, V, seq, torch.from_numpy(lists.astype(np.int32).reshape(B, Hkv, k)), cnt, (B, Hq, Hkv, P, k)


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_pool_gives_the_synchronous_results_bit_for_bit(name):
    """scout_cpu_attend_async on a caller-owned pool computes exactly what scout_cpu_attend does."""
    s = SHAPES[name]
    wl, Kb, Vb, cpu, cnt, _ = _setup(s)
    O_ref, L_ref = _run(s, wl, Kb, Vb, cpu, cnt)
    with bs.CpuPool(3) as pool:
        assert pool.threads == 3
        for _ in range(2):  # the pool takes job after job
            O_p = torch.full_like(O_ref, 7.0)
            L_p = torch.full_like(L_ref, 7.0)
            pool.submit(_bf16(wl.q), _bf16(Kb), _bf16(Vb), torch.from_numpy(wl.seq_len.astype(np.int32)),
                        torch.from_numpy(cpu.reshape(s.B, s.Hkv, s.k)), torch.from_numpy(cnt.reshape(s.B, s.Hkv)),
                        s.B, s.Hq, s.Hkv, s.P, s.k, s.scale, O_p, L_p)
            assert pool.wait(60.0)
            assert torch.equal(O_p, O_ref) and torch.equal(L_p, L_ref)


def test_late_cpu_partial_is_a_timeout_not_a_stall():
    """A CPU partial that is not ready within the caller's bound comes back as SCOUT_ERR_TIMEOUT
    (the pipeline's signal that the CPU side is late); the job goes on, a second submission is
    refused meanwhile, and a later wait finds the results exact."""
    q, K, V, seq, lists, cnt, (B, Hq, Hkv, P, k) = _random_job()
    O_ref, L_ref = bs.cpu_attend(q, K, V, seq, lists, cnt, B, Hq, Hkv, P, k, 0.088, n_threads=2)
    pool = bs.CpuPool(1)  # one worker: the job takes tens of milliseconds
    O_p, L_p = torch.zeros_like(O_ref), torch.zeros_like(L_ref)
    pool.submit(q, K, V, seq, lists, cnt, B, Hq, Hkv, P, k, 0.088, O_p, L_p)
    L = bs.lib()
    assert L.scout_cpu_pool_wait(pool._p, 0) == 5  # SCOUT_ERR_TIMEOUT
    with pytest.raises(bs.ScoutError, match="INVALID_ARG"):
        pool.submit(q, K, V, seq, lists, cnt, B, Hq, Hkv, P, k, 0.088, O_p, L_p)
    assert pool.wait(120.0)
    assert torch.equal(O_p, O_ref) and torch.equal(L_p, L_ref)
    assert L.scout_cpu_pool_wait(pool._p, -1) == 1  # a negative bound is refused
    # closing the pool while a job runs waits for it
    pool.submit(q, K, V, seq, lists, cnt, B, Hq, Hkv, P, k, 0.088, O_p, L_p)
    pool.close()
    assert torch.equal(O_p, O_ref)
