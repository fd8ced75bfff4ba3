"""bench.py's CPU-side leg (scout_cpu_attend on the host cores) on host tensors shaped as the
step's: it gathers each unit's blocks from the pool into logical order, counts the K/V bytes of
the listed blocks' valid tokens, and reports a failure instead of raising."""
import numpy as np
import torch

import bench
import oracle as O
from block_sparse_kv_pred_gb300 import workload as W
from _parity import ensure_built


def _step_like(s, rng):
    """Host stand-ins for the step's tensors: a permuted pool, Q_pred, the CPU work list."""
    wl = W.Workload(s)
    U, nb = s.units, s.nblk
    K = np.stack([wl.unit_kv(u) for u in range(U)]).reshape(U * nb, s.P, s.D)
    V = np.stack([wl.unit_kv(u, "V") for u in range(U)]).reshape(U * nb, s.P, s.D)
    perm = rng.permutation(U * nb)  # slot of logical block i is perm[i]
    K_pool, V_pool = np.empty_like(K), np.empty_like(V)
    K_pool[perm], V_pool[perm] = K, V
    cpu = np.full((s.B, s.Hkv, s.k), -1, np.int32)
    cnt = np.zeros((s.B, s.Hkv), np.int32)
    for u in range(U):
        b, kvh = divmod(u, s.Hkv)
        c = np.sort(rng.choice(nb, size=int(rng.integers(0, s.k + 1)), replace=False))
        cpu[b, kvh, :len(c)] = c
        cnt[b, kvh] = len(c)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)  # noqa: E731
    t = {"K_pool": bf(K_pool), "V_pool": bf(V_pool),
         "page_table": torch.from_numpy(perm.astype(np.int32).reshape(s.B, s.Hkv, nb)),
         "Qp1": bf(wl.q.reshape(s.B, s.Hq * s.D)), "cpu1": torch.from_numpy(cpu), "cpu_count1": torch.from_numpy(cnt),
         "seq_len": torch.from_numpy(wl.seq_len.astype(np.int32))}
    return wl, t, cpu, cnt


def test_cpu_side_leg_reports_throughput_and_bytes():
    ensure_built()
    s = W.Shape("side", B=3, Hq=8, Hkv=2, T=1500, P=32, k=10, resident_frac=0.0, seq_lens=(1500, 777, 64))
    wl, t, cpu, cnt = _step_like(s, np.random.default_rng(5))
    r = bench.cpu_side(s, t, seconds=0.05, max_seqs=2)
    assert "unavailable" not in r, r
    tokens = sum(len(O.block_tokens(cpu[b, h, :cnt[b, h]], s.P, int(wl.seq_len[b]))) for b in range(2)
                 for h in range(s.Hkv))
    assert r["kv_bytes_per_call"] == tokens * s.D * 2 * 2
    assert r["value"] > 0 and r["threads"] >= 1 and r["unit"] == "GB/s"
    assert "2 of 3 sequences" in r["sample"]


def test_cpu_side_leg_reports_a_failure_instead_of_raising():
    s = W.Shape("side", B=1, Hq=8, Hkv=2, T=256, P=32, k=4, resident_frac=0.0)
    wl, t, _, _ = _step_like(s, np.random.default_rng(6))
    t["page_table"][0, 0, 0] = -1
    assert "unavailable" in bench.cpu_side(s, t)
    del t["Qp1"]
    t["page_table"][0, 0, 0] = 0
    assert "KeyError" in bench.cpu_side(s, t)["unavailable"]
