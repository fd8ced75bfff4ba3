"""Helpers shared by the GPU parity tests: device inputs, oracle references, tolerances.

Tolerances (from the acceptance rules of this library):
  digests       min/max bit-exact; mean |gpu - oracle| <= 1e-6 |oracle| + 1e-6 * mean|K|
  scores        |gpu - oracle| <= 1e-4 * (largest |score| of the unit)
  selection     lists bit-exact; when the fp64 and fp32 rankings differ, only
                blocks within 1e-4 (relative) of the k-th score may differ
  attention     |gpu - oracle| <= 2e-3 + 1e-2 |oracle| for O and LSE
  Q_pred        ||gpu - oracle||_F <= 1e-2 ||oracle||_F
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle as O
import block_sparse_kv_pred_gb300 as bs
from block_sparse_kv_pred_gb300 import build as B

ATOL, RTOL = 2e-3, 1e-2
SCORE_REL = 1e-4


def ensure_built():
    if not (os.path.exists(bs.lib_path()) and os.path.exists(os.path.join(os.path.dirname(bs.lib_path()),
                                                                          "libscoutgen.so"))):
        B.build()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_dev(a, device="cuda"):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).to(device)
    return torch.from_numpy(a).to(device)


def pools_from_units(K_units, V_units, P, rng):
    """Paged pools [slots][P][D] from logical [U][nb*P][D] arrays, with a random page table."""
    U, Tp, D = K_units.shape
    nb = Tp // P
    perm = rng.permutation(U * nb).astype(np.int32)
    table = perm.reshape(U, nb)
    Kp = np.empty((U * nb, P, D), dtype=np.uint16)
    Vp = np.empty_like(Kp)
    Kr = K_units.reshape(U, nb, P, D)
    Vr = V_units.reshape(U, nb, P, D)
    Kp[table.ravel()] = Kr.reshape(U * nb, P, D)
    Vp[table.ravel()] = Vr.reshape(U * nb, P, D)
    return Kp, Vp, table


def bits_from_mask(mask: np.ndarray) -> np.ndarray:
    """uint32 [U][words] residency bitmap from a bool [U][nb] mask."""
    U, nb = mask.shape
    words = -(-nb // 32)
    out = np.zeros((U, words), dtype=np.uint32)
    for j in range(nb):
        out[:, j // 32] |= mask[:, j].astype(np.uint32) << np.uint32(j % 32)
    return out


def nvalid(seq_len: int, P: int) -> int:
    return -(-int(seq_len) // P)


def check_attention(o_gpu, l_gpu, o_ref, l_ref, what=""):
    if l_ref == -np.inf:
        assert l_gpu == -np.inf and np.all(o_gpu == 0), what
        return
    assert abs(l_gpu - l_ref) <= ATOL + RTOL * abs(l_ref), (what, l_gpu, l_ref)
    err = np.abs(o_gpu - o_ref) - (ATOL + RTOL * np.abs(o_ref))
    assert np.all(err <= 0), (what, float(np.max(np.abs(o_gpu - o_ref))))


def oracle_qpred(s):
    """The oracle's Q_pred of a step's synthetic layer in fp64 [B][Hq*D], from the seeded X and
    W_Q (the host side of the generator that filled the device buffers)."""
    from block_sparse_kv_pred_gb300 import workload as W

    X = W.normal_bf16(s.seed, W.STREAM_X, (s.B, s.hidden))
    Wq = W.normal_bf16(s.seed, W.STREAM_W, (s.Hq * s.D, s.hidden), s.w_sigma)
    return O.predict_q(X, Wq)


def check_qpred(got_bits, ref):
    """The Q_pred bar against the unrounded fp64 product: every entry within bf16 rounding
    (2^-8 relative) plus 1e-3 of the largest entry."""
    got = O.bf16_to_f64(got_bits)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-3 * np.abs(ref).max())


def check_selection(U_ref, k, S_gpu, what=""):
    """GPU top-k set equals the fp64 one except for blocks within SCORE_REL of the k-th score."""
    S_ref = O.select_topk(U_ref, k)
    a, b = set(S_ref.tolist()), set(int(x) for x in S_gpu)
    if a == b:
        return True
    kth = np.sort(U_ref)[::-1][min(k, len(U_ref)) - 1]
    for j in a ^ b:
        assert abs(U_ref[j] - kth) <= SCORE_REL * max(abs(kth), 1e-30), (what, j, U_ref[j], kth)
    return False


def check_topk_property(scores, S, k, nv, what=""):
    """Validity of a selection against its own scores: every member beats every non-member."""
    S = [int(x) for x in S]
    assert len(S) == min(k, nv) and S == sorted(S) and len(set(S)) == len(S), what
    sel = np.zeros(nv, bool)
    sel[S] = True
    if sel.all() or not sel.any():
        return
    worst_in = min(S, key=lambda j: (scores[j], -j))
    rest = np.nonzero(~sel)[0]
    best_out = max(rest, key=lambda j: (scores[j], -j))
    assert (scores[worst_in] > scores[best_out]) or (scores[worst_in] == scores[best_out] and worst_in < best_out), what


def _mask(lst, cnt, nb):
    """bool [U][nb]: the first cnt[u] entries of each list; raises on a duplicate or a bad entry."""
    U, k = lst.shape
    live = np.arange(k)[None, :] < cnt[:, None]
    assert np.all((lst[live] >= 0) & (lst[live] < nb)) and np.all(lst[~live] == -1)
    m = np.zeros((U, nb + 1), bool)
    m[np.arange(U)[:, None], np.where(live, lst, nb)] = True
    m = m[:, :nb]
    assert np.array_equal(m.sum(1), cnt)  # no entry twice
    return m


def check_list_algebra(s, rec, nb):
    """The lists of every unit of a sweep record: top-k count, each list ascending and without
    repeats, res and cpu the split of top-k by residency, delta = cpu minus the previous cpu."""
    U, k = s.units, s.k
    nvalid = -(-rec["seq"].astype(np.int64) // s.P)
    tc = rec["topk_count"]
    assert np.array_equal(tc, np.minimum(k, np.repeat(nvalid, s.Hkv)))
    for n in ("topk", "res", "cpu", "delta"):
        lst, c = rec[n], rec[n + "_count"]
        live = np.arange(k)[None, :] < c[:, None]
        d = np.diff(np.where(live, lst, np.iinfo(np.int32).max), axis=1)
        assert np.all(d[live[:, 1:]] > 0), n  # ascending
    T = _mask(rec["topk"], tc, nb)
    Rm = _mask(rec["res"], rec["res_count"], nb)
    Cm = _mask(rec["cpu"], rec["cpu_count"], nb)
    Dm = _mask(rec["delta"], rec["delta_count"], nb)
    assert np.array_equal(Rm | Cm, T) and not np.any(Rm & Cm)
    assert np.array_equal(Rm, T & rec["resident"]) and np.array_equal(Cm, T & ~rec["resident"])
    prev = np.zeros_like(Cm) if rec["prev_cpu"] is None else _mask(*rec["prev_cpu"], nb)
    assert np.array_equal(Dm, Cm & ~prev)
