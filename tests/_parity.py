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
