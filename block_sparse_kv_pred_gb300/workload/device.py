"""Device-resident copies of a :class:`Workload`, filled by libscoutgen.so.

The device generator uses the same counter-based definition as the host one,
so ``Workload.unit_kv(u)`` equals the pool pages of unit u bit for bit.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import STREAM_K, STREAM_V, STREAM_W, STREAM_X, Workload

_GEN = None


def gen_lib():
    global _GEN
    if _GEN is None:
        path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "libscoutgen.so")
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run `python -m block_sparse_kv_pred_gb300.build`")
        L = ctypes.CDLL(path)
        p, i, i64, u64, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
        L.scoutgen_fill_normal_bf16.argtypes = [p, i64, u64, u64, f, i64, p]
        L.scoutgen_fill_normal_bf16.restype = i
        L.scoutgen_fill_pool_bf16.argtypes = [p, i64, i, i, p, i, u64, u64, p, p, p, p]
        L.scoutgen_fill_pool_bf16.restype = i
        _GEN = L
    return _GEN


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def fill_normal(t: torch.Tensor, seed: int, stream_id: int, sigma: float = 1.0, offset: int = 0):
    assert t.dtype == torch.bfloat16 and t.is_contiguous()
    rc = gen_lib().scoutgen_fill_normal_bf16(t.data_ptr(), t.numel(), seed, stream_id, sigma, offset, _stream())
    if rc:
        raise RuntimeError(f"scoutgen_fill_normal_bf16 failed ({rc})")
    return t


def to_dev(a: np.ndarray, device) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).to(device)
    return torch.from_numpy(a).to(device)


def materialize(wl: Workload, device="cuda", with_gemm: bool = True) -> dict:
    """All device inputs of one decode step (pool holds every block of every unit)."""
    s = wl.s
    dev = torch.device(device)
    out = {}
    out["q"] = to_dev(wl.q, dev)
    out["seq_len"] = to_dev(wl.seq_len, dev)
    out["page_table"] = to_dev(wl.page_table.reshape(s.B, s.Hkv, s.nblk), dev)
    out["resident_bits"] = to_dev(wl.resident_bits(), dev)
    owner = to_dev(wl.slot_owner, dev)
    chan = to_dev(wl.chan_scale, dev)
    heavy = to_dev(wl.heavy, dev)
    hdir = to_dev(wl.hdir, dev)
    for name, sid, hv in (("K_pool", STREAM_K, True), ("V_pool", STREAM_V, False)):
        pool = torch.empty((wl.n_slots, s.P, s.D), dtype=torch.bfloat16, device=dev)
        rc = gen_lib().scoutgen_fill_pool_bf16(pool.data_ptr(), wl.n_slots, s.P, s.D, owner.data_ptr(), s.nblk,
                                               s.seed, sid, chan.data_ptr(), heavy.data_ptr() if hv else None,
                                               hdir.data_ptr() if hv else None, _stream())
        if rc:
            raise RuntimeError(f"scoutgen_fill_pool_bf16 failed ({rc})")
        out[name] = pool
    if with_gemm and s.hidden:
        out["X"] = fill_normal(torch.empty((s.B, s.hidden), dtype=torch.bfloat16, device=dev), s.seed, STREAM_X)
        out["W"] = fill_normal(torch.empty((s.Hq * s.D, s.hidden), dtype=torch.bfloat16, device=dev), s.seed,
                               STREAM_W, s.w_sigma)
    o, lse = wl.cpu_partial()
    out["O_cpu"] = to_dev(o, dev)
    out["lse_cpu"] = to_dev(lse, dev)
    return out


def materialize_pool(wl: Workload, keep: np.ndarray, device="cuda", seed_offset: int = 7919):
    """A K/V pool holding only the blocks marked in ``keep`` (bool [units][nblk]), each in a slot of
    a seeded permutation, as a GPU holding part of the cache keeps them.  Returns (K_pool, V_pool,
    page_table int32 [B][Hkv][nblk] with -1 for blocks without a slot, n_slots); the pages equal
    ``Workload.unit_kv`` bit for bit."""
    s = wl.s
    dev = torch.device(device)
    idx = np.flatnonzero(np.asarray(keep, dtype=bool).reshape(-1)).astype(np.int32)  # u * nblk + j
    n = int(idx.size)
    if n == 0:
        raise ValueError("the pool would hold no block")
    perm = np.random.Generator(np.random.PCG64(s.seed + seed_offset)).permutation(n).astype(np.int32)
    owner = np.empty(n, dtype=np.int32)
    owner[perm] = idx  # slot perm[i] holds block idx[i]
    table = np.full(s.units * s.nblk, -1, dtype=np.int32)
    table[idx] = perm
    d_owner = to_dev(owner, dev)
    chan = to_dev(wl.chan_scale, dev)
    heavy = to_dev(wl.heavy, dev)
    hdir = to_dev(wl.hdir, dev)
    pools = []
    for sid, hv in ((STREAM_K, True), (STREAM_V, False)):
        pool = torch.empty((n, s.P, s.D), dtype=torch.bfloat16, device=dev)
        rc = gen_lib().scoutgen_fill_pool_bf16(pool.data_ptr(), n, s.P, s.D, d_owner.data_ptr(), s.nblk, s.seed, sid,
                                               chan.data_ptr(), heavy.data_ptr() if hv else None,
                                               hdir.data_ptr() if hv else None, _stream())
        if rc:
            raise RuntimeError(f"scoutgen_fill_pool_bf16 failed ({rc})")
        pools.append(pool)
    return pools[0], pools[1], to_dev(table.reshape(s.B, s.Hkv, s.nblk), dev), n
