"""Python binding of libscout (block-sparse decode attention for GB300, sm_103a).

Argument marshalling only: every entry point forwards device pointers of torch
tensors, sizes and the current CUDA stream to the C ABI declared in
``include/scout.h``; all arithmetic runs in the library's CUDA kernels.  There is
no fallback: if ``libscout.so`` is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "ScoutError", "lib", "MINMAX", "MEAN", "predict_q", "build_digest", "score_topk", "score_topk_workspace",
    "sparse_attn", "sparse_attn_merge", "sparse_attn_workspace", "merge", "recall_async", "commit_residency",
    "plan_recall", "plan_recall_pages", "recall_intervals", "cpu_attend", "RecallOp", "Launch", "Prepared",
    "INJECT_NONE", "INJECT_ABANDON", "INJECT_COPY_FAIL", "recall_gather_async", "CpuPool", "resident_list",
    "POOL_SUM",
]

MINMAX = 0
MEAN = 1
POOL_SUM = 0x10  # OR-ed into the kind: the group's scores summed instead of their maximum
_KIND = {"minmax": MINMAX, "mean": MEAN, MINMAX: MINMAX, MEAN: MEAN}

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB = None

_p = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_f = ctypes.c_float
_sz = ctypes.c_size_t


class ScoutError(RuntimeError):
    pass


class RecallOp(ctypes.Structure):
    _fields_ = [("unit", ctypes.c_int32), ("block", ctypes.c_int32), ("slot", ctypes.c_int32),
                ("evict_block", ctypes.c_int32)]


_SIGS = {
    "scout_status_string": ([_i], ctypes.c_char_p),
    "scout_version": ([], _i),
    "scout_predict_q": ([_p, _p, _p, _i, _i, _i, _p, _p, _p], _i),
    "scout_build_digest": ([_i, _p, _i64, _p, _p, _i, _i, _i, _i, _i, _p, _i, _p, _p, _p], _i),
    "scout_score_topk_workspace_bytes": ([_i, _i, _i], _sz),
    "scout_score_topk": ([_i, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _p,
                          _p, _p, _sz, _p, _p, _p], _i),
    "scout_score_topk_noalloc_max_bytes": ([], _sz),
    "scout_score_topk_noalloc": ([_i, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p,
                                  _p, _p, _p, _p], _i),
    "scout_sparse_attn_workspace_bytes": ([_i, _i, _i, _i, _i], _sz),
    "scout_sparse_attn": ([_p, _p, _p, _i64, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _p, _p, _p, _sz, _p,
                           _p, _p], _i),
    "scout_sparse_attn_merge": ([_p, _p, _p, _i64, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _p, _p, _p, _p,
                                 _p, _sz, _p, _p, _p], _i),
    "scout_merge": ([_p, _p, _p, _p, _i, _i, _p, _p, _p], _i),
    "scout_recall_async": ([_p, _i, _p, _p, _p, _p, _i64, _i, _i, _i, _i, _i, _p, _p, _p, _p], _i),
    "scout_recall_gather_async": ([_p, _i, _p, _p, _p, _p, _i64, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p], _i),
    "scout_commit_residency": ([_p, _i, _p, _p, _i64, _i, _i, _i, _p, _p], _i),
    "scout_plan_recall": ([_p, _p, _p, _p, _p, _i, _i, _i, _p, _i, _p], _i),
    "scout_cpu_attend": ([_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _p, _p, _i], _i),
    "scout_cpu_attend_scalar": ([_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _p, _p, _i], _i),
    "scout_recall_intervals": ([_p, _i, _i, _f, _p], _i),
    "scout_resident_list": ([_p, _p, _i, _i, _i, _i, _i, _p, _p, _p, _p], _i),
    "scout_cpu_pool_create": ([_i], _p),
    "scout_cpu_pool_threads": ([_p], _i),
    "scout_cpu_pool_destroy": ([_p], None),
    "scout_cpu_attend_async": ([_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _p, _p], _i),
    "scout_cpu_pool_wait": ([_p, _i64], _i),
    "scout_plan_recall_pages": ([_p, _p, _p, _p, _p, _i, _i, _i, _i, _p, _i, _p], _i),
}


class Launch(ctypes.Structure):
    """scout_launch: launch options of the persistent kernels.  max_ctas 0 = one CTA per SM;
    pdl 1 = start early after the previous kernel on the stream; early_event = a
    cudaEvent_t (timing disabled) this launch records programmatically, so that one of the
    three persistent kernels on a stream waiting for it may start early; inject = a
    SCOUT_INJECT_* fault for tests (0 in normal use)."""
    _fields_ = [("max_ctas", ctypes.c_int), ("pdl", ctypes.c_int), ("early_event", ctypes.c_void_p),
                ("inject", ctypes.c_int)]


INJECT_NONE = 0
INJECT_ABANDON = 1
INJECT_COPY_FAIL = 2


def _launch(max_ctas, pdl=False, early_event=None, inject=INJECT_NONE):
    """Launch options, or None for the defaults.  ``early_event``: a torch.cuda.Event created
    without timing and already recorded once (so that it exists), or a raw handle."""
    if max_ctas is None and not pdl and early_event is None and not inject:
        return None
    if max_ctas is not None and max_ctas < 0:
        raise ScoutError("max_ctas must be >= 0")
    if early_event is not None and not isinstance(early_event, int):
        if not early_event.cuda_event:
            raise ScoutError("early_event has not been created yet: record it once first")
        early_event = early_event.cuda_event
    return ctypes.pointer(Launch(int(max_ctas or 0), int(bool(pdl)), early_event, int(inject)))


def lib_path() -> str:
    return os.path.join(_PKG, "libscout.so")


def lib():
    """The loaded libscout (raises ScoutError when it is not built)."""
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise ScoutError(f"{path} is missing: run `python -m block_sparse_kv_pred_gb300.build`")
        L = ctypes.CDLL(path)
        for name, (args, res) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = L
    return _LIB


def _check(rc: int, what: str):
    if rc != 0:
        raise ScoutError(f"{what}: {lib().scout_status_string(rc).decode()}")


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _dev(t: torch.Tensor, dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ScoutError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ScoutError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ScoutError(f"{name} must be contiguous")
    return t.data_ptr()


def _opt(t, dtype, name):
    return None if t is None else _dev(t, dtype, name)


# ---------------------------------------------------------------------------
def predict_q(X: torch.Tensor, W: torch.Tensor, Q: torch.Tensor | None = None, status=None, max_ctas=None,
              stream=None) -> torch.Tensor:
    """Q_pred = X W^T (bf16 in, fp32 accumulate, bf16 out)."""
    M, K = X.shape
    N = W.shape[0]
    if Q is None:
        Q = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    _check(lib().scout_predict_q(_dev(X, torch.bfloat16, "X"), _dev(W, torch.bfloat16, "W"),
                                 _dev(Q, torch.bfloat16, "Q"), M, N, K, _opt(status, torch.int32, "status"),
                                 _launch(max_ctas), _stream(stream)), "scout_predict_q")
    return Q


def build_digest(kind, K_pool, page_table, seq_len, B, Hkv, P, digest, block_list=None, status=None,
                 stream=None):
    kind = _KIND[kind]
    nblk_cap = page_table.shape[-1]
    n_slots = K_pool.shape[0]
    ddt = torch.bfloat16 if kind == MINMAX else torch.float32
    n_list = 0 if block_list is None else block_list.shape[0]
    _check(lib().scout_build_digest(kind, _dev(K_pool, torch.bfloat16, "K_pool"), n_slots,
                                    _dev(page_table, torch.int32, "page_table"), _dev(seq_len, torch.int32, "seq_len"),
                                    B, Hkv, K_pool.shape[-1], P, nblk_cap, _opt(block_list, torch.int32, "block_list"),
                                    n_list, _dev(digest, ddt, "digest"), _opt(status, torch.int32, "status"),
                                    _stream(stream)), "scout_build_digest")
    return digest


def score_topk_workspace(B, Hkv, nblk_cap, device="cuda") -> torch.Tensor:
    n = lib().scout_score_topk_workspace_bytes(B, Hkv, nblk_cap)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def score_topk(kind, q, digest, seq_len, resident_bits, B, Hq, Hkv, P, nblk_cap, k, workspace, out=None,
               prev_cpu=None, scores=None, status=None, max_ctas=None, inject=INJECT_NONE, pool="max",
               stream=None) -> dict:
    """Score digests, select top-k per unit, split by residency.

    ``out`` (optional) is a dict of preallocated outputs with the keys returned.
    ``prev_cpu`` is an optional (list, count) pair from the previous step.
    ``status`` (optional int32 device tensor) receives SCOUT_DEV_TIMEOUT (2) if a bounded wait
    expired.  ``inject`` is a test hook (INJECT_ABANDON).  ``pool``: "max" (the group's scores
    pooled by their maximum) or "sum".
    """
    kind = _KIND[kind]
    if pool not in ("max", "sum"):
        raise ScoutError(f"pool must be 'max' or 'sum', got {pool!r}")
    dev = q.device
    U = B * Hkv
    if out is None:
        out = {}
        for name in ("topk", "res", "cpu", "delta"):
            out[name] = torch.empty((B, Hkv, k), dtype=torch.int32, device=dev)
            out[name + "_count"] = torch.empty((B, Hkv), dtype=torch.int32, device=dev)
    pl, pc = (None, None) if prev_cpu is None else prev_cpu
    ddt = torch.bfloat16 if kind == MINMAX else torch.float32
    _check(lib().scout_score_topk(
        kind | (POOL_SUM if pool == "sum" else 0), _dev(q, torch.bfloat16, "q"), _dev(digest, ddt, "digest"), _dev(seq_len, torch.int32, "seq_len"),
        _dev(resident_bits, torch.int32, "resident_bits"), _opt(pl, torch.int32, "prev_cpu_list"),
        _opt(pc, torch.int32, "prev_cpu_count"), B, Hq, Hkv, q.shape[-1], P, nblk_cap, k,
        _opt(scores, torch.float32, "scores"),
        _dev(out["topk"], torch.int32, "topk"), _dev(out["topk_count"], torch.int32, "topk_count"),
        _dev(out["res"], torch.int32, "res"), _dev(out["res_count"], torch.int32, "res_count"),
        _dev(out["cpu"], torch.int32, "cpu"), _dev(out["cpu_count"], torch.int32, "cpu_count"),
        _dev(out["delta"], torch.int32, "delta"), _dev(out["delta_count"], torch.int32, "delta_count"),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _opt(status, torch.int32, "status"),
        _launch(max_ctas, inject=inject), _stream(stream)), "scout_score_topk")
    if scores is not None:
        out["scores"] = scores
    del U
    return out


def resident_list(resident_bits, seq_len, B, Hkv, P, nblk_cap, cap, out=None, status=None, stream=None):
    """Every valid resident block of each unit, ascending -> (list int32 [B][Hkv][cap], count
    int32 [B][Hkv]); the GPU's blocks under the "all resident blocks" reading."""
    dev = resident_bits.device
    lst, cnt = out if out is not None else (torch.empty((B, Hkv, cap), dtype=torch.int32, device=dev),
                                            torch.empty((B, Hkv), dtype=torch.int32, device=dev))
    _check(lib().scout_resident_list(_dev(resident_bits, torch.int32, "resident_bits"),
                                     _dev(seq_len, torch.int32, "seq_len"), B, Hkv, P, nblk_cap, cap,
                                     _dev(lst, torch.int32, "list"), _dev(cnt, torch.int32, "count"),
                                     _opt(status, torch.int32, "status"), _stream(stream)), "scout_resident_list")
    return lst, cnt


def sparse_attn_workspace(B, Hq, Hkv, P, D=128, device="cuda") -> torch.Tensor:
    n = lib().scout_sparse_attn_workspace_bytes(B, Hq, Hkv, D, P)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def sparse_attn(q, K_pool, V_pool, page_table, seq_len, res_list, res_count, B, Hq, Hkv, P, k, scale, workspace,
                O=None, lse=None, status=None, max_ctas=None, stream=None):
    """GPU partial attention over the resident selected blocks -> (O fp32 [B][Hq][D], lse fp32 [B][Hq])."""
    D = q.shape[-1]
    if O is None:
        O = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _check(lib().scout_sparse_attn(
        _dev(q, torch.bfloat16, "q"), _dev(K_pool, torch.bfloat16, "K_pool"), _dev(V_pool, torch.bfloat16, "V_pool"),
        K_pool.shape[0], _dev(page_table, torch.int32, "page_table"), _dev(seq_len, torch.int32, "seq_len"),
        _dev(res_list, torch.int32, "res_list"), _dev(res_count, torch.int32, "res_count"), B, Hq, Hkv, D, P,
        page_table.shape[-1], k, float(scale), _dev(O, torch.float32, "O"), _dev(lse, torch.float32, "lse"),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _opt(status, torch.int32, "status"),
        _launch(max_ctas), _stream(stream)), "scout_sparse_attn")
    return O, lse


def sparse_attn_merge(q, K_pool, V_pool, page_table, seq_len, res_list, res_count, B, Hq, Hkv, P, k, scale,
                      workspace, O_cpu, lse_cpu, O_out=None, lse_out=None, status=None, max_ctas=None,
                      stream=None):
    """GPU partial attention merged with the CPU partial -> (O bf16 [B][Hq][D], lse fp32 [B][Hq])."""
    D = q.shape[-1]
    if O_out is None:
        O_out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    if lse_out is None:
        lse_out = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _check(lib().scout_sparse_attn_merge(
        _dev(q, torch.bfloat16, "q"), _dev(K_pool, torch.bfloat16, "K_pool"), _dev(V_pool, torch.bfloat16, "V_pool"),
        K_pool.shape[0], _dev(page_table, torch.int32, "page_table"), _dev(seq_len, torch.int32, "seq_len"),
        _dev(res_list, torch.int32, "res_list"), _dev(res_count, torch.int32, "res_count"), B, Hq, Hkv, D, P,
        page_table.shape[-1], k, float(scale), _dev(O_cpu, torch.float32, "O_cpu"),
        _dev(lse_cpu, torch.float32, "lse_cpu"), _dev(O_out, torch.bfloat16, "O_out"),
        _dev(lse_out, torch.float32, "lse_out"), _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        _opt(status, torch.int32, "status"), _launch(max_ctas), _stream(stream)), "scout_sparse_attn_merge")
    return O_out, lse_out


def merge(O_a, lse_a, O_b, lse_b, O_out=None, lse_out=None, stream=None):
    """LSE merge of two partials -> (O bf16, lse fp32)."""
    D = O_a.shape[-1]
    rows = O_a.numel() // D
    if O_out is None:
        O_out = torch.empty(O_a.shape, dtype=torch.bfloat16, device=O_a.device)
    if lse_out is None:
        lse_out = torch.empty(lse_a.shape, dtype=torch.float32, device=O_a.device)
    _check(lib().scout_merge(_dev(O_a, torch.float32, "O_a"), _dev(lse_a, torch.float32, "lse_a"),
                             _dev(O_b, torch.float32, "O_b"), _dev(lse_b, torch.float32, "lse_b"), rows, D,
                             _dev(O_out, torch.bfloat16, "O_out"), _dev(lse_out, torch.float32, "lse_out"),
                             _stream(stream)), "scout_merge")
    return O_out, lse_out


def recall_async(ops, host_K, host_V, K_pool, V_pool, B, Hkv, P, nblk_cap, side_stream, wait_event=None,
                 done_event=None, inject=INJECT_NONE):
    """Queue host->pool copies of recalled blocks on side_stream (one cudaMemcpyAsync per run of
    consecutive blocks and slots). ``ops``: list of (unit, block, slot, evict)."""
    arr = (RecallOp * max(1, len(ops)))(*[RecallOp(*o) for o in ops])
    for t, n in ((host_K, "host_K"), (host_V, "host_V")):
        if t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ScoutError(f"{n} must be a contiguous bf16 host tensor")
    _check(lib().scout_recall_async(arr, len(ops), host_K.data_ptr(), host_V.data_ptr(),
                                    _dev(K_pool, torch.bfloat16, "K_pool"), _dev(V_pool, torch.bfloat16, "V_pool"),
                                    K_pool.shape[0], B, Hkv, K_pool.shape[-1], P, nblk_cap, _launch(None, inject=inject),
                                    None if wait_event is None else wait_event.cuda_event, side_stream.cuda_stream,
                                    None if done_event is None else done_event.cuda_event), "scout_recall_async")


def recall_gather_async(d_ops, host_K, host_V, K_pool, V_pool, B, Hkv, P, nblk_cap, side_stream, wait_event=None,
                        done_event=None, status=None, inject=INJECT_NONE):
    """Move the recalled blocks with one gather kernel on side_stream that reads them straight from
    pinned, mapped host memory.  ``d_ops``: device int32 [n][4] (unit, block, slot, evict)."""
    for t, n in ((host_K, "host_K"), (host_V, "host_V")):
        if t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16 or not t.is_pinned():
            raise ScoutError(f"{n} must be a contiguous, pinned bf16 host tensor")
    n = 0 if d_ops is None else d_ops.shape[0]
    _check(lib().scout_recall_gather_async(
        _opt(d_ops, torch.int32, "ops"), n, host_K.data_ptr(), host_V.data_ptr(), _dev(K_pool, torch.bfloat16, "K_pool"),
        _dev(V_pool, torch.bfloat16, "V_pool"), K_pool.shape[0], B, Hkv, K_pool.shape[-1], P, nblk_cap,
        _opt(status, torch.int32, "status"), _launch(None, inject=inject),
        None if wait_event is None else wait_event.cuda_event, side_stream.cuda_stream,
        None if done_event is None else done_event.cuda_event), "scout_recall_gather_async")


def commit_residency(d_ops, page_table, resident_bits, n_slots, B, Hkv, wait_event=None, stream=None):
    """Apply recall ops (device int32 [n][4]) to the page table and residency bits after wait_event."""
    n = 0 if d_ops is None else d_ops.shape[0]
    _check(lib().scout_commit_residency(_opt(d_ops, torch.int32, "ops"), n, _dev(page_table, torch.int32, "page_table"),
                                        _dev(resident_bits, torch.int32, "resident_bits"), n_slots, B, Hkv,
                                        page_table.shape[-1], None if wait_event is None else wait_event.cuda_event,
                                        _stream(stream)), "scout_commit_residency")


def _check_plan_shapes(sc, ti, tc, rb, pt, units, nblk, k):
    """The host planners read these arrays by (units, nblk_cap, k): refuse any other shape."""
    words = -(-nblk // 32)
    if sc.size != units * nblk or sc.shape[0] != units:
        raise ScoutError(f"scores must be [{units}][{nblk}], got {sc.shape}")
    if ti.size != units * k or ti.shape[-1] != k:
        raise ScoutError(f"topk_idx must be [{units}][{k}], got {ti.shape}")
    if tc.size != units:
        raise ScoutError(f"topk_count must hold {units} counts, got {tc.shape}")
    if rb.size != units * words or rb.shape[-1] != words:
        raise ScoutError(f"resident_bits must be [{units}][{words}], got {rb.shape}")
    if pt.size != units * nblk or pt.shape[-1] != nblk:
        raise ScoutError(f"page_table must be [{units}][{nblk}], got {pt.shape}")


def plan_recall(scores, topk_idx, topk_count, resident_bits, page_table, k):
    """Recall ops (unit, block, slot, evicted block) for one recall step, planned on the host.

    All arguments are host numpy arrays: scores fp32 [units][nblk_cap], topk_idx int32
    [units][k], topk_count int32 [units], resident_bits uint32 [units][words], page_table
    int32 [units][nblk_cap].  Returns an int32 array [n][4].
    """
    import numpy as np

    sc = np.ascontiguousarray(scores, dtype=np.float32)
    ti = np.ascontiguousarray(topk_idx, dtype=np.int32)
    tc = np.ascontiguousarray(topk_count, dtype=np.int32)
    rb = np.ascontiguousarray(resident_bits, dtype=np.uint32)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    units, nblk = sc.shape
    _check_plan_shapes(sc, ti, tc, rb, pt, units, nblk, k)
    cap = max(1, int(tc.clip(0, k).sum()))
    ops = (RecallOp * cap)()
    n = ctypes.c_int(0)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    _check(lib().scout_plan_recall(ptr(sc), ptr(ti), ptr(tc), ptr(rb), ptr(pt), units, nblk, k, ops, cap,
                                   ctypes.byref(n)), "scout_plan_recall")
    return np.array([[o.unit, o.block, o.slot, o.evict_block] for o in ops[: n.value]], dtype=np.int32).reshape(-1, 4)


def plan_recall_pages(scores, topk_idx, topk_count, resident_bits, page_table, B, Hkv, k):
    """Recall ops with residency per page (one block of a sequence for all its KV heads).

    Host arrays as for plan_recall (units = B * Hkv; the residency bits of a sequence's heads
    must be identical).  Returns int32 [n][4] (unit, block in, slot, block out): one op per KV
    head and page pair, grouped by unit, ascending block in."""
    import numpy as np

    sc = np.ascontiguousarray(scores, dtype=np.float32)
    ti = np.ascontiguousarray(topk_idx, dtype=np.int32)
    tc = np.ascontiguousarray(topk_count, dtype=np.int32)
    rb = np.ascontiguousarray(resident_bits, dtype=np.uint32)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    nblk = sc.shape[-1]
    _check_plan_shapes(sc.reshape(-1, nblk), ti, tc, rb, pt, B * Hkv, nblk, k)
    cap = max(1, int(tc.clip(0, k).sum()) * Hkv)
    ops = (RecallOp * cap)()
    n = ctypes.c_int(0)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    _check(lib().scout_plan_recall_pages(ptr(sc), ptr(ti), ptr(tc), ptr(rb), ptr(pt), B, Hkv, nblk, k, ops, cap,
                                         ctypes.byref(n)), "scout_plan_recall_pages")
    return np.array([[o.unit, o.block, o.slot, o.evict_block] for o in ops[: n.value]], dtype=np.int32).reshape(-1, 4)


def recall_intervals(ratio, beta=0.12):
    """Per-layer recall intervals (section 3.4) from CPU-compute-ratio traces.

    ``ratio``: host array [layers][steps], layer l's ratio at the (s+1)-th decoding step after
    a refresh, from a profiling run without recalls.  Returns int32 [layers]: the largest number
    of leading steps whose ratio is below ``beta``, at least 1 and at most ``steps``."""
    import numpy as np

    r = np.ascontiguousarray(ratio, dtype=np.float32)
    if r.ndim != 2:
        raise ScoutError("ratio must be [layers][steps]")
    out = np.zeros(r.shape[0], dtype=np.int32)
    _check(lib().scout_recall_intervals(r.ctypes.data_as(ctypes.c_void_p), r.shape[0], r.shape[1], float(beta),
                                        out.ctypes.data_as(ctypes.c_void_p)), "scout_recall_intervals")
    return out


def _host(t, dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ScoutError(f"{name} must be a host tensor")
    if t.dtype != dtype:
        raise ScoutError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ScoutError(f"{name} must be contiguous")
    return t.data_ptr()


def cpu_attend(q, K, V, seq_len, cpu_list, cpu_count, B, Hq, Hkv, P, k, scale, O_cpu=None, lse_cpu=None,
               n_threads=0, scalar=False):
    """CPU-side attention over the CPU work list, on the host cores (synchronous).

    Host tensors: q bf16 [B][Hq][D]; K, V bf16 [B][Hkv][nblk_cap][P][D] (every block of the
    layer in logical order); seq_len int32 [B]; cpu_list int32 [B][Hkv][k] and cpu_count
    int32 [B][Hkv] as scout_score_topk writes them.  Returns (O_cpu fp32 [B][Hq][D],
    lse_cpu fp32 [B][Hq]), the partial that scout_merge / scout_sparse_attn_merge take.
    The foreign call releases the GIL, so other Python threads run meanwhile.  ``scalar``: the
    plain-loop form (scout_cpu_attend_scalar) instead of the register-tiled one."""
    D = q.shape[-1]
    per_block = B * Hkv * P * D
    if K.numel() != V.numel() or K.numel() % per_block:
        raise ScoutError("K and V must hold [B][Hkv][nblk_cap][P][D] elements")
    nblk_cap = K.numel() // per_block
    if O_cpu is None:
        O_cpu = torch.empty((B, Hq, D), dtype=torch.float32)
    if lse_cpu is None:
        lse_cpu = torch.empty((B, Hq), dtype=torch.float32)
    fn = lib().scout_cpu_attend_scalar if scalar else lib().scout_cpu_attend
    _check(fn(_host(q, torch.bfloat16, "q"), _host(K, torch.bfloat16, "K"), _host(V, torch.bfloat16, "V"),
              _host(seq_len, torch.int32, "seq_len"), _host(cpu_list, torch.int32, "cpu_list"),
              _host(cpu_count, torch.int32, "cpu_count"), B, Hq, Hkv, D, P, nblk_cap, k, float(scale),
              _host(O_cpu, torch.float32, "O_cpu"), _host(lse_cpu, torch.float32, "lse_cpu"), int(n_threads)),
           "scout_cpu_attend_scalar" if scalar else "scout_cpu_attend")
    return O_cpu, lse_cpu


class CpuPool:
    """A caller-owned pool of CPU worker threads (scout_cpu_pool): ``submit`` starts the CPU-side
    attention of one layer and returns at once; ``wait(timeout_s)`` returns True when it is done
    and False when it is still running after the timeout (a late CPU partial).  ``close`` (or
    leaving a ``with`` block) waits for a running job and joins the workers."""

    def __init__(self, n_threads: int = 0):
        self._p = lib().scout_cpu_pool_create(int(n_threads))
        if not self._p:
            raise ScoutError("scout_cpu_pool_create: no worker thread could be started")
        self.threads = lib().scout_cpu_pool_threads(self._p)
        self._keep = ()

    def submit(self, q, K, V, seq_len, cpu_list, cpu_count, B, Hq, Hkv, P, k, scale, O_cpu, lse_cpu):
        """Host tensors as for ``cpu_attend``; O_cpu / lse_cpu are written when the job is done."""
        if not self._p:
            raise ScoutError("the pool is closed")
        D = q.shape[-1]
        per_block = B * Hkv * P * D
        if K.numel() != V.numel() or K.numel() % per_block:
            raise ScoutError("K and V must hold [B][Hkv][nblk_cap][P][D] elements")
        nblk_cap = K.numel() // per_block
        args = (_host(q, torch.bfloat16, "q"), _host(K, torch.bfloat16, "K"), _host(V, torch.bfloat16, "V"),
                _host(seq_len, torch.int32, "seq_len"), _host(cpu_list, torch.int32, "cpu_list"),
                _host(cpu_count, torch.int32, "cpu_count"))
        outs = (_host(O_cpu, torch.float32, "O_cpu"), _host(lse_cpu, torch.float32, "lse_cpu"))
        _check(lib().scout_cpu_attend_async(self._p, *args, B, Hq, Hkv, D, P, nblk_cap, k, float(scale), *outs),
               "scout_cpu_attend_async")
        self._keep = (q, K, V, seq_len, cpu_list, cpu_count, O_cpu, lse_cpu)  # alive until the job is done

    def wait(self, timeout_s: float) -> bool:
        rc = lib().scout_cpu_pool_wait(self._p, max(0, int(timeout_s * 1e6)))
        if rc == 5:
            return False
        _check(rc, "scout_cpu_pool_wait")
        return True

    def close(self):
        if self._p:
            lib().scout_cpu_pool_destroy(self._p)
            self._p = None
            self._keep = ()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001  (interpreter shutdown)
            pass


class Prepared:
    """One C-ABI call with its arguments converted once; calling it re-issues the call.

    Used by timing loops so that per-step host work is a single foreign call.
    Buffers named by the arguments must outlive the object.
    """

    def __init__(self, name: str, *args):
        self.name = name
        self.fn = getattr(lib(), name)
        self.args = tuple(args)

    def __call__(self):
        rc = self.fn(*self.args)
        if rc != 0:
            raise ScoutError(f"{self.name}: {lib().scout_status_string(rc).decode()}")
