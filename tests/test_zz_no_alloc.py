"""The allocation-free selection entry point against the workspace one.

scout_score_topk_noalloc serves callers that cannot allocate device memory at
selection time (a fixed start-up memory pool, or a plugin host without an
allocator).  It must give exactly what scout_score_topk gives with a caller
workspace, call after call, although its scratch array keeps the previous
call's contents.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_sparse_kv_pred_gb300 as bs
from block_sparse_kv_pred_gb300 import workload as W
from block_sparse_kv_pred_gb300.workload import device as WD
from _parity import SCORE_REL, ensure_built

pytestmark = pytest.mark.gpu

CASES = [W.tiny(), W.Shape("noalloc_ragged", B=3, Hq=10, Hkv=2, T=5000, P=32, k=8, resident_frac=0.25,
                           seq_lens=(5000, 4097, 33)),
         W.Shape("noalloc_mean", B=2, Hq=8, Hkv=2, T=4100, P=16, k=20, resident_frac=0.25, kind="mean")]


def _outputs(s):
    o = {}
    for name in ("topk", "res", "cpu", "delta"):
        o[name] = torch.full((s.B, s.Hkv, s.k), -7, dtype=torch.int32, device="cuda")
        o[name + "_count"] = torch.full((s.B, s.Hkv), -7, dtype=torch.int32, device="cuda")
    o["scores"] = torch.zeros((s.B, s.Hkv, s.nblk), dtype=torch.float32, device="cuda")
    o["status"] = torch.zeros(1, dtype=torch.int32, device="cuda")
    return o


def _noalloc(s, d, dg, o, prev):
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    kind = bs.MINMAX if s.kind == "minmax" else bs.MEAN
    rc = bs.lib().scout_score_topk_noalloc(
        kind, p(d["q"]), p(dg), p(d["seq_len"]), p(d["resident_bits"]), p(prev[0]), p(prev[1]), s.B, s.Hq, s.Hkv,
        s.D, s.P, s.nblk, s.k, p(o["scores"]), p(o["topk"]), p(o["topk_count"]), p(o["res"]), p(o["res_count"]),
        p(o["cpu"]), p(o["cpu_count"]), p(o["delta"]), p(o["delta_count"]), p(o["status"]),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, bs.lib().scout_status_string(rc)


@pytest.mark.parametrize("s", CASES, ids=lambda s: s.name)
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(s):
    ensure_built()
    wl = W.Workload(s)
    d = WD.materialize(wl, with_gemm=False)
    if s.kind == "minmax":
        dg = torch.empty((s.B, s.Hkv, s.nblk, 2, s.D), dtype=torch.bfloat16, device="cuda")
    else:
        dg = torch.empty((s.B, s.Hkv, s.nblk, s.D), dtype=torch.float32, device="cuda")
    bs.build_digest(s.kind, d["K_pool"], d["page_table"], d["seq_len"], s.B, s.Hkv, s.P, dg)
    rng = np.random.default_rng(4)
    prev_l = torch.as_tensor(np.sort(rng.integers(0, 4, size=(s.B, s.Hkv, s.k)), axis=-1).astype(np.int32),
                             device="cuda")
    prev_c = torch.full((s.B, s.Hkv), min(2, s.k), dtype=torch.int32, device="cuda")
    ref = _outputs(s)
    ws = bs.score_topk_workspace(s.B, s.Hkv, s.nblk)
    bs.score_topk(s.kind, d["q"], dg, d["seq_len"], d["resident_bits"], s.B, s.Hq, s.Hkv, s.P, s.nblk, s.k, ws,
                  out=ref, prev_cpu=(prev_l, prev_c), scores=ref["scores"])
    torch.cuda.synchronize()
    for call in range(2):
        got = _outputs(s)
        _noalloc(s, d, dg, got, (prev_l, prev_c))
        torch.cuda.synchronize()
        assert int(got["status"].item()) == 0, call
        for key in ("topk", "res", "cpu", "delta", "topk_count", "res_count", "cpu_count", "delta_count"):
            assert torch.equal(got[key], ref[key]), (call, key)
        big = ref["scores"][torch.isfinite(ref["scores"])].abs().max()
        diff = (got["scores"] - ref["scores"]).nan_to_num(0.0).abs()
        assert torch.equal(torch.isinf(got["scores"]), torch.isinf(ref["scores"]))
        assert float(diff.max()) <= SCORE_REL * float(big), call


def test_noalloc_rejects_problems_beyond_its_fixed_scratch():
    ensure_built()
    L = bs.lib()
    cap = L.scout_score_topk_noalloc_max_bytes()
    assert cap == 4 << 20
    # 262,144 x 8 units need 8 MiB of counters: rejected before any launch
    fake = ctypes.c_void_p(256)
    args = [0, fake, fake, fake, fake, None, None, 262144, 40, 8, 128, 16, 64, 32] + [None] + [fake] * 8 + [None, None]
    assert L.scout_score_topk_noalloc(*args) == 3
    # 131,072 x 8 units (1,048,576) is the largest problem the array takes; one more sequence is not
    args[7] = 131073
    assert L.scout_score_topk_noalloc(*args) == 3
    # a bad argument is rejected before the shared array is touched (no stream work at all)
    args[7], args[0] = 4, 7
    assert L.scout_score_topk_noalloc(*args) == 1
