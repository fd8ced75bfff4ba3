"""The C-ABI library loads, exports every declared entry point, and rejects bad
arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

import block_sparse_kv_pred_gb300 as bs
from block_sparse_kv_pred_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(bs.lib_path()):
        B.build()
    return bs.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "scout.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(scout_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version(L):
    for code in range(6):
        assert L.scout_status_string(code).decode().startswith("SCOUT_")
    assert L.scout_status_string(99) == b"unknown scout status"
    assert L.scout_version() == 10000


def test_workspace_sizes(L):
    assert L.scout_score_topk_workspace_bytes(40, 8, 1024) == 1280
    assert L.scout_score_topk_workspace_bytes(0, 8, 1024) == 0
    assert L.scout_sparse_attn_workspace_bytes(40, 40, 8, 128, 32) > 1024 * 2 * 8 * 128 * 4


def test_host_validation_rejects_without_launch(L):
    # null pointers, bad shapes and unsupported sizes come back before any CUDA call
    fake = ctypes.c_void_p(4096)
    assert L.scout_merge(None, None, None, None, 4, 128, None, None, None) == 1
    assert L.scout_merge(fake, fake, fake, fake, 4, 64, fake, fake, None) == 2  # D != 128
    assert L.scout_predict_q(fake, fake, fake, 8, 100, 64, None, None, None) == 2  # N % 128
    assert L.scout_predict_q(fake, fake, fake, 0, 128, 64, None, None, None) == 1
    assert L.scout_predict_q(fake, fake, fake, 257, 128, 64, None, None, None) == 2  # M > 256
    assert L.scout_build_digest(0, fake, 10, fake, fake, 1, 1, 128, 48, 4, None, 0, fake, None, None) == 2  # P
    assert L.scout_build_digest(7, fake, 10, fake, fake, 1, 1, 128, 32, 4, None, 0, fake, None, None) == 1  # kind
    args = [0, fake, fake, fake, fake, None, None, 1, 18, 2, 128, 32, 64, 8, None] + [fake] * 8 + [fake, 1 << 20, None,
                                                                                                   None, None]
    assert L.scout_score_topk(*args) == 2  # G = 9 > 8
    args[7:10] = [1, 8, 2]
    args[-4] = 16
    assert L.scout_score_topk(*args) == 3  # workspace too small
    args[5] = fake  # prev list without prev count
    assert L.scout_score_topk(*args) == 1
    assert L.scout_sparse_attn(fake, fake, fake, 100, fake, fake, fake, fake, 1, 8, 2, 128, 32, 8, 4, 0.0, fake,
                               fake, fake, 1 << 24, None, None, None) == 1  # scale <= 0
    assert L.scout_sparse_attn(fake, ctypes.c_void_p(4097), fake, 100, fake, fake, fake, fake, 1, 8, 2, 128, 32, 8,
                               4, 0.1, fake, fake, fake, 1 << 24, None, None, None) == 2  # misaligned pool
    assert L.scout_sparse_attn(fake, fake, fake, 100, fake, fake, fake, fake, 1, 8, 2, 128, 32, 8, (1 << 27) + 1,
                               0.1, fake, fake, fake, 1 << 24, None, None, None) == 2  # B Hkv k > 2^28 entries
    assert L.scout_sparse_attn(fake, fake, fake, 100, fake, fake, fake, fake, 2049, 8, 2, 128, 32, 8, 4, 0.1, fake,
                               fake, fake, 1 << 30, None, None, None) == 2  # B Hkv = 4098 units > 4096
    neg = ctypes.pointer(bs.Launch(-1))
    assert L.scout_predict_q(fake, fake, fake, 8, 128, 64, None, neg, None) == 1  # max_ctas < 0
    assert L.scout_sparse_attn_merge(fake, fake, fake, 100, fake, fake, fake, fake, 1, 8, 2, 128, 32, 8, 4, 0.1,
                                     None, fake, fake, fake, fake, 1 << 24, None, None, None) == 1  # no O_cpu
    assert L.scout_sparse_attn_merge(fake, fake, fake, 100, fake, fake, fake, fake, 1, 8, 2, 128, 32, 8, 4, 0.1,
                                     fake, fake, fake, fake, fake, 1 << 24, None, neg, None) == 1  # max_ctas < 0
    ops = (bs.RecallOp * 1)(bs.RecallOp(0, 5, 3, -1))
    assert L.scout_recall_async(ops, 1, fake, fake, fake, fake, 2, 1, 1, 128, 32, 8, None, None, None,
                                None) == 1  # slot 3 >= 2
    assert L.scout_recall_gather_async(fake, 1, fake, fake, fake, fake, 2, 1, 1, 128, 48, 8, None, None, None, None,
                                       None) == 2  # P = 48
    bad = ctypes.pointer(bs.Launch(0, 0, None, bs.INJECT_ABANDON))  # not an injection the recall knows
    assert L.scout_recall_gather_async(fake, 1, fake, fake, fake, fake, 2, 1, 1, 128, 32, 8, None, bad, None, None,
                                       None) == 1


def test_generator_library_exports():
    import block_sparse_kv_pred_gb300.workload.device as WD

    if not os.path.exists(os.path.join(os.path.dirname(bs.lib_path()), "libscoutgen.so")):
        B.build()
    L = WD.gen_lib()
    assert hasattr(L, "scoutgen_fill_normal_bf16") and hasattr(L, "scoutgen_fill_pool_bf16")


def test_launch_options_layout_and_step_checks():
    """scout_launch as the binding lays it out (two ints, then the event handle), an event that
    does not exist yet refused, and the step's early-start options checked before any device work."""
    assert ctypes.sizeof(bs.Launch) == 24 and bs.Launch.early_event.offset == 8 and bs.Launch.inject.offset == 16
    lp = bs._launch(0, early_event=0x1234)
    assert (lp.contents.max_ctas, lp.contents.pdl, lp.contents.early_event) == (0, 0, 0x1234)
    assert bs._launch(None, pdl=True).contents.pdl == 1
    assert bs._launch(None) is None

    class Uncreated:  # a torch.cuda.Event before its first record
        cuda_event = 0

    with pytest.raises(bs.ScoutError):
        bs._launch(0, early_event=Uncreated())
    from block_sparse_kv_pred_gb300 import workload as W
    from block_sparse_kv_pred_gb300.step import setup_step

    with pytest.raises(ValueError, match="serial"):
        setup_step(W.tiny(), "cpu", pdl=True)
    with pytest.raises(ValueError, match="early starters"):
        setup_step(W.tiny(), "cpu", early=("build_digest",))


def test_packed_step_buffers_are_aligned_and_disjoint():
    """The step's per-parity input and output sets are views of one byte buffer each (one copy
    moves a set): every view starts on a 256-byte boundary (TMA needs 16), has its shape and
    dtype, and no two views overlap."""
    import torch

    from block_sparse_kv_pred_gb300.step import packed

    specs = [("X", (40, 5120), torch.bfloat16), ("lse", (40, 40), torch.float32), ("cnt", (3, 5), torch.int32),
             ("q", (40, 40, 128), torch.bfloat16)]
    buf, views = packed(specs, "cpu")
    base = buf.data_ptr()
    spans = []
    for name, shape, dtype in specs:
        v = views[name]
        assert v.shape == shape and v.dtype == dtype and v.is_contiguous()
        off = v.data_ptr() - base
        assert off % 256 == 0
        spans.append((off, off + v.numel() * v.element_size()))
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:])) and spans[-1][1] <= buf.numel()
    for i, (name, _, _) in enumerate(specs):
        views[name].fill_(i + 1)
    for i, (name, _, _) in enumerate(specs):
        assert torch.all(views[name] == i + 1)
