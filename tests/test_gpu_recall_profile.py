"""Section 3.4's offline recall-interval profile at the sweep shape (batch 16, 40/8 heads, 64K
context, k = 64 blocks held per KV head): seeded layers decode without recalls through the
library, and each layer's interval is the oracle's rule applied to its CPU compute ratio trace.
"""
import numpy as np
import pytest

import oracle as O
from block_sparse_kv_pred_gb300.sweep import profile_recall_intervals
from _parity import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_recall_interval_profile():
    traces, iv = profile_recall_intervals(2, 4, 0.12)
    assert traces.shape == (2, 4) and np.all((traces >= 0) & (traces <= 1))
    assert list(iv) == O.recall_intervals(traces.tolist(), np.float32(0.12))
