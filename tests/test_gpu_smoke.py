"""The smoke entry point itself: one tiny decode step checked against the oracle."""
import os
import sys

import pytest

pytestmark = pytest.mark.gpu
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def test_smoke_entry_point():
    import __graft_entry__ as g

    g.smoke()
