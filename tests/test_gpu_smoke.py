"""The entry point's smoke check (one small forward + backward against the
oracle, with the feature set of the windowed GQA workload) as part of the GPU
suite."""

import os
import sys

import pytest

pytestmark = pytest.mark.gpu

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def test_smoke_entry_point():
    import __graft_entry__

    __graft_entry__.smoke()
