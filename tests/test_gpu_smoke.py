"""The round-end smoke call (the tiny pipeline through the library, plain and
with every store fused, against the oracle) stays green."""
import os
import sys

import pytest

pytestmark = pytest.mark.gpu


def test_smoke():
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import __graft_entry__
    __graft_entry__.smoke()
