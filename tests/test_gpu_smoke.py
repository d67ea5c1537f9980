"""The driver's smoke entry point (one small forward on cuda:0 against the oracle) runs clean."""
import os
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_smoke_entry_point(capsys):
    sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__.smoke()
    assert "smoke ok" in capsys.readouterr().out
