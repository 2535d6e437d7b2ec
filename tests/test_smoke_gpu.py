"""The smoke check (__graft_entry__.smoke: a small product on each path,
checked against the oracle) as a GPU test, so that a change in the dispatch
rules its shapes rely on fails here too (needs a GB300)."""
import os
import sys

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def test_smoke():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import __graft_entry__
    __graft_entry__.smoke()
