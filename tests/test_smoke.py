"""The entry point's own smoke check (one small forward and backward on
cuda:0, compared with the oracle) runs as a GPU test too."""
import pytest

pytestmark = pytest.mark.gpu


def test_graft_entry_smoke():
    import __graft_entry__
    __graft_entry__.smoke()
