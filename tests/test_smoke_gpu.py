"""The package smoke check (one small forward + L2 + backward on cuda:0,
checked against the oracle) runs as a GPU test too."""
import pytest

pytestmark = pytest.mark.gpu


def test_smoke():
    import __graft_entry__
    __graft_entry__.smoke()
