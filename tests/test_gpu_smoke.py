"""The build entry point's smoke check (one small layer forward + backward on
cuda:0 against the oracle) runs as part of the GPU suite, so that a change to
the buffers or the binding cannot break it unnoticed.  GPU only."""
import pytest

pytestmark = pytest.mark.gpu


def test_graft_entry_smoke(moe_gpu):
    import __graft_entry__ as g
    g.smoke()
