import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes)")


def pytest_collection_modifyitems(config, items):
    # GPU tests cannot run without a device; make that an explicit skip rather
    # than a failure when someone runs the whole suite on a CPU-only machine.
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def moe_gpu():
    """Build the library, initialise it on cuda:0 and return (module, device)."""
    import torch

    import moe_expert_layer_softmax_gb300 as m
    from moe_expert_layer_softmax_gb300 import _build

    _build.build()
    torch.cuda.set_device(0)
    m.init(0)
    return m, torch.device("cuda", 0)


@pytest.fixture(autouse=True)
def _checks_build_guards(request):
    """With MOE_GB300_CHECKS=1 (the checks build: device-side bounds checks and
    guard bands around every buffer of allocate()), every GPU test must leave
    the bounds-check words at zero and every guard band intact."""
    yield
    if os.environ.get("MOE_GB300_CHECKS", "") != "1" or "gpu" not in request.keywords:
        return
    import moe_expert_layer_softmax_gb300 as m
    flags = m.checks_read(reset=True)
    bad = m.check_canaries()
    assert flags == 0, f"bounds check words {flags:#x}"
    assert not bad, bad
