import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def load_builder():
    """cascaded_reductions_gb300/_build.py loaded by path (the package's
    __init__ needs the library it builds)."""
    import importlib.util
    path = os.path.join(ROOT, "cascaded_reductions_gb300", "_build.py")
    spec = importlib.util.spec_from_file_location("rf_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def pytest_sessionstart(session):
    # nvcc is present wherever the tests run; a no-op when librf.so is current
    load_builder().build()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    # GPU tests cannot run without a device; make that explicit instead of
    # letting them fail on a CPU-only machine.
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def _no_refused_index(request):
    """Under the bounds-checked library (RF_LIBRARY names it), every GPU test
    must also leave no refused index behind in rf_device_error."""
    yield
    if "gpu" not in request.keywords or not os.environ.get("RF_LIBRARY"):
        return
    import torch
    if not torch.cuda.is_available():
        return
    import cascaded_reductions_gb300 as rf
    if rf.rf_bounds_checked():
        status = rf.rf_device_error()
        assert status == rf.RF_OK, f"device status {status} after the test (6 = RF_ERR_BOUNDS)"
