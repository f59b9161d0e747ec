import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the kernels)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def _device_error_word_clean(request):
    """After every GPU test, the library's sticky device error word of the default
    workspace must be clear: a kernel that flagged a timed-out wait or a bad index (and
    carried on) fails the test even when its outputs happened to match."""
    yield
    if "gpu" not in request.keywords:
        return
    import torch
    if not torch.cuda.is_available():
        return
    pkg = sys.modules.get("retrieval_sparse_attention_causal_gb300")
    if pkg is None or not getattr(pkg, "_default_ws", None):
        return
    for key in list(pkg._default_ws):
        pkg._default_ws[key].check()
