import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def _checked_library_loaded():
    lib = os.environ.get("FMHA_GB300_LIB")
    return bool(lib) and os.path.basename(lib) == "libfmha_gb300_checked.so"


@pytest.fixture(autouse=True)
def _index_checks_clean(request):
    """Under the checked build (FMHA_GB300_LIB names libfmha_gb300_checked.so),
    every GPU test ends by reading the device status word, so a failed index
    check in any kernel it ran fails the test with the check's site."""
    yield
    if "gpu" not in request.keywords or not _checked_library_loaded():
        return
    from head_attention_forward_fmha_gb300 import binding
    assert binding.fmha_build_flags() == binding.FMHA_BUILD_CHECKED, "FMHA_GB300_LIB did not load the checked build"
    binding.fmha_check_device_status()
