import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped (not failed) when no GPU is visible; on a machine with one the
    # library must load, and a missing library is a test failure.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device visible")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(autouse=True)
def _tensor_core_path_for_gpu_tests(request):
    """GPU tests drive the tensor-core decode kernel at every size: small bf16 calls would
    otherwise go to the CUDA-core kernel (tests/test_gpu_small_path.py covers that one and
    sets the limit itself)."""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    try:
        from mla_latent_kv_split_gb300 import binding as mb
        old = mb.mla_decode_set_small_call_limit(0)
    except Exception:  # library not built yet: the test's own fixtures build it
        yield
        return
    try:
        yield
    finally:
        mb.mla_decode_set_small_call_limit(old)
