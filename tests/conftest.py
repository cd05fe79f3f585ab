import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large shapes; still part of the default run")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    return oracle.load()


@pytest.fixture(autouse=True)
def _debug_build_index_checks(request):
    """Under GQA_ATTN_DEBUG=1 (the debug build of the library, with device-side index checks),
    every GPU test must end with no failed index check in the device status word."""
    yield
    if os.environ.get("GQA_ATTN_DEBUG", "") != "1" or request.node.get_closest_marker("gpu") is None:
        return
    import causal_gqa_attention_gb300 as cga

    status = cga.device_status()
    assert not status & cga.ATTN_DEV_INDEX_CHECK, f"index check failed (status {status:#x})"
