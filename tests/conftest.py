import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, TESTS):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload, tens of seconds")


@pytest.fixture(scope="session")
def golden():
    with open(os.path.join(TESTS, "golden", "crafted_cases.json")) as f:
        return json.load(f)


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle


def _gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def rp():
    """The product library's Python binding, on a GPU machine only."""
    if not _gpu_available():
        pytest.skip("no CUDA device")
    import verifiable_repops_gemm_gb300 as rp
    rp.load()
    return rp


@pytest.fixture(autouse=True)
def _no_pending_device_failure(request):
    """After every test that used the library on the GPU, its shared status
    word must be clear: no bounded wait gave up and -- when REPOPS_LIBRARY
    names the access-checking build -- no access fell outside its buffer.
    Tests that provoke a failure on purpose read (and so clear) it themselves."""
    yield
    if "rp" not in request.fixturenames or not _gpu_available():
        return
    import verifiable_repops_gemm_gb300 as lib
    from verifiable_repops_gemm_gb300 import _capi
    st = lib.device_status()
    assert st == 0, "device status %d (%s) left by the test" % (st, _capi.status_string(st))
