import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a library)")


@pytest.fixture(autouse=True)
def _no_kernel_wait_timed_out(request):
    """After every GPU test: no kernel wait of the library ran out (the watchdog flag is
    clear).  A timed-out wait leaves outputs incomplete, so a test whose tolerances
    happened to hold would otherwise pass on them.  Tests that provoke a timeout on
    purpose read and clear the flag themselves."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    from top_kl_distill_gb300 import vloss
    if vloss._lib is None:            # the test never loaded the library
        return
    import torch
    if not torch.cuda.is_available():
        return
    flag = vloss.vl_watchdog_flag(torch.cuda.current_device(), True)
    assert flag == 0, f"a kernel wait timed out during this test (watchdog flag {flag})"
