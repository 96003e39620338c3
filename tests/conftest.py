import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
for _p in (ROOT, TESTS):
    if _p not in sys.path:
        sys.path.insert(0, _p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


@pytest.fixture(params=["chunked", "sequential", "sequential-1run", "sequential-chain3"])
def scan_mode(request):
    """Runs a GPU test once per scan strategy of wkv_forward / wkv_backward
    (forced through the library's test hooks; back to automatic after):
    the chunked scan, the sequential walk with its runs per column chosen by
    the library, the sequential walk with one run per column, and the
    sequential forward as chained runs of 3 chunks."""
    from rwkv_linear_attention_backward_b300 import binding

    binding.set_scan_mode(request.param.split("-")[0])
    binding.set_max_runs(1 if request.param.endswith("1run") else 0)
    binding.set_chain_len(3 if request.param.endswith("chain3") else 0)
    yield request.param
    binding.set_scan_mode("auto")
    binding.set_max_runs(0)
    binding.set_chain_len(0)


@pytest.fixture(scope="session")
def oracle():
    import oracle as _oracle

    return _oracle.load()


def pytest_sessionfinish(session, exitstatus):
    """Every parity comparison of the run (both gates' numbers), written as
    JSON to the file named by WKV_PARITY_LOG when it is set."""
    import json

    path = os.environ.get("WKV_PARITY_LOG")
    if not path:
        return
    try:
        from parity import PARITY_LOG
    except ImportError:
        return
    if PARITY_LOG:
        with open(path, "w") as f:
            json.dump(PARITY_LOG, f, indent=0)
