import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload; minutes of device or host time")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


def pytest_terminal_summary(terminalreporter):
    # The largest oracle error of each full-size workload run on the GPU.
    mod = sys.modules.get("test_configs_gpu")
    errors = getattr(mod, "MAX_ERRORS", None)
    if errors:
        terminalreporter.write_sep("-", "max |C - C_ref| / (|alpha| sum|a||b| + |beta||c_old|)")
        for key, err in errors.items():
            terminalreporter.write_line("%-60s %.3g" % (key, err))
