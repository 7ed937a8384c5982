import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload checks")


@pytest.fixture(scope="session")
def golden():
    import json
    with open(os.path.join(ROOT, "tests", "golden", "hand_worked.json")) as f:
        return json.load(f)


def pytest_terminal_summary(terminalreporter):
    """The largest relative L2 error each test measured (parity margins)."""
    from tests import _util
    per = {}
    for test, val in _util.MEASURED:
        per[test] = max(per.get(test, 0.0), val)
    if not per:
        return
    terminalreporter.write_sep("-", "largest relative L2 error measured, per test")
    for test in sorted(per):
        terminalreporter.write_line(f"{per[test]:.3e}  {test}")
    path = os.environ.get("HH_ERROR_REPORT")
    if path:
        with open(path, "w") as f:
            json.dump(per, f, indent=1, sort_keys=True)

