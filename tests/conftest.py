import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long CPU test (exhaustive sweeps)")


def read_table(name):
    """Rows of a '|'-separated golden table, comments skipped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c.strip() for c in line.split("|")])
    return rows


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    from oracle.build import build
    build()
    return oracle


def pytest_addoption(parser):
    parser.addoption("--runslow", action="store_true", default=False,
                     help="also run the exhaustive sweeps marked slow")


def pytest_collection_modifyitems(config, items):
    if config.getoption("--runslow") or os.environ.get("KIVI_RUNSLOW") == "1":
        return
    skip = pytest.mark.skip(reason="exhaustive sweep: run with --runslow")
    for item in items:
        if "slow" in item.keywords:
            item.add_marker(skip)
