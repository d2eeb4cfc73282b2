import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session", autouse=True)
def index_checks_clean():
    """With TV_DEBUG_CHECKS=1 (set by tests/test_zx_debug_checks.py for the
    session it runs on the index-checked build): after the whole session, no
    index check of the library may have failed."""
    yield
    if os.environ.get("TV_DEBUG_CHECKS") != "1":
        return
    import tree_speculative_decoding_build_gb300 as tv
    assert tv.tv_debug_checks_enabled(), "TV_DEBUG_CHECKS=1 but the release library is loaded"
    n, where, line = tv.tv_debug_check_failures()
    assert n == 0, f"{n} failed index checks, the first in {where} line {line}"
