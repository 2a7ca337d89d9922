import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for _p in (ROOT, os.path.dirname(os.path.abspath(__file__))):
    if _p not in sys.path:
        sys.path.insert(0, _p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def uly():
    """The CUDA library binding, built in-tree if needed."""
    import long_context_sequence_head_gb300 as m
    from long_context_sequence_head_gb300 import build as b
    b.build(debug=m.debug_build_selected())
    m.load()
    # tests bound every device-side wait to 250 ms so a broken pipeline fails fast
    m.ulysses_set_wait_limit_ns(250_000_000)
    return m
