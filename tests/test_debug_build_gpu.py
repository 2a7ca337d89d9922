"""The bounds-checked debug build of the library (-DULY_DEBUG): every
raw-pointer global access of the swap and attention kernels is checked
against its buffer, and a failed check is reported as ULY_ERR_BOUNDS
instead of being made.  The attention and swap parity suites run again in a
child process that loads this build: every case must match the oracle as
before and no check may fire.  The reporting path itself is exercised by a
self-test whose check is handed an offset past its extent (no memory is
touched)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ULY_ERR_BOUNDS = 9


def test_bounds_selftest_reports(uly):
    if not uly.debug_build_selected():
        pytest.skip("runs in the child process that loads the debug build")
    assert uly.ulysses_selftest_bounds() == 0
    st, site = uly.ulysses_get_device_status()
    assert st == ULY_ERR_BOUNDS and site == 0x8000 | 0x7F, (st, hex(site))
    assert uly.ulysses_get_device_status()[0] == 0  # cleared


def test_parity_suites_under_the_debug_build(uly):
    if uly.debug_build_selected():
        pytest.skip("already inside the debug-build process")
    from long_context_sequence_head_gb300 import build as b
    b.build(debug=True)
    env = dict(os.environ, ULY_DEBUG_BUILD="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_attn_gpu.py", "tests/test_swap_gpu.py", "tests/test_fused_seq_gpu.py",
           "tests/test_debug_build_gpu.py::test_bounds_selftest_reports"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "failed" not in r.stdout, r.stdout[-2000:]
