"""The debug build's bounds check (include/nvfp4_testing.h) on the GPU: the
cases run in a child process (tests/bounds_debug_cases.py) that loads only
the debug library, so this process keeps the regular one."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_build_bounds_check():
    """Clean in every mode on ragged shapes, equal to the oracle, and firing
    (skipped stores, fill kept) on a range shortened by 16 bytes."""
    r = subprocess.run([sys.executable, os.path.join(HERE, "bounds_debug_cases.py")], capture_output=True,
                       text=True, timeout=1200, cwd=os.path.dirname(HERE))
    assert r.returncode == 0, (r.stdout[-4000:], r.stderr[-4000:])
    assert "bounds check: clean in every mode" in r.stdout
