"""The debug-bounds build on the GPU: every kernel's copy and store
coordinates are checked against their operands (RG_DEBUG_BOUNDS=1), on the
edge cases of grouping (empty, single-row, ragged and half-tile groups,
multi-chunk experts, narrow and one-stage tiles, outer groups, fused
epilogues, MXFP8).  Every case must leave the status word at 0 and give the
oracle's results.  Nothing is planted: the check logic itself is tested on
the host (test_bounds_host.py)."""
import os
import subprocess
import sys

import pytest

from moe_grouped_gemm_device_gb300 import _build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_bounds_build_runs_the_edge_cases_clean():
    lib = _build.build_bounds()
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_bounds_cases.py"), lib],
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "ALL OK" in r.stdout
