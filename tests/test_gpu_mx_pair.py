"""The MXFP8 Mgemm's CTA-pair comparison build (RG_MX_PAIR=1: 256 x 256
tiles with the block-scaled tcgen05.mma.cta_group::2, every CTA of a pair
holding the B scales of all 256 columns) gives the oracle's results, with
the debug-bounds checks on and the status word clean."""
import os
import subprocess
import sys

import pytest

from moe_grouped_gemm_device_gb300 import _build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_mx_pair_build_matches_the_oracle():
    lib = _build.build(extra_flags=("-DRG_MX_PAIR=1", "-DRG_DEBUG_BOUNDS=1"),
                       out_dir=os.path.join(_build.OUT_DIR, "mx_pair"))
    r = subprocess.run([sys.executable, os.path.join(HERE, "mx_pair_cases.py"), lib],
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "ALL OK" in r.stdout
