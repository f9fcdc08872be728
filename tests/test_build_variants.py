"""The single-CTA comparison build (RG_CTA_PAIR=0: tcgen05 MMAs of one CTA,
M=128, instead of CTA pairs) keeps compiling: every translation unit of the
library is compiled for sm_103a with that switch into a scratch directory.
No GPU is needed (nvcc cross-compiles); skipped where nvcc is missing."""
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

import pytest

from moe_grouped_gemm_device_gb300 import _build


def _nvcc():
    try:
        return _build.nvcc()
    except RuntimeError:
        return None


@pytest.mark.skipif(_nvcc() is None, reason="nvcc not available")
def test_single_cta_build_compiles(tmp_path):
    cc = _nvcc()

    def compile_one(src):
        cmd = [cc, *_build.ARCH, *_build.NVCC_FLAGS, "-DRG_CTA_PAIR=0", "-c",
               os.path.join(_build.CSRC, src), "-o", str(tmp_path / (src + ".o"))]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, r.returncode, r.stderr[-2000:]

    with ThreadPoolExecutor(len(_build.SOURCES)) as ex:
        results = list(ex.map(compile_one, _build.SOURCES))
    failed = [(s, err) for s, rc, err in results if rc != 0]
    assert not failed, failed
    shutil.rmtree(tmp_path, ignore_errors=True)
