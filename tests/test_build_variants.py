"""Comparison builds keep compiling: the single-CTA build (RG_CTA_PAIR=0:
tcgen05 MMAs of one CTA, M=128, instead of CTA pairs; every translation unit
of the library, compiled for sm_103a into a scratch directory), the MXFP8
weight gradient with 128-column tiles (RG_MXK_BN=128) and the MXFP8 Mgemm
with CTA pairs (RG_MX_PAIR=1).  No GPU is needed
(nvcc cross-compiles); skipped where nvcc is missing."""
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


@pytest.mark.skipif(_nvcc() is None, reason="nvcc not available")
def test_mx_wgrad_128_column_build_compiles(tmp_path):
    """The MXFP8 weight gradient's comparison build with 128-column tiles and
    two tensor-memory accumulators (RG_MXK_BN=128)."""
    cmd = [_nvcc(), *_build.ARCH, *_build.NVCC_FLAGS, "-DRG_MXK_BN=128", "-c",
           os.path.join(_build.CSRC, "mxgemm.cu"), "-o", str(tmp_path / "mxgemm.o")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]


@pytest.mark.skipif(_nvcc() is None, reason="nvcc not available")
def test_mx_pair_build_compiles(tmp_path):
    """The MXFP8 Mgemm's comparison build with CTA pairs (RG_MX_PAIR=1); the
    host side (tensor-map boxes, grid) is in api.cu."""
    cc = _nvcc()
    for src in ("mxgemm.cu", "api.cu"):
        cmd = [cc, *_build.ARCH, *_build.NVCC_FLAGS, "-DRG_MX_PAIR=1", "-c",
               os.path.join(_build.CSRC, src), "-o", str(tmp_path / (src + ".o"))]
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, (src, r.stderr[-2000:])
