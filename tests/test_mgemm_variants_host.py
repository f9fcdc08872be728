"""The M-grouped GEMM's tile-variant selection (csrc/internal.h), compiled
as plain C++ on the host: for each (transpose_B, N, K) the CTA-pair build
picks 64-column pair tiles for forward outputs at most 64 wide, single-CTA
128 x 256 tiles for contractions of one 64-deep stage, and 256 x 256 pair
tiles otherwise, and B's tensor-map box holds the B rows one CTA of that
tile loads (32, 256, 128).  The single-CTA build (RG_CTA_PAIR=0) has one
variant, 256 B rows per box.  The LoRA shapes of the benchmark land where
intended: the shrink (N = 32, K = 3072) on the narrow pair tiles, the expand
(N = 1280, K = 16) on single CTAs."""
import os
import shutil
import subprocess

import pytest

from moe_grouped_gemm_device_gb300 import _build

PROGRAM = r"""
#include <cstdio>
#include "internal.h"
int main() {
  const int cases[][3] = {{0, 32, 3072}, {0, 1280, 16}, {0, 64, 64}, {0, 65, 64}, {0, 2560, 3072}, {1, 3072, 1280},
                          {1, 384, 64}, {1, 200, 16}, {1, 48, 320}, {0, 48, 320}, {0, 384, 65}, {0, 8, 8}};
  for (const auto& c : cases) {
    const bool tb = c[0] != 0;
    std::printf("%d %d %d %d %d %d\n", c[0], c[1], c[2], rg::mgemm_narrow(tb, c[1]) ? 1 : 0,
                rg::mgemm_one_cta(tb, c[1], c[2]) ? 1 : 0, rg::mgemm_b_box_rows(tb, c[1], c[2]));
  }
  return 0;
}
"""


def _cuda_include():
    try:
        inc = os.path.join(os.path.dirname(os.path.dirname(_build.nvcc())), "include")
    except RuntimeError:
        return None
    return inc if os.path.exists(os.path.join(inc, "cuda.h")) else None


def _run(tmp_path, flags):
    src = tmp_path / "variants.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "variants"
    r = subprocess.run(["g++", "-std=c++17", "-O1", *flags, "-I", _build.CSRC, "-I", _cuda_include(), str(src),
                        "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60).stdout.split("\n")
    return {tuple(map(int, ln.split()[:3])): tuple(map(int, ln.split()[3:])) for ln in out if ln.strip()}


@pytest.mark.skipif(shutil.which("g++") is None or _cuda_include() is None, reason="g++ or CUDA headers missing")
def test_pair_build_variant_selection(tmp_path):
    got = _run(tmp_path, [])
    for (tb, n, k), (narrow, one_cta, box) in got.items():
        want_narrow = tb == 0 and n <= 64
        want_one = not want_narrow and k <= 64
        assert (narrow, one_cta) == (int(want_narrow), int(want_one)), (tb, n, k)
        assert box == (32 if want_narrow else 256 if want_one else 128), (tb, n, k)
    assert got[(0, 32, 3072)] == (1, 0, 32)     # LoRA shrink
    assert got[(0, 1280, 16)] == (0, 1, 256)    # LoRA expand
    assert got[(0, 2560, 3072)] == (0, 0, 128)  # a3b forward gate-up


@pytest.mark.skipif(shutil.which("g++") is None or _cuda_include() is None, reason="g++ or CUDA headers missing")
def test_single_cta_build_has_one_variant(tmp_path):
    got = _run(tmp_path, ["-DRG_CTA_PAIR=0"])
    assert all(v == (0, 0, 256) for v in got.values()), got
