"""The coordinate checks of the debug-bounds build (csrc/bounds.cuh), compiled
as plain C++ on the host: boxes the kernels issue pass, and boxes that break
each rule -- an unaligned innermost coordinate, a K-grouped box reaching a
row of the next expert or before its own, an output box straddling a group
end or the output width, an index past its stack -- fail."""
import os
import shutil
import subprocess

import pytest

from moe_grouped_gemm_device_gb300 import _build

PROGRAM = r"""
#include <cstdio>
#include "bounds.cuh"
using namespace rg::bounds;
int fails = 0;
#define EXPECT(c) do { if (!(c)) { std::printf("FAILED: %s (line %d)\n", #c, __LINE__); ++fails; } } while (0)
int main() {
  // 16-byte rule on the innermost coordinate
  EXPECT(inner_aligned(64, 2) && inner_aligned(8, 2) && inner_aligned(4, 4) && inner_aligned(16, 1));
  EXPECT(!inner_aligned(4, 2) && !inner_aligned(2, 4) && !inner_aligned(8, 1) && !inner_aligned(-8, 2));
  // K-grouped views, rows [lo, hi) = [100, 230), BR = 96
  EXPECT(kgemm_rows(100, 0, 96, 100, 230));            // a full block
  EXPECT(kgemm_rows(196, 34 - 96, 96, 100, 230));      // the ragged last block: 34 rows
  EXPECT(kgemm_rows(229, 1 - 96, 96, 100, 230));       // a last block of one row
  EXPECT(!kgemm_rows(196, 0, 96, 100, 230));           // would read 62 rows of the next expert
  EXPECT(!kgemm_rows(196, 35 - 96, 96, 100, 230));     // one row too many
  EXPECT(!kgemm_rows(99, 0, 96, 100, 230));            // starts in the previous expert
  EXPECT(!kgemm_rows(230, -95, 96, 100, 230));         // starts past the expert
  EXPECT(!kgemm_rows(150, -96, 96, 100, 230));         // no row in range
  EXPECT(!kgemm_rows(150, 1, 96, 100, 230));           // positive start inside the view
  // M-grouped tiles start inside their group
  EXPECT(mgemm_rows(100, 100, 230, 1000) && mgemm_rows(229, 100, 230, 1000));
  EXPECT(!mgemm_rows(230, 100, 230, 1000) && !mgemm_rows(99, 100, 230, 1000));
  // output boxes: 64 x 32 bf16 at (col0, row0), group [100, 230), width 384
  EXPECT(out_box(320, 64, 198, 32, 100, 230, 384, 2));
  EXPECT(!out_box(320, 64, 199, 32, 100, 230, 384, 2));   // straddles the group's end
  EXPECT(!out_box(352, 64, 100, 32, 100, 230, 384, 2));   // past the output width
  EXPECT(!out_box(4, 64, 100, 32, 100, 230, 384, 2));     // unaligned start
  EXPECT(!out_box(0, 64, 98, 32, 100, 230, 384, 2));      // starts in the previous group
  // partial boxes clipped by the tensor map, indices into stacks
  EXPECT(within(3040, 32, 3072) && within(3056, 32, 3072) && !within(3072, 32, 3072) && !within(0, 0, 10));
  EXPECT(index_ok(0, 1) && index_ok(31, 32) && !index_ok(32, 32) && !index_ok(-1, 32));
  std::printf("%s\n", fails ? "SOME CHECKS FAILED" : "ALL CHECKS PASSED");
  return fails != 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="g++ not available")
def test_bounds_predicates_on_the_host(tmp_path):
    src = tmp_path / "bounds_test.cc"
    src.write_text(PROGRAM)
    exe = tmp_path / "bounds_test"
    r = subprocess.run(["g++", "-std=c++17", "-O1", "-I", _build.CSRC, str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and "ALL CHECKS PASSED" in r.stdout, r.stdout


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="nvcc not available")
def test_debug_bounds_build_compiles(tmp_path):
    lib = _build.build(force=True, extra_flags=_build.BOUNDS_FLAGS, out_dir=str(tmp_path))
    assert os.path.exists(lib)
