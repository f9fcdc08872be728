// Coordinate checks of the debug-bounds build (RG_DEBUG_BOUNDS=1).
//
// Every tensor copy and store a kernel issues is described by the box it
// starts and the operand it addresses; the predicates below say whether that
// box keeps the rules the kernels rely on:
//   * the innermost coordinate of a tiled copy times the element size is a
//     multiple of 16 bytes (the copy engine does not check it);
//   * every element of the box that lies inside the tensor map's extents
//     lies inside the operand the kernel meant to read or write (for the
//     overlapping zero-filling views of the K-grouped GEMM: inside the
//     expert's own rows).  A load box may start past a plain map's extent
//     (the second CTA's half of a last, partial column block): all of its
//     elements are then out of range and zero-filled without a memory
//     access, so only its alignment and its group index are checked;
//   * an output box covers only rows of its own group and columns below the
//     output width.
// In the debug build a failed check sets RG_DEV_BOUNDS in the status word and
// the access is skipped (a skipped load's bytes are counted as arrived on its
// stage barrier, so the pipeline neither hangs nor reads the bad address).
// The predicates are plain host/device functions so that the host tests can
// exercise them, including boxes that break each rule.
#pragma once

#ifndef RG_HD
#if defined(__CUDACC__)
#define RG_HD __host__ __device__ __forceinline__
#else
#define RG_HD inline
#endif
#endif

namespace rg {
namespace bounds {

// Innermost coordinate x of a tiled copy of elements of `elem_bytes` bytes:
// the copy must start on a 16-byte boundary.
RG_HD bool inner_aligned(long long x, int elem_bytes) { return x >= 0 && (x * elem_bytes) % 16 == 0; }

// A box of `box` elements starting at `start` along one dimension of extent
// `extent`: at least one element in range, and the start not past the end.
RG_HD bool within(long long start, long long box, long long extent) {
  return box > 0 && start < extent && start + box > 0;
}

// K-grouped operand views (element (c, i, j) is row i + j, i < br): a box at
// (c, i0, r) of br rows reads rows r + i0 .. r + i0 + br - 1 of which those
// with i = i0 + k >= 0 are in range.  The box must start inside the expert
// [lo, hi) and every in-range row must belong to it: r in [lo, hi),
// -br < i0 <= 0 and r + i0 + br <= hi.
RG_HD bool kgemm_rows(long long r, long long i0, long long br, long long lo, long long hi) {
  return lo <= r && r < hi && -br < i0 && i0 <= 0 && r + i0 + br <= hi;
}

// M-grouped A box: rows row0 .. row0 + box_rows - 1 of a tile that starts
// inside its group [lo, hi) (rows past hi may be read; they are never
// stored) and inside the tensor of m rows.
RG_HD bool mgemm_rows(long long row0, long long lo, long long hi, long long m) {
  return lo <= row0 && row0 < hi && row0 < m;
}

// Output box of `rows` x `cols` elements at (col0, row0): all rows inside the
// group [lo, hi), all columns below `width`, innermost coordinate aligned.
RG_HD bool out_box(long long col0, long long cols, long long row0, long long rows, long long lo, long long hi,
                   long long width, int elem_bytes) {
  return inner_aligned(col0, elem_bytes) && col0 + cols <= width && lo <= row0 && row0 + rows <= hi;
}

// An index into a stack of `count` matrices (expert, group, or outer group).
RG_HD bool index_ok(long long i, long long count) { return 0 <= i && i < count; }

#if defined(__CUDACC__)
// A failed check of the debug build: set the status bit, and tell the caller
// to skip the access.
__device__ __forceinline__ bool report(bool ok, unsigned int* status) {
  if (!ok) atomicOr(status, 0x8u);
  return ok;
}
#endif

}  // namespace bounds
}  // namespace rg

#ifndef RG_DEBUG_BOUNDS
#define RG_DEBUG_BOUNDS 0
#endif
// RG_BOUNDS_OK(cond, status): the debug build evaluates `cond` and reports a
// failure; every other build evaluates nothing and passes.
#define RG_BOUNDS_OK(cond, status) (!RG_DEBUG_BOUNDS || ::rg::bounds::report((cond), (status)))
