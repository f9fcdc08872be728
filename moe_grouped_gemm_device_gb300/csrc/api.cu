// C-ABI host layer of librg.so: argument validation, TMA tensor-map encoding,
// per-device setup and kernel launch.  Declared in include/rg.h.
//
// Nothing here allocates device or host memory.  The per-device status words
// are module-scope __device__ variables (one instance per device context);
// their device addresses are looked up once per device.  Tensor maps are
// encoded on the host for every call and passed by value as kernel
// parameters, so no host workspace outlives a call.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "rg.h"

namespace {

__device__ unsigned int g_status_word;    // bits set by the GEMM and conversion kernels
__device__ unsigned int g_selftest_word;  // bits set by the wait self-test
__device__ unsigned int g_status_taken;   // last value taken from a status word, read by the host

// Hand-over flags of rg_kgemm_noalloc: the scratch of the chunk-mode Kgemm
// for callers that cannot allocate, held by every GPU that loads the library
// until the process exits.  Host code must not pass this name to a kernel
// (on the host it is a stand-in, not a device address): its device address
// is looked up once per device in device_state() and kept in DeviceState.
static __device__ __align__(256) int g_kgemm_noalloc_flags[RG_KGEMM_NOALLOC_MAX_FLAGS];

// Read a status word and clear it in one atomic step, on the caller's stream.
__global__ void take_status_kernel(unsigned int* word, unsigned int* taken) { *taken = atomicExch(word, 0u); }

constexpr int kMaxDevices = 64;
// Smallest accepted bound on a pipeline wait: a wait can legitimately last a
// whole tile's mainloop, or longer on a GPU shared with other work.
constexpr unsigned long long kMinWaitLimitNs = 1000000ull;
thread_local int t_last_cuda_error = 0;
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};

struct DeviceState {
  bool ready = false;
  bool supported = false;
  int num_sms = 0;
  int mg_grid = 0;      // persistent grid of each kernel (CTAs)
  int kg_grid = 0;
  int mx_grid = 0;      // MXFP8 Mgemm
  size_t max_smem = 0;  // opt-in dynamic shared memory per block
  unsigned int* status = nullptr;    // &g_status_word on this device
  unsigned int* selftest = nullptr;  // &g_selftest_word
  unsigned int* taken = nullptr;     // &g_status_taken
  int* noalloc_flags = nullptr;      // &g_kgemm_noalloc_flags on this device
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
std::mutex g_take_mu[kMaxDevices];  // one reader of g_status_taken per device at a time

int fail_cuda(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return RG_ERR_CUDA;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Per-device one-time setup.  Returns RG_OK / RG_ERR_UNSUPPORTED / RG_ERR_CUDA
// and, on success, the state of the current device.
int device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return RG_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& ds = g_dev[dev];
  if (!ds.ready) {
    int major = 0, minor = 0, sms = 0, smem = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
      return fail_cuda(e);
    ds.supported = (major == 10 && minor == 3);
    ds.num_sms = sms;
    ds.max_smem = static_cast<size_t>(smem);
    if (ds.supported) {
      void* p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_status_word)) != cudaSuccess) return fail_cuda(e);
      ds.status = static_cast<unsigned int*>(p);
      if ((e = cudaGetSymbolAddress(&p, g_selftest_word)) != cudaSuccess) return fail_cuda(e);
      ds.selftest = static_cast<unsigned int*>(p);
      if ((e = cudaGetSymbolAddress(&p, g_status_taken)) != cudaSuccess) return fail_cuda(e);
      ds.taken = static_cast<unsigned int*>(p);
      int* flags = nullptr;
      if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&flags), g_kgemm_noalloc_flags)) != cudaSuccess)
        return fail_cuda(e);
      ds.noalloc_flags = flags;
      if ((e = rg::mgemm_setup(smem)) != cudaSuccess) return fail_cuda(e);
      if ((e = rg::kgemm_setup(smem)) != cudaSuccess) return fail_cuda(e);
      if ((e = rg::mx_setup(smem)) != cudaSuccess) return fail_cuda(e);
      if ((e = rg::mxk_setup(smem)) != cudaSuccess) return fail_cuda(e);
      if (encode_fn() == nullptr) return fail_cuda(cudaErrorNotSupported);
      // One CTA per SM (shared memory limits residency to one); with CTA
      // pairs, as many 2-CTA clusters as can be resident at once.
      ds.mg_grid = ds.kg_grid = ds.mx_grid = sms;
      if (rg::kCtaGroup == 2) {
        int mc = 0, kc = 0;
        if ((e = rg::mgemm_max_clusters(&mc, smem)) != cudaSuccess) return fail_cuda(e);
        if ((e = rg::kgemm_max_clusters(&kc, smem)) != cudaSuccess) return fail_cuda(e);
        if (mc < 1 || kc < 1) return fail_cuda(cudaErrorLaunchOutOfResources);
        ds.mg_grid = 2 * std::min(mc, sms / 2);
        ds.kg_grid = 2 * std::min(kc, sms / 2);
      }
      if (rg::mxm::CG == 2) {
        int xc = 0;
        if ((e = rg::mx_max_clusters(&xc, smem)) != cudaSuccess) return fail_cuda(e);
        if (xc < 1) return fail_cuda(cudaErrorLaunchOutOfResources);
        ds.mx_grid = 2 * std::min(xc, sms / 2);
      }
    }
    ds.ready = true;
  }
  if (!ds.supported) return RG_ERR_UNSUPPORTED;
  *out = &ds;
  return RG_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Take (read and clear atomically) the status word `word` of the current
// device after the work queued on `stream`, and wait for the result.
// Returns the bits (>= 0) or RG_ERR_CUDA.
int take_status(const DeviceState* ds, unsigned int* word, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  std::lock_guard<std::mutex> lock(g_take_mu[dev]);
  take_status_kernel<<<1, 1, 0, stream>>>(word, ds->taken);
  if ((e = cudaGetLastError()) != cudaSuccess) return fail_cuda(e);
  unsigned int v = 0;
  if ((e = cudaMemcpyFromSymbolAsync(&v, g_status_taken, sizeof v, 0, cudaMemcpyDeviceToHost, stream)) !=
      cudaSuccess)
    return fail_cuda(e);
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return fail_cuda(e);
  return static_cast<int>(v & 0x7fffffffu);
}

// Encode a tiled tensor map; dims/box innermost first, strides in bytes for
// dims 1..rank-1.
bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr, const uint64_t* dims,
            const uint64_t* strides, const uint32_t* box) {
  const uint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  const CUresult r = encode_fn()(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), dims,
                                 strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tiled tensor map with an explicit swizzle mode.
bool encode_sw(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr, const uint64_t* dims,
               const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw) {
  const uint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  const CUresult r = encode_fn()(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), dims, strides,
                                 box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Transposed weights w [G, K, N] (N contiguous) as read by the input-gradient
// Mgemm: 64 columns x 64 K rows per box.  With N a multiple of 64 the map is
// the 4-D view {64 cols, K, column block, group} (column-block stride 128
// bytes), whose boxes of box_cols / 64 column blocks (two for pair tiles,
// four for single-CTA tiles) land in shared memory exactly as that many
// 64-column boxes side by side: one copy per atom instead of one per box.
// Returns the view used (1 = 4-D) or -1 when encoding fails.
// kbox K rows per box (64, or 16 / 32 for the narrow boxes of single-CTA
// one-stage tiles; the rows stay 128 bytes of N, 128-byte swizzle).
int encode_weight_t(CUtensorMap* m, const void* w, int G, int N, int K, int box_cols = rg::mg::BN_CTA,
                    int kbox = rg::mg::BK) {
  if (N % 64 == 0) {
    const uint64_t dims[4] = {64, static_cast<uint64_t>(K), static_cast<uint64_t>(N / 64),
                              static_cast<uint64_t>(G)};
    const uint64_t str[3] = {static_cast<uint64_t>(N) * 2, 128, static_cast<uint64_t>(K) * N * 2};
    const uint32_t box[4] = {64, static_cast<uint32_t>(kbox), static_cast<uint32_t>(box_cols / 64), 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, w, dims, str, box) ? 1 : -1;
  }
  const uint64_t dims[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K), static_cast<uint64_t>(G)};
  const uint64_t str[2] = {static_cast<uint64_t>(N) * 2, static_cast<uint64_t>(K) * N * 2};
  const uint32_t box[3] = {64, static_cast<uint32_t>(kbox), 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, w, dims, str, box) ? 0 : -1;
}

// Swizzle of a K-major box whose rows are kbox bf16 (32, 64 or 128 bytes):
// the swizzle of the row's width, as the kernels' shared-memory descriptors
// expect.
CUtensorMapSwizzle kswizzle(int kbox) {
  return kbox == 16 ? CU_TENSOR_MAP_SWIZZLE_32B : kbox == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
}

// Row-major bf16 [rows, cols] tensor, boxes of kbox columns x box_rows rows.
bool encode_rows(CUtensorMap* m, const void* ptr, int64_t rows, int cols, uint32_t box_rows,
                 int kbox = rg::mg::BK) {
  const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
  const uint64_t str[1] = {static_cast<uint64_t>(cols) * 2};
  const uint32_t box[2] = {static_cast<uint32_t>(kbox), box_rows};
  return encode_sw(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, str, box, kswizzle(kbox));
}

// Forward weight [E, N, K] (K contiguous): boxes of kbox K x (B rows per CTA
// of the tile the launch uses).
bool encode_weight(CUtensorMap* m, const void* w, int E, int N, int K, int box_rows, int kbox = rg::mg::BK) {
  const uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(E)};
  const uint64_t str[2] = {static_cast<uint64_t>(K) * 2, static_cast<uint64_t>(N) * K * 2};
  const uint32_t box[3] = {static_cast<uint32_t>(kbox), static_cast<uint32_t>(box_rows), 1};
  return encode_sw(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, w, dims, str, box, kswizzle(kbox));
}

rg::GroupArgs group_args(const DeviceState* ds, const int32_t* offsets, int E, int64_t M, int N, int K,
                         void* out) {
  rg::GroupArgs a;
  a.offsets = offsets;
  a.E = E;
  a.M = static_cast<int>(M);
  a.N = N;
  a.K = K;
  a.out = out;
  a.out2 = nullptr;
  a.status = ds->status;
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.accumulate = 0;
  a.outer = 1;
  a.kg_wide = 0;
  a.mg_wide_b = 0;
  a.flags = nullptr;
  return a;
}

int check_common(const int32_t* offsets, int E, int64_t M, int N, int K) {
  if (offsets == nullptr || (reinterpret_cast<uintptr_t>(offsets) & 3u) != 0) return RG_ERR_INVALID_ARG;
  if (E < 1 || E > RG_MAX_EXPERTS) return RG_ERR_INVALID_ARG;
  if (M < 0 || M > INT32_MAX) return RG_ERR_INVALID_ARG;
  if (N < 8 || K < 8 || (N % 8) != 0 || (K % 8) != 0) return RG_ERR_INVALID_ARG;
  return RG_OK;
}

// The M-grouped GEMM of both entry points: O outer groups over the columns
// of x and y (1 = plain Mgemm), L row groups.
int mgemm_impl(const void* x, const void* w, const int32_t* offsets, int O, int L, int64_t M, int N, int K,
               int transpose_B, void* y, cudaStream_t stream) {
  if (O < 1 || O > RG_MAX_OUTER) return RG_ERR_INVALID_ARG;
  int rc = check_common(offsets, L, M, N, K);
  if (rc != RG_OK) return rc;
  if (static_cast<int64_t>(O) * N > INT32_MAX || static_cast<int64_t>(O) * K > INT32_MAX ||
      static_cast<int64_t>(O) * L > INT32_MAX)
    return RG_ERR_INVALID_ARG;
  if (w == nullptr || !aligned16(w)) return RG_ERR_INVALID_ARG;
  if (M > 0 && (x == nullptr || y == nullptr || !aligned16(x) || !aligned16(y)))
    return RG_ERR_INVALID_ARG;
  // the tile list is indexed with 32-bit integers (the launch's tiles have
  // TILE_M rows, or BM for the single-CTA one-stage tiles)
  const int64_t tile_rows = rg::mgemm_one_cta(transpose_B != 0, N, K) ? rg::mg::BM : rg::mg::TILE_M;
  const int64_t max_tiles = (M / tile_rows + L) * ((N + rg::mg::BN - 1) / rg::mg::BN) * O;
  if (max_tiles > INT32_MAX) return RG_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds)) != RG_OK) return rc;
  if (rg::mgemm_smem_bytes(L) > ds->max_smem) return RG_ERR_INVALID_ARG;  // too many groups
  if (M == 0) return RG_OK;  // no rows, nothing to write

  // The weights of all (outer, inner) groups form one stack of O*L matrices.
  const int G = O * L;
  const int kbox = rg::mgemm_kbox(transpose_B != 0, N, K);  // K columns per operand box
  CUtensorMap tmA, tmAh, tmB, tmY;
  if (O == 1) {
    if (!encode_rows(&tmA, x, M, K, rg::mg::BM, kbox)) return RG_ERR_INVALID_ARG;
    if (!encode_rows(&tmAh, x, M, K, rg::mg::BM / 2, kbox)) return RG_ERR_INVALID_ARG;
    if (!encode_rows(&tmY, y, M, N, 32)) return RG_ERR_INVALID_ARG;
  } else {
    // x [M, O*K] as {K, O, M}; y [M, O*N] as {N, O, M}: one outer group's
    // column block per box, so a box never reads or writes a neighbour's columns
    const uint64_t xd[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(O), static_cast<uint64_t>(M)};
    const uint64_t xs[2] = {static_cast<uint64_t>(K) * 2, static_cast<uint64_t>(O) * K * 2};
    const uint32_t xb[3] = {static_cast<uint32_t>(kbox), 1, rg::mg::BM};
    if (!encode_sw(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, x, xd, xs, xb, kswizzle(kbox)))
      return RG_ERR_INVALID_ARG;
    const uint32_t xbh[3] = {static_cast<uint32_t>(kbox), 1, rg::mg::BM / 2};
    if (!encode_sw(&tmAh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, x, xd, xs, xbh, kswizzle(kbox)))
      return RG_ERR_INVALID_ARG;
    const uint64_t yd[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(O), static_cast<uint64_t>(M)};
    const uint64_t ys[2] = {static_cast<uint64_t>(N) * 2, static_cast<uint64_t>(O) * N * 2};
    const uint32_t yb[3] = {64, 1, 32};
    if (!encode(&tmY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, y, yd, ys, yb)) return RG_ERR_INVALID_ARG;
  }
  int wide_b = 0;
  if (!transpose_B) {  // w [G, N, K], K contiguous: one 64-wide K box of the tile's B rows per stage and CTA
    if (!encode_weight(&tmB, w, G, N, K, rg::mgemm_b_box_rows(false, N, K), kbox)) return RG_ERR_INVALID_ARG;
  } else if ((wide_b = encode_weight_t(&tmB, w, G, N, K, rg::mgemm_b_box_rows(true, N, K), kbox)) < 0) {
    // w [G, K, N], N contiguous
    return RG_ERR_INVALID_ARG;
  }
  rg::GroupArgs args = group_args(ds, offsets, L, M, N, K, y);
  args.outer = O;
  args.mg_wide_b = wide_b;
  const cudaError_t e =
      rg::launch_mgemm(transpose_B != 0, tmA, tmAh, tmB, tmY, args, ds->mg_grid, ds->num_sms, stream);
  if (e != cudaSuccess) return fail_cuda(e);
  return RG_OK;
}

}  // namespace

extern "C" {

int rg_mgemm(const void* x, const void* w, const int32_t* offsets, int E, int64_t M, int N, int K,
             int transpose_B, void* y, cudaStream_t stream) {
  return mgemm_impl(x, w, offsets, 1, E, M, N, K, transpose_B, y, stream);
}

int rg_mgemm_nested(const void* x, const void* w, const int32_t* offsets, int O, int L, int64_t M, int N,
                    int K, int transpose_B, void* y, cudaStream_t stream) {
  return mgemm_impl(x, w, offsets, O, L, M, N, K, transpose_B, y, stream);
}

int rg_mgemm_swiglu(const void* x, const void* w13, const int32_t* offsets, int E, int64_t M, int F,
                    int K, void* y13, void* h, cudaStream_t stream) {
  if (F < 8 || F % 8 != 0 || F > INT32_MAX / 2) return RG_ERR_INVALID_ARG;  // h rows: 16-byte strides
  const int N = 2 * F;
  int rc = check_common(offsets, E, M, N, K);
  if (rc != RG_OK) return rc;
  if (w13 == nullptr || !aligned16(w13)) return RG_ERR_INVALID_ARG;
  if (M > 0 && (x == nullptr || h == nullptr || !aligned16(x) || !aligned16(h)))
    return RG_ERR_INVALID_ARG;
  if (y13 != nullptr && !aligned16(y13)) return RG_ERR_INVALID_ARG;
  const int64_t max_tiles = (M / rg::mg::TILE_M + E) * ((F + rg::mg::BN_CTA - 1) / rg::mg::BN_CTA);
  if (max_tiles > INT32_MAX) return RG_ERR_INVALID_ARG;
  if (rg::kCtaGroup != 2) return RG_ERR_UNSUPPORTED;  // gate and up halves come from the two CTAs
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds)) != RG_OK) return rc;
  if (rg::mgemm_smem_bytes(E) > ds->max_smem) return RG_ERR_INVALID_ARG;
  if (M == 0) return RG_OK;

  CUtensorMap tmA, tmB, tmH, tmY13;
  if (!encode_rows(&tmA, x, M, K, rg::mg::BM)) return RG_ERR_INVALID_ARG;
  if (!encode_weight(&tmB, w13, E, N, K, rg::mg::BN_CTA)) return RG_ERR_INVALID_ARG;  // fused epilogue: default tile
  if (!encode_rows(&tmH, h, M, F, 32)) return RG_ERR_INVALID_ARG;
  if (y13 != nullptr) {
    if (!encode_rows(&tmY13, y13, M, N, 32)) return RG_ERR_INVALID_ARG;
  } else {
    tmY13 = tmH;  // not used
  }
  rg::GroupArgs args = group_args(ds, offsets, E, M, N, K, h);
  args.out2 = y13;
  const cudaError_t e = rg::launch_mgemm_swiglu(tmA, tmB, tmH, tmY13, args, ds->mg_grid, stream);
  if (e != cudaSuccess) return fail_cuda(e);
  return RG_OK;
}

int rg_mgemm_swiglu_dgrad(const void* dy, const void* w2, const int32_t* offsets, int E, int64_t M,
                          int F, int K, const void* y13, void* dy13, cudaStream_t stream) {
  if (F < 8 || F % 8 != 0 || F > INT32_MAX / 2) return RG_ERR_INVALID_ARG;
  int rc = check_common(offsets, E, M, 2 * F, K);
  if (rc != RG_OK) return rc;
  if (w2 == nullptr || !aligned16(w2)) return RG_ERR_INVALID_ARG;
  if (M > 0) {
    if (dy == nullptr || y13 == nullptr || dy13 == nullptr || !aligned16(dy) || !aligned16(y13) ||
        !aligned16(dy13))
      return RG_ERR_INVALID_ARG;
    // y13 is read through the non-coherent cache while dy13 is written
    const uintptr_t a = reinterpret_cast<uintptr_t>(y13), b = reinterpret_cast<uintptr_t>(dy13);
    const uintptr_t bytes = static_cast<uintptr_t>(M) * static_cast<uintptr_t>(2 * F) * 2;
    if (a < b + bytes && b < a + bytes) return RG_ERR_INVALID_ARG;
  }
  const int64_t max_tiles = (M / rg::mg::TILE_M + E) * ((F + rg::mg::BN - 1) / rg::mg::BN);
  if (max_tiles > INT32_MAX) return RG_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds)) != RG_OK) return rc;
  if (rg::mgemm_smem_bytes(E) > ds->max_smem) return RG_ERR_INVALID_ARG;
  if (M == 0) return RG_OK;

  CUtensorMap tmA, tmB, tmD;
  if (!encode_rows(&tmA, dy, M, K, rg::mg::BM)) return RG_ERR_INVALID_ARG;
  const int wide_b = encode_weight_t(&tmB, w2, E, F, K);  // w2 [E, K, F], F contiguous
  if (wide_b < 0) return RG_ERR_INVALID_ARG;
  if (!encode_rows(&tmD, dy13, M, 2 * F, 32)) return RG_ERR_INVALID_ARG;
  rg::GroupArgs args = group_args(ds, offsets, E, M, F, K, dy13);
  args.mg_wide_b = wide_b;
  args.out2 = const_cast<void*>(y13);
  const cudaError_t e = rg::launch_mgemm_swiglu_dgrad(tmA, tmB, tmD, args, ds->mg_grid, stream);
  if (e != cudaSuccess) return fail_cuda(e);
  return RG_OK;
}

}  // extern "C"

extern "C" {

int64_t rg_mx_blocked_bytes(int64_t R, int KS, int G) {
  if (R < 0 || KS < 1 || G < 1) return -1;
  return (R / 128 + G) * ((KS + 3) / 4) * 512;
}

int rg_mx_scales_blocked(const uint8_t* scales, const int32_t* offsets, int G, int64_t R, int KS, uint8_t* out,
                         int64_t out_bytes, cudaStream_t stream) {
  if (offsets == nullptr || (reinterpret_cast<uintptr_t>(offsets) & 3u) != 0) return RG_ERR_INVALID_ARG;
  if (G < 1 || G > RG_MAX_EXPERTS || R < 0 || R > INT32_MAX || KS < 1) return RG_ERR_INVALID_ARG;
  if (R * static_cast<int64_t>(KS) > INT64_MAX / 2) return RG_ERR_INVALID_ARG;
  if (out == nullptr || !aligned16(out) || out_bytes < rg_mx_blocked_bytes(R, KS, G)) return RG_ERR_INVALID_ARG;
  if (R > 0 && scales == nullptr) return RG_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != RG_OK) return rc;
  const cudaError_t e = rg::launch_mx_blocked(scales, offsets, G, static_cast<int>(R), KS, out, ds->status,
                                              ds->num_sms, stream);
  if (e != cudaSuccess) return fail_cuda(e);
  return RG_OK;
}

int rg_mgemm_mxfp8(const void* xq, const void* sx_blocked, const void* wq, const void* sw_blocked,
                   const int32_t* offsets, int E, int64_t M, int N, int K, int transpose_B, void* y,
                   cudaStream_t stream) {
  if (offsets == nullptr || (reinterpret_cast<uintptr_t>(offsets) & 3u) != 0) return RG_ERR_INVALID_ARG;
  if (E < 1 || E > RG_MAX_EXPERTS || M < 0 || M > INT32_MAX) return RG_ERR_INVALID_ARG;
  if (N < 16 || N % 16 != 0 || K < 32 || K % 32 != 0) return RG_ERR_INVALID_ARG;
  if (wq == nullptr || sw_blocked == nullptr || !aligned16(wq) || !aligned16(sw_blocked)) return RG_ERR_INVALID_ARG;
  if (M > 0 && (xq == nullptr || sx_blocked == nullptr || y == nullptr || !aligned16(xq) ||
                !aligned16(sx_blocked) || !aligned16(y)))
    return RG_ERR_INVALID_ARG;
  const int64_t max_tiles = (M / 128 + E) * ((N + 255) / 256);
  if (max_tiles > INT32_MAX) return RG_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != RG_OK) return rc;
  if (rg::mx_smem_bytes(E) > ds->max_smem) return RG_ERR_INVALID_ARG;
  if (M == 0) return RG_OK;

  CUtensorMap tmA, tmB, tmY;
  {  // xq [M, K] bytes: 128 x 128 boxes
    const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
    const uint64_t str[1] = {static_cast<uint64_t>(K)};
    const uint32_t box[2] = {128, 128};
    if (!encode_sw(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, xq, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return RG_ERR_INVALID_ARG;
  }
  if (!transpose_B) {  // wq [E, N, K]: one 128 (K) x BN_CTA (N) box per stage (256 N, or 128 per CTA of a pair)
    const uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(E)};
    const uint64_t str[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N) * K};
    const uint32_t box[3] = {128, static_cast<uint32_t>(rg::mxm::BN_CTA), 1};
    if (!encode_sw(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, wq, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return RG_ERR_INVALID_ARG;
  } else {  // wq [E, K, N]: 128 (N) x 128 (K) boxes, two per stage (one per CTA of a pair)
    const uint64_t dims[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K), static_cast<uint64_t>(E)};
    const uint64_t str[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K) * N};
    const uint32_t box[3] = {128, 128, 1};
    if (!encode_sw(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, wq, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return RG_ERR_INVALID_ARG;
  }
  {  // y [M, N] bf16: 32 x 32 boxes, 64-byte swizzle
    const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M)};
    const uint64_t str[1] = {static_cast<uint64_t>(N) * 2};
    const uint32_t box[2] = {32, 32};
    if (!encode_sw(&tmY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, y, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B))
      return RG_ERR_INVALID_ARG;
  }
  // CTA pairs: the blocked scale buffers as rows of 256 bytes (a 512-byte
  // chunk is two rows); a single CTA reads them with plain bulk copies
  CUtensorMap tmSA = {}, tmSB = {};
  if (rg::mxm::CG == 2) {
    const uint64_t rows_a = static_cast<uint64_t>(rg_mx_blocked_bytes(M, K / 32, E)) / 256;
    const uint64_t rows_b = static_cast<uint64_t>(rg_mx_blocked_bytes(static_cast<int64_t>(E) * N, K / 32, E)) / 256;
    const uint64_t da[2] = {256, rows_a}, db[2] = {256, rows_b};
    const uint64_t str[1] = {256};
    const uint32_t box[2] = {256, 2};
    if (!encode_sw(&tmSA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, sx_blocked, da, str, box, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_sw(&tmSB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, sw_blocked, db, str, box, CU_TENSOR_MAP_SWIZZLE_NONE))
      return RG_ERR_INVALID_ARG;
  }
  rg::MxArgs a;
  a.offsets = offsets;
  a.sfa = static_cast<const uint8_t*>(sx_blocked);
  a.sfb = static_cast<const uint8_t*>(sw_blocked);
  a.E = E;
  a.M = static_cast<int>(M);
  a.N = N;
  a.K = K;
  a.out = y;
  a.status = ds->status;
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.accumulate = 0;
  const cudaError_t e = rg::launch_mx_mgemm(transpose_B != 0, tmA, tmB, tmY, tmSA, tmSB, a, ds->mx_grid, stream);
  if (e != cudaSuccess) return fail_cuda(e);
  return RG_OK;
}

int64_t rg_mx_blocked_k_bytes(int64_t R, int KS, int G) {
  if (R < 1 || KS < 1 || G < 1) return -1;
  return (R + 127) / 128 * (KS / 4 + G) * 512;
}

int rg_mx_scales_blocked_k(const uint8_t* scales, const int32_t* offsets, int G, int64_t R, int KS, uint8_t* out,
                           int64_t out_bytes, cudaStream_t stream) {
  if (offsets == nullptr || (reinterpret_cast<uintptr_t>(offsets) & 3u) != 0) return RG_ERR_INVALID_ARG;
  if (G < 1 || G > RG_MAX_EXPERTS || R < 1 || R > INT32_MAX || KS < 1 || KS > INT32_MAX / 32)
    return RG_ERR_INVALID_ARG;
  if (scales == nullptr || out == nullptr || !aligned16(out) || out_bytes < rg_mx_blocked_k_bytes(R, KS, G))
    return RG_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != RG_OK) return rc;
  const cudaError_t e = rg::launch_mx_blocked_k(scales, offsets, G, static_cast<int>(R), KS, out, ds->status,
                                                ds->num_sms, stream);
  if (e != cudaSuccess) return fail_cuda(e);
  return RG_OK;
}

int rg_kgemm_mxfp8(const void* gq, const void* sg_blocked, const void* xq, const void* sx_blocked,
                   const int32_t* offsets, int E, int64_t M, int N, int K, float* dW, int accumulate,
                   cudaStream_t stream) {
  if (offsets == nullptr || (reinterpret_cast<uintptr_t>(offsets) & 3u) != 0) return RG_ERR_INVALID_ARG;
  if (E < 1 || E > RG_MAX_EXPERTS || M < 0 || M > INT32_MAX || M % 32 != 0) return RG_ERR_INVALID_ARG;
  if (N < 16 || N % 16 != 0 || K < 16 || K % 16 != 0) return RG_ERR_INVALID_ARG;
  if (dW == nullptr || !aligned16(dW)) return RG_ERR_INVALID_ARG;
  if (M > 0 && (gq == nullptr || xq == nullptr || sg_blocked == nullptr || sx_blocked == nullptr ||
                !aligned16(gq) || !aligned16(xq) || !aligned16(sg_blocked) || !aligned16(sx_blocked)))
    return RG_ERR_INVALID_ARG;
  const int64_t tiles = static_cast<int64_t>(E) * ((N + 127) / 128) * ((K + 255) / 256);
  if (tiles > INT32_MAX) return RG_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != RG_OK) return rc;
  if (rg::mxk_smem_bytes(E) > ds->max_smem) return RG_ERR_INVALID_ARG;

  // With M == 0 every valid offsets vector is all zeros: only zero tiles are
  // written, and the operand maps describe one row of dW that is never read.
  const void* g_ptr = M > 0 ? gq : static_cast<const void*>(dW);
  const void* x_ptr = M > 0 ? xq : static_cast<const void*>(dW);
  const uint64_t rows = M > 0 ? static_cast<uint64_t>(M) : 1;
  CUtensorMap tmG, tmX, tmD;
  {  // gq [M, N] bytes: 128 (n) x 128 (rows) boxes
    const uint64_t dims[2] = {static_cast<uint64_t>(N), rows};
    const uint64_t str[1] = {static_cast<uint64_t>(N)};
    const uint32_t box[2] = {128, 128};
    if (!encode_sw(&tmG, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, g_ptr, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return RG_ERR_INVALID_ARG;
  }
  {  // xq [M, K] bytes: 128 (k) x 128 (rows) boxes
    const uint64_t dims[2] = {static_cast<uint64_t>(K), rows};
    const uint64_t str[1] = {static_cast<uint64_t>(K)};
    const uint32_t box[2] = {128, 128};
    if (!encode_sw(&tmX, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, x_ptr, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return RG_ERR_INVALID_ARG;
  }
  {  // dW [E, N, K] fp32: BOX_COLS (k) x 32 (n) boxes, one swizzle row per box row
    const uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(E)};
    const uint64_t str[2] = {static_cast<uint64_t>(K) * 4, static_cast<uint64_t>(N) * K * 4};
    const uint32_t box[3] = {static_cast<uint32_t>(rg::mxk::BOX_COLS), 32, 1};
    const CUtensorMapSwizzle sw = rg::mxk::BOX_COLS == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (!encode_sw(&tmD, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dW, dims, str, box, sw)) return RG_ERR_INVALID_ARG;
  }
  rg::MxArgs a;
  a.offsets = offsets;
  a.sfa = static_cast<const uint8_t*>(sg_blocked);
  a.sfb = static_cast<const uint8_t*>(sx_blocked);
  a.E = E;
  a.M = static_cast<int>(M);
  a.N = N;
  a.K = K;
  a.out = dW;
  a.status = ds->status;
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.accumulate = accumulate != 0;
  const cudaError_t e = rg::launch_mx_kgemm(tmG, tmX, tmD, a, ds->num_sms, stream);
  if (e != cudaSuccess) return fail_cuda(e);
  return RG_OK;
}

}  // extern "C"

namespace {
// Bytes of chunk-mode flags: one int per (expert, dW tile, CTA of the pair).
int64_t kgemm_flag_bytes(int E, int N, int K) {
  return static_cast<int64_t>(E) * ((N + rg::kg::TILE_M - 1) / rg::kg::TILE_M) * ((K + rg::kg::BN - 1) / rg::kg::BN) *
         rg::kCtaGroup * static_cast<int64_t>(sizeof(int));
}

// flags: null (tile mode) or device memory of kgemm_flag_bytes(E, N, K) bytes that the
// call zeroes on `stream` before the kernel (chunk mode) -- when the shape has more
// tiles per expert than the grid has CTA pairs; otherwise the kernel cannot take the
// chunk-major schedule, and the flags are neither cleared nor passed.
int kgemm_impl(const void* grad, const void* X, const int32_t* offsets, int E, int64_t M, int N, int K,
               float* dW, int accumulate, int* flags, cudaStream_t stream) {
  int rc = check_common(offsets, E, M, N, K);
  if (rc != RG_OK) return rc;
  if (dW == nullptr || !aligned16(dW)) return RG_ERR_INVALID_ARG;
  if (M > 0 && (grad == nullptr || X == nullptr || !aligned16(grad) || !aligned16(X)))
    return RG_ERR_INVALID_ARG;
  const int64_t tiles = static_cast<int64_t>(E) * ((N + rg::kg::TILE_M - 1) / rg::kg::TILE_M) *
                        ((K + rg::kg::BN - 1) / rg::kg::BN);
  if (tiles > INT32_MAX) return RG_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds)) != RG_OK) return rc;
  if (rg::kgemm_smem_bytes(E, ds->max_smem) > ds->max_smem) return RG_ERR_INVALID_ARG;

  // With M == 0 every valid offsets vector is all zeros, so the kernel only
  // writes zero tiles; the operand maps then describe one row of dW, which is
  // never loaded.
  const void* g_ptr = M > 0 ? grad : static_cast<const void*>(dW);
  const void* x_ptr = M > 0 ? X : static_cast<const void*>(dW);
  const uint64_t rows = M > 0 ? static_cast<uint64_t>(M) : 1;

  // Operands as overlapping views in which element (.., i, .., j) is row
  // j + i (i < BR): a box starting at i = v - BR < 0 zero-fills its leading
  // BR - v rows (an expert's ragged last block), and every element the
  // kernel reads lies in rows offsets[e] .. offsets[e+1]-1 of some expert.
  // With N and K multiples of 64 the views are 4-D {64 cols, i, column
  // block, j} and one copy brings a CTA's 64-column boxes of an operand
  // (column block stride 128 bytes); otherwise 3-D {cols, i, j}, one copy
  // per box.
  const bool wide = N % 64 == 0 && K % 64 == 0;
  CUtensorMap tmG, tmX, tmD;
  auto operand_map = [&](CUtensorMap* m, const void* p, int cols, int boxes) {
    const uint64_t pitch = static_cast<uint64_t>(cols) * 2;
    if (wide) {
      const uint64_t dims[4] = {64, rg::kg::BR, static_cast<uint64_t>(cols / 64), rows};
      const uint64_t str[3] = {pitch, 128, pitch};
      const uint32_t box[4] = {64, rg::kg::BR, static_cast<uint32_t>(boxes), 1};
      return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p, dims, str, box);
    }
    const uint64_t dims[3] = {static_cast<uint64_t>(cols), rg::kg::BR, rows};
    const uint64_t str[2] = {pitch, pitch};
    const uint32_t box[3] = {64, rg::kg::BR, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p, dims, str, box);
  };
  if (!operand_map(&tmG, g_ptr, N, rg::kg::BM / 64)) return RG_ERR_INVALID_ARG;
  if (!operand_map(&tmX, x_ptr, K, rg::kg::BN_CTA / 64)) return RG_ERR_INVALID_ARG;
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(E)};
    const uint64_t str[2] = {static_cast<uint64_t>(K) * 4, static_cast<uint64_t>(N) * K * 4};
    const uint32_t box[3] = {static_cast<uint32_t>(rg::kg::BOX_COLS), 32, 1};
    const CUtensorMapSwizzle sw = rg::kg::BOX_COLS == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (!encode_sw(&tmD, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dW, dims, str, box, sw)) return RG_ERR_INVALID_ARG;
  }
  rg::GroupArgs args = group_args(ds, offsets, E, M, N, K, dW);
  args.accumulate = accumulate;
  args.kg_wide = wide ? 1 : 0;
  const int64_t tiles_per_expert = kgemm_flag_bytes(1, N, K) / (rg::kCtaGroup * static_cast<int64_t>(sizeof(int)));
  if (flags != nullptr && tiles_per_expert > ds->kg_grid / rg::kCtaGroup) {
    cudaError_t e = cudaMemsetAsync(flags, 0, static_cast<size_t>(kgemm_flag_bytes(E, N, K)), stream);
    if (e != cudaSuccess) return fail_cuda(e);
    args.flags = flags;
  }
  const cudaError_t e = rg::launch_kgemm(tmG, tmX, tmD, args, ds->kg_grid, ds->max_smem, stream);
  if (e != cudaSuccess) return fail_cuda(e);
  return RG_OK;
}

}  // namespace

extern "C" {

int rg_kgemm(const void* grad, const void* X, const int32_t* offsets, int E, int64_t M, int N, int K,
             float* dW, cudaStream_t stream) {
  return kgemm_impl(grad, X, offsets, E, M, N, K, dW, 0, nullptr, stream);
}

int rg_kgemm_acc(const void* grad, const void* X, const int32_t* offsets, int E, int64_t M, int N,
                 int K, float* dW, cudaStream_t stream) {
  return kgemm_impl(grad, X, offsets, E, M, N, K, dW, 1, nullptr, stream);
}

int64_t rg_kgemm_workspace_bytes(int E, int N, int K) {
  if (E < 1 || E > RG_KGEMM_MAX_EXPERTS || N < 1 || K < 1) return -1;
  return kgemm_flag_bytes(E, N, K);
}

int rg_kgemm_noalloc(const void* grad, const void* X, const int32_t* offsets, int E, int64_t M, int N, int K,
                     float* dW, int accumulate, cudaStream_t stream) {
  const int64_t need = rg_kgemm_workspace_bytes(E, N, K);
  if (need < 0) return RG_ERR_INVALID_ARG;
  if (need > static_cast<int64_t>(sizeof(g_kgemm_noalloc_flags))) return RG_ERR_SCRATCH;
  DeviceState* ds = nullptr;
  const int rc = device_state(&ds);
  if (rc != RG_OK) return rc;
  // kgemm_impl zeroes the flags the problem uses (cudaMemsetAsync on
  // `stream`) before it launches the kernel, where the kernel may use them;
  // nothing is allocated
  return kgemm_impl(grad, X, offsets, E, M, N, K, dW, accumulate != 0, ds->noalloc_flags, stream);
}

int rg_kgemm_ws(const void* grad, const void* X, const int32_t* offsets, int E, int64_t M, int N, int K,
                float* dW, int accumulate, void* workspace, int64_t workspace_bytes, cudaStream_t stream) {
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 3u) != 0) return RG_ERR_INVALID_ARG;
  const int64_t need = rg_kgemm_workspace_bytes(E, N, K);
  if (need < 0 || workspace_bytes < need) return RG_ERR_INVALID_ARG;
  return kgemm_impl(grad, X, offsets, E, M, N, K, dW, accumulate != 0, static_cast<int*>(workspace), stream);
}

int rg_get_device_status(cudaStream_t stream) {
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != RG_OK) return rc;
  return take_status(ds, ds->status, stream);
}

int rg_set_wait_timeout_ns(uint64_t ns) {
  if (ns < kMinWaitLimitNs) return RG_ERR_INVALID_ARG;
  g_wait_limit_ns.store(ns);
  return RG_OK;
}

int rg_selftest_wait_timeout(uint64_t ns, cudaStream_t stream, uint32_t* status) {
  if (ns == 0 || status == nullptr) return RG_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != RG_OK) return rc;
  // the self-test reports through its own word: bits pending in the status
  // word of the GEMM kernels stay there for rg_get_device_status
  if ((rc = take_status(ds, ds->selftest, stream)) < 0) return rc;
  const cudaError_t e = rg::launch_wait_selftest(ds->selftest, ns, stream);
  if (e != cudaSuccess) return fail_cuda(e);
  if ((rc = take_status(ds, ds->selftest, stream)) < 0) return rc;
  *status = static_cast<uint32_t>(rc);
  return RG_OK;
}

int rg_shutdown(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (DeviceState& ds : g_dev) ds = DeviceState{};
  return RG_OK;
}

int rg_last_cuda_error(void) { return t_last_cuda_error; }

int rg_device_supported(void) {
  DeviceState* ds = nullptr;
  return device_state(&ds) == RG_OK ? 1 : 0;
}

const char* rg_version(void) { return "rg 0.1.0 (sm_103a tcgen05 grouped GEMM)"; }

}  // extern "C"
