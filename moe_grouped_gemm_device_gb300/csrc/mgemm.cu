// M-grouped BF16 GEMM for sm_103a: forward (y = x . w[e]^T) and input
// gradient (transpose_B: y = x . w[e]) over expert row groups given by a
// cumulative offsets vector (RapidGEMM README, "Kernels", Mgemm).
//
// Design
//   * Persistent grid, one CTA per SM.  Every CTA reads offsets[0..E] into
//     shared memory, validates it, and builds the tile list itself: expert e
//     contributes ceil(M_e/128) x ceil(N/256) tiles, laid out expert by expert
//     (prefix sums in shared memory).  CTA b takes tiles b, b+G, b+2G, ... so
//     no host synchronisation and no global scratch are needed; empty experts
//     contribute no tiles, tiny ones a single ragged tile.
//   * A tile is rows [offsets[e] + 128 m, +128) x columns [256 n, +256).  Its
//     row window starts at the expert's first row, so it never straddles a
//     group start; rows past the expert's end (which belong to the next
//     expert) are loaded but never stored.
//   * Warp roles (192 threads): warp 0 lane 0 issues TMA loads into a
//     4-stage ring of 48 KB stages (A 128x64 and B 256x64 bf16, 128-byte
//     swizzle); warp 1 owns tensor memory and lane 0 issues tcgen05.mma
//     (M=128, N=256, K=16) into one of two 256-column fp32 accumulators;
//     warps 2-5 drain the other accumulator (tcgen05.ld -> bf16 -> shared
//     memory -> TMA store), so the epilogue overlaps the next tile's MMAs.
//   * Tail rows: a warp whose 32 rows are all inside the expert stores them
//     with one TMA store per 64 columns; otherwise each valid row is written
//     with plain 16-byte stores.
//   * Every mbarrier wait is bounded (WaitGuard).  A wait that runs out sets
//     the device status, all roles stop, in-flight copies and MMAs are drained
//     with bounded waits, and tensor memory is freed before the CTA exits.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace rg {
namespace {

using namespace mg;

constexpr int NUM_BARS = 2 * STAGES + 5;  // full[S], empty[S], tfull[2], tempty[2], drain
constexpr int SMEM_FIXED = 1024 /* alignment slack */ + STAGES * STAGE_BYTES +
                           EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES + NUM_BARS * 8 + 16;
constexpr uint32_t TMEM_COLS = 512;

template <bool TRANS_B>
__global__ void __launch_bounds__(THREADS, 1)
    mgemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmY, const GroupArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);

  uint8_t* epi = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES);
  int* misc = reinterpret_cast<int*>(bars + NUM_BARS);  // [0] tmem base, [1] abort
  int* s_off = misc + 4;                                // [E+1] offsets
  int* s_pre = s_off + (args.E + 1);                    // [E+1] tile prefix

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = args.E;
  const int N = args.N;
  const int K = args.K;
  const int nbn = (N + BN - 1) / BN;
  const int nk = (K + BK - 1) / BK;

  // ---- offsets -> shared memory, validation ---------------------------------
  if (threadIdx.x == 0) misc[1] = 0;
  for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = args.offsets[i];
  __syncthreads();
  int bad = 0;
  for (int i = threadIdx.x; i < E; i += blockDim.x) bad |= (s_off[i + 1] < s_off[i]);
  if (threadIdx.x == 0) bad |= (s_off[0] != 0) | (s_off[E] > args.M);
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(args.status, kDevBadOffsets);
    return;
  }

  // ---- per-expert tile prefix (warp 0, warp-wide scan) ----------------------
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int lo = min(E, lane * per), hi = min(E, lo + per);
    int s = 0;
    for (int e = lo; e < hi; ++e) s += ((s_off[e + 1] - s_off[e] + BM - 1) / BM) * nbn;
    int incl = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - s;
    for (int e = lo; e < hi; ++e) {
      s_pre[e] = run;
      run += ((s_off[e + 1] - s_off[e] + BM - 1) / BM) * nbn;
    }
    if (lane == 31) s_pre[E] = incl;
  }
  __syncthreads();
  const int T = s_pre[E];
  if (static_cast<int>(blockIdx.x) >= T) return;

  // ---- barriers and tensor memory -------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), EPI_WARPS * 32);
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&misc[0]), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const WaitGuard guard{args.status, args.wait_limit_ns, reinterpret_cast<volatile int*>(&misc[1])};

  if (warp == 0) {
    // ======================= TMA producer (one thread) =======================
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;  // stages with a load issued, and its parity
      bool ok = true;
      int e = 0;
      for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
        while (s_pre[e + 1] <= t) ++e;
        const int local = t - s_pre[e];
        const int row0 = s_off[e] + (local / nbn) * BM;
        const int n0 = (local % nbn) * BN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(guard, empty_bar(stage), phase ^ 1u)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          tma_load_2d(sa, &tmA, fb, kb * BK, row0);
          if constexpr (!TRANS_B) {
            tma_load_3d(sb, &tmB, fb, kb * BK, n0, e);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j) tma_load_3d(sb + j * 8192, &tmB, fb, n0 + 64 * j, kb * BK, e);
          }
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {  // let issued loads land before the CTA exits
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s)) mbar_wait_drain(full_bar(s), (armed_par >> s) & 1u, guard.limit_ns);
      }
    }
  } else if (warp == 1) {
    // ========================= MMA issuer (warp 1) ===========================
    constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, false, TRANS_B);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < T; t += gridDim.x, ++acc) {
      const int buf = acc & 1;
      const uint32_t tph = (acc >> 1) & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(guard, tempty_bar(buf), tph ^ 1u));
      if (!ok) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem + buf * BN;
      for (int kb = 0; kb < nk; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(guard, full_bar(stage), phase));
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = sdesc_sw128(sa + 32 * k, 16, 1024);
            const uint64_t bd = TRANS_B ? sdesc_sw128(sb + 2048 * k, 8192, 1024)
                                        : sdesc_sw128(sb + 32 * k, 16, 1024);
            umma_bf16(d_tmem, ad, bd, IDESC, (kb | k) != 0);
          }
          umma_commit(empty_bar(stage));  // frees the stage once these MMAs finish
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) umma_commit(tfull_bar(buf));  // accumulator ready for the epilogue
      __syncwarp();
    }
    if (!ok && lane == 0) {  // wait for issued MMAs before tensor memory is freed
      umma_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0, guard.limit_ns);
    }
    __syncwarp();
  } else {
    // ======================= epilogue (warps 2..5) ===========================
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r_in_tile = q * 32 + lane;
    uint8_t* ebuf = epi + (warp - 2) * EPI_BUFS * EPI_BUF_BYTES;
    const uint32_t ebuf_s = smem_u32(ebuf);
    __nv_bfloat16* y = static_cast<__nv_bfloat16*>(args.out);
    int acc = 0;
    int e = 0;
    for (int t = blockIdx.x; t < T; t += gridDim.x, ++acc) {
      while (s_pre[e + 1] <= t) ++e;
      const int local = t - s_pre[e];
      const int row0 = s_off[e] + (local / nbn) * BM;
      const int rows_valid = min(BM, s_off[e + 1] - row0);
      const int n0 = (local % nbn) * BN;
      const int buf = acc & 1;
      const uint32_t tph = (acc >> 1) & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(guard, tfull_bar(buf), tph))) break;
      tc_fence_after();
      const bool warp_full = q * 32 + 32 <= rows_valid;
      const bool row_ok = r_in_tile < rows_valid;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 64; ++c) {
        uint32_t v0[32], v1[32];
        tmem_ld_32x32b_x32(taddr + 64 * c, v0);
        tmem_ld_32x32b_x32(taddr + 64 * c + 32, v1);
        tmem_ld_wait();
        if (c == BN / 64 - 1) {  // accumulator fully read: hand it back to the MMA warp
          tc_fence_before();
          mbar_arrive(tempty_bar(buf));
        }
        uint32_t p[32];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          p[j] = pack_bf16x2(v0[2 * j], v0[2 * j + 1]);
          p[16 + j] = pack_bf16x2(v1[2 * j], v1[2 * j + 1]);
        }
        const int col0 = n0 + 64 * c;
        if (col0 >= N) continue;
        if (warp_full) {
          if (lane == 0) bulk_wait_read<0>();  // previous store has left the buffer
          __syncwarp();
          uint4* rowp = reinterpret_cast<uint4*>(ebuf + lane * 128);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            rowp[j ^ (lane & 7)] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmY, ebuf_s, col0, row0 + q * 32);
            bulk_commit();
          }
        } else if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(y + (static_cast<int64_t>(row0 + r_in_tile) * N + col0));
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (col0 + 8 * j < N) dst[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
        }
      }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  // ---- teardown --------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

size_t mgemm_smem_bytes(int E) { return SMEM_FIXED + 2 * (static_cast<size_t>(E) + 1) * 4; }

cudaError_t mgemm_setup(int max_smem) {
  const int max_bytes = static_cast<int>(std::min<size_t>(mgemm_smem_bytes(1024), max_smem));
  cudaError_t e = cudaFuncSetAttribute(mgemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mgemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_bytes);
}

cudaError_t launch_mgemm(bool transpose_B, const CUtensorMap& tmA, const CUtensorMap& tmB,
                         const CUtensorMap& tmY, const GroupArgs& args, int grid,
                         cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = mgemm_smem_bytes(args.E);
  cfg.stream = stream;
  if (transpose_B) return cudaLaunchKernelEx(&cfg, mgemm_kernel<true>, tmA, tmB, tmY, args);
  return cudaLaunchKernelEx(&cfg, mgemm_kernel<false>, tmA, tmB, tmY, args);
}

}  // namespace rg
