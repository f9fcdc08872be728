// K-grouped weight gradient with FP32 output for sm_103a:
//   dW[e] = grad[rows of e]^T . X[rows of e]      (RapidGEMM README, "Kernels", Kgemm)
// grad is [M,N], X is [M,K], dW is [E,N,K]; the contraction runs over the rows
// offsets[e] .. offsets[e+1]-1 of expert e, whose bounds may fall anywhere.
//
// Design
//   * Output tiles are (e, n-block of 128, k-block of 256); every expert has
//     the same number of tiles, so the tile list is E x ceil(N/128) x
//     ceil(K/256).  Experts are visited in decreasing row count (ties by
//     index), which every CTA computes itself in shared memory; CTA b takes
//     tiles b, b+G, ..., so each round of G tiles has near-equal cost
//     (longest-first list scheduling) without global scratch or host sync.
//   * The contraction is fed 64 rows at a time: A = grad[r:r+64, n0:n0+128]
//     and B = X[r:r+64, k0:k0+256], both N/K-contiguous, i.e. MN-major
//     operands of tcgen05.mma (M=128, N=256, K=16).  Rows of the last block
//     that lie past the expert's end belong to the next expert: the MMA warp
//     zeroes them in shared memory (both operands, so no NaN/Inf can leak)
//     and fences them into the async proxy before issuing the MMAs.
//   * The fp32 accumulator (128 lanes x 256 columns, double-buffered in
//     tensor memory) holds at most CHUNK_ROWS rows of one expert: a longer
//     expert is summed chunk by chunk, the first chunk's partial stored to dW
//     and each later one added to it by a TMA fp32 reduce-add, in order.  This
//     bounds the fp32 accumulation chain inside the tensor cores (whose error
//     grows with its length) without any scratch memory.  The path to dW is
//     tcgen05.ld -> swizzled shared memory -> TMA store / reduce-add of 32x32
//     fp32 boxes.  Experts without rows produce zero tiles without touching
//     the tensor cores.
//   * Same bounded-wait / abort / drain scheme as the M-grouped kernel.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace rg {
namespace {

using namespace kg;

constexpr int NUM_BARS = 2 * STAGES + 5;
// The dynamic shared-memory window of a CTA without static shared memory
// starts 1024-byte aligned; the kernel checks this instead of padding for it.
constexpr int SMEM_FIXED = STAGES * STAGE_BYTES + EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES +
                           NUM_BARS * 8 + 16;
constexpr uint32_t TMEM_COLS = 512;
constexpr int BOX_BYTES = BR * 128;  // one 64-element-wide box of BR rows

__global__ void __launch_bounds__(THREADS, 1)
    kgemm_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmX,
                 const __grid_constant__ CUtensorMap tmD, const GroupArgs args) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // swizzled TMA boxes and MMA descriptors need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(args.status, kDevLaunchConfig);
    return;
  }

  uint8_t* epi = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES);
  int* misc = reinterpret_cast<int*>(bars + NUM_BARS);  // [0] tmem base, [1] abort
  int* s_off = misc + 4;                                // [E+1] offsets
  int* s_ord = s_off + (args.E + 1);                    // [E] experts by decreasing rows

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
  const int nbn = (N + BM - 1) / BM;
  const int nbk = (K + BN - 1) / BN;
  const int tpe = nbn * nbk;
  const int T = E * tpe;

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
  if (static_cast<int>(blockIdx.x) >= T) return;

  // ---- experts ordered by decreasing row count (stable) ---------------------
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int ce = s_off[e + 1] - s_off[e];
    int rank = 0;
    for (int f = 0; f < E; ++f) {
      const int cf = s_off[f + 1] - s_off[f];
      rank += (cf > ce) | ((cf == ce) & (f < e));
    }
    s_ord[rank] = e;
  }

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
      tma_prefetch_desc(&tmG);
      tma_prefetch_desc(&tmX);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
        const int p = t / tpe;
        const int e = s_ord[p];
        const int local = t - p * tpe;
        const int n0 = (local / nbk) * BM;
        const int k0 = (local % nbk) * BN;
        const int r_begin = s_off[e], r_end = s_off[e + 1];
        for (int r = r_begin; r < r_end; r += BR) {
          if (!mbar_wait(guard, empty_bar(stage), phase ^ 1u)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
#pragma unroll
          for (int j = 0; j < BM / 64; ++j) tma_load_2d(sa + j * BOX_BYTES, &tmG, fb, n0 + 64 * j, r);
#pragma unroll
          for (int j = 0; j < BN / 64; ++j) tma_load_2d(sb + j * BOX_BYTES, &tmX, fb, k0 + 64 * j, r);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s)) mbar_wait_drain(full_bar(s), (armed_par >> s) & 1u, guard.limit_ns);
      }
    }
  } else if (warp == 1) {
    // ========================= MMA issuer (warp 1) ===========================
    constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, true, true);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
      const int e = s_ord[t / tpe];
      const int r_begin = s_off[e], r_end = s_off[e + 1];
      // zero tile (no rows): no MMA, no accumulator.  Otherwise one
      // accumulator per chunk of at most CHUNK_ROWS rows.
      for (int cr = r_begin; cr < r_end && ok; cr += CHUNK_ROWS) {
        const int c_end = min(r_end, cr + CHUNK_ROWS);
        const int buf = acc & 1;
        const uint32_t tph = (acc >> 1) & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(guard, tempty_bar(buf), tph ^ 1u));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * BN;
        for (int r = cr; r < c_end; r += BR) {
          ok = __all_sync(0xffffffffu, mbar_wait(guard, full_bar(stage), phase));
          if (!ok) break;
          const int valid = min(BR, r_end - r);
          if (valid < BR) {
            // rows [valid, BR) belong to the next expert (or lie past M): zero
            // them in all six boxes of the stage before the tensor cores read it
            uint8_t* st = smem + stage * STAGE_BYTES;
            const int units = (BR - valid) * 8;  // 16-byte units per box
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
            for (int b = 0; b < STAGE_BYTES / BOX_BYTES; ++b) {
              uint4* bp = reinterpret_cast<uint4*>(st + b * BOX_BYTES + valid * 128);
              for (int u = lane; u < units; u += 32) bp[u] = z;
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
          tc_fence_after();
          if (lane == 0) {
            const uint32_t sa = sbase + stage * STAGE_BYTES;
            const uint32_t sb = sa + A_BYTES;
#pragma unroll
            for (int k = 0; k < BR / 16; ++k) {
              const uint64_t ad = sdesc_sw128(sa + 2048 * k, BOX_BYTES, 1024);
              const uint64_t bd = sdesc_sw128(sb + 2048 * k, BOX_BYTES, 1024);
              umma_bf16(d_tmem, ad, bd, IDESC, (r != cr) | (k != 0));
            }
            umma_commit(empty_bar(stage));
          }
          __syncwarp();
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (lane == 0) umma_commit(tfull_bar(buf));
        __syncwarp();
        ++acc;
      }
    }
    if (!ok && lane == 0) {
      umma_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0, guard.limit_ns);
    }
    __syncwarp();
  } else {
    // ======================= epilogue (warps 2..5) ===========================
    // Warp q owns rows n0 + 32q .. +31 of the tile; each 32x32 fp32 box goes
    // through one of EPI_BUFS rotating staging buffers.  The first chunk of
    // an expert's rows is stored, later chunks are reduce-added; before a
    // later chunk the warp waits until its previous writes have landed, so
    // the adds are applied in chunk order (deterministic).
    const int q = warp & 3;
    uint8_t* ebase = epi + (warp - 2) * EPI_BUFS * EPI_BUF_BYTES;
    int acc = 0;
    uint32_t nstore = 0;
    bool ok = true;
    auto stage_buf = [&](const uint32_t (&v)[32]) -> uint32_t {
      const uint32_t b = nstore % EPI_BUFS;
      if (lane == 0) bulk_wait_read<EPI_BUFS - 1>();  // buffer b is no longer read
      __syncwarp();
      uint4* rowp = reinterpret_cast<uint4*>(ebase + b * EPI_BUF_BYTES + lane * 128);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        rowp[j ^ (lane & 7)] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      ++nstore;
      return smem_u32(ebase + b * EPI_BUF_BYTES);
    };
    for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
      const int p = t / tpe;
      const int e = s_ord[p];
      const int local = t - p * tpe;
      const int n0 = (local / nbk) * BM;
      const int k0 = (local % nbk) * BN;
      const int r_begin = s_off[e], r_end = s_off[e + 1];
      const bool warp_rows = n0 + q * 32 < N;  // this warp's 32 rows of dW exist
      if (r_end == r_begin) {  // expert without rows: dW tile = 0
        if (!warp_rows) continue;
        uint32_t z[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) z[j] = 0u;
#pragma unroll 1
        for (int c = 0; c < BN / 32 && k0 + 32 * c < K; ++c) {
          const uint32_t src = stage_buf(z);
          if (lane == 0) {
            tma_store_3d(&tmD, src, k0 + 32 * c, n0 + q * 32, e);
            bulk_commit();
          }
        }
        continue;
      }
      for (int cr = r_begin; cr < r_end; cr += CHUNK_ROWS) {
        const bool first = cr == r_begin;
        const int buf = acc & 1;
        const uint32_t tph = (acc >> 1) & 1;
        ++acc;
        ok = __all_sync(0xffffffffu, mbar_wait(guard, tfull_bar(buf), tph));
        if (!ok) break;
        tc_fence_after();
        if (!first && lane == 0) bulk_wait<0>();  // previous partial of this tile is in dW
        const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(taddr + 32 * c, v);
          tmem_ld_wait();
          if (c == BN / 32 - 1) {  // accumulator fully read: hand it back
            tc_fence_before();
            mbar_arrive(tempty_bar(buf));
          }
          if (!warp_rows || k0 + 32 * c >= K) continue;
          const uint32_t src = stage_buf(v);
          if (lane == 0) {
            if (first)
              tma_store_3d(&tmD, src, k0 + 32 * c, n0 + q * 32, e);
            else
              tma_reduce_add_3d(&tmD, src, k0 + 32 * c, n0 + q * 32, e);
            bulk_commit();
          }
        }
      }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

__global__ void wait_selftest_kernel(unsigned int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitGuard g{status, limit_ns, &abort_flag};
  // Nothing ever arrives on `bar`: the wait must give up after limit_ns.
  if (threadIdx.x == 0) mbar_wait(g, smem_u32(&bar), 0);
  __syncthreads();
}

}  // namespace

size_t kgemm_smem_bytes(int E) { return SMEM_FIXED + (2 * static_cast<size_t>(E) + 1) * 4; }

cudaError_t kgemm_setup(int max_smem) {
  return cudaFuncSetAttribute(kgemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(std::min<size_t>(kgemm_smem_bytes(1024), max_smem)));
}

cudaError_t launch_kgemm(const CUtensorMap& tmG, const CUtensorMap& tmX, const CUtensorMap& tmD,
                         const GroupArgs& args, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = kgemm_smem_bytes(args.E);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kgemm_kernel, tmG, tmX, tmD, args);
}

cudaError_t launch_wait_selftest(unsigned int* status, unsigned long long limit_ns,
                                 cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, wait_selftest_kernel, status, limit_ns);
}

}  // namespace rg
