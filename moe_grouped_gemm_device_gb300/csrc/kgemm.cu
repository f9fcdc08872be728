// K-grouped weight gradient with FP32 output for sm_103a:
//   dW[e] = grad[rows of e]^T . X[rows of e]      (RapidGEMM README, "Kernels", Kgemm)
// grad is [M,N], X is [M,K], dW is [E,N,K]; the contraction runs over the rows
// offsets[e] .. offsets[e+1]-1 of expert e, whose bounds may fall anywhere.
//
// Design
//   * Output tiles are (e, n-block of TILE_M, k-block of 256); every expert
//     has the same number of tiles, so the tile list is E x ceil(N/TILE_M) x
//     ceil(K/256).  Every CTA sorts the experts by decreasing row count (ties
//     by index) in shared memory; worker w takes tiles w, w+W, ... of that
//     list, so every round of W tiles has near-equal cost (longest-first list
//     scheduling) -- without global scratch or host sync.  A worker issues
//     the tiles of its experts below LIGHT_ROWS rows (whose stores outlast
//     their MMAs) one at a time between the row blocks of its other tiles,
//     so that their stores overlap tensor-core work (kgemm_plan.cuh).  With a
//     flag workspace (chunk mode) a long expert's tiles instead share each
//     row chunk in one round, handing the partial sums on through flags.
//   * The contraction is fed BR = 96 rows at a time, six MMA steps of 16
//     rows per barrier round of the MMA warp, through a ring of four stages
//     (48 KB per CTA each): three stages ahead of the tensor cores hide the
//     copies' latency better than two of 128 rows.  With CG = 2 (default) a CTA
//     pair computes a 256x256 dW tile with tcgen05.mma.cta_group::2: for the
//     row block starting at r, CTA c loads grad[r:r+BR, n0+128c : +128] (A,
//     its 128 rows of dW) and X[r:r+BR, k0+128c : +128] (its half of B); both
//     are N/K-contiguous, i.e. MN-major operands.  CG = 1: one CTA, 128x256
//     tiles, two 72 KB stages.
//   * Both operands are read through 3-D views {columns, i < BR, j} of the
//     row-major tensors in which element (c, i, j) is row i + j (both row
//     strides equal the pitch).  A full block loads box (c, 0, r): rows
//     r .. r+BR-1.  An expert's ragged last block of v < BR rows loads box
//     (c, v-BR, r): its first BR-v rows have i < 0 and are zero-filled by the
//     copy engine, the expert's rows r .. r+v-1 land in the last v rows, and
//     no row past the expert is read.  The MMAs skip the leading all-zero
//     16-row steps.  With N and K multiples of 64 the views are 4-D,
//     {64 cols, i, column block, j}, and one copy per operand and stage
//     brings both of the CTA's 64-column boxes.  So no block needs fixing up
//     in shared memory, and the copies of both CTAs complete their bytes on
//     the issuing CTA's stage barrier (.cta_group::2) for every block alike.
//   * The fp32 accumulator (128 lanes x 256 columns per CTA, double-buffered
//     in tensor memory) holds at most CHUNK_ROWS rows of one expert: a longer
//     expert is summed chunk by chunk, the first chunk's partial stored to dW
//     and each later one added to it by a TMA fp32 reduce-add, in order.  This
//     bounds the fp32 accumulation chain inside the tensor cores (whose error
//     grows with its length) without any scratch memory.  The path to dW is
//     tcgen05.ld -> swizzled shared memory -> TMA store / reduce-add of 32x32
//     fp32 boxes (whole 128-byte lines) with an L2 evict-first policy (dW is
//     written once and not read here).  Experts without rows produce zero
//     tiles without touching the tensor cores.
//   * Same bounded-wait / abort / drain scheme as the M-grouped kernel: every
//     wait is bounded, a wait that runs out stops every role of the CTA, and
//     at the end the issuing CTA waits for every copy either CTA issued.
#include <algorithm>

#include "bounds.cuh"
#include "internal.h"
#include "kgemm_plan.cuh"
#include "ptx.cuh"
#include "rg.h"

namespace rg {
namespace {

template <int CG, int ST>
struct Cfg {
  static constexpr int BM = 128;           // dW rows per CTA (MMA M per CTA)
  static constexpr int TILE_M = BM * CG;   // dW rows per tile
  static constexpr int BN = 256;           // dW columns per tile (MMA N)
  static constexpr int BN_CTA = BN / CG;   // X columns loaded per CTA
  static constexpr int BR = kg::BR;        // rows of the contraction per stage
  static constexpr int STAGES = ST;
  static constexpr int BOX_BYTES = BR * 128;  // one 64-element-wide box of BR rows
  static constexpr int A_BYTES = BM * BR * 2;
  static constexpr int B_BYTES = BN_CTA * BR * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int EPI_WARPS = 8;              // two per TMEM lane quarter
  static constexpr int EPI_GROUP = kg::EPI_GROUP;  // dW boxes staged per bulk group
  static constexpr int BOX_COLS = kg::BOX_COLS;    // fp32 columns of a 32-row dW box
  static constexpr int DW_BOX_BYTES = 32 * BOX_COLS * 4;
  static constexpr int EPI_BUF_BYTES = DW_BOX_BYTES * EPI_GROUP;  // per epilogue warp
  // warp 0 and the last warp: TMA producers (alternate stages), warp 1: MMA,
  // warps 2..9: epilogue
  static constexpr int PRODUCER2 = 2 + EPI_WARPS;
  static constexpr int THREADS = 32 * (PRODUCER2 + 1);
  // full[S], empty[S], tfull[2], tempty[2], drain, published
  static constexpr int NUM_BARS = 2 * STAGES + 6;
  // The dynamic shared-memory window of a CTA without static shared memory
  // starts 1024-byte aligned; the kernel checks this instead of padding.
  static constexpr int SMEM_FIXED = STAGES * STAGE_BYTES + EPI_WARPS * EPI_BUF_BYTES + NUM_BARS * 8 +
                                    static_cast<int>(sizeof(IssueLog<STAGES>)) + 16;
};

constexpr uint32_t TMEM_COLS = 512;
constexpr int CHUNK_ROWS = kg::CHUNK_ROWS;
constexpr int LIGHT_ROWS = kg::LIGHT_ROWS;
// An expert whose operand rows take more than half of the 126 MB L2 cannot
// keep them there between two rounds of its tiles.
constexpr long long kKmajorBytes = 64ll << 20;


template <int CG, int ST>
__global__ void __launch_bounds__(Cfg<CG, ST>::THREADS, 1)
    kgemm_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmX,
                 const __grid_constant__ CUtensorMap tmD, const GroupArgs args) {
  using C = Cfg<CG, ST>;
  constexpr int BM = C::BM, TILE_M = C::TILE_M, BN = C::BN, BN_CTA = C::BN_CTA, BR = C::BR;
  constexpr int STAGES = C::STAGES, A_BYTES = C::A_BYTES, STAGE_BYTES = C::STAGE_BYTES;
  constexpr int BOX_BYTES = C::BOX_BYTES, EPI_BUF_BYTES = C::EPI_BUF_BYTES;

  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // swizzled TMA boxes and MMA descriptors need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(args.status, kDevLaunchConfig);
    return;
  }
  uint8_t* epi = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + C::EPI_WARPS * EPI_BUF_BYTES);
  IssueLog<STAGES>* ilog = reinterpret_cast<IssueLog<STAGES>*>(bars + C::NUM_BARS);
  int* misc = reinterpret_cast<int*>(ilog + 1);  // [0] tmem base, [1] abort
  int* s_off = misc + 4;                                   // [E+1] offsets
  int* s_ord = s_off + (args.E + 1);                       // [E] experts by decreasing rows
  int* s_up = s_ord + args.E;                              // [E+1] chunk mode: first item of each

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  // chunk mode: every epilogue warp's writes of a chunk that a later chunk
  // of the same tile adds to have completed
  const uint32_t pub_bar = bar0 + 8u * (2 * STAGES + 5);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;  // rank 0 issues the MMAs
  const int worker = blockIdx.x / CG;
  const int nworkers = gridDim.x / CG;
  const int E = args.E;
  const int N = args.N;
  const int K = args.K;
  const int nbn = (N + TILE_M - 1) / TILE_M;
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
  if (__syncthreads_or(bad)) {  // both CTAs of a pair see the same offsets and leave together
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(args.status, kDevBadOffsets);
    return;
  }
  // Chunk mode changes the schedule only where an expert's tiles outnumber
  // the workers (they then run in more than one round) and some expert is
  // longer than one chunk; otherwise all of an expert's tiles walk its rows
  // together in one round, which reads them once, and the tile list is used.
  // (The first two conditions are the same in every CTA.)
  bool chunked = args.flags != nullptr && tpe > nworkers;
  if (chunked) {
    int longest = 0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) longest |= (s_off[e + 1] - s_off[e]) > CHUNK_ROWS;
    chunked = __syncthreads_or(longest);
  }
  if (!chunked && worker >= T) return;  // (chunk mode: once its item count is known)

  // ---- experts ordered by decreasing row count (stable) ---------------------
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int ce = s_off[e + 1] - s_off[e];
    int rank_e = 0;
    for (int f = 0; f < E; ++f) {
      const int cf = s_off[f + 1] - s_off[f];
      rank_e += (cf > ce) | ((cf == ce) & (f < e));
    }
    s_ord[rank_e] = e;
  }
  // Work items.  Tile mode (no flags): item i is tile i of the list, with all
  // of its row chunks.  Chunk mode (args.flags): item i is one row chunk of
  // one tile; each expert's items run chunk by chunk (chunk 0 of all its
  // tiles, then chunk 1, ...), so that the tiles of an expert too long for
  // one chunk read each chunk of its rows from DRAM once, in the same round
  // of the grid; a chunk's reduce-add into dW waits for the previous chunk's
  // writes (a flag per tile half), so the chunks are still added in row order.
  const kgplan::Tables tb{s_off, s_ord, s_up, E, tpe, chunked, CHUNK_ROWS};
  if (chunked) {
    __syncthreads();  // s_ord complete
    if (warp == 0) {  // s_up[p] = items of the experts before position p of the order (warp scan)
      const int per = (E + 31) / 32;
      const int lo = min(E, lane * per), hi = min(E, lo + per);
      int sum = 0;
      for (int p = lo; p < hi; ++p) sum += tb.nchunks(s_ord[p]) * tpe;
      int incl = sum;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
      }
      int run = incl - sum;
      for (int p = lo; p < hi; ++p) {
        s_up[p] = run;
        run += tb.nchunks(s_ord[p]) * tpe;
      }
      if (lane == 31) s_up[E] = incl;
    }
    __syncthreads();
    if (worker >= s_up[E]) return;  // same decision in both CTAs of a pair
  }

  // ---- barriers and tensor memory -------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), C::EPI_WARPS * CG);
    }
    mbar_init(drain_bar, 1);
    mbar_init(pub_bar, C::EPI_WARPS);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<CG>(smem_u32(&misc[0]), TMEM_COLS);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const WaitGuard guard{args.status, args.wait_limit_ns, reinterpret_cast<volatile int*>(&misc[1])};
  auto wait_pair = [&](uint32_t bar, uint32_t par) {
    if constexpr (CG == 2) return mbar_wait_cl(guard, bar, par);
    else return mbar_wait(guard, bar, par);
  };
  // (n block, k block) of an expert's tile.  The tiles of an expert run over
  // more than one round of the grid; if its operand rows overflow L2 between
  // rounds, the second round reads again the operand whose blocks the first
  // round did not finish.  Tiles go n-major (k blocks vary fastest: grad's
  // n blocks are finished in turn, X is read again) unless the expert is that
  // large and grad is the narrower operand (N < K): then k-major.
  auto kmajor = [&](int e) {
    const long long bytes = 2ll * (s_off[e + 1] - s_off[e]) * (N + K);
    return N < K && bytes > kKmajorBytes;
  };
  auto nblk = [&](int e, int local) { return kmajor(e) ? local % nbn : local / nbk; };
  auto kblk = [&](int e, int local) { return kmajor(e) ? local / nbn : local % nbk; };
  // The worker's issue order: heavy items' row blocks with the light items
  // interleaved (kgemm_plan.cuh).
  using kgplan::Acc;
  using kgplan::Item;
  const kgplan::Plan plan = kgplan::make_plan(tb, worker, nworkers, BR, LIGHT_ROWS);
  auto walk = [&](auto&& on_segment, auto&& on_zero) { return kgplan::walk(tb, plan, on_segment, on_zero); };
  if (warp == 0 || warp == C::PRODUCER2) {
    // ============ TMA producers (lane 0 of warp 0 and of the last warp) =====
    // One thread issuing every copy caps the copy rate of a CTA below what
    // the tensor cores consume, so two threads take turns: each walks the
    // whole (tile, row-block) sequence and fills every other stage.
    if (lane == 0) {
      tma_prefetch_desc(&tmG);
      tma_prefetch_desc(&tmX);
      [[maybe_unused]] const uint64_t op_policy = RG_KG_LOAD_HINT ? l2_policy_evict_last() : 0;
      const uint32_t pid = warp == 0 ? 0u : 1u;
      issue_log_init(ilog, pid);
      uint32_t it = 0;
      int stage = 0;
      uint32_t phase = 0;
      const uint32_t full_issuer = CG == 2 ? mapa_shared(full_bar(0), 0) : full_bar(0);
      int e = -1, local = -1, n0 = 0, k0 = 0, r_begin = 0, r_end = 0;  // the item of the last copy
      walk(
          [&](const Item& itm, int, int, int, int r0, int r1, Acc, bool, bool) {
            if (itm.e != e || itm.local != local) {
              e = itm.e;
              local = itm.local;
              n0 = nblk(e, local) * TILE_M + static_cast<int>(rank) * BM;
              k0 = kblk(e, local) * BN + static_cast<int>(rank) * BN_CTA;
              r_begin = s_off[e];
              r_end = s_off[e + 1];
            }
            for (int r = r0; r < r1; r += BR) {
              if ((it++ & 1u) != pid) {  // the other producer's stage
                if (++stage == STAGES) {
                  stage = 0;
                  phase ^= 1u;
                }
                continue;
              }
              // Everything about the copy is worked out before the wait: between
              // the stage becoming free and its copy starting is the critical path.
              const uint32_t sa = sbase + stage * STAGE_BYTES;
              const uint32_t sb = sa + A_BYTES;
              // i0 < 0 for the expert's ragged last block: its leading -i0 rows
              // are zero-filled and its last rows are r .. r_end-1.
              const int i0 = min(0, r_end - r - BR);
              const uint32_t fb = full_issuer + 8u * stage;
              // (debug-bounds build: every in-range row of the box must be a row
              // of expert e; a refused copy's bytes are counted as arrived)
              const bool rows_ok = !RG_DEBUG_BOUNDS || bounds::kgemm_rows(r, i0, BR, r_begin, r_end);
              if (!wait_pair(empty_bar(stage), phase ^ 1u)) return false;
              if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), STAGE_BYTES * CG);
              if (args.kg_wide) {  // one copy per operand: column blocks n0/64 .. and k0/64 ..
                if (RG_BOUNDS_OK(rows_ok && n0 % 64 == 0, args.status)) {
                  if constexpr (RG_KG_LOAD_HINT && CG == 2) tma_load_4d_pair_hint(sa, &tmG, fb, 0, i0, n0 / 64, r, op_policy);
                  else tma_load_4d_cg<CG>(sa, &tmG, fb, 0, i0, n0 / 64, r);
                } else {
                  mbar_complete_tx_cluster(fb, A_BYTES);
                }
                if (RG_BOUNDS_OK(rows_ok && k0 % 64 == 0, args.status)) {
                  if constexpr (RG_KG_LOAD_HINT && CG == 2) tma_load_4d_pair_hint(sb, &tmX, fb, 0, i0, k0 / 64, r, op_policy);
                  else tma_load_4d_cg<CG>(sb, &tmX, fb, 0, i0, k0 / 64, r);
                } else {
                  mbar_complete_tx_cluster(fb, C::B_BYTES);
                }
              } else {
    #pragma unroll
                for (int j = 0; j < BM / 64; ++j) {
                  if (RG_BOUNDS_OK(rows_ok && bounds::inner_aligned(n0 + 64 * j, 2), args.status))
                    tma_load_3d_cg<CG>(sa + j * BOX_BYTES, &tmG, fb, n0 + 64 * j, i0, r);
                  else
                    mbar_complete_tx_cluster(fb, BOX_BYTES);
                }
    #pragma unroll
                for (int j = 0; j < BN_CTA / 64; ++j) {
                  if (RG_BOUNDS_OK(rows_ok && bounds::inner_aligned(k0 + 64 * j, 2), args.status))
                    tma_load_3d_cg<CG>(sb + j * BOX_BYTES, &tmX, fb, k0 + 64 * j, i0, r);
                  else
                    mbar_complete_tx_cluster(fb, BOX_BYTES);
                }
              }
              ilog->it[pid][stage] = static_cast<int>(it - 1);
              ilog->bytes[pid][stage] = STAGE_BYTES;
              if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
              }
            }
            return true;
          },
          [](const Item&) { return true; });
    }
  } else if (warp == 1 && rank == 0) {
    // ========================= MMA issuer (warp 1) ===========================
    constexpr uint32_t IDESC = idesc_bf16_f32(TILE_M, BN, true, true);
    int stage = 0;
    uint32_t phase = 0;
    // One accumulator per chunk of at most CHUNK_ROWS rows of an item; an
    // item without rows has neither MMAs nor an accumulator.
    const bool ok = walk(
        [&](const Item&, int, int cs, int ce, int r0, int r1, Acc a, bool first, bool last) {
          const uint32_t d_tmem = tmem + a.buf * BN;
          if (first) {
            if (!__all_sync(0xffffffffu, wait_pair(tempty_bar(a.buf), a.par ^ 1u))) return false;
            tc_fence_after();
          }
          for (int r = r0; r < r1; r += BR) {
            // the expert's ragged last block starts with all-zero 16-row steps
            // (a chunk that ends before the expert ends is whole row blocks)
            const int k_first = max(0, r + BR - ce) / 16;
            const uint32_t sa = sbase + stage * STAGE_BYTES;
            const uint32_t sb = sa + A_BYTES;
            if (!__all_sync(0xffffffffu, wait_pair(full_bar(stage), phase))) return false;
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
              for (int k = 0; k < BR / 16; ++k) {
                if (k >= k_first) {
                  const uint64_t ad = sdesc_sw128(sa + 2048 * k, BOX_BYTES, 1024);
                  const uint64_t bd = sdesc_sw128(sb + 2048 * k, BOX_BYTES, 1024);
                  umma_bf16<CG>(d_tmem, ad, bd, IDESC, (r != cs) | (k != k_first));
                }
              }
              umma_commit<CG>(empty_bar(stage));
            }
            __syncwarp();
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (last) {
            if (lane == 0) umma_commit<CG>(tfull_bar(a.buf));
            __syncwarp();
          }
          return true;
        },
        [](const Item&) { return true; });
    if (!ok && lane == 0) {  // wait for issued MMAs before tensor memory is freed
      umma_commit_local<CG>(drain_bar);
      mbar_wait_drain(drain_bar, 0);
    }
    __syncwarp();
  } else if (warp == 1) {
    // peer CTA of a pair: its tensor cores are driven by the issuing CTA
  } else {
    // ======================= epilogue (warps 2..9) ===========================
    // Warp w owns TMEM lane quarter q = w % 4 (dW rows n0 + 32q .. +31 of this
    // CTA's half of the tile) and column half h (128 of the 256 columns).  It
    // pulls its whole 32x128 slice into registers with four back-to-back
    // tcgen05.ld, hands the accumulator back at once -- so the MMAs of the
    // next-but-one tile never wait for the stores -- and then writes the
    // fp32 boxes: registers -> swizzled staging buffer -> TMA store (whole
    // 128-byte lines).  The first chunk of an expert's rows is stored
    // (reduce-added when accumulating into dW), later chunks are TMA
    // reduce-added, in chunk order: in tile mode the warp waits until its
    // previous writes have landed; in chunk mode, where the chunks of a tile
    // run on different CTAs, it waits for the tile half's flag, which the CTA
    // that wrote the previous chunk raises once all of its writes are in dW.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    uint8_t* ebuf = epi + (warp - 2) * EPI_BUF_BYTES;
    const uint32_t ebuf_s = smem_u32(ebuf);
    constexpr int GB = C::EPI_GROUP;
    constexpr int BC = C::BOX_COLS, BOXB = C::DW_BOX_BYTES;
    constexpr int NBOX = (BN / 2) / BC;  // boxes of this warp's 128 columns
    // staging swizzle: 16-byte chunk ^= row % 8 (128-byte rows) or (row / 2) % 4 (64-byte rows)
    const int sw = BC == 32 ? (lane & 7) : ((lane >> 1) & 3);
    const uint32_t tempty_issuer = CG == 2 ? mapa_shared(tempty_bar(0), 0) : tempty_bar(0);
    // dW is written once and never read here: first out of L2, so that the
    // operand rows other tiles of the expert still need stay resident
    const uint64_t dw_policy = l2_policy_evict_first();
    // Stage the boxes of one bulk group: the values of box b at v + BC b
    // (v = null: zeros) into slot b of this warp's buffer, after the previous
    // group has left the buffer; one proxy fence for all of them.
    auto stage_group = [&](const uint32_t* v, int nb) {
      if (lane == 0) bulk_wait_read<0>();
      __syncwarp();
#pragma unroll
      for (int b = 0; b < GB; ++b) {
        if (b >= nb) break;
        uint4* rowp = reinterpret_cast<uint4*>(ebuf + b * BOXB + lane * BC * 4);
#pragma unroll
        for (int j = 0; j < BC / 4; ++j)
          rowp[j ^ sw] = v ? make_uint4(v[BC * b + 4 * j], v[BC * b + 4 * j + 1], v[BC * b + 4 * j + 2],
                                        v[BC * b + 4 * j + 3])
                           : make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
      __syncwarp();
    };
    // boxes of this warp's 128 columns at kh that lie below K, from box c0 on, at most GB
    auto group_boxes = [&](int kh, int c0) { return min(GB, (K - kh - BC * c0 + BC - 1) / BC); };
    auto release_acc = [&](int buf) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 2) mbar_arrive_cluster(tempty_issuer + 8u * buf);
        else mbar_arrive(tempty_bar(buf));
      }
    };
    // a 32-row x BC-column fp32 box of dW[e] at (column k, row n): inside dW, 16-byte aligned start
    auto dw_box_ok = [&](int k, int n, int ee) {
      return bounds::inner_aligned(k, 4) && bounds::within(k, BC, K) && bounds::within(n, 32, N) &&
             bounds::index_ok(ee, E);
    };
    uint32_t pub_par = 0;  // chunk mode, warp 2: parity of pub_bar's next phase
    walk(  // the accumulators in the order they end
        [&](const Item& itm, int c, int, int, int, int, Acc a, bool, bool last) {
          if (!last) return true;
          const int e = itm.e;
          const int n0 = nblk(e, itm.local) * TILE_M + static_cast<int>(rank) * BM;
          const int kh = kblk(e, itm.local) * BN + h * (BN / 2);  // first dW column of this warp
          const bool warp_rows = n0 + q * 32 < N;  // this warp's 32 rows of dW exist
          // chunk mode: this CTA's half of the tile is handed from chunk to
          // chunk through its flag (the number of chunks whose writes are in dW)
          int* flag = chunked ? args.flags + (static_cast<int64_t>(e) * tpe + itm.local) * CG + rank : nullptr;
          const bool first = c == 0;
          const bool overwrite = first && !args.accumulate;
          if (!warp_wait_acc<CG>(guard, tfull_bar(a.buf), a.par)) return false;
          tc_fence_after();
          if (!warp_rows) {
            release_acc(a.buf);
          } else {
            uint32_t v[BN / 2];
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + a.buf * BN + h * (BN / 2);
#pragma unroll
            for (int b = 0; b < BN / 64; ++b)
              tmem_ld_32x32b_x32(taddr + 32 * b, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * b));
            tmem_ld_wait();
            release_acc(a.buf);  // accumulator fully read: hand it back
            if (!first) {  // the previous chunk of this tile half must be in dW
              if (!chunked) {
                if (lane == 0) bulk_wait<0>();
              } else if (__shfl_sync(0xffffffffu, lane == 0 ? (flag_wait_ge(guard, flag, c) ? 1 : 0) : 0, 0) == 0) {
                return false;
              }
            }
#pragma unroll
            for (int c0 = 0; c0 < NBOX; c0 += GB) {
              if (kh + BC * c0 >= K) break;
              const int nb = group_boxes(kh, c0);
              stage_group(v + BC * c0, nb);
              if (lane == 0) {
                for (int b = 0; b < nb; ++b) {
                  const int kb = kh + BC * (c0 + b);
                  if (!RG_BOUNDS_OK(dw_box_ok(kb, n0 + q * 32, e), args.status)) continue;
                  if (overwrite)
                    tma_store_3d_hint(&tmD, ebuf_s + b * BOXB, kb, n0 + q * 32, e, dw_policy);
                  else
                    tma_reduce_add_3d_hint(&tmD, ebuf_s + b * BOXB, kb, n0 + q * 32, e, dw_policy);
                }
                bulk_commit();
              }
            }
          }
          if (chunked && c + 1 < itm.nch) {  // a later chunk of this tile adds onto these writes
            if (lane == 0) {
              bulk_wait<0>();  // this warp's writes are complete
              fence_proxy_async_global();
              mbar_arrive(pub_bar);
            }
            bool pub_ok = true;
            if (warp == 2) {  // once all eight warps' writes are complete: publish
              pub_ok = __shfl_sync(0xffffffffu, lane == 0 ? (mbar_wait(guard, pub_bar, pub_par) ? 1 : 0) : 0, 0) != 0;
              pub_par ^= 1u;
              if (pub_ok && lane == 0) flag_publish(flag, c + 1);
            }
            __syncwarp();
            if (!pub_ok) return false;
          }
          return true;
        },
        [&](const Item& itm) {  // expert without rows: dW tile = 0 (unchanged when accumulating)
          const int e = itm.e;
          const int n0 = nblk(e, itm.local) * TILE_M + static_cast<int>(rank) * BM;
          const int kh = kblk(e, itm.local) * BN + h * (BN / 2);
          if (n0 + q * 32 >= N || args.accumulate) return true;
#pragma unroll 1
          for (int c0 = 0; c0 < NBOX && kh + BC * c0 < K; c0 += GB) {
            const int nb = group_boxes(kh, c0);
            stage_group(nullptr, nb);
            if (lane == 0) {
              for (int b = 0; b < nb; ++b)
                if (RG_BOUNDS_OK(dw_box_ok(kh + BC * (c0 + b), n0 + q * 32, e), args.status))
                  tma_store_3d(&tmD, ebuf_s + b * BOXB, kh + BC * (c0 + b), n0 + q * 32, e);
              bulk_commit();
            }
          }
          return true;
        });
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  // ---- teardown --------------------------------------------------------------
  // Once no producer of either CTA issues any more, the issuing CTA settles
  // every stage (drain_stages) -- after a normal run a formality, after an
  // abort the wait for copies still in flight -- and the peer leaves only
  // after that, since its copies complete on the issuer's barriers.
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();
  if (threadIdx.x == 0 && rank == 0)
    drain_stages<STAGES>(full_bar(0), ilog, CG == 2 ? mapa_shared(smem_u32(ilog), 1) : 0u);
  if constexpr (CG == 2) cluster_sync();
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem, TMEM_COLS);
  }
}

// Ring depth.  The shared-memory tables of the experts sit beside the ring:
// a launch whose tables do not fit beside the deep ring (more than 239
// experts with CTA pairs) runs the same kernel with one stage fewer, which
// leaves room for RG_MAX_EXPERTS_CFG experts.
constexpr int kStagesDeep = kCtaGroup == 2 ? kg::STAGES : 2;
constexpr int kStagesShallow =
    Cfg<kCtaGroup, kStagesDeep>::SMEM_FIXED + (3 * RG_MAX_EXPERTS_CFG + 2) * 4 <= 232448 ? kStagesDeep
                                                                                         : kStagesDeep - 1;
static_assert(kStagesShallow >= 2, "the shallow ring keeps two stages");
static_assert(Cfg<kCtaGroup, kStagesShallow>::SMEM_FIXED + (3 * RG_MAX_EXPERTS_CFG + 2) * 4 <= 232448,
              "the expert tables of RG_MAX_EXPERTS_CFG experts must fit beside the shallow ring");

// Ring and barriers, then offsets [E+1], order [E] and (chunk mode) item prefix [E+1].
template <int ST>
size_t smem_bytes(int E) {
  return Cfg<kCtaGroup, ST>::SMEM_FIXED + (3 * static_cast<size_t>(E) + 2) * 4;
}

// The deep ring when the expert tables fit beside it in `max_smem` bytes.
bool use_deep(int E, size_t max_smem) { return smem_bytes<kStagesDeep>(E) <= max_smem; }

void fill_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int grid, size_t smem,
                 cudaStream_t stream) {
  *cfg = cudaLaunchConfig_t{};
  cfg->gridDim = dim3(grid);
  cfg->blockDim = dim3(Cfg<kCtaGroup, kStagesDeep>::THREADS);
  cfg->dynamicSmemBytes = smem;
  cfg->stream = stream;
  if (kCtaGroup == 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
  }
}

}  // namespace

size_t kgemm_smem_bytes(int E, size_t max_smem) {
  return use_deep(E, max_smem) ? smem_bytes<kStagesDeep>(E) : smem_bytes<kStagesShallow>(E);
}

cudaError_t kgemm_setup(int max_smem) {
  cudaError_t e = cudaFuncSetAttribute(
      kgemm_kernel<kCtaGroup, kStagesDeep>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      static_cast<int>(std::min<size_t>(smem_bytes<kStagesDeep>(RG_MAX_EXPERTS_CFG), max_smem)));
  if (e != cudaSuccess || kStagesShallow == kStagesDeep) return e;
  return cudaFuncSetAttribute(
      kgemm_kernel<kCtaGroup, kStagesShallow>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      static_cast<int>(std::min<size_t>(smem_bytes<kStagesShallow>(RG_MAX_EXPERTS_CFG), max_smem)));
}

cudaError_t kgemm_max_clusters(int* clusters, int max_smem) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  fill_config(&cfg, attr, 2 * kCtaGroup, std::min<size_t>(smem_bytes<kStagesDeep>(1), max_smem), nullptr);
  return cudaOccupancyMaxActiveClusters(clusters, kgemm_kernel<kCtaGroup, kStagesDeep>, &cfg);
}

cudaError_t launch_kgemm(const CUtensorMap& tmG, const CUtensorMap& tmX, const CUtensorMap& tmD,
                         const GroupArgs& args, int grid, size_t max_smem, cudaStream_t stream) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  if (use_deep(args.E, max_smem)) {
    fill_config(&cfg, attr, grid, smem_bytes<kStagesDeep>(args.E), stream);
    return cudaLaunchKernelEx(&cfg, kgemm_kernel<kCtaGroup, kStagesDeep>, tmG, tmX, tmD, args);
  }
  fill_config(&cfg, attr, grid, smem_bytes<kStagesShallow>(args.E), stream);
  return cudaLaunchKernelEx(&cfg, kgemm_kernel<kCtaGroup, kStagesShallow>, tmG, tmX, tmD, args);
}

}  // namespace rg
