// M-grouped BF16 GEMM for sm_103a: forward (y = x . w[e]^T) and input
// gradient (transpose_B: y = x . w[e]) over expert row groups given by a
// cumulative offsets vector (RapidGEMM README, "Kernels", Mgemm).
//
// Design
//   * Persistent grid.  Every CTA reads offsets[0..E] into shared memory,
//     validates it, and builds the tile list itself: expert e contributes
//     ceil(M_e/TILE_M) x ceil(N/256) tiles, laid out expert by expert (prefix
//     sums in shared memory).  Worker w (a CTA pair, or a CTA) takes tiles
//     w, w+W, w+2W, ... so no host synchronisation and no global scratch are
//     needed; empty experts contribute no tiles, tiny ones a single ragged one.
//   * A tile is rows [offsets[e] + TILE_M m, +TILE_M) x columns [256 n, +256).
//     Its row window starts at the expert's first row, so it never straddles a
//     group start; rows past the expert's end (they belong to the next expert)
//     are loaded but never stored.
//   * CG = 2 (default): a CTA pair (cluster of 2) computes a 256x256 tile with
//     tcgen05.mma.cta_group::2 (M=256, N=256, K=16).  Each CTA loads its own
//     128 rows of A and 128 rows of B (output columns); a stage holds two
//     64-deep atoms of both (64 KB per CTA, eight MMAs per barrier round of
//     the MMA warp) and three stages are in flight.  Each CTA's tensor memory
//     receives its 128 rows of D.  The peer CTA's TMA copies complete their
//     bytes directly on the issuing CTA's stage barrier (.cta_group::2), and
//     MMA completion is multicast to the barriers of both CTAs.
//     CG = 1: one CTA computes a 128x256 tile (tcgen05 M=128), four 48 KB stages.
//   * Tile variants (CTA-pair build; the host picks one per launch and
//     encodes B's map for it): forward outputs at most 64 wide run 64-column
//     pair tiles (N = 64 MMAs, five stages); contractions of one 64-deep stage
//     run on single CTAs (128 x 256 tiles, no cluster, eight epilogue warps),
//     whose accumulator hand-over between the MMA issuer and the epilogue
//     is much shorter than a pair's and sets the pace when a tile has one
//     MMA, with operand boxes as deep as the contraction (16 or 32 K columns,
//     32- or 64-byte swizzle) instead of 64-column boxes mostly zero-filled.
//   * Transposed B (input gradient, w [E, K, N]) is read N-contiguous in
//     64-column boxes; with N a multiple of 64 the map is a 4-D view whose
//     box of two column blocks fills both boxes of a CTA's atom in one copy.
//   * Half tiles (CTA pairs, plain epilogue): an expert's last row block of at
//     most 128 rows runs as an M=128 pair MMA; each CTA loads only its 64 rows
//     of A, through a second tensor map with 64-row boxes.
//   * Warp roles (224 threads per CTA): lane 0 of warps 0 and 6 issue the TMA
//     loads of alternate stages;
//     warp 1 owns tensor memory, and in the issuing CTA lane 0 issues the MMAs
//     into one of two 256-column fp32 accumulators; warps 2-5 drain the other
//     accumulator
//     (tcgen05.ld -> bf16 -> swizzled shared memory -> TMA store), so the
//     epilogue overlaps the next tile's MMAs.
//   * Tail rows: a warp whose 32 rows are all inside the expert stores them
//     with one TMA store per 64 columns; otherwise each valid row is written
//     with plain 16-byte stores.
//   * Every mbarrier wait is bounded (WaitGuard).  A wait that runs out sets
//     the device status and all roles stop; issued MMAs are waited for, and
//     at the end the issuing CTA waits for every copy either CTA of the pair
//     issued (drain_stages), with bounded waits, before tensor memory is freed
//     and the CTAs exit.
#include <algorithm>

#include "bounds.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace rg {
namespace {

// BNT: tile columns (256; 64 for outputs at most 64 wide, whose MMAs would
// otherwise be mostly padding).  EPIW: epilogue warps (4; 8 when the
// contraction fits one stage and the epilogue, not the MMAs, sets the pace --
// two warps per tensor-memory lane quarter then split the columns).
// operand stages of the narrow-box one-stage tiles (3, 4 and 6 measured
// alike; 10 slower)
#ifndef RG_MG_NARROW_STAGES
#define RG_MG_NARROW_STAGES 4
#endif
// BKW: K columns per operand box (64: rows of 128 bytes, 128-byte swizzle;
// 16 or 32 for the single-CTA one-stage tiles of contractions that short,
// rows of 32 or 64 bytes with the swizzle of that width, instead of boxes
// three quarters or half zero-filled).
template <int CG, int BNT = 256, int EPIW = 4, int BKW = 64>
struct Cfg {
  static constexpr int BM = 128;            // rows of A (and of D) per CTA
  static constexpr int TILE_M = BM * CG;    // rows per tile
  static constexpr int BN = BNT;            // tile columns = MMA N
  static constexpr int BN_CTA = BN / CG;    // B rows (output columns) loaded per CTA
  static constexpr int BK = BKW;            // K of one operand box (bf16)
  // Atoms per stage: two for the 256- and 64-column tiles, so that one
  // barrier round of the MMA warp issues eight MMAs (four cost a fixed share
  // of its time); the 8-epilogue-warp tile (K <= 64) has one.
  static constexpr int KATOMS = CG == 2 && (EPIW == 4) ? 2 : 1;
  static constexpr int BKS = BK * KATOMS;   // K per stage
  // 256-column tiles: three 64 KB stages; 64-column tiles (N = 64 MMAs, a
  // quarter as long): five 40 KB stages; single CTAs: four 48 KB stages, or
  // three beside the staging of eight epilogue warps (one-stage contractions;
  // RG_MG_NARROW_STAGES with narrow operand boxes)
  static constexpr int STAGES = CG == 2 ? (BNT == 64 ? 5 : 3) : (EPIW == 8 ? (BKW == 64 ? 3 : RG_MG_NARROW_STAGES) : 4);
  static constexpr int A_ATOM = BM * BK * 2;       // one atom of A (bytes)
  static constexpr int B_ATOM = BN_CTA * BK * 2;   // one atom of B
  static constexpr int A_BYTES = A_ATOM * KATOMS;
  static constexpr int B_BYTES = B_ATOM * KATOMS;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int EPI_WARPS = EPIW;
  // sleep between the epilogue's polls of its accumulator barrier (CTA
  // pairs): 1 us for tiles of many stages (polling costs the copies and MMAs
  // shared-memory bandwidth), RG_MG_SHORT_POLL_NS for pair tiles with eight
  // epilogue warps (single CTAs use the suspending wait instead)
  static constexpr uint32_t ACC_POLL_NS = EPIW == 8 ? RG_MG_SHORT_POLL_NS : 1000;
  // staging per epilogue warp: one 32-row x 64-column bf16 box, or with 8
  // epilogue warps (two chunks per warp and tile) two, written together
  static constexpr int EPI_BUF_BYTES = 32 * 128 * (EPIW == 8 ? 2 : 1);
  // warp 0 and warp 2 + EPIW: TMA producers (alternate stages), warp 1: MMA,
  // warps 2 .. 1 + EPIW: epilogue
  static constexpr int PRODUCER2 = 2 + EPIW;
  static constexpr int THREADS = 32 * (3 + EPIW);
  // full[S], empty[S], tfull[2], tempty[2], drain
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  // The dynamic shared-memory window of a CTA without static shared memory
  // starts 1024-byte aligned; the kernel checks this instead of padding.
  static constexpr int SMEM_FIXED = STAGES * STAGE_BYTES + EPI_WARPS * EPI_BUF_BYTES + NUM_BARS * 8 +
                                    static_cast<int>(sizeof(IssueLog<STAGES>)) + 16;
};

constexpr uint32_t TMEM_COLS = 512;

// Epilogue variants.
//   kEpiPlain:     y = accumulator (bf16).
//   kEpiSwiglu:    forward gate-up GEMM with h = SiLU(gate) * up in the
//                  epilogue.  B is w13 [E, 2F, K] with the gate rows first; a
//                  tile covers output features [f0, f0+128): CTA 0 of the pair
//                  loads gate rows f0.., CTA 1 up rows F+f0.., so every
//                  accumulator holds gate in columns 0..127 and up in 128..255.
//   kEpiSwigluBwd: input gradient of the down projection (transpose_B,
//                  N = F) followed by the SwiGLU backward: the accumulator is
//                  dh, args.out2 holds the saved gate-up output y13 [M, 2F],
//                  and the epilogue writes dy13 = [dh*up*SiLU'(gate), dh*SiLU(gate)].
constexpr int kEpiPlain = 0, kEpiSwiglu = 1, kEpiSwigluBwd = 2;

// Shared-memory descriptor of a K-major operand whose rows are SW bytes
// (SW = 32, 64 or 128) with the SW-byte swizzle: 8-row atoms of 8 x SW bytes
// packed one after the other (SBO), the K extent of one MMA inside a row
// (LBO unused).  Swizzle mode bits: 2 = 128 B, 4 = 64 B, 6 = 32 B.
template <int SW>
__device__ __forceinline__ uint64_t sdesc_kmajor(uint32_t saddr) {
  static_assert(SW == 32 || SW == 64 || SW == 128, "swizzle width");
  constexpr uint64_t mode = SW == 128 ? 2 : SW == 64 ? 4 : 6;
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(16 >> 4) << 16) |
         (static_cast<uint64_t>((8 * SW) >> 4) << 32) | (1ull << 46) | (mode << 61);
}

template <bool TRANS_B, int CG, int EPI = kEpiPlain, int BNT = 256, int EPIW = 4, int BKW = 64>
__global__ void __launch_bounds__(Cfg<CG, BNT, EPIW, BKW>::THREADS, 1)
    mgemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAh,
                 const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmY2,
                 const GroupArgs args) {
  constexpr bool SWIGLU = EPI == kEpiSwiglu;
  static_assert(!SWIGLU || (CG == 2 && !TRANS_B), "SwiGLU variant: forward, CTA pairs");
  static_assert(EPI != kEpiSwigluBwd || TRANS_B, "SwiGLU backward: input-gradient GEMM");
  static_assert((BNT == 256 && (EPIW == 4 || EPIW == 8)) || (BNT == 64 && EPIW == 4 && CG == 2 && !TRANS_B),
                "tile variants: 256 columns with 4 or 8 epilogue warps; 64 columns (forward, CTA pairs)");
  static_assert(EPI == kEpiPlain || (BNT == 256 && EPIW == 4), "fused epilogues use the default tile");
  static_assert(BKW == 64 || ((BKW == 16 || BKW == 32) && CG == 1 && EPIW == 8 && BNT == 256 && EPI == kEpiPlain),
                "narrow operand boxes: single-CTA one-stage tiles only");
  using C = Cfg<CG, BNT, EPIW, BKW>;
  constexpr int BM = C::BM, TILE_M = C::TILE_M, BN = C::BN, BN_CTA = C::BN_CTA, BK = C::BK;
  constexpr int KATOMS = C::KATOMS, BKS = C::BKS, A_ATOM = C::A_ATOM, B_ATOM = C::B_ATOM;
  constexpr int STAGES = C::STAGES, A_BYTES = C::A_BYTES, STAGE_BYTES = C::STAGE_BYTES;

  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // swizzled TMA boxes and MMA descriptors need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(args.status, kDevLaunchConfig);
    return;
  }
  uint8_t* epi = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + C::EPI_WARPS * C::EPI_BUF_BYTES);
  IssueLog<STAGES>* ilog = reinterpret_cast<IssueLog<STAGES>*>(bars + C::NUM_BARS);
  int* misc = reinterpret_cast<int*>(ilog + 1);  // [0] tmem base, [1] abort
  int* s_off = misc + 4;                                   // [E+1] offsets
  int* s_pre = s_off + (args.E + 1);                       // [E+1] tile prefix

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;  // rank 0 issues the MMAs
  const int worker = blockIdx.x / CG;
  const int nworkers = gridDim.x / CG;
  const int E = args.E;
  const int N = args.N;
  const int K = args.K;
  const int F = N / 2;  // SwiGLU: output features
  // output-column blocks per row block: 256 columns, or 128 SwiGLU features
  const int nbn = SWIGLU ? (F + BN_CTA - 1) / BN_CTA : (N + BN - 1) / BN;
  const int nk = (K + BKS - 1) / BKS;  // stages per tile

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

  // ---- per-expert tile prefix (warp 0, warp-wide scan) ----------------------
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int lo = min(E, lane * per), hi = min(E, lo + per);
    int s = 0;
    for (int e = lo; e < hi; ++e) s += ((s_off[e + 1] - s_off[e] + TILE_M - 1) / TILE_M) * nbn;
    int incl = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - s;
    for (int e = lo; e < hi; ++e) {
      s_pre[e] = run;
      run += ((s_off[e + 1] - s_off[e] + TILE_M - 1) / TILE_M) * nbn;
    }
    if (lane == 31) s_pre[E] = incl;
  }
  __syncthreads();
  // Outer groups (nested grouped GEMM): every inner tile is repeated for
  // o = 0..O-1, tile t = inner tile (t / O), outer group (t % O).
  const int O = args.outer;
  const int T = s_pre[E] * O;
  if (worker >= T) return;  // same decision in both CTAs of a pair

  // Half tiles: an expert's last row block with at most 128 rows runs as an
  // M=128 pair MMA (64 rows per CTA) instead of an M=256 one with half of it
  // padding.  Each CTA's 64 rows x 256 columns then sit in 128 tensor-memory
  // columns: lanes 0..63 hold output columns 0..127, lanes 64..127 columns
  // 128..255.  Plain epilogue, 256-column tiles, CTA pairs only.
  constexpr bool HALF_TILES = EPI == kEpiPlain && BNT == 256 && CG == 2;
  auto is_half = [&](int e, int local) {
    if constexpr (!HALF_TILES) {
      return false;
    } else {
      const int rows = s_off[e + 1] - s_off[e];
      const int mt = local / nbn;
      return mt == (rows - 1) / TILE_M && rows - mt * TILE_M <= BM;
    }
  };

  // ---- barriers and tensor memory -------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), C::EPI_WARPS * CG);  // one arrival per epilogue warp of the pair
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<CG>(smem_u32(&misc[0]), TMEM_COLS);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // peer barriers initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const WaitGuard guard{args.status, args.wait_limit_ns, reinterpret_cast<volatile int*>(&misc[1])};
  // barriers that threads of the peer CTA (or its tensor-core commits) arrive on
  auto wait_pair = [&](uint32_t bar, uint32_t par) {
    if constexpr (CG == 2) return mbar_wait_cl(guard, bar, par);
    else return mbar_wait(guard, bar, par);
  };

  if (warp == 0 || warp == C::PRODUCER2) {
    // ============ TMA producers (lane 0 of warps 0 and 6) ====================
    // One thread issuing every copy caps the copy rate of a CTA below what
    // the tensor cores consume, so two threads take turns: each walks the
    // whole (tile, k-block) sequence and fills every other stage.
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      if constexpr (HALF_TILES) tma_prefetch_desc(&tmAh);
      tma_prefetch_desc(&tmB);
      const uint32_t pid = warp == 0 ? 0u : 1u;
      issue_log_init(ilog, pid);
      uint32_t it = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int e = 0;
      const uint32_t full_issuer = CG == 2 ? mapa_shared(full_bar(0), 0) : full_bar(0);
      for (int t = worker; t < T && ok; t += nworkers) {
        const int ti = t / O, o = t - ti * O;
        while (s_pre[e + 1] <= ti) ++e;
        const int local = ti - s_pre[e];
        const int eb = o * E + e;  // weight slot: w[o][e]
        // a half tile's rows are split 64 / 64 between the CTAs, each loading
        // its 64 rows of A through the 64-row map
        const bool half = is_half(e, local);
        const CUtensorMap* am = half ? &tmAh : &tmA;
        const uint32_t stage_tx = (half ? STAGE_BYTES - A_BYTES / 2 : STAGE_BYTES) * CG;
        const int tile_row0 = s_off[e] + (local / nbn) * TILE_M;
        const int row0 = tile_row0 + static_cast<int>(rank) * (half ? BM / 2 : BM);
        // B rows this CTA loads: its half of the 256 output columns, or (SwiGLU)
        // the gate rows (CTA 0) / the matching up rows (CTA 1) of 128 features
        const int n0 = SWIGLU ? (local % nbn) * BN_CTA + static_cast<int>(rank) * F
                              : (local % nbn) * BN + static_cast<int>(rank) * BN_CTA;
        for (int kb = 0; kb < nk; ++kb) {
          if ((it++ & 1u) == pid) {
            if (!wait_pair(empty_bar(stage), phase ^ 1u)) {
              ok = false;
              break;
            }
            // both CTAs' copies complete on the issuing CTA's full barrier,
            // which expects the bytes of the whole pair
            const uint32_t fb = full_issuer + 8u * stage;
            const uint32_t sa = sbase + stage * STAGE_BYTES;
            const uint32_t sb = sa + A_BYTES;
            if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), stage_tx);
            // one copy of A and of B per 64-deep atom (atoms past K are
            // zero-filled boxes; the MMA warp skips them)
#pragma unroll
            for (int j = 0; j < KATOMS; ++j) {
              const int kc = kb * BKS + BK * j;
              const uint32_t saj = sa + j * A_ATOM, sbj = sb + j * B_ATOM;
              // (debug-bounds build: a refused copy's bytes are counted as
              // arrived, so the stage completes without it)
              if (RG_BOUNDS_OK(bounds::inner_aligned(kc, 2) && bounds::mgemm_rows(tile_row0, s_off[e], s_off[e + 1], args.M) &&
                                   bounds::index_ok(o, O),
                               args.status)) {
                if (O == 1) tma_load_2d_cg<CG>(saj, am, fb, kc, row0);
                else tma_load_3d_cg<CG>(saj, am, fb, kc, o, row0);
              } else {
                mbar_complete_tx_cluster(fb, half ? A_ATOM / 2 : A_ATOM);
              }
              if constexpr (!TRANS_B) {
                if (RG_BOUNDS_OK(bounds::inner_aligned(kc, 2) && bounds::index_ok(eb, O * E), args.status))
                  tma_load_3d_cg<CG>(sbj, &tmB, fb, kc, n0, eb);
                else
                  mbar_complete_tx_cluster(fb, B_ATOM);
              } else if (args.mg_wide_b) {  // both 64-column boxes in one copy (4-D view)
                if (RG_BOUNDS_OK(n0 % 64 == 0 && bounds::index_ok(eb, O * E), args.status))
                  tma_load_4d_cg<CG>(sbj, &tmB, fb, 0, kc, n0 / 64, eb);
                else
                  mbar_complete_tx_cluster(fb, B_ATOM);
              } else {
#pragma unroll
                for (int jj = 0; jj < BN_CTA / 64; ++jj) {  // 64 columns x BK K rows per box
                  if (RG_BOUNDS_OK(bounds::inner_aligned(n0 + 64 * jj, 2) && bounds::index_ok(eb, O * E), args.status))
                    tma_load_3d_cg<CG>(sbj + jj * (BK * 128), &tmB, fb, n0 + 64 * jj, kc, eb);
                  else
                    mbar_complete_tx_cluster(fb, BK * 128);
                }
              }
            }
            ilog->it[pid][stage] = static_cast<int>(it - 1);
            ilog->bytes[pid][stage] = stage_tx / CG;
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1 && rank == 0) {
    // ================= MMA issuer (warp 1 of the issuing CTA) =================
    constexpr uint32_t IDESC = idesc_bf16_f32(TILE_M, BN, false, TRANS_B);
    constexpr uint32_t IDESC_HALF = idesc_bf16_f32(TILE_M / 2, BN, false, TRANS_B);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    bool ok = true;
    int e = 0;
    for (int t = worker; t < T; t += nworkers, ++acc) {
      const int ti = t / O;
      while (s_pre[e + 1] <= ti) ++e;
      const uint32_t idesc = is_half(e, ti - s_pre[e]) ? IDESC_HALF : IDESC;
      const int buf = acc & 1;
      const uint32_t tph = (acc >> 1) & 1;
      ok = __all_sync(0xffffffffu, wait_pair(tempty_bar(buf), tph ^ 1u));
      if (!ok) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem + buf * BN;
      for (int kb = 0; kb < nk; ++kb) {
        ok = __all_sync(0xffffffffu, wait_pair(full_bar(stage), phase));
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int k = 0; k < BKS / 16; ++k) {
            const int j = k / (BK / 16), kk = k % (BK / 16);  // atom, 16-deep step in it
            // steps at or past K multiply zero-filled columns: skipped (bit-identical)
            if (kb * BKS + BK * j + 16 * kk < K) {
              const uint32_t saj = sa + j * A_ATOM, sbj = sb + j * B_ATOM;
              const uint64_t ad = sdesc_kmajor<BK * 2>(saj + 32 * kk);
              // transposed B: 128-byte rows of 64 columns, BK K rows per 64-column block
              const uint64_t bd = TRANS_B ? sdesc_sw128(sbj + 2048 * kk, BK * 128, 1024)
                                          : sdesc_kmajor<BK * 2>(sbj + 32 * kk);
              umma_bf16<CG>(d_tmem, ad, bd, idesc, (kb | k) != 0);
            }
          }
          umma_commit<CG>(empty_bar(stage));  // frees the stage (in both CTAs) once these MMAs finish
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) umma_commit<CG>(tfull_bar(buf));  // accumulator ready for the epilogue(s)
      __syncwarp();
    }
    if (!ok && lane == 0) {  // wait for issued MMAs before tensor memory is freed
      umma_commit_local<CG>(drain_bar);
      mbar_wait_drain(drain_bar, 0);
    }
    __syncwarp();
  } else if (warp == 1) {
    // warp 1 of the peer CTA only takes part in the tensor-memory allocation
  } else {
    // =================== epilogue (warps 2 .. 1 + EPIW) ======================
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    // 64-column chunks of the tile this warp converts: all of them, or with 8
    // epilogue warps the first or second half
    constexpr int CH = BN / 64 / (C::EPI_WARPS / 4);
    const int c_first = ((warp - 2) >> 2) * CH;
    const int r_in_cta = q * 32 + lane;
    uint8_t* ebuf = epi + (warp - 2) * C::EPI_BUF_BYTES;
    const uint32_t ebuf_s = smem_u32(ebuf);
    __nv_bfloat16* y = static_cast<__nv_bfloat16*>(args.out);
    const uint32_t tempty_issuer = CG == 2 ? mapa_shared(tempty_bar(0), 0) : tempty_bar(0);
    auto release_acc = [&](int buf) {  // this warp is done with accumulator `buf`
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 2) mbar_arrive_cluster(tempty_issuer + 8u * buf);
        else mbar_arrive(tempty_bar(buf));
      }
    };
    int o = 0;  // outer group of the current tile
    int e = 0;  // its inner group (expert)
    // Write one 32-row x 64-column bf16 chunk of this warp (packed pairs p)
    // to out[row0 + q*32 + lane, col0 ..]: a TMA store when all 32 rows
    // belong to the expert and all 64 columns are below col_limit, otherwise
    // masked 16-byte stores of the valid rows and columns.  With outer groups
    // the map is 3-D (o selects the column block) and `out` already points
    // at column block o of a row of length ld.
    int wrow = q * 32;  // first row (within this CTA's rows of the tile) of this warp's lanes
    auto emit = [&](const uint32_t (&p)[32], const CUtensorMap* map, __nv_bfloat16* out, int ld,
                    int row0, int rows_valid, int col0, int col_limit) {
      if (col0 >= col_limit) return;
      if (wrow + 32 <= rows_valid && col0 + 64 <= col_limit) {
        if (lane == 0) bulk_wait_read<0>();  // previous store has left the buffer
        __syncwarp();
        uint4* rowp = reinterpret_cast<uint4*>(ebuf + lane * 128);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          rowp[j ^ (lane & 7)] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (RG_BOUNDS_OK(bounds::out_box(col0, 64, row0 + wrow, 32, s_off[e], s_off[e + 1], col_limit, 2) &&
                               bounds::index_ok(o, O),
                           args.status)) {
            if (O == 1) tma_store_2d(map, ebuf_s, col0, row0 + wrow);
            else tma_store_3d(map, ebuf_s, col0, o, row0 + wrow);
          }
          bulk_commit();
        }
      } else if (wrow + lane < rows_valid) {
        uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<int64_t>(row0 + wrow + lane) * ld + col0));
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (col0 + 8 * j < col_limit &&
              RG_BOUNDS_OK(bounds::out_box(col0 + 8 * j, 8, row0 + wrow + lane, 1, s_off[e], s_off[e + 1], col_limit, 2),
                           args.status))
            dst[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
      }
    };
    int acc = 0;
    for (int t = worker; t < T; t += nworkers, ++acc) {
      const int ti = t / O;
      o = t - ti * O;
      while (s_pre[e + 1] <= ti) ++e;
      const int local = ti - s_pre[e];
      const bool half = is_half(e, local);
      const int cta_rows = half ? BM / 2 : BM;  // rows of the tile this CTA holds
      const int row0 = s_off[e] + (local / nbn) * TILE_M + static_cast<int>(rank) * cta_rows;
      const int rows_valid = min(cta_rows, s_off[e + 1] - row0);  // <= 0: this CTA's part is past the expert
      // a half tile's lane quarter q holds rows 32 (q % 2) .. and columns 128 (q / 2) ..
      wrow = half ? (q & 1) * 32 : q * 32;
      const int buf = acc & 1;
      const uint32_t tph = (acc >> 1) & 1;
      if (!warp_wait_acc<CG, C::ACC_POLL_NS>(guard, tfull_bar(buf), tph)) break;
      tc_fence_after();
      if (wrow >= rows_valid) {  // none of this warp's rows belong to the expert
        release_acc(buf);
        continue;
      }
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN;
      if constexpr (EPI == kEpiSwigluBwd) {
        // dh columns n0.. of this tile; gate/up of the same rows from y13
        const int n0 = (local % nbn) * BN;
        const __nv_bfloat16* y13 = static_cast<const __nv_bfloat16*>(args.out2);
        const bool row_ok = r_in_cta < rows_valid;
        const int64_t rbase = static_cast<int64_t>(row0 + r_in_cta) * (2 * N);
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          const int col0 = n0 + 64 * c;
          uint4 gq[8], uq[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (row_ok && col0 + 8 * j < N) {
              gq[j] = __ldg(reinterpret_cast<const uint4*>(y13 + rbase + col0 + 8 * j));
              uq[j] = __ldg(reinterpret_cast<const uint4*>(y13 + rbase + N + col0 + 8 * j));
            } else {
              gq[j] = make_uint4(0, 0, 0, 0);
              uq[j] = make_uint4(0, 0, 0, 0);
            }
          }
          uint32_t v[64];
          tmem_ld_32x32b_x32(taddr + 64 * c, *reinterpret_cast<uint32_t(*)[32]>(v));
          tmem_ld_32x32b_x32(taddr + 64 * c + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
          tmem_ld_wait();
          if (c == BN / 64 - 1 || col0 + 64 >= N) release_acc(buf);
          const uint32_t* gw = reinterpret_cast<const uint32_t*>(gq);
          const uint32_t* uw = reinterpret_cast<const uint32_t*>(uq);
          uint32_t pg[32], pu[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {  // fp32 math on the fp32 dh and bf16 gate/up
            // (__expf / __fdividef: fast intrinsics, relative error ~1e-6, far
            // below the final bf16 rounding; e^-g = inf for g << 0 gives s = 0)
            float dg[2], du[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const float gv = __uint_as_float(k ? (gw[j] & 0xffff0000u) : (gw[j] << 16));
              const float uv = __uint_as_float(k ? (uw[j] & 0xffff0000u) : (uw[j] << 16));
              const float dh = __uint_as_float(v[2 * j + k]);
              const float sg = __fdividef(1.0f, 1.0f + __expf(-gv));
              du[k] = dh * (gv * sg);
              dg[k] = dh * uv * (sg * (1.0f + gv * (1.0f - sg)));
            }
            pg[j] = pack_bf16x2(__float_as_uint(dg[0]), __float_as_uint(dg[1]));
            pu[j] = pack_bf16x2(__float_as_uint(du[0]), __float_as_uint(du[1]));
          }
          emit(pg, &tmY, y, 2 * N, row0, rows_valid, col0, N);
          emit(pu, &tmY, y, 2 * N, row0, rows_valid, N + col0, 2 * N);
          if (col0 + 64 >= N) break;
        }
      } else if constexpr (!SWIGLU) {
        // chunk c: tensor-memory columns 64c.., output columns n0 + 64c.. (full
        // tile) or n0 + 128 (q / 2) + 64c.. (half tile, 128 columns per lane quarter)
        const int n0 = (local % nbn) * BN + (half ? (q >> 1) * 128 : 0);
        const int nch = half ? CH / 2 : CH;
        const int cf = half ? c_first / 2 : c_first;
        if constexpr (C::EPI_WARPS == 8) {
          // both chunks of this warp in one go when both are whole boxes:
          // two staging buffers, one proxy fence, one bulk group
          const int col0 = n0 + 64 * cf;
          if (nch == 2 && wrow + 32 <= rows_valid && col0 + 128 <= N) {
            uint32_t p[2][32];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              uint32_t v0[32], v1[32];
              tmem_ld_32x32b_x32(taddr + 64 * (cf + h2), v0);
              tmem_ld_32x32b_x32(taddr + 64 * (cf + h2) + 32, v1);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                p[h2][j] = pack_bf16x2(v0[2 * j], v0[2 * j + 1]);
                p[h2][16 + j] = pack_bf16x2(v1[2 * j], v1[2 * j + 1]);
              }
            }
            release_acc(buf);
            if (lane == 0) bulk_wait_read<0>();  // the previous stores have left both buffers
            __syncwarp();
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              uint4* rowp = reinterpret_cast<uint4*>(ebuf + h2 * 4096 + lane * 128);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                rowp[j ^ (lane & 7)] =
                    make_uint4(p[h2][4 * j], p[h2][4 * j + 1], p[h2][4 * j + 2], p[h2][4 * j + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {
                if (!RG_BOUNDS_OK(bounds::out_box(col0 + 64 * h2, 64, row0 + wrow, 32, s_off[e], s_off[e + 1], N, 2) &&
                                      bounds::index_ok(o, O),
                                  args.status))
                  continue;
                if (O == 1) tma_store_2d(&tmY, ebuf_s + h2 * 4096, col0 + 64 * h2, row0 + wrow);
                else tma_store_3d(&tmY, ebuf_s + h2 * 4096, col0 + 64 * h2, o, row0 + wrow);
              }
              bulk_commit();
            }
            continue;
          }
        }
#pragma unroll 1
        for (int c = cf; c < cf + nch; ++c) {
          uint32_t v0[32], v1[32];
          tmem_ld_32x32b_x32(taddr + 64 * c, v0);
          tmem_ld_32x32b_x32(taddr + 64 * c + 32, v1);
          tmem_ld_wait();
          if (c == cf + nch - 1) release_acc(buf);
          uint32_t p[32];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            p[j] = pack_bf16x2(v0[2 * j], v0[2 * j + 1]);
            p[16 + j] = pack_bf16x2(v1[2 * j], v1[2 * j + 1]);
          }
          emit(p, &tmY, y + static_cast<int64_t>(o) * N, O * N, row0, rows_valid, n0 + 64 * c, N);
        }
      } else {
        // columns 0..127 hold gate(f0 + j), 128..255 up(f0 + j)
        const int f0 = (local % nbn) * BN_CTA;
        __nv_bfloat16* y13 = static_cast<__nv_bfloat16*>(args.out2);
#pragma unroll 1
        for (int c = 0; c < BN_CTA / 64; ++c) {
          uint32_t g[64], u[64];
          tmem_ld_32x32b_x32(taddr + 64 * c, *reinterpret_cast<uint32_t(*)[32]>(g));
          tmem_ld_32x32b_x32(taddr + 64 * c + 32, *reinterpret_cast<uint32_t(*)[32]>(g + 32));
          tmem_ld_32x32b_x32(taddr + BN_CTA + 64 * c, *reinterpret_cast<uint32_t(*)[32]>(u));
          tmem_ld_32x32b_x32(taddr + BN_CTA + 64 * c + 32, *reinterpret_cast<uint32_t(*)[32]>(u + 32));
          tmem_ld_wait();
          if (c == BN_CTA / 64 - 1) release_acc(buf);
          uint32_t p[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {  // SiLU(gate) * up in fp32, then bf16
            float hv[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const float gv = __uint_as_float(g[2 * j + k]);
              hv[k] = __fdividef(gv, 1.0f + __expf(-gv)) * __uint_as_float(u[2 * j + k]);
            }
            p[j] = pack_bf16x2(__float_as_uint(hv[0]), __float_as_uint(hv[1]));
          }
          emit(p, &tmY, y, F, row0, rows_valid, f0 + 64 * c, F);
          if (y13 != nullptr) {  // keep the pre-activation for the backward pass
#pragma unroll
            for (int j = 0; j < 32; ++j) p[j] = pack_bf16x2(g[2 * j], g[2 * j + 1]);
            emit(p, &tmY2, y13, N, row0, rows_valid, f0 + 64 * c, F);
#pragma unroll
            for (int j = 0; j < 32; ++j) p[j] = pack_bf16x2(u[2 * j], u[2 * j + 1]);
            emit(p, &tmY2, y13, N, row0, rows_valid, F + f0 + 64 * c, N);
          }
        }
      }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  // ---- teardown --------------------------------------------------------------
  // Once no producer of either CTA issues any more, the issuing CTA settles
  // every stage (drain_stages): after a normal run a formality, after an
  // abort the wait for copies still in flight.  The peer leaves only after
  // that, since its copies complete on the issuer's barriers.
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // no remote arrive or MMA still targets either CTA
  if (threadIdx.x == 0 && rank == 0)
    drain_stages<STAGES>(full_bar(0), ilog, CG == 2 ? mapa_shared(smem_u32(ilog), 1) : 0u);
  if constexpr (CG == 2) cluster_sync();
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem, TMEM_COLS);
  }
}

// every variant holds the tables of RG_MAX_EXPERTS_CFG groups beside its pipeline
// (the 64-column pair tiles and the single-CTA one-stage tiles exist in the
// CTA-pair build only)
constexpr int kOneEpiw = RG_MG_ONE_STAGE_EPIW;
static_assert(kOneEpiw == 4 || kOneEpiw == 8, "single-CTA one-stage tiles: 4 or 8 epilogue warps");
static_assert(Cfg<kCtaGroup, 256, 4>::SMEM_FIXED + 2 * (RG_MAX_EXPERTS_CFG + 1) * 4 <= 232448 &&
                  (kCtaGroup == 1 ||
                   (Cfg<kCtaGroup, 64, 4>::SMEM_FIXED + 2 * (RG_MAX_EXPERTS_CFG + 1) * 4 <= 232448 &&
                    Cfg<1, 256, kOneEpiw>::SMEM_FIXED + 2 * (RG_MAX_EXPERTS_CFG + 1) * 4 <= 232448)),
              "an Mgemm variant exceeds the shared memory of a CTA at the largest group count");

template <int BNT, int EPIW, int CG = kCtaGroup, int BKW = 64>
size_t smem_of(int E) {
  return Cfg<CG, BNT, EPIW, BKW>::SMEM_FIXED + 2 * (static_cast<size_t>(E) + 1) * 4;
}

template <bool TB, int EPI = kEpiPlain, int BNT = 256, int EPIW = 4, int CG = kCtaGroup, int BKW = 64>
cudaError_t set_smem(int max_smem) {
  const int bytes =
      static_cast<int>(std::min<size_t>(smem_of<BNT, EPIW, CG, BKW>(RG_MAX_EXPERTS_CFG), max_smem));
  return cudaFuncSetAttribute(mgemm_kernel<TB, CG, EPI, BNT, EPIW, BKW>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// launch configuration; CTA pairs (cg == 2) as clusters of two
void fill_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int grid, size_t smem, int threads,
                 cudaStream_t stream, int cg = kCtaGroup) {
  *cfg = cudaLaunchConfig_t{};
  cfg->gridDim = dim3(grid);
  cfg->blockDim = dim3(threads);
  cfg->dynamicSmemBytes = smem;
  cfg->stream = stream;
  if (cg == 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
  }
}

template <bool TB, int EPI = kEpiPlain, int BNT = 256, int EPIW = 4, int CG = kCtaGroup, int BKW = 64>
cudaError_t launch_variant(const CUtensorMap& tmA, const CUtensorMap& tmAh, const CUtensorMap& tmB,
                           const CUtensorMap& tmY, const CUtensorMap& tmY2, const GroupArgs& args, int grid,
                           cudaStream_t stream) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  fill_config(&cfg, attr, grid, smem_of<BNT, EPIW, CG, BKW>(args.E), Cfg<CG, BNT, EPIW, BKW>::THREADS, stream,
              CG);
  return cudaLaunchKernelEx(&cfg, mgemm_kernel<TB, CG, EPI, BNT, EPIW, BKW>, tmA, tmAh, tmB, tmY, tmY2, args);
}

// the single-CTA one-stage tile with operand boxes BKW deep
template <bool TB>
cudaError_t launch_one_cta(const CUtensorMap& tmA, const CUtensorMap& tmAh, const CUtensorMap& tmB,
                           const CUtensorMap& tmY, const GroupArgs& args, int sms, cudaStream_t stream) {
  switch (mgemm_kbox(TB, args.N, args.K)) {
    case 16:
      return launch_variant<TB, kEpiPlain, 256, kOneEpiw, 1, 16>(tmA, tmAh, tmB, tmY, tmY, args, sms, stream);
    case 32:
      return launch_variant<TB, kEpiPlain, 256, kOneEpiw, 1, 32>(tmA, tmAh, tmB, tmY, tmY, args, sms, stream);
    default:
      return launch_variant<TB, kEpiPlain, 256, kOneEpiw, 1>(tmA, tmAh, tmB, tmY, tmY, args, sms, stream);
  }
}

}  // namespace

size_t mgemm_smem_bytes(int E) {  // the largest of the variants built
  if constexpr (kCtaGroup == 1) return smem_of<256, 4>(E);
  return std::max({smem_of<256, 4>(E), smem_of<64, 4>(E), smem_of<256, kOneEpiw, 1>(E)});
}

cudaError_t mgemm_setup(int max_smem) {
  cudaError_t e = set_smem<false>(max_smem);
  if (e != cudaSuccess) return e;
  if ((e = set_smem<true>(max_smem)) != cudaSuccess) return e;
  if ((e = set_smem<true, kEpiSwigluBwd>(max_smem)) != cudaSuccess) return e;
  if constexpr (kCtaGroup == 2) {
    if ((e = set_smem<false, kEpiSwiglu>(max_smem)) != cudaSuccess) return e;
    if ((e = set_smem<false, kEpiPlain, 64, 4>(max_smem)) != cudaSuccess) return e;
    if ((e = set_smem<false, kEpiPlain, 256, kOneEpiw, 1>(max_smem)) != cudaSuccess) return e;
    if ((e = set_smem<true, kEpiPlain, 256, kOneEpiw, 1>(max_smem)) != cudaSuccess) return e;
    if constexpr (kOneEpiw == 8) {
      if ((e = set_smem<false, kEpiPlain, 256, 8, 1, 16>(max_smem)) != cudaSuccess) return e;
      if ((e = set_smem<true, kEpiPlain, 256, 8, 1, 16>(max_smem)) != cudaSuccess) return e;
      if ((e = set_smem<false, kEpiPlain, 256, 8, 1, 32>(max_smem)) != cudaSuccess) return e;
      if ((e = set_smem<true, kEpiPlain, 256, 8, 1, 32>(max_smem)) != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

cudaError_t mgemm_max_clusters(int* clusters, int max_smem) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  fill_config(&cfg, attr, 2 * kCtaGroup, std::min<size_t>(smem_of<256, 4>(RG_MAX_EXPERTS_CFG), max_smem),
              Cfg<kCtaGroup>::THREADS, nullptr);
  return cudaOccupancyMaxActiveClusters(clusters, mgemm_kernel<false, kCtaGroup>, &cfg);
}

cudaError_t launch_mgemm(bool transpose_B, const CUtensorMap& tmA, const CUtensorMap& tmAh,
                         const CUtensorMap& tmB, const CUtensorMap& tmY, const GroupArgs& args, int grid,
                         int sms, cudaStream_t stream) {
  if constexpr (kCtaGroup == 2) {
    if (mgemm_narrow(transpose_B != 0, args.N))
      return launch_variant<false, kEpiPlain, 64, 4>(tmA, tmAh, tmB, tmY, tmY, args, grid, stream);
    if (mgemm_one_cta(transpose_B != 0, args.N, args.K)) {
      if (transpose_B) return launch_one_cta<true>(tmA, tmAh, tmB, tmY, args, sms, stream);
      return launch_one_cta<false>(tmA, tmAh, tmB, tmY, args, sms, stream);
    }
  }
  if (transpose_B) return launch_variant<true>(tmA, tmAh, tmB, tmY, tmY, args, grid, stream);
  return launch_variant<false>(tmA, tmAh, tmB, tmY, tmY, args, grid, stream);
}

cudaError_t launch_mgemm_swiglu(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmH,
                                const CUtensorMap& tmY13, const GroupArgs& args, int grid,
                                cudaStream_t stream) {
  if constexpr (kCtaGroup != 2) {
    return cudaErrorNotSupported;
  } else {
    return launch_variant<false, kEpiSwiglu>(tmA, tmA, tmB, tmH, tmY13, args, grid, stream);  // no half tiles
  }
}

cudaError_t launch_mgemm_swiglu_dgrad(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                      const CUtensorMap& tmDy13, const GroupArgs& args, int grid,
                                      cudaStream_t stream) {
  return launch_variant<true, kEpiSwigluBwd>(tmA, tmA, tmB, tmDy13, tmDy13, args, grid, stream);  // no half tiles
}

}  // namespace rg
