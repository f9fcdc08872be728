// MXFP8 M-grouped GEMM for sm_103a (FP8 E4M3 operands, one E8M0 scale per 32
// elements along the contraction, fp32 accumulation, bf16 output), and the
// conversion of grouped E8M0 scales into the blocked ("128x4") layout the
// tensor cores read them in.  The MXFP8 grouped GEMM of the torchao MoE
// training PR and the block-scaled FP8 GEMMs of the DeepGEMM issue thread,
// over the Mgemm grouping of the RapidGEMM README ("Kernels").
//
// Blocked scale layout (rg_mx_scales_blocked).  The rows of a scale matrix
// [R, KS] are grouped by an offsets vector; every group is cut into blocks of
// 128 rows starting at its first row, and the blocks of all groups are
// numbered in order.  Block b, chunk c (scale columns 4c..4c+3) is the
// 512-byte range at (b * ceil(KS/4) + c) * 512; row i of the block and column
// j of the chunk sit at byte 16*(i%32) + 4*(i/32) + j.  Positions past a
// group's end or past column KS-1 hold 0x7F (scale 1.0).  One such range is
// exactly what tcgen05.cp.32x128b.warpx4 moves into tensor memory: lane l
// (of every 32-lane quarter) receives rows l, l+32, l+64, l+96 in four
// consecutive 32-bit columns, one scale byte per 32-element K block.
//
// GEMM design (mx_mgemm_kernel)
//   * Persistent grid.  The tile list is built on the device from the offsets
//     exactly as in the BF16 Mgemm (expert by expert, n fastest); worker w (a
//     CTA pair, or a CTA) takes tiles w, w+W, ...
//   * CG = 1 (default): one CTA computes 128 rows of one expert x 256 output
//     columns with tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale
//     (M=128, N=256, K=32), four stages; scale blocks arrive by bulk copies.
//   * CG = 2 (RG_MX_PAIR=1, comparison build): a CTA pair computes 256 rows
//     x 256 columns with the cta_group::2 form (M=256).  Each CTA loads its
//     own 128 rows of A and its 128 rows of B, 32 KB of operands per stage
//     instead of 48 KB, in six stages.  The peer CTA's copies complete on the
//     issuing CTA's stage barrier; scale blocks come through tensor maps
//     over the blocked buffers (rows of 256 bytes) for that reason.  Each
//     CTA's tensor memory needs the B scales of all 256 columns, so a pair
//     copies as many scale blocks into tensor memory per MMA as a single
//     CTA.  Measured on the 30B-A3B layer, the pair is 13-22% slower: with
//     neither operand nor scale copies it reaches 2.9 PFLOP/s on the
//     forward gate-up, the scale copies into tensor memory take a fifth of
//     that away and the operand copies a further 8%.
//   * One stage = 128 K elements: A 128x128 B, this CTA's B rows (K-major; or
//     128-column MN-major boxes for transpose_B), the A scale block of this
//     CTA's rows (512 B) and both B scale blocks of the tile (1 KB).
//   * Lane 0 of warps 0 and 10: copies of alternate stages (one thread cannot
//     issue copies fast enough).  Warp 1: tensor memory; in the issuing CTA
//     its lane 0 copies each stage's scales into a per-stage slot of tensor
//     memory (tcgen05.cp; with pairs every CTA's own blocks into its own
//     tensor memory) and issues the four MMAs of the stage, scale byte k of
//     each 32-bit scale word for MMA k.  Warps 2..9: epilogue, two per
//     tensor-memory lane quarter (128 columns each).
//   * Tensor memory: the fp32 accumulator (256 columns) and STAGES x 16
//     scale columns; a second accumulator does not fit, so the epilogue
//     drains the accumulator into registers and releases it before
//     converting and storing, which lets the next tile's MMAs start almost at
//     once.
//   * Epilogue: bf16 (round to nearest even), 32-row x 32-column TMA stores
//     through a 64-byte-swizzled staging buffer when all 32 rows belong to
//     the expert, masked 16-byte stores otherwise.  A pair tile's second CTA
//     may hold no row of the expert (its last tile of at most 128 rows); it
//     stores nothing.
//   * Bounded waits as in the BF16 kernels (WaitGuard): a wait that runs out
//     sets the device status, the CTA drains and frees tensor memory.
#include <algorithm>

#include "bounds.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace rg {
namespace {

template <int CG>
struct MxCfg {
  static constexpr int BM = 128;             // rows of A (and of D) per CTA
  static constexpr int TILE_M = BM * CG;     // rows per tile
  static constexpr int BN = 256;             // tile columns = MMA N
  static constexpr int BN_CTA = BN / CG;     // B rows (output columns) loaded per CTA
  static constexpr int BK = 128;             // K elements (bytes) per stage
  static constexpr int STAGES = CG == 2 ? 6 : 4;
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = BN_CTA * BK;
  static constexpr int SFA_BYTES = 512;
  // both 128-column B scale blocks of the tile, in every CTA of a pair: each
  // CTA's tensor core reads the scales of all N columns from its own tensor
  // memory (measured: a CTA holding only its own columns' block gives wrong
  // products in the other half)
  static constexpr int SFB_BYTES = 1024;
  static constexpr int AB_BYTES = A_BYTES + B_BYTES;   // operand tiles of a stage (1024-aligned)
  static constexpr int SF_BYTES = SFA_BYTES + SFB_BYTES;
  static constexpr int STAGE_BYTES = AB_BYTES + SF_BYTES;  // bytes one stage's copies deliver to a CTA
  static constexpr int EPI_WARPS = 8;
  static constexpr int EPI_BUF_BYTES = 32 * 64;  // 32 rows x 32 bf16 columns
  // warps 0 and 10: producers (alternate stages), 1: MMA, 2..9: epilogue
  static constexpr int PRODUCER2 = 2 + EPI_WARPS;
  static constexpr int THREADS = 32 * (PRODUCER2 + 1);
  // full[S], empty[S], tfull, tempty, drain
  static constexpr int NUM_BARS = 2 * STAGES + 3;
  // [operand tiles of every stage][scale blocks of every stage][epilogue buffers][barriers][misc]
  static constexpr int SMEM_FIXED = STAGES * STAGE_BYTES + EPI_WARPS * EPI_BUF_BYTES + NUM_BARS * 8 +
                                    static_cast<int>(sizeof(IssueLog<STAGES>)) + 16;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t SF_COL0 = 256;  // scale slots: stage s at SF_COL0 + 16 s (A: 4 cols, B: 8 cols)
};
static_assert(MxCfg<mxm::CG>::AB_BYTES % 1024 == 0, "operand tiles must keep the 1024-byte swizzle alignment");
static_assert(MxCfg<mxm::CG>::SF_COL0 + 16 * MxCfg<mxm::CG>::STAGES <= MxCfg<mxm::CG>::TMEM_COLS,
              "the accumulator and the scale slots must fit in tensor memory");

template <bool TRANS_B, int CG>
__global__ void __launch_bounds__(MxCfg<CG>::THREADS, 1)
    mx_mgemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmSA,
                    const __grid_constant__ CUtensorMap tmSB, const MxArgs args) {
  using C = MxCfg<CG>;
  constexpr int BM = C::BM, TILE_M = C::TILE_M, BN = C::BN, BN_CTA = C::BN_CTA, BK = C::BK;
  constexpr int STAGES = C::STAGES;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicOr(args.status, kDevLaunchConfig);
    return;
  }
  uint8_t* epi = smem + STAGES * C::STAGE_BYTES;  // after the operand tiles and the scale blocks
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + C::EPI_WARPS * C::EPI_BUF_BYTES);
  IssueLog<STAGES>* ilog = reinterpret_cast<IssueLog<STAGES>*>(bars + C::NUM_BARS);
  int* misc = reinterpret_cast<int*>(ilog + 1);  // [0] tmem base, [1] abort
  int* s_off = misc + 4;
  int* s_pre = s_off + (args.E + 1);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  const uint32_t tfull_bar = bar0 + 8u * (2 * STAGES);
  const uint32_t tempty_bar = bar0 + 8u * (2 * STAGES + 1);
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;  // rank 0 issues the MMAs
  const int worker = blockIdx.x / CG;
  const int nworkers = gridDim.x / CG;
  const int E = args.E, N = args.N, K = args.K;
  const int nbn = (N + BN - 1) / BN;
  const int nkc = (K + BK - 1) / BK;      // stages per tile = scale chunks per block
  const int nb_w = (N + 127) / 128;       // 128-row scale blocks of one expert's B

  // ---- offsets -> shared memory, validation, tile prefix ---------------------
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
  const int T = s_pre[E];
  if (worker >= T) return;  // same decision in both CTAs of a pair

  // ---- barriers and tensor memory -------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, C::EPI_WARPS * CG);  // one arrival per epilogue warp of the pair
    mbar_init(drain_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<CG>(smem_u32(&misc[0]), C::TMEM_COLS);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // peer barriers initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const WaitGuard guard{args.status, args.wait_limit_ns, reinterpret_cast<volatile int*>(&misc[1])};
  // barriers that the peer CTA (or the issuing CTA's tensor-core commits) arrive on
  auto wait_pair = [&](uint32_t bar, uint32_t par) {
    if constexpr (CG == 2) return mbar_wait_cl(guard, bar, par);
    else return mbar_wait(guard, bar, par);
  };
  // stage s: A at s*AB_BYTES and B after it; its scale blocks after all operand tiles
  auto sa_of = [&](int s) { return sbase + s * C::AB_BYTES; };
  auto sb_of = [&](int s) { return sa_of(s) + C::A_BYTES; };
  auto sfa_of = [&](int s) { return sbase + STAGES * C::AB_BYTES + s * C::SF_BYTES; };
  auto sfb_of = [&](int s) { return sfa_of(s) + C::SFA_BYTES; };

  if (warp == 0 || warp == C::PRODUCER2) {
    // ================ producers (lane 0 of warps 0 and 10) ===================
    // Two threads take turns: each walks the whole (tile, k-chunk) sequence
    // and fills every other stage, doubling the rate at which copies issue.
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      if constexpr (CG == 2) {
        tma_prefetch_desc(&tmSA);
        tma_prefetch_desc(&tmSB);
      }
      const uint32_t pid = warp == 0 ? 0u : 1u;
      issue_log_init(ilog, pid);
      uint32_t it = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int e = 0;
      int blk_e = 0;  // 128-row scale blocks of A of the experts before e
      const uint32_t full_issuer = CG == 2 ? mapa_shared(full_bar(0), 0) : full_bar(0);
      for (int t = worker; t < T && ok; t += nworkers) {
        while (s_pre[e + 1] <= t) {
          blk_e += (s_off[e + 1] - s_off[e] + BM - 1) / BM;
          ++e;
        }
        const int local = t - s_pre[e];
        const int mb = local / nbn, nt = local % nbn;
        const int tile_row0 = s_off[e] + mb * TILE_M;
        const int row0 = tile_row0 + static_cast<int>(rank) * BM;  // this CTA's rows
        const int n0 = nt * BN + static_cast<int>(rank) * BN_CTA;  // this CTA's B rows
        // scale blocks: A's block of this CTA's rows (a pair tile's second
        // CTA past the expert's end repeats the expert's last block: its
        // rows are never stored, any finite scale will do), B blocks 2nt and
        // 2nt+1 of expert e (the second repeats the first past the last
        // block: those B rows are zero-filled)
        const int nblk = (s_off[e + 1] - s_off[e] + BM - 1) / BM;
        const int blk_a = blk_e + min(mb * CG + static_cast<int>(rank), nblk - 1);
        const int blk_b0 = e * nb_w + 2 * nt;
        const int blk_b1 = e * nb_w + min(2 * nt + 1, nb_w - 1);
        for (int kc = 0; kc < nkc; ++kc) {
          if ((it++ & 1u) != pid) {  // the other producer's stage
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if (!wait_pair(empty_bar(stage), phase ^ 1u)) {
            ok = false;
            break;
          }
          // both CTAs' copies complete on the issuing CTA's full barrier,
          // which expects the bytes of the whole pair
          const uint32_t fb = full_issuer + 8u * stage;
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), C::STAGE_BYTES * CG);
          // (debug-bounds build: a refused copy's bytes are counted as arrived)
          if (RG_BOUNDS_OK(bounds::inner_aligned(kc * BK, 1) &&
                               bounds::mgemm_rows(tile_row0, s_off[e], s_off[e + 1], args.M),
                           args.status))
            tma_load_2d_cg<CG>(sa_of(stage), &tmA, fb, kc * BK, row0);
          else
            mbar_complete_tx_cluster(fb, C::A_BYTES);
          if (n0 >= N) {
            // a pair tile's second CTA past the last output column (N tail):
            // no B rows to load, and the columns they would give are not stored
            mbar_complete_tx_cluster(fb, C::B_BYTES);
          } else if constexpr (!TRANS_B) {
            if (RG_BOUNDS_OK(bounds::inner_aligned(kc * BK, 1) && bounds::index_ok(n0, N) && bounds::index_ok(e, E),
                             args.status))
              tma_load_3d_cg<CG>(sb_of(stage), &tmB, fb, kc * BK, n0, e);
            else
              mbar_complete_tx_cluster(fb, C::B_BYTES);
          } else {
#pragma unroll
            for (int j = 0; j < BN_CTA / 128; ++j) {
              if (RG_BOUNDS_OK(bounds::inner_aligned(n0 + 128 * j, 1) && bounds::index_ok(e, E), args.status))
                tma_load_3d_cg<CG>(sb_of(stage) + 16384 * j, &tmB, fb, n0 + 128 * j, kc * BK, e);
              else
                mbar_complete_tx_cluster(fb, 16384);
            }
          }
          // scale blocks lie inside the blocked buffers: (M/128 + E) blocks of
          // A's scales, (E*N/128 + E) of B's, nkc chunks of 512 bytes each
          if (RG_BOUNDS_OK(bounds::index_ok(blk_a, args.M / 128 + E) && bounds::index_ok(blk_b0, E * N / 128 + E) &&
                               bounds::index_ok(blk_b1, E * N / 128 + E),
                           args.status)) {
            if constexpr (CG == 2) {  // 512-byte chunk = two 256-byte rows of the maps
              tma_load_2d_cg<2>(sfa_of(stage), &tmSA, fb, 0, 2 * (blk_a * nkc + kc));
              tma_load_2d_cg<2>(sfb_of(stage), &tmSB, fb, 0, 2 * (blk_b0 * nkc + kc));
              tma_load_2d_cg<2>(sfb_of(stage) + 512, &tmSB, fb, 0, 2 * (blk_b1 * nkc + kc));
            } else {
              bulk_load(sfa_of(stage), args.sfa + (static_cast<int64_t>(blk_a) * nkc + kc) * 512, 512, fb);
              bulk_load(sfb_of(stage), args.sfb + (static_cast<int64_t>(blk_b0) * nkc + kc) * 512, 512, fb);
              bulk_load(sfb_of(stage) + 512, args.sfb + (static_cast<int64_t>(blk_b1) * nkc + kc) * 512, 512, fb);
            }
          } else {
            mbar_complete_tx_cluster(fb, C::SF_BYTES);
          }
          ilog->it[pid][stage] = static_cast<int>(it - 1);
          ilog->bytes[pid][stage] = C::STAGE_BYTES;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1 && rank == 0) {
    // ============= scale copies and MMAs (warp 1 of the issuing CTA) ==========
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    bool ok = true;
    for (int t = worker; t < T; t += nworkers, ++acc) {
      ok = __all_sync(0xffffffffu, wait_pair(tempty_bar, (acc & 1) ^ 1u));
      if (!ok) break;
      tc_fence_after();
      for (int kc = 0; kc < nkc; ++kc) {
        ok = __all_sync(0xffffffffu, wait_pair(full_bar(stage), phase));
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sfa_t = tmem + C::SF_COL0 + 16u * stage;
          const uint32_t sfb_t = sfa_t + 4u;
          tmem_cp_32x128b_x4<CG>(sfa_t, sdesc_plain16(sfa_of(stage)));
          tmem_cp_32x128b_x4<CG>(sfb_t, sdesc_plain16(sfb_of(stage)));
          tmem_cp_32x128b_x4<CG>(sfb_t + 4u, sdesc_plain16(sfb_of(stage) + 512));
          const uint32_t sa = sa_of(stage), sb = sb_of(stage);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k) {
            const uint64_t ad = sdesc_sw128(sa + 32 * k, 16, 1024);
            const uint64_t bd = TRANS_B ? sdesc_sw128(sb + 4096 * k, 16384, 1024)
                                        : sdesc_sw128(sb + 32 * k, 16, 1024);
            umma_mxf8<CG>(tmem, ad, bd, idesc_mxf8_f32(TILE_M, BN, false, TRANS_B, k), sfa_t, sfb_t,
                          (kc | k) != 0);
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
      if (lane == 0) umma_commit<CG>(tfull_bar);  // accumulator ready for the epilogue(s)
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
    // ======================= epilogue (warps 2..9) ===========================
    // Warp w reads TMEM lane quarter q = w % 4 and column half h.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int r_in = q * 32 + lane;
    uint8_t* ebuf = epi + (warp - 2) * C::EPI_BUF_BYTES;
    const uint32_t ebuf_s = smem_u32(ebuf);
    __nv_bfloat16* y = static_cast<__nv_bfloat16*>(args.out);
    const uint32_t tempty_issuer = CG == 2 ? mapa_shared(tempty_bar, 0) : tempty_bar;
    int acc = 0;
    int e = 0;
    for (int t = worker; t < T; t += nworkers, ++acc) {
      while (s_pre[e + 1] <= t) ++e;
      const int local = t - s_pre[e];
      const int row0 = s_off[e] + (local / nbn) * TILE_M + static_cast<int>(rank) * BM;
      const int n0 = (local % nbn) * BN + 128 * h;
      const int rows_valid = min(BM, s_off[e + 1] - row0);  // <= 0: this CTA's rows are past the expert
      // the single accumulator is on the MMAs' critical path: lane 0 polls
      // without sleeping (CTA pairs), the warp waits (one CTA)
      if (!warp_wait_acc<CG, 32>(guard, tfull_bar, acc & 1)) break;
      tc_fence_after();
      uint32_t v[128];
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + 128u * h;
      tmem_ld_32x32b_x32(taddr, *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld_32x32b_x32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld_32x32b_x32(taddr + 64, *reinterpret_cast<uint32_t(*)[32]>(v + 64));
      tmem_ld_32x32b_x32(taddr + 96, *reinterpret_cast<uint32_t(*)[32]>(v + 96));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {  // the accumulator is free for the next tile
        if constexpr (CG == 2) mbar_arrive_cluster(tempty_issuer);
        else mbar_arrive(tempty_bar);
      }
      if (q * 32 >= rows_valid || n0 >= N) continue;
      uint32_t p[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) p[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
      if (q * 32 + 32 <= rows_valid) {
        // 4 TMA stores of 32 rows x 32 columns; columns >= N are clipped by the map
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (n0 + 32 * c >= N) break;
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
          uint4* rowp = reinterpret_cast<uint4*>(ebuf + lane * 64);
          const int sw = (lane >> 1) & 3;  // 64-byte swizzle: 16-byte chunk ^= (row / 2) % 4
#pragma unroll
          for (int j = 0; j < 4; ++j)
            rowp[j ^ sw] = make_uint4(p[16 * c + 4 * j], p[16 * c + 4 * j + 1], p[16 * c + 4 * j + 2],
                                      p[16 * c + 4 * j + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (RG_BOUNDS_OK(bounds::inner_aligned(n0 + 32 * c, 2) && bounds::within(n0 + 32 * c, 32, N) &&
                                 s_off[e] <= row0 + q * 32 && row0 + q * 32 + 32 <= s_off[e + 1],
                             args.status))
              tma_store_2d(&tmY, ebuf_s, n0 + 32 * c, row0 + q * 32);
            bulk_commit();
          }
        }
      } else if (r_in < rows_valid) {
        uint4* dst = reinterpret_cast<uint4*>(y + static_cast<int64_t>(row0 + r_in) * N + n0);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (n0 + 8 * j < N) dst[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
      }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  // ---- teardown --------------------------------------------------------------
  // The last phase each stage was filled in has landed (after an abort, the
  // wait for copies still in flight) before the CTAs exit; with pairs the
  // issuing CTA settles the stages of both (drain_stages), and the peer
  // leaves only after that, since its copies complete on the issuer's
  // barriers.
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // no remote arrive or MMA still targets either CTA
  if (threadIdx.x == 0 && rank == 0)
    drain_stages<STAGES>(full_bar(0), ilog, CG == 2 ? mapa_shared(smem_u32(ilog), 1) : 0u);
  if constexpr (CG == 2) cluster_sync();
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------- blocked scale conversions
//
// Both conversions stage a 128-row slab of the scale matrix in shared memory
// with coalesced loads (consecutive threads read consecutive bytes) and then
// emit 512-byte blocks, one warp per block: lane l gathers rows l, l+32,
// l+64, l+96 (4 scale columns each) and writes its 16 bytes, so every block
// is one contiguous store line.  A pass covers at most PASS_COLS scale
// columns (PASS_COLS / 4 chunks).
constexpr int kConvThreads = 256;
constexpr int kPassCols = 256;

// Offsets -> shared memory, validation (leading zero, non-decreasing, last
// <= limit, multiples of `align`), and s_pre[g] = sum over g' < g of
// ceil((offsets[g'+1] - offsets[g']) / 128).  Returns false (after setting
// the status bit once) when the offsets are invalid.
__device__ bool conv_prologue(const int32_t* offsets, int G, int64_t limit, int align, int* s_off, int* s_pre,
                              unsigned int* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i <= G; i += blockDim.x) s_off[i] = offsets[i];
  __syncthreads();
  int bad = 0;
  for (int i = threadIdx.x; i < G; i += blockDim.x) bad |= (s_off[i + 1] < s_off[i]);
  for (int i = threadIdx.x; i <= G; i += blockDim.x) bad |= (s_off[i] % align) != 0;
  if (threadIdx.x == 0) bad |= (s_off[0] != 0) | (static_cast<int64_t>(s_off[G]) > limit);
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(status, kDevBadOffsets);
    return false;
  }
  if (warp == 0) {
    const int per = (G + 31) / 32;
    const int lo = min(G, lane * per), hi = min(G, lo + per);
    int s = 0;
    for (int g = lo; g < hi; ++g) s += (s_off[g + 1] - s_off[g] + 127) / 128;
    int incl = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - s;
    for (int g = lo; g < hi; ++g) {
      s_pre[g] = run;
      run += (s_off[g + 1] - s_off[g] + 127) / 128;
    }
    if (lane == 31) s_pre[G] = incl;
  }
  __syncthreads();
  return true;
}

// The last g with s_pre[g] <= x (the group owning block / chunk x).
__device__ __forceinline__ int group_of(const int* s_pre, int G, int x) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_pre[mid] <= x) lo = mid;
    else hi = mid;
  }
  return lo;
}

// One warp: the 512-byte block made of chunk columns [4c, 4c+4) of the
// 128-row slab `tile` (row stride `ld` bytes), written to dst.
__device__ __forceinline__ void emit_block(const uint8_t* tile, int ld, int c, uint8_t* dst, int lane) {
  uint32_t w[4];
#pragma unroll
  for (int qq = 0; qq < 4; ++qq) w[qq] = *reinterpret_cast<const uint32_t*>(tile + (lane + 32 * qq) * ld + 4 * c);
  reinterpret_cast<uint4*>(dst)[lane] = make_uint4(w[0], w[1], w[2], w[3]);
}

// Groups along the rows: block b = rows base .. base+127 of group g.
__global__ void __launch_bounds__(kConvThreads) mx_blocked_kernel(const uint8_t* __restrict__ src,
                                                                  const int32_t* __restrict__ offsets, int G,
                                                                  int R, int KS, uint8_t* __restrict__ dst,
                                                                  unsigned int* status) {
  __shared__ __align__(16) uint8_t tile[128 * kPassCols];
  extern __shared__ int s_tab[];
  int* s_off = s_tab;
  int* s_pre = s_tab + G + 1;
  if (!conv_prologue(offsets, G, R, 1, s_off, s_pre, status)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nc = (KS + 3) / 4;
  const int NB = s_pre[G];
  for (int b = blockIdx.x; b < NB; b += gridDim.x) {
    const int g = group_of(s_pre, G, b);
    const int base = s_off[g] + 128 * (b - s_pre[g]);
    const int rows = min(128, s_off[g + 1] - base);
    for (int c0 = 0; c0 < nc; c0 += kPassCols / 4) {
      const int cols = min(kPassCols, 4 * (nc - c0));  // staged width (whole chunks)
      const int col0 = 4 * c0;
      if (cols == KS && (reinterpret_cast<uintptr_t>(src) & 3) == 0) {
        // the pass covers whole rows: the slab is one contiguous run of
        // 32-bit words (KS is a multiple of 4 here); eight loads in flight
        const uint32_t* s32 = reinterpret_cast<const uint32_t*>(src + static_cast<int64_t>(base) * KS);
        uint32_t* t32 = reinterpret_cast<uint32_t*>(tile);
        const int valid_w = rows * KS / 4, total_w = 128 * KS / 4;
        for (int i0 = threadIdx.x; i0 < total_w; i0 += 8 * blockDim.x) {
          uint32_t v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * blockDim.x;
            v[u] = i < valid_w ? __ldg(s32 + i) : 0x7F7F7F7Fu;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * blockDim.x;
            if (i < total_w) t32[i] = v[u];
          }
        }
      } else {
        for (int i0 = threadIdx.x; i0 < 128 * cols; i0 += 8 * blockDim.x) {
          uint8_t v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * blockDim.x;
            const int r = i / cols, col = col0 + (i - r * cols);
            v[u] = (i < 128 * cols && r < rows && col < KS) ? src[static_cast<int64_t>(base + r) * KS + col] : 0x7F;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * blockDim.x;
            if (i < 128 * cols) tile[i] = v[u];
          }
        }
      }
      __syncthreads();
      for (int c = warp; c < cols / 4; c += blockDim.x >> 5)
        emit_block(tile, cols, c, dst + (static_cast<int64_t>(b) * nc + c0 + c) * 512, lane);
      __syncthreads();
    }
  }
}

// Groups along the contraction: chunk q of group g covers scale columns
// cb = offsets[g]/32 + 4 (q - s_pre[g]) .. cb+3, those at or past
// offsets[g+1]/32 are padding.  A work item is a 128-row slab times up to
// kKChunks consecutive chunks, whose columns form one contiguous range; the
// range is staged from its start rounded down to 4 bytes, so that rows whose
// length is a multiple of 4 are read as aligned 32-bit words.
constexpr int kKChunks = 32;
constexpr int kKStride = 4 * kKChunks + 8;  // staged bytes per row (range + alignment slack)

__global__ void __launch_bounds__(kConvThreads) mx_blocked_k_kernel(const uint8_t* __restrict__ src,
                                                                    const int32_t* __restrict__ offsets, int G,
                                                                    int R, int KS, uint8_t* __restrict__ dst,
                                                                    unsigned int* status) {
  __shared__ __align__(16) uint8_t tile[128 * kKStride];
  __shared__ int s_cb[kKChunks], s_c1[kKChunks];
  extern __shared__ int s_tab[];
  int* s_off = s_tab;
  int* s_pre = s_tab + G + 1;
  if (!conv_prologue(offsets, G, 32ll * KS, 32, s_off, s_pre, status)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NQ = s_pre[G];
  const int nrb = (R + 127) / 128;
  const int nqp = (NQ + kKChunks - 1) / kKChunks;
  const bool words = (KS & 3) == 0 && (reinterpret_cast<uintptr_t>(src) & 3) == 0;
  for (int it = blockIdx.x; it < nrb * nqp; it += gridDim.x) {
    const int rb = it / nqp, q0 = (it - rb * nqp) * kKChunks;
    const int nq = min(kKChunks, NQ - q0);
    for (int k = threadIdx.x; k < nq; k += blockDim.x) {
      const int g = group_of(s_pre, G, q0 + k);
      s_cb[k] = s_off[g] / 32 + 4 * (q0 + k - s_pre[g]);
      s_c1[k] = s_off[g + 1] / 32;
    }
    __syncthreads();
    const int cs = words ? (s_cb[0] & ~3) : s_cb[0];   // first staged column
    const int ce = min(KS, s_cb[nq - 1] + 4);          // one past the last needed column
    if (words) {
      const int wpr = (ce - cs + 3) / 4;  // ends inside the row: KS is a multiple of 4
      for (int i0 = threadIdx.x; i0 < 128 * wpr; i0 += 8 * blockDim.x) {
        uint32_t v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + u * blockDim.x;
          const int r = i / wpr, row = 128 * rb + r;
          v[u] = (i < 128 * wpr && row < R)
                     ? __ldg(reinterpret_cast<const uint32_t*>(src + static_cast<int64_t>(row) * KS + cs) + (i - r * wpr))
                     : 0x7F7F7F7Fu;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + u * blockDim.x;
          const int r = i / wpr;
          if (i < 128 * wpr) reinterpret_cast<uint32_t*>(tile + r * kKStride)[i - r * wpr] = v[u];
        }
      }
    } else {
      const int width = ce - cs;
      for (int i0 = threadIdx.x; i0 < 128 * width; i0 += 8 * blockDim.x) {
        uint8_t v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + u * blockDim.x;
          const int r = i / width, row = 128 * rb + r;
          v[u] = (i < 128 * width && row < R) ? src[static_cast<int64_t>(row) * KS + cs + (i - r * width)] : 0x7F;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + u * blockDim.x;
          const int r = i / width;
          if (i < 128 * width) tile[r * kKStride + (i - r * width)] = v[u];
        }
      }
    }
    __syncthreads();
    for (int k = warp; k < nq; k += blockDim.x >> 5) {
      const int cb = s_cb[k] - cs, c1 = s_c1[k] - cs;  // relative to the staged range
      uint32_t w[4];
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        uint32_t v = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t byte = cb + j < c1 ? tile[(lane + 32 * qq) * kKStride + cb + j] : 0x7Fu;
          v |= byte << (8 * j);
        }
        w[qq] = v;
      }
      reinterpret_cast<uint4*>(dst + (static_cast<int64_t>(rb) * NQ + q0 + k) * 512)[lane] =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ MX Kgemm
//
// dW[e] (fp32, [E, N, K]) = sum over the rows of expert e of
// (gq * 2^sg)^T (xq * 2^sx): FP8 E4M3 operands quantized along the rows
// (one E8M0 scale per column and 32-row block), every expert's row range a
// whole number of 32-row blocks.  Tile = 128 dW rows (n) x 256 dW columns (k)
// of one expert (BN = 256; a comparison build takes BN = 128 with two
// tensor-memory accumulators, since the scale slots leave no room for two
// 256-column ones), tcgen05 M=128 N=BN with both operands MN-major.  A stage is 128 rows of the expert: the MMAs of the
// 32-row steps that lie inside the expert are issued, so no row of the next
// expert enters an accumulation and nothing needs zeroing.  Scales come from the layout for groups along the
// contraction.  Tiles are taken longest expert first; rows are summed in
// tensor memory in chunks of at most CHUNK_ROWS, the first chunk's partial
// stored (or reduce-added when accumulating into dW), later ones TMA
// reduce-added in row order.  Empty experts get dW[e] = 0 (unchanged when
// accumulating).
struct MxkCfg {
  static constexpr int BM = 128;        // dW rows per tile (MMA M)
  static constexpr int BN = mxk::BN;    // dW columns per tile (MMA N)
  static constexpr int XB = BN / 128;   // 128-column boxes of X (and scale chunks of X) per stage
  static constexpr int ACC_BUFS = BN == 128 ? 2 : 1;  // accumulators in tensor memory
  static constexpr int BR = 128;        // expert rows per stage (4 scale blocks)
  static constexpr int STAGES = mxk::STAGES;
  static constexpr int A_BYTES = BM * BR;
  static constexpr int B_BYTES = BN * BR;
  static constexpr int AB_BYTES = A_BYTES + B_BYTES;
  static constexpr int SF_BYTES = 512 + 512 * XB;
  static constexpr int STAGE_BYTES = AB_BYTES + SF_BYTES;
  static constexpr int CHUNK_STAGES = mxk::CHUNK_ROWS / BR;
  static constexpr int EPI_WARPS = 8;
  static constexpr int BOX_COLS = mxk::BOX_COLS;
  static constexpr int BOX_BYTES = 32 * BOX_COLS * 4;      // 32 rows x BOX_COLS fp32 (one TMA box)
  static constexpr int EPI_GROUP = mxk::EPI_GROUP;
  static constexpr int EPI_BUF_BYTES = BOX_BYTES * EPI_GROUP;  // per epilogue warp
  // warps 0 and 10: producers (alternate stages), 1: MMA, 2..9: epilogue
  static constexpr int PRODUCER2 = 2 + EPI_WARPS;
  static constexpr int THREADS = 32 * (PRODUCER2 + 1);
  // full[S], empty[S], tfull[ACC_BUFS], tempty[ACC_BUFS], drain
  static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC_BUFS + 1;
  static constexpr int SMEM_FIXED = STAGES * STAGE_BYTES + EPI_WARPS * EPI_BUF_BYTES + NUM_BARS * 8 +
                                    static_cast<int>(sizeof(IssueLog<STAGES>)) + 16;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t SF_COL0 = ACC_BUFS * BN;  // scale slots (16 columns per stage) after the accumulators
};
static_assert(MxkCfg::SF_COL0 + 16 * MxkCfg::STAGES <= MxkCfg::TMEM_COLS,
              "accumulators and scale slots must fit in tensor memory");
static_assert(MxkCfg::AB_BYTES % 1024 == 0 && MxkCfg::EPI_BUF_BYTES % (MxkCfg::BOX_COLS * 32) == 0,
              "operand tiles and epilogue boxes must keep their swizzle alignment");
static_assert(MxkCfg::SMEM_FIXED + 3 * (RG_MAX_EXPERTS_CFG + 1) * 4 <= 232448,
              "MXFP8 wgrad configuration exceeds the shared memory of a CTA");
static_assert(mxk::CHUNK_ROWS % MxkCfg::BR == 0, "chunks must hold whole stages");

__global__ void __launch_bounds__(MxkCfg::THREADS, 1)
    mx_kgemm_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmD, const MxArgs args) {
  using C = MxkCfg;
  constexpr int BM = C::BM, BN = C::BN, BR = C::BR, STAGES = C::STAGES;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicOr(args.status, kDevLaunchConfig);
    return;
  }
  // [operand tiles of every stage][epilogue buffers][scale blocks][barriers][misc]
  // (the 128-byte-swizzled epilogue boxes need 1024-byte alignment)
  uint8_t* epi = smem + STAGES * C::AB_BYTES;
  uint8_t* sf_area = epi + C::EPI_WARPS * C::EPI_BUF_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sf_area + STAGES * C::SF_BYTES);
  IssueLog<STAGES>* ilog = reinterpret_cast<IssueLog<STAGES>*>(bars + C::NUM_BARS);
  int* misc = reinterpret_cast<int*>(ilog + 1);  // [0] tmem base, [1] abort
  int* s_off = misc + 4;           // [E+1]
  int* s_qp = s_off + (args.E + 1);  // [E+1] first scale chunk of each expert
  int* s_ord = s_qp + (args.E + 1);  // [E] experts by decreasing rows

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + C::ACC_BUFS + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * C::ACC_BUFS);
  constexpr int XB = C::XB, ACC_BUFS = C::ACC_BUFS;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = args.E, N = args.N, K = args.K;
  const int nbn = (N + BM - 1) / BM;
  const int nbk = (K + BN - 1) / BN;
  const int nrb_x = (K + 127) / 128;  // 128-row scale blocks of X's columns
  const int tpe = nbn * nbk;
  const int T = E * tpe;

  // ---- offsets -> shared memory, validation, chunk prefix, order -----------
  if (threadIdx.x == 0) misc[1] = 0;
  for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = args.offsets[i];
  __syncthreads();
  int bad = 0;
  for (int i = threadIdx.x; i < E; i += blockDim.x) bad |= (s_off[i + 1] < s_off[i]);
  for (int i = threadIdx.x; i <= E; i += blockDim.x) bad |= (s_off[i] & 31) != 0;
  if (threadIdx.x == 0) bad |= (s_off[0] != 0) | (s_off[E] > args.M);
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(args.status, kDevBadOffsets);
    return;
  }
  if (static_cast<int>(blockIdx.x) >= T) return;
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int lo = min(E, lane * per), hi = min(E, lo + per);
    int s = 0;
    for (int e = lo; e < hi; ++e) s += (s_off[e + 1] - s_off[e] + BR - 1) / BR;
    int incl = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - s;
    for (int e = lo; e < hi; ++e) {
      s_qp[e] = run;
      run += (s_off[e + 1] - s_off[e] + BR - 1) / BR;
    }
    if (lane == 31) s_qp[E] = incl;
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int ce = s_off[e + 1] - s_off[e];
    int rank_e = 0;
    for (int f = 0; f < E; ++f) {
      const int cf = s_off[f + 1] - s_off[f];
      rank_e += (cf > ce) | ((cf == ce) & (f < e));
    }
    s_ord[rank_e] = e;
  }
  __syncthreads();
  const int NQ = s_qp[E];

  // ---- barriers and tensor memory -------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < ACC_BUFS; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), C::EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<1>(smem_u32(&misc[0]), C::TMEM_COLS);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const WaitGuard guard{args.status, args.wait_limit_ns, reinterpret_cast<volatile int*>(&misc[1])};
  auto sa_of = [&](int s) { return sbase + s * C::AB_BYTES; };
  auto sb_of = [&](int s) { return sa_of(s) + C::A_BYTES; };
  const uint32_t sf_base = smem_u32(sf_area);
  auto sfa_of = [&](int s) { return sf_base + s * C::SF_BYTES; };
  auto sfb_of = [&](int s) { return sfa_of(s) + 512; };
  auto tile_at = [&](int t, int& e, int& nb, int& kb) {
    const int pe = t / tpe, local = t - pe * tpe;
    e = s_ord[pe];
    nb = local / nbk;
    kb = local - nb * nbk;
  };

  if (warp == 0 || warp == C::PRODUCER2) {
    // ======== producers (lane 0 of warps 0 and 10, alternate stages) =========
    if (lane == 0) {
      tma_prefetch_desc(&tmG);
      tma_prefetch_desc(&tmX);
      const uint32_t pid = warp == 0 ? 0u : 1u;
      issue_log_init(ilog, pid);
      uint32_t it = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
        int e, nb, kb;
        tile_at(t, e, nb, kb);
        const int r_begin = s_off[e], r_end = s_off[e + 1];
        const int n0 = nb * BM, k0 = kb * BN;
        // X's 128-column scale blocks of this tile (past K: zero-filled rows, any scale)
        const int xb0 = XB * kb, xb1 = min(XB * kb + XB - 1, nrb_x - 1);
        for (int r = r_begin, c = 0; r < r_end; r += BR, ++c) {
          if ((it++ & 1u) != pid) {  // the other producer's stage
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if (!mbar_wait(guard, empty_bar(stage), phase ^ 1u)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
          // (debug-bounds build: a refused copy's bytes are counted as arrived)
          const bool rows_ok = !RG_DEBUG_BOUNDS || (r_begin <= r && r < r_end && (r & 31) == 0);
          if (RG_BOUNDS_OK(rows_ok && bounds::inner_aligned(n0, 1) && bounds::index_ok(n0, N) &&
                               bounds::inner_aligned(k0, 1) && bounds::index_ok(k0, K),
                           args.status)) {
            tma_load_2d(sa_of(stage), &tmG, fb, n0, r);
#pragma unroll
            for (int x = 0; x < XB; ++x) tma_load_2d(sb_of(stage) + 16384 * x, &tmX, fb, k0 + 128 * x, r);
          } else {
            mbar_complete_tx_cluster(fb, C::AB_BYTES);
          }
          const int q = s_qp[e] + c;
          // scale chunks inside the blocked buffers: ceil(N/128) (or
          // ceil(K/128)) row blocks of NQ chunks of 512 bytes
          if (RG_BOUNDS_OK(bounds::index_ok(q, NQ) && bounds::index_ok(nb, (N + 127) / 128) && bounds::index_ok(xb1, nrb_x),
                           args.status)) {
            bulk_load(sfa_of(stage), args.sfa + (static_cast<int64_t>(nb) * NQ + q) * 512, 512, fb);
            bulk_load(sfb_of(stage), args.sfb + (static_cast<int64_t>(xb0) * NQ + q) * 512, 512, fb);
            if (XB == 2) bulk_load(sfb_of(stage) + 512, args.sfb + (static_cast<int64_t>(xb1) * NQ + q) * 512, 512, fb);
          } else {
            mbar_complete_tx_cluster(fb, (1 + XB) * 512);
          }
          ilog->it[pid][stage] = static_cast<int>(it - 1);
          ilog->bytes[pid][stage] = C::STAGE_BYTES;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ============= scale copies and MMAs (warp 1, lane 0) =====================
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
      int e, nb, kb;
      tile_at(t, e, nb, kb);
      const int rows = s_off[e + 1] - s_off[e];
      const int nst = (rows + BR - 1) / BR;
      for (int c0 = 0; c0 < nst && ok; c0 += C::CHUNK_STAGES, ++acc) {
        const int buf = acc % ACC_BUFS;
        const uint32_t tph = static_cast<uint32_t>(acc / ACC_BUFS) & 1u;
        ok = __all_sync(0xffffffffu, mbar_wait(guard, tempty_bar(buf), tph ^ 1u));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * BN;
        const int c1 = min(nst, c0 + C::CHUNK_STAGES);
        for (int c = c0; c < c1; ++c) {
          ok = __all_sync(0xffffffffu, mbar_wait(guard, full_bar(stage), phase));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t sfa_t = tmem + C::SF_COL0 + 16u * stage;
            const uint32_t sfb_t = sfa_t + 4u;
            tmem_cp_32x128b_x4(sfa_t, sdesc_plain16(sfa_of(stage)));
#pragma unroll
            for (int x = 0; x < XB; ++x) tmem_cp_32x128b_x4(sfb_t + 4u * x, sdesc_plain16(sfb_of(stage) + 512 * x));
            const int ksteps = min(4, (rows - BR * c) / 32);  // 32-row steps inside the expert
            const uint32_t sa = sa_of(stage), sb = sb_of(stage);
            for (int k = 0; k < ksteps; ++k) {
              const uint64_t ad = sdesc_sw128(sa + 4096 * k, 16384, 1024);
              const uint64_t bd = sdesc_sw128(sb + 4096 * k, 16384, 1024);
              umma_mxf8(d_tmem, ad, bd, idesc_mxf8_f32(BM, BN, true, true, k), sfa_t, sfb_t,
                        (c != c0) | (k != 0));
            }
            umma_commit<1>(empty_bar(stage));
          }
          __syncwarp();
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (lane == 0) umma_commit<1>(tfull_bar(buf));
        __syncwarp();
      }
    }
    if (!ok && lane == 0) {
      umma_commit<1>(drain_bar);
      mbar_wait_drain(drain_bar, 0);
    }
    __syncwarp();
  } else {
    // ======================= epilogue (warps 2..9) ===========================
    // Warp w owns TMEM lane quarter q = w % 4 (dW rows n0 + 32q ..) and
    // column half h (WC = BN / 2 columns), stored as boxes of 32 rows x
    // BOX_COLS fp32 through one staging buffer per warp.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    uint8_t* ebuf = epi + (warp - 2) * C::EPI_BUF_BYTES;
    const uint32_t ebuf_s = smem_u32(ebuf);
    int acc = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
      int e, nb, kb;
      tile_at(t, e, nb, kb);
      const int rows = s_off[e + 1] - s_off[e];
      const int nst = (rows + BR - 1) / BR;
      constexpr int WC = BN / 2;  // dW columns of this warp
      const int n0 = nb * BM + 32 * q;
      const int kc0 = kb * BN + WC * h;
      const bool mine = n0 < N && kc0 < K;  // this warp's boxes hold valid dW elements
      // a 32-row x BOX_COLS box of dW[e] at column k: inside dW, 16-byte aligned start
      auto dw_box_ok = [&](int k) {
        return bounds::inner_aligned(k, 4) && bounds::within(k, C::BOX_COLS, K) && bounds::within(n0, 32, N) &&
               bounds::index_ok(e, E);
      };
      if (rows == 0) {  // no rows: dW[e] = 0 (left unchanged when accumulating)
        if (!args.accumulate && mine) {
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
#pragma unroll
          for (int u = 0; u < C::EPI_BUF_BYTES / 512; ++u)
            reinterpret_cast<uint4*>(ebuf)[lane + 32 * u] = make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            for (int b = 0; b < WC / C::BOX_COLS && kc0 + C::BOX_COLS * b < K; ++b)
              if (RG_BOUNDS_OK(dw_box_ok(kc0 + C::BOX_COLS * b), args.status))
                tma_store_3d(&tmD, ebuf_s, kc0 + C::BOX_COLS * b, n0, e);
            bulk_commit();
          }
        }
        continue;
      }
      for (int c0 = 0; c0 < nst; c0 += C::CHUNK_STAGES, ++acc) {
        const int buf = acc % ACC_BUFS;
        if (!__all_sync(0xffffffffu, mbar_wait(guard, tfull_bar(buf), static_cast<uint32_t>(acc / ACC_BUFS) & 1u))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v[WC];
        const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + WC * h;
#pragma unroll
        for (int b = 0; b < WC / 32; ++b)
          tmem_ld_32x32b_x32(taddr + 32 * b, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * b));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(buf));  // the accumulator is free again
        if (!mine) continue;
        const bool reduce = args.accumulate || c0 > 0;
        // a later chunk is added onto the earlier chunk's writes: let them land first
        if (lane == 0 && c0 > 0) bulk_wait<0>();
        constexpr int BC = C::BOX_COLS, CH = BC / 4;  // 16-byte chunks per box row
        // swizzle: chunk ^= row % 8 (128-byte rows) or (row / 2) % 4 (64-byte rows)
        const int sw = BC == 32 ? (lane & 7) : ((lane >> 1) & 3);
        // groups of GB boxes: staged together after the previous group has
        // left the buffer, one proxy fence, their stores in one bulk group
        constexpr int GB = C::EPI_GROUP;
#pragma unroll
        for (int b0 = 0; b0 < WC / BC; b0 += GB) {
          if (kc0 + BC * b0 >= K) break;
          const int nb = min(GB, (K - kc0 - BC * b0 + BC - 1) / BC);
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
#pragma unroll
          for (int g = 0; g < GB; ++g) {
            if (g >= nb) break;
            const int b = b0 + g;
            uint4* rowp = reinterpret_cast<uint4*>(ebuf + g * C::BOX_BYTES + lane * BC * 4);
#pragma unroll
            for (int j = 0; j < CH; ++j)
              rowp[j ^ sw] = make_uint4(v[BC * b + 4 * j], v[BC * b + 4 * j + 1], v[BC * b + 4 * j + 2],
                                        v[BC * b + 4 * j + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            for (int g = 0; g < nb; ++g) {
              const int kb = kc0 + BC * (b0 + g);
              const uint32_t src = ebuf_s + g * C::BOX_BYTES;
              if (!RG_BOUNDS_OK(dw_box_ok(kb), args.status)) continue;
              if (reduce) tma_reduce_add_3d(&tmD, src, kb, n0, e);
              else tma_store_3d(&tmD, src, kb, n0, e);
            }
            bulk_commit();
          }
        }
      }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  // ---- teardown --------------------------------------------------------------
  // the last phase each stage was filled in has landed (after an abort, the
  // wait for copies still in flight) before the CTA exits
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) drain_stages<STAGES>(full_bar(0), ilog, 0u);
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<1>(tmem, C::TMEM_COLS);
  }
}

}  // namespace

using MxSel = MxCfg<mxm::CG>;
static_assert(MxSel::SMEM_FIXED + 2 * (RG_MAX_EXPERTS_CFG + 1) * 4 <= 232448,
              "MXFP8 Mgemm configuration exceeds the shared memory of a CTA at the largest group count");
size_t mx_smem_bytes(int E) { return MxSel::SMEM_FIXED + 2 * (static_cast<size_t>(E) + 1) * 4; }

cudaError_t mx_setup(int max_smem) {
  const int bytes = static_cast<int>(std::min<size_t>(mx_smem_bytes(RG_MAX_EXPERTS_CFG), max_smem));
  cudaError_t e = cudaFuncSetAttribute(mx_mgemm_kernel<false, mxm::CG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mx_mgemm_kernel<true, mxm::CG>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t mx_max_clusters(int* clusters, int max_smem) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(4);
  cfg.blockDim = dim3(MxSel::THREADS);
  cfg.dynamicSmemBytes = std::min<size_t>(mx_smem_bytes(RG_MAX_EXPERTS_CFG), max_smem);
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters, mx_mgemm_kernel<false, mxm::CG>, &cfg);
}

// grid: CTAs (a multiple of 2 with CTA pairs, launched as clusters of 2)
cudaError_t launch_mx_mgemm(bool transpose_B, const CUtensorMap& tmA, const CUtensorMap& tmB,
                            const CUtensorMap& tmY, const CUtensorMap& tmSA, const CUtensorMap& tmSB,
                            const MxArgs& args, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(MxSel::THREADS);
  cfg.dynamicSmemBytes = mx_smem_bytes(args.E);
  cfg.stream = stream;
  if (mxm::CG == 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  if (transpose_B)
    return cudaLaunchKernelEx(&cfg, mx_mgemm_kernel<true, mxm::CG>, tmA, tmB, tmY, tmSA, tmSB, args);
  return cudaLaunchKernelEx(&cfg, mx_mgemm_kernel<false, mxm::CG>, tmA, tmB, tmY, tmSA, tmSB, args);
}

cudaError_t launch_mx_blocked(const uint8_t* src, const int32_t* offsets, int G, int R, int KS, uint8_t* dst,
                              unsigned int* status, int num_sms, cudaStream_t stream) {
  const int64_t blocks_ub = static_cast<int64_t>(R) / 128 + G;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(blocks_ub, 8 * num_sms)));
  const size_t smem = 2 * (static_cast<size_t>(G) + 1) * sizeof(int);
  mx_blocked_kernel<<<grid, kConvThreads, smem, stream>>>(src, offsets, G, R, KS, dst, status);
  return cudaGetLastError();
}

}  // namespace rg

namespace rg {

size_t mxk_smem_bytes(int E) { return MxkCfg::SMEM_FIXED + 3 * (static_cast<size_t>(E) + 1) * 4; }

cudaError_t mxk_setup(int max_smem) {
  const int bytes = static_cast<int>(std::min<size_t>(mxk_smem_bytes(RG_MAX_EXPERTS_CFG), max_smem));
  return cudaFuncSetAttribute(mx_kgemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t launch_mx_kgemm(const CUtensorMap& tmG, const CUtensorMap& tmX, const CUtensorMap& tmD,
                            const MxArgs& args, int grid, cudaStream_t stream) {
  mx_kgemm_kernel<<<grid, MxkCfg::THREADS, mxk_smem_bytes(args.E), stream>>>(tmG, tmX, tmD, args);
  return cudaGetLastError();
}

cudaError_t launch_mx_blocked_k(const uint8_t* src, const int32_t* offsets, int G, int R, int KS, uint8_t* dst,
                                unsigned int* status, int num_sms, cudaStream_t stream) {
  const int64_t items_ub = (static_cast<int64_t>(R) + 127) / 128 * ((KS / 4 + G + kKChunks - 1) / kKChunks);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(items_ub, 8 * num_sms)));
  const size_t smem = 2 * (static_cast<size_t>(G) + 1) * sizeof(int);
  mx_blocked_k_kernel<<<grid, kConvThreads, smem, stream>>>(src, offsets, G, R, KS, dst, status);
  return cudaGetLastError();
}

}  // namespace rg
