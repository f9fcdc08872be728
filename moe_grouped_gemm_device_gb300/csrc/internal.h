// Host-side declarations shared by the C-ABI layer and the kernel translation
// units.  Not part of the public interface.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace rg {

// Arguments every grouped-GEMM kernel receives besides its tensor maps.
struct GroupArgs {
  const int32_t* offsets;   // device [E+1]
  int E;
  int M;                    // rows of the activation tensors
  int N;
  int K;
  void* out;                // y (bf16) for Mgemm (h for the SwiGLU variant), dW (fp32) for Kgemm
  void* out2;               // SwiGLU: the gate-up output y13 (bf16) -- written (forward, or
                            // null) or read (backward)
  unsigned int* status;     // device status word
  unsigned long long wait_limit_ns;
  int accumulate;           // Kgemm: 1 = dW += result, 0 = dW = result
  int outer;                // Mgemm: outer groups O along the columns of x and y (1 = plain);
                            // with O > 1 the x and y maps are 3-D {cols, O, rows}
  int kg_wide;              // Kgemm: 1 = operand maps are 4-D {64 cols, BR rows, column block,
                            // row} and one copy loads both 64-column boxes of a CTA (N and K
                            // multiples of 64); 0 = 3-D maps {cols, BR rows, row}, one copy per box
  int mg_wide_b;            // Mgemm with transpose_B: 1 = the w map is 4-D {64 cols, K, column
                            // block, group} and one copy loads both 64-column boxes of a CTA's
                            // atom (N a multiple of 64); 0 = 3-D {N, K, group}, one copy per box
  int* flags;               // Kgemm chunk mode: zeroed device flags, one per (expert, tile, CTA
                            // of the pair); null = tile mode
};

// Arguments of the MXFP8 Mgemm besides its tensor maps.
struct MxArgs {
  const int32_t* offsets;   // device [E+1]
  const uint8_t* sfa;       // blocked E8M0 scales of A (rows grouped by offsets)
  const uint8_t* sfb;       // blocked E8M0 scales of B (E groups of N rows)
  int E, M, N, K;
  void* out;                // y (bf16), or dW (fp32) for the K-grouped GEMM
  unsigned int* status;
  unsigned long long wait_limit_ns;
  int accumulate;           // K-grouped: 1 = dW += result, 0 = dW = result
};

// CTA group of the tensor-core MMAs: 2 (default) = a CTA pair computes one
// tile with tcgen05.mma.cta_group::2; 1 = one CTA per tile.
#ifndef RG_CTA_PAIR
#define RG_CTA_PAIR 1
#endif
constexpr int kCtaGroup = RG_CTA_PAIR ? 2 : 1;
// MXFP8 weight-gradient pipeline: stages of 128 expert rows, and the fp32
// epilogue's TMA boxes (32 rows x BOX_COLS columns; 16 columns use a 64-byte
// swizzle, 32 a 128-byte one), one staging buffer per epilogue warp.
// Compile-time switches for comparison builds.
// dW columns per tile: 256 (one tensor-memory accumulator beside the scale
// slots) or 128 (two accumulators, so the stores of one tile overlap the next
// tile's MMAs; a comparison build: each stage then carries half the MMA work
// for two thirds of the operand bytes, and the kernel is bound by operand
// delivery, not by the stores)
#ifndef RG_MXK_BN
#define RG_MXK_BN 256
#endif
#ifndef RG_MXK_STAGES
#define RG_MXK_STAGES (RG_MXK_BN == 128 ? 6 : 4)
#endif
#ifndef RG_MXK_BOX_COLS
#define RG_MXK_BOX_COLS 16
#endif
#ifndef RG_MXK_EPI_GROUP
#define RG_MXK_EPI_GROUP 1
#endif
namespace mxk {
constexpr int STAGES = RG_MXK_STAGES;
constexpr int BN = RG_MXK_BN;
static_assert(BN == 128 || BN == 256, "MXFP8 wgrad tiles are 128 or 256 dW columns wide");
constexpr int BOX_COLS = RG_MXK_BOX_COLS;
constexpr int EPI_GROUP = RG_MXK_EPI_GROUP;  // dW boxes staged and stored per bulk group
static_assert(EPI_GROUP == 1 || EPI_GROUP == 2 || EPI_GROUP == 4, "1, 2 or 4 boxes per bulk group");
constexpr int CHUNK_ROWS = 4096;  // rows summed in tensor memory per partial (32 stages of 128)
static_assert(BOX_COLS == 16 || BOX_COLS == 32, "dW boxes are 16 or 32 fp32 columns wide");
}  // namespace mxk

// MXFP8 Mgemm: 0 (default) = one CTA per 128 x 256 tile; 1 = a CTA pair
// computes a 256 x 256 tile with the block-scaled tcgen05.mma.cta_group::2
// (comparison build: measured 13-22% slower on the 30B-A3B layer, the
// per-stage scale copies into tensor memory costing a pair more than a CTA).
#ifndef RG_MX_PAIR
#define RG_MX_PAIR 0
#endif
namespace mxm {
constexpr int CG = RG_MX_PAIR ? 2 : 1;
constexpr int BN_CTA = 256 / CG;  // B rows (output columns) loaded per CTA
}  // namespace mxm

// Largest E the kernels are set up for (shared-memory tables of E+1 ints).
constexpr int RG_MAX_EXPERTS_CFG = 1024;


// Tile geometry the host needs for tensor-map boxes and size checks.
namespace mg {
constexpr int BM = 128;                  // rows per CTA
constexpr int TILE_M = BM * kCtaGroup;   // rows per tile
constexpr int BN = 256;                  // output columns per tile
constexpr int BN_CTA = BN / kCtaGroup;   // B rows loaded per CTA
constexpr int BK = 64;
}  // namespace mg

// K-grouped pipeline shape (compile-time switches for comparison builds):
// rows of the contraction per stage, stages in the ring (CTA pairs), and the
// 32 x 32 fp32 dW boxes an epilogue warp stages and stores per bulk group.
#ifndef RG_KG_BR
#define RG_KG_BR 96
#endif
#ifndef RG_KG_STAGES
#define RG_KG_STAGES 4
#endif
#ifndef RG_KG_EPI_GROUP
#define RG_KG_EPI_GROUP 1
#endif
// Columns of a dW box (32 x 32 fp32 with a 128-byte swizzle, or 32 x 16 with a 64-byte one).
#ifndef RG_KG_BOX_COLS
#define RG_KG_BOX_COLS 32
#endif
// An L2 evict-last hint on the operand copies (1) or none (0).
#ifndef RG_KG_LOAD_HINT
#define RG_KG_LOAD_HINT 1
#endif
// Experts of fewer rows than this are light in the K-grouped schedule: their
// tiles are interleaved with the row blocks of the longer experts' tiles.
#ifndef RG_KG_LIGHT_ROWS
#define RG_KG_LIGHT_ROWS 512
#endif
namespace kg {
constexpr int BM = 128;                  // dW rows per CTA
constexpr int TILE_M = BM * kCtaGroup;   // dW rows per tile
constexpr int BN = 256;                  // dW columns per tile
constexpr int BN_CTA = BN / kCtaGroup;   // X columns loaded per CTA
constexpr int BR = RG_KG_BR;             // contraction rows per stage (BR / 16 MMA steps)
constexpr int STAGES = RG_KG_STAGES;
constexpr int EPI_GROUP = RG_KG_EPI_GROUP;
constexpr int BOX_COLS = RG_KG_BOX_COLS;
static_assert(BOX_COLS == 16 || BOX_COLS == 32, "dW boxes are 16 or 32 fp32 columns wide");
static_assert(BR % 16 == 0 && BR >= 16 && BR <= 256, "stages hold whole 16-row MMA steps");
static_assert(EPI_GROUP == 1 || EPI_GROUP == 2 || EPI_GROUP == 4, "1, 2 or 4 dW boxes per bulk group");
// Rows of one expert accumulated in tensor memory before the partial sum is
// folded into dW (store for the first chunk, fp32 reduce-add for the rest):
// whole stages, at most 4096 rows.  Bounds the length of each fp32
// accumulation chain inside the tensor cores.
constexpr int CHUNK_ROWS = 4096 / BR * BR;
constexpr int LIGHT_ROWS = RG_KG_LIGHT_ROWS;
static_assert(LIGHT_ROWS >= 1 && LIGHT_ROWS <= CHUNK_ROWS, "a light expert has rows, and fewer than one chunk");
}  // namespace kg

// Sleep between polls of the accumulator barrier by the epilogue of Mgemm
// pair tiles with eight epilogue warps (comparison builds; the one-stage
// tiles run on single CTAs, whose epilogue uses the suspending wait).
#ifndef RG_MG_SHORT_POLL_NS
#define RG_MG_SHORT_POLL_NS 1000
#endif

// Mgemm tile variants of the CTA-pair build: 64-column pair tiles for
// forward outputs at most 64 wide; a contraction that fits one 64-deep stage
// (one MMA per tile, the epilogue and the accumulator hand-over set the pace)
// runs on single CTAs, 128 x 256 tiles with RG_MG_ONE_STAGE_EPIW epilogue
// warps: the hand-over between the MMA and the epilogue inside one CTA is
// much shorter than across a pair.  The host encodes B's tensor map for the
// tile the launch uses and launches single-CTA tiles on a grid of one CTA
// per SM.
#ifndef RG_MG_ONE_STAGE_EPIW
#define RG_MG_ONE_STAGE_EPIW 8
#endif
inline bool mgemm_narrow(bool transpose_B, int N) { return kCtaGroup == 2 && !transpose_B && N <= 64; }
inline bool mgemm_one_cta(bool transpose_B, int N, int K) {
  return kCtaGroup == 2 && !mgemm_narrow(transpose_B, N) && K <= mg::BK;
}
// K columns per operand box: 64 (128-byte rows), or for single-CTA
// one-stage tiles of shorter contractions 16 or 32 (rows of 32 or 64 bytes
// with the swizzle of that width), so that the copies do not fill three
// quarters or half of each box with zeros.
inline int mgemm_kbox(bool transpose_B, int N, int K) {
  if (!mgemm_one_cta(transpose_B, N, K) || RG_MG_ONE_STAGE_EPIW != 8) return mg::BK;
  return K <= 16 ? 16 : K <= 32 ? 32 : mg::BK;
}
// B rows (output columns) per CTA of the launch's tile
inline int mgemm_b_box_rows(bool transpose_B, int N, int K) {
  return mgemm_narrow(transpose_B, N) ? 32 : mgemm_one_cta(transpose_B, N, K) ? mg::BN : mg::BN_CTA;
}

// Bytes of dynamic shared memory a launch with E experts needs.
size_t mgemm_smem_bytes(int E);
size_t kgemm_smem_bytes(int E, size_t max_smem);  // of the ring a launch with E experts uses

// One-time per-device kernel attribute setup: allow up to `max_smem` bytes
// of dynamic shared memory (the device's opt-in limit).
cudaError_t mgemm_setup(int max_smem);
cudaError_t kgemm_setup(int max_smem);

// Number of 2-CTA clusters of each kernel that can be resident at once.
cudaError_t mgemm_max_clusters(int* clusters, int max_smem);
cudaError_t kgemm_max_clusters(int* clusters, int max_smem);

// tmA: x with boxes of 128 rows; tmAh: the same tensor with boxes of 64 rows
// (an expert's last row block of at most 128 rows, split 64 / 64 between the
// CTAs of a pair).
// grid: CTAs of the pair tiles; sms: CTAs of the single-CTA tiles (one per SM)
cudaError_t launch_mgemm(bool transpose_B, const CUtensorMap& tmA, const CUtensorMap& tmAh,
                         const CUtensorMap& tmB, const CUtensorMap& tmY, const GroupArgs& args, int grid,
                         int sms, cudaStream_t stream);
// Forward gate-up GEMM with the SwiGLU activation in the epilogue: B = w13
// [E, 2F, K] (gate rows then up rows), args.N = 2F, tmH/args.out = h [M, F],
// tmY13/args.out2 = y13 [M, 2F] or null.  CTA pairs only.
cudaError_t launch_mgemm_swiglu(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmH,
                                const CUtensorMap& tmY13, const GroupArgs& args, int grid,
                                cudaStream_t stream);
// Input gradient of the down projection fused with the SwiGLU backward:
// A = dy [M, K], B = w2 [E, K, F] (transpose_B), args.N = F, args.out2 = y13
// [M, 2F] (read), tmDy13/args.out = dy13 [M, 2F] (written).
cudaError_t launch_mgemm_swiglu_dgrad(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                      const CUtensorMap& tmDy13, const GroupArgs& args, int grid,
                                      cudaStream_t stream);
// Four-stage ring, or three stages when the expert tables would not fit beside four.
cudaError_t launch_kgemm(const CUtensorMap& tmG, const CUtensorMap& tmX, const CUtensorMap& tmD,
                         const GroupArgs& args, int grid, size_t max_smem, cudaStream_t stream);
// MXFP8 Mgemm (FP8 E4M3 operands, E8M0 scales per 32 K elements in the
// blocked layout) and the conversion of grouped scales to that layout.
size_t mx_smem_bytes(int E);
cudaError_t mx_setup(int max_smem);
// CTA pairs: 2-CTA clusters of the MXFP8 Mgemm resident at once.
cudaError_t mx_max_clusters(int* clusters, int max_smem);
// tmSA / tmSB: the blocked scale buffers of A and B as rows of 256 bytes
// (the CTA-pair kernel copies its scale blocks through them).
cudaError_t launch_mx_mgemm(bool transpose_B, const CUtensorMap& tmA, const CUtensorMap& tmB,
                            const CUtensorMap& tmY, const CUtensorMap& tmSA, const CUtensorMap& tmSB,
                            const MxArgs& args, int grid, cudaStream_t stream);
cudaError_t launch_mx_blocked(const uint8_t* src, const int32_t* offsets, int G, int R, int KS, uint8_t* dst,
                              unsigned int* status, int num_sms, cudaStream_t stream);
// MXFP8 Kgemm (FP8 operands quantized along the rows, experts on 32-row
// boundaries) and the scale layout for groups along the contraction.
size_t mxk_smem_bytes(int E);
cudaError_t mxk_setup(int max_smem);
cudaError_t launch_mx_kgemm(const CUtensorMap& tmG, const CUtensorMap& tmX, const CUtensorMap& tmD,
                            const MxArgs& args, int grid, cudaStream_t stream);
cudaError_t launch_mx_blocked_k(const uint8_t* src, const int32_t* offsets, int G, int R, int KS, uint8_t* dst,
                                unsigned int* status, int num_sms, cudaStream_t stream);
cudaError_t launch_wait_selftest(unsigned int* status, unsigned long long limit_ns,
                                 cudaStream_t stream);

}  // namespace rg
