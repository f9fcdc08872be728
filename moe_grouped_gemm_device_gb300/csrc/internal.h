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
  void* out;                // y (bf16) for Mgemm, dW (fp32) for Kgemm
  unsigned int* status;     // device status word
  unsigned long long wait_limit_ns;
};

// Tile shapes (also used by the host to size shared memory).
namespace mg {
constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 4, EPI_BUFS = 1, EPI_BUF_BYTES = 32 * 128;
constexpr int THREADS = 192;
}  // namespace mg

#ifndef RG_KG_STAGES
#define RG_KG_STAGES 4
#endif
#ifndef RG_KG_EPI_BUFS
#define RG_KG_EPI_BUFS 1
#endif
namespace kg {
constexpr int BM = 128, BN = 256, BR = 64, STAGES = RG_KG_STAGES;
constexpr int A_BYTES = BM * BR * 2, B_BYTES = BN * BR * 2, STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 4, EPI_BUFS = RG_KG_EPI_BUFS, EPI_BUF_BYTES = 32 * 128;
constexpr int THREADS = 192;
// Rows of one expert accumulated in tensor memory before the partial sum is
// folded into dW (store for the first chunk, fp32 reduce-add for the rest).
// Bounds the length of each fp32 accumulation chain inside the tensor cores.
constexpr int CHUNK_ROWS = 4096;
static_assert(CHUNK_ROWS % BR == 0, "chunks must hold whole row blocks");
}  // namespace kg

// Bytes of dynamic shared memory a launch with E experts needs.
size_t mgemm_smem_bytes(int E);
size_t kgemm_smem_bytes(int E);

// One-time per-device kernel attribute setup: allow up to `max_smem` bytes
// of dynamic shared memory (the device's opt-in limit).
cudaError_t mgemm_setup(int max_smem);
cudaError_t kgemm_setup(int max_smem);

cudaError_t launch_mgemm(bool transpose_B, const CUtensorMap& tmA, const CUtensorMap& tmB,
                         const CUtensorMap& tmY, const GroupArgs& args, int grid,
                         cudaStream_t stream);
cudaError_t launch_kgemm(const CUtensorMap& tmG, const CUtensorMap& tmX, const CUtensorMap& tmD,
                         const GroupArgs& args, int grid, cudaStream_t stream);
cudaError_t launch_zero_f32(float* p, int64_t n, int grid, cudaStream_t stream);
cudaError_t launch_wait_selftest(unsigned int* status, unsigned long long limit_ns,
                                 cudaStream_t stream);

}  // namespace rg
