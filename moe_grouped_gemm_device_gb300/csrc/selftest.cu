// Self-test of the bounded barrier waits, the failure-detection path of every
// pipeline kernel, run without a fault or a hang: each form of wait that the
// kernels use waits on a barrier that nothing signals and has to give up once
// its bound has passed, with the timeout status.
#include "internal.h"
#include "ptx.cuh"

namespace rg {
namespace {

// Warp 0 (lane 0): the suspending wait of single-CTA barriers.  Warp 1 (all
// lanes, as the MMA warp waits): the cluster-scope poll for barriers the peer
// CTA of a pair arrives on.  Warp 2: the epilogues' accumulator wait, one lane
// polling with a sleep.  Each wait has its own abort flag and status word, so
// that one running out does not end the others early; the device status gets
// kDevTimeout only when all three ran out, and nothing when any of them
// returned as if its barrier had completed.
__global__ void wait_selftest_kernel(unsigned int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar[3];
  __shared__ int abort_flag[3];
  __shared__ unsigned int st[3];
  __shared__ int gave_up[3];
  const int w = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 3; ++i) {
      mbar_init(smem_u32(&bar[i]), 1);
      abort_flag[i] = 0;
      st[i] = 0;
      gave_up[i] = 0;
    }
    fence_mbar_init();
  }
  __syncthreads();
  const WaitGuard g{&st[w], limit_ns, &abort_flag[w]};
  const uint32_t b = smem_u32(&bar[w]);
  bool done = true;
  if (w == 0) {
    if (lane == 0) done = mbar_wait(g, b, 0);
  } else if (w == 1) {
    done = __all_sync(0xffffffffu, mbar_wait_cl(g, b, 0)) != 0;
  } else {
    done = warp_wait_acc<2>(g, b, 0);
  }
  __syncwarp();
  if (lane == 0) gave_up[w] = !done && (st[w] & kDevTimeout) != 0;
  __syncthreads();
  if (threadIdx.x == 0 && gave_up[0] && gave_up[1] && gave_up[2]) atomicOr(status, kDevTimeout);
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned int* status, unsigned long long limit_ns,
                                 cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(96);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, wait_selftest_kernel, status, limit_ns);
}

}  // namespace rg
