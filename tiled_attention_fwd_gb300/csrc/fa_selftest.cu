// Diagnostic of the bounded device-side waits (no counterpart in the pages:
// the attention kernels' failure handling is this library's own).  One block
// waits on shared-memory barriers that nothing ever signals, through the same
// wait_bar / warp_wait_bar as the attention kernels: the first wait to pass
// the time limit raises the block's abort flag and records its code in the
// device status word, every other wait then returns at once, and the kernel
// ends.  It holds no tensor memory, issues no copies and touches no memory of
// the caller, so a test can make a wait expire without faulting or hanging
// the GPU.
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

__global__ void __launch_bounds__(128, 1) fa_selftest_wait_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitGuard g{&abort_flag, status, limit_ns};
  // Warp 0 waits warp-wide (the softmax and correction form); the other warps
  // wait lane by lane on the second barrier (the producer form).  Phase 0 of
  // either barrier never completes.
  if (warp == 0)
    (void)warp_wait_bar(smem_u32(&bars[0]), 0, g, kStatusTimeoutSoftmax);
  else
    (void)wait_bar(smem_u32(&bars[1]), 0, g, kStatusTimeoutLoad);
}

}  // namespace

int launch_selftest_wait(const LaunchCtx& ctx) {
  fa_selftest_wait_kernel<<<1, 128, 0, ctx.stream>>>(ctx.status, ctx.limit_ns);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace fa
