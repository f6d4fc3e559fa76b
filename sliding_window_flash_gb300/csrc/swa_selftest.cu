// swa_selftest.cu — exercises the failure path every kernel relies on: a bounded mbarrier wait
// that runs out.  One thread waits on a barrier that nothing arrives on, with the same bounded
// wait the attention kernels use (about a second of SM clock); when the bound runs out the wait
// raises the block's abort flag and the per-device error word and returns, and the kernel exits.
// No trap, no fault, no endless loop: the context stays usable and swa_check_device reports
// SWA_ERR_DEVICE_TIMEOUT.
#include "swa_kernels.h"
#include "swa_ptx.cuh"

namespace swa {
namespace {

__global__ void __launch_bounds__(32, 1) swa_wait_timeout_selftest_kernel(unsigned* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncwarp();
  // nothing ever arrives on `bar`: the wait must run out and report it
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, err);
  __syncwarp();
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(unsigned* err, cudaStream_t stream) {
  swa_wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(err);
  return cudaGetLastError();
}

}  // namespace swa
