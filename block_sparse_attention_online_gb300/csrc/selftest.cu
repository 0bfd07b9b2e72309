// Diagnostic kernel for the failure path of the bounded waits: a CTA that
// holds TMEM waits, with every thread, on an mbarrier phase that nothing
// completes.  The first wait to give up (after the 1 s limit) raises the
// CTA's abort flag and ORs kErrTimeout into the device error word, the other
// waits then fail at once, and the CTA frees its TMEM and exits, so the
// context stays usable and the host reads the timeout as a status.
#include "internal.h"
#include "tc_common.cuh"

namespace attn_skip {
namespace {

using namespace tc;

__global__ void __launch_bounds__(64, 1) selftest_wait_kernel(unsigned *err) {
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // one arrival expected; none is ever made
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_base), 32);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  volatile int *abort = &abort_flag;
  mbar_wait_warp(smem_u32(&bar), 0, abort, err, kErrTimeout);  // gives up; result unused
  __syncwarp();
  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem_base, 32);
  }
}

}  // namespace

cudaError_t launch_selftest_wait(unsigned *err, cudaStream_t s) {
  selftest_wait_kernel<<<1, 64, 0, s>>>(err);
  return cudaGetLastError();
}

}  // namespace attn_skip
