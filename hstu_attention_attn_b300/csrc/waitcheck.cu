// waitcheck.cu -- self-check of the bounded-wait path of the tcgen05 kernels.
// One CTA holds tensor memory and waits on an mbarrier that nothing completes,
// with the two wait forms the kernels use (the tight one of the MMA and
// epilogue warps, the sleeping warp-wide one of the TMA producers).  The waits
// give up after their limit, the CTA records the timeout in the status word,
// raises its abort flag, frees its tensor memory and returns, exactly as an
// attention or GEMM kernel does when a partner stops making progress.
#include "common.cuh"

namespace mtgr {

__global__ void __launch_bounds__(64, 1) wait_timeout_kernel(int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_word;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // no thread ever arrives
    abort_word = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  volatile int* abort_flag = &abort_word;
  const bool ok = warp == 0 ? mbar_wait(&bar, 0, abort_flag) : mbar_wait_warp_sleepy(&bar, 0, abort_flag);
  if (!ok) {
    *abort_flag = 1;
    atomicOr(status, DEV_ERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 32);
  }
}

cudaError_t launch_wait_timeout(int32_t* status, cudaStream_t s) {
  TraceScope tr("wait_timeout", s);
  wait_timeout_kernel<<<1, 64, 0, s>>>(status);
  return cudaGetLastError();
}

}  // namespace mtgr
