// rx_selftest_wait_timeout: exercises the bounded mbarrier wait every tcgen05 kernel uses, on a
// barrier that nothing arrives at, so the timeout path is tested without faulting or hanging a GPU.
#include <cuda_runtime.h>

#include "rx_internal.h"
#include "tc.cuh"

namespace {

// One CTA: thread 0 initialises a barrier expecting one arrival, then every thread waits for its
// first phase with the given limit; no thread arrives.  The wait gives up, raises the CTA's abort
// flag and records RX_ERR_TIMEOUT in *status (first error wins).
__global__ void wait_timeout_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t mbar;
  __shared__ int abort_flag;
  const uint32_t bar = rx::smem_u32(&mbar);
  if (threadIdx.x == 0) {
    rx::tc::mbar_init(bar, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  rx::tc::mbar_wait(bar, 0, &abort_flag, status, limit_ns);
}

}  // namespace

extern "C" rx_status rx_selftest_wait_timeout(int32_t* status, int64_t limit_ns,
                                              rx_stream_t stream) {
  if (!status || limit_ns <= 0 || limit_ns > 2000000000LL)
    return rx::set_error(RX_ERR_INVALID, "rx_selftest_wait_timeout: status NULL or limit not in (0, 2 s]");
  wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status, (uint64_t)limit_ns);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? RX_OK : rx::set_error(RX_ERR_CUDA, cudaGetErrorString(e));
}
