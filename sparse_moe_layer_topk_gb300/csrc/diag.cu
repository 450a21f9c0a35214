// Diagnostic of the bounded waits: every mbarrier wait in the library's
// kernels (mbar_wait) gives up after a time limit, records MOE_FLAG_TIMEOUT in
// the caller's error word and lets its kernel return, instead of spinning
// forever. This kernel runs that same wait, with a caller-chosen limit, on a
// barrier that nothing ever arrives at, so the give-up path can be exercised
// without a fault: no TMA copy, tensor map or tensor memory is involved.
#include "common.cuh"
#include "gemm.h"
#include "timing.h"

namespace moe {
namespace {

__global__ void wait_timeout_kernel(unsigned long long limit_ns, int* err_flag,
                                    long long* waited_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // expects one arrival; none comes
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long t0 = globaltimer_ns();
    const bool done = mbar_wait(&bar, 0, &abort_flag, limit_ns);
    *waited_ns = static_cast<long long>(globaltimer_ns() - t0);
    if (!done) set_flag(err_flag, MOE_FLAG_TIMEOUT);
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_diag_wait_timeout(long long limit_ns, int32_t* err_flag, long long* waited_ns,
                                     void* stream) {
  if (!err_flag || !waited_ns) return MOE_ERR_ARG;
  if (limit_ns < 1000 || limit_ns > 1000000000ll) return MOE_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  {
    LaunchTimer lt("diag_wait_timeout", st);
    wait_timeout_kernel<<<1, 32, 0, st>>>(static_cast<unsigned long long>(limit_ns), err_flag,
                                          waited_ns);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
