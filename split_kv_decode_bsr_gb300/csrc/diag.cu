// Failure-detection check: a kernel waits, through the same bounded mbarrier wait
// the attention and decode kernels use, on a barrier phase that nothing completes.
// The wait gives up after the caller's short limit, records its code in the device
// error word and the kernel returns; the context stays usable. No fault, trap or
// unbounded wait is involved.
#include "internal.h"
#include "ptx.cuh"

namespace sta {
namespace {

constexpr int kDiagWaitCode = 0x7f1;

__global__ void bounded_wait_check_kernel(int* err, unsigned long long limit_ns, int* outcome) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival completes phase 0; none is ever made
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) *outcome = mbar_wait(&bar, 0, err, kDiagWaitCode, limit_ns) ? 1 : 0;
}

}  // namespace
}  // namespace sta

using namespace sta;

extern "C" sta_status sta_check_bounded_wait(int64_t limit_ns, int* outcome_dev, sta_stream stream) {
  if (limit_ns < 1000 || limit_ns > (int64_t)kWaitLimitNs || !outcome_dev) return STA_ERR_INVALID_ARG;
  if ((uintptr_t)outcome_dev & 3u) return STA_ERR_UNSUPPORTED;
  int* err = device_error_word();
  if (!err) return STA_ERR_CUDA;
  bounded_wait_check_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err, (unsigned long long)limit_ns, outcome_dev);
  STA_LAUNCH_CHECK();
  return STA_OK;
}
