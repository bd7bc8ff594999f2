// Self-test of the bounded device waits every kernel of the library uses.
//
// The kernel waits on an mbarrier that nothing ever completes.  Warp 0 waits
// with the caller's short limit; when it runs out it raises the CTA's abort
// flag and reports BCA_ERR_TIMEOUT.  Warps 1-3 wait with a limit 50x longer
// and must notice the abort flag and return at once, the way the producer,
// MMA and softmax roles of the attention kernel give up together.  Nothing is
// faulted and nothing hangs: the kernel ends after about limit_ns and the
// context stays usable.
#include "common.cuh"
#include "ptx.cuh"

namespace bca {
namespace {

__global__ void __launch_bounds__(128)
    wait_timeout_selftest_kernel(uint64_t limit_ns, int32_t* status, uint64_t* elapsed_ns) {
  __shared__ uint64_t never;   // no thread ever arrives on it
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&never, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  const uint64_t t0 = globaltimer_ns();
  if (warp == 0) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&never, 0, &abort_flag, limit_ns));
    if (!ok && lane == 0) {
      abort_flag = 1;
      report_status(status, BCA_ERR_TIMEOUT);
    }
  } else {
    mbar_wait(&never, 0, &abort_flag, 50 * limit_ns);
  }
  __syncthreads();
  if (threadIdx.x == 0 && elapsed_ns != nullptr) *elapsed_ns = globaltimer_ns() - t0;
}

}  // namespace
}  // namespace bca

extern "C" bca_status bca_selftest_wait_timeout(uint64_t limit_ns, int32_t* status_dev,
                                                uint64_t* elapsed_ns_dev, void* stream) {
  if (status_dev == nullptr || limit_ns == 0 || limit_ns > 1000000000ull)
    return BCA_ERR_INVALID_ARG;
  bca::wait_timeout_selftest_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      limit_ns, status_dev, elapsed_ns_dev);
  return cudaGetLastError() == cudaSuccess ? BCA_OK : BCA_ERR_CUDA;
}
