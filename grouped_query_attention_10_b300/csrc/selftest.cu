// selftest.cu -- exercises the kernels' failure path on the device without a
// fault: the bounded barrier wait every role of every kernel uses is run
// against a barrier that nothing ever arrives at. It gives up after the given
// limit, raises the CTA's abort flag and the kernel reports GQA_ERR_TIMEOUT in
// the status word, exactly as a stalled prefill or decode would; the context
// stays usable.
#include "../../include/gqa.h"
#include "launch.h"
#include "ptx.cuh"

namespace gqa {

__global__ void bounded_wait_selftest_kernel(int32_t* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // nothing arrives on `bar`: every lane's wait must end by the limit
  const bool ok = mbar_wait_for(&bar, 0, &abort_flag, limit_ns);
  __syncthreads();
  if (threadIdx.x == 0 && (!ok || abort_flag)) record_status(status, GQA_ERR_TIMEOUT);
}

cudaError_t launch_bounded_wait_selftest(int32_t* status, long long limit_ns, cudaStream_t s) {
  bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(status,
                                                static_cast<unsigned long long>(limit_ns));
  return cudaGetLastError();
}

}  // namespace gqa
