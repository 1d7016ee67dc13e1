// inkling_rel_attn_selftest_timeout: exercises the bounded pipeline wait that
// every kernel of the library uses, without a fault: one thread waits on an
// mbarrier that nothing ever arrives on, gives up after `timeout_ms`, reports
// INKLING_DEVERR_TIMEOUT in the caller's error word and returns, leaving the
// context usable.
#include "internal.h"
#include "plan.cuh"
#include "ptx.cuh"

namespace ira {

__global__ void timeout_probe_kernel(int32_t* err, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing arrives on `bar`: phase 0 never completes
    if (!mbar_wait(smem_u32(&bar), 0, &abort_flag, timeout_ns)) report(err, INKLING_DEVERR_TIMEOUT);
  }
}

}  // namespace ira

extern "C" int inkling_rel_attn_selftest_timeout(int32_t* device_error, int32_t timeout_ms,
                                                 void* stream) {
  if (!device_error || timeout_ms < 1 || timeout_ms > 10000) return INKLING_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(device_error) & 3) != 0) return INKLING_ERR_ALIGN;
  ira::timeout_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      device_error, (unsigned long long)timeout_ms * 1000000ull);
  return cudaGetLastError() == cudaSuccess ? INKLING_OK : INKLING_ERR_CUDA;
}
