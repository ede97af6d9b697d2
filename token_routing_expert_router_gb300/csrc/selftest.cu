// Diagnostic: the bounded mbarrier wait every tcgen05 kernel of the library uses, run on a
// barrier that nothing ever arrives on. It must give up after the limit, record
// MOE_ERR_TIMEOUT in the status word and return, leaving the context usable. Nothing else
// is in flight in this kernel (no TMA copy, no MMA, no TMEM), so giving up is harmless.
#include "tc_common.cuh"

namespace moe {
namespace {

__global__ void bounded_wait_kernel(uint64_t timeout_ns, DeviceStatus* st) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) tc::mbar_wait(&bar, 0, &abort_flag, timeout_ns, st);  // phase 0 never completes
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_selftest_bounded_wait(int64_t timeout_ns, int32_t* device_status,
                                                  moe_stream_t stream) {
  if (!device_status || ((uintptr_t)device_status & 7u) || timeout_ns <= 0 || timeout_ns > 10000000000LL)
    return MOE_ERR_INVALID_ARG;
  moe::bounded_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(
      (uint64_t)timeout_ns, reinterpret_cast<moe::DeviceStatus*>(device_status));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
