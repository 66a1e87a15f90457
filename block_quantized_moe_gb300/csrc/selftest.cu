// Self-test of the bounded pipeline waits (failure detection; the pages have no
// counterpart). Every TMA/tensor-core pipeline wait in this library gives up after a time
// limit, raises FTMOE_ERR_WAIT_TIMEOUT in the device error word and lets the kernel return
// normally. This kernel makes exactly that wait run out: one thread waits, through the same
// mbar_wait the GEMMs use, on a shared-memory mbarrier that nothing ever arrives on, with a
// short limit. No TMA load, MMA or tensor memory is involved, so nothing is left in flight.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace ftmoe {

__global__ void __launch_bounds__(32) wait_timeout_selftest_kernel(unsigned long long limit_ns,
                                                                    unsigned long long* elapsed_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(smem_u32(&bar), 1);  // one arrival completes phase 0; none ever comes
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const unsigned long long t0 = globaltimer();
  const bool done = mbar_wait(smem_u32(&bar), 0, &abort_flag, limit_ns);
  const unsigned long long t1 = globaltimer();
  if (elapsed_ns != nullptr) *elapsed_ns = done ? 0ull : t1 - t0;
}

FTMOE_DEFINE_ERR_READER(read_err_selftest)

}  // namespace ftmoe

extern "C" ftmoe_status ftmoe_selftest_wait_timeout(uint64_t timeout_ns, unsigned long long* elapsed_ns,
                                                    void* stream) {
  if (timeout_ns < 1000ull || timeout_ns > 1000000000ull) return FTMOE_INVALID_ARG;
  const cudaError_t e = ftmoe::launch_kernel(ftmoe::wait_timeout_selftest_kernel, dim3(1), dim3(32), 0,
                                             reinterpret_cast<cudaStream_t>(stream), false,
                                             (unsigned long long)timeout_ns, elapsed_ns);
  return e == cudaSuccess ? FTMOE_OK : FTMOE_CUDA_ERROR;
}
