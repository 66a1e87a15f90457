// Self-tests. First, the bounded pipeline waits (failure detection; the pages have no
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

// Self-test of the division by a shared divisor (common.cuh SharedDivisor, Markstein's
// correction) against the IEEE quotient (__fdiv_rn), bit for bit:
//   mode 0: every mantissa of the divisor in [1, 2) scaled by 2^es, 4096 dividends each (8 of
//           them next to the divisor, the rest of random mantissas and signs with |x / d| from
//           2^-31 to 2^10), plus +0 and -0;
//   mode 1: 1024 divisors of random mantissas and exponents, each against every dividend
//           mantissa at a chosen exponent.
// One thread per mantissa (2^23 threads); counts[0] += quotients checked, counts[1] +=
// quotients that differ.
__device__ __forceinline__ uint32_t st_mix(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352dU;
  x ^= x >> 15;
  x *= 0x846ca68bU;
  x ^= x >> 16;
  return x;
}

__global__ void __launch_bounds__(256) shared_division_selftest_kernel(int mode, int es,
                                                                       unsigned long long* counts) {
  const uint32_t m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= (1u << 23)) return;
  unsigned long long n = 0, bad = 0;
  if (mode == 0) {
    const float d = __uint_as_float(((uint32_t)(127 + es) << 23) | m);
    const SharedDivisor ds(d);
    for (int j = 0; j < 4096; ++j) {
      const uint32_t h = st_mix(m * 4096u + (uint32_t)j + (uint32_t)(es + 64) * 977u);
      const int ex = (int)(h % 40u) - 30 + es;
      uint32_t bits = ((uint32_t)(127 + ex) << 23) | (st_mix(h) & 0x7FFFFFu);
      if (j < 8) bits = __float_as_uint(d) + (uint32_t)j - 4u;
      const float x = (h & 0x80000000u) ? -__uint_as_float(bits) : __uint_as_float(bits);
      bad += __float_as_uint(ds.div(x)) != __float_as_uint(__fdiv_rn(x, d)) ? 1 : 0;
      ++n;
    }
    bad += __float_as_uint(ds.div(-0.0f)) != __float_as_uint(__fdiv_rn(-0.0f, d)) ? 1 : 0;
    bad += __float_as_uint(ds.div(0.0f)) != __float_as_uint(__fdiv_rn(0.0f, d)) ? 1 : 0;
    n += 2;
  } else {
    for (int k = 0; k < 1024; ++k) {
      const uint32_t h = st_mix((uint32_t)k * 2654435761u + 12345u);
      const int dexp = (int)(h % 60u) - 30;
      const float d = __uint_as_float(((uint32_t)(127 + dexp) << 23) | (st_mix(h ^ 0x9e3779b9u) & 0x7FFFFFu));
      const SharedDivisor ds(d);
      const float x = __uint_as_float(((uint32_t)(127 + dexp + (k % 40) - 30) << 23) | m);
      bad += __float_as_uint(ds.div(x)) != __float_as_uint(__fdiv_rn(x, d)) ? 1 : 0;
      ++n;
    }
  }
  atomicAdd(&counts[0], n);
  if (bad) atomicAdd(&counts[1], bad);
}

FTMOE_DEFINE_ERR_READER(read_err_selftest)

}  // namespace ftmoe

extern "C" ftmoe_status ftmoe_selftest_shared_division(unsigned long long* counts, void* stream) {
  if (!counts) return FTMOE_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(counts, 0, 2 * sizeof(unsigned long long), st);
  const int es[3] = {-20, 0, 17};
  for (int i = 0; i < 3 && e == cudaSuccess; ++i)
    e = ftmoe::launch_kernel(ftmoe::shared_division_selftest_kernel, dim3((1u << 23) / 256), dim3(256), 0, st, false,
                             0, es[i], counts);
  if (e == cudaSuccess)
    e = ftmoe::launch_kernel(ftmoe::shared_division_selftest_kernel, dim3((1u << 23) / 256), dim3(256), 0, st, false,
                             1, 0, counts);
  return e == cudaSuccess ? FTMOE_OK : FTMOE_CUDA_ERROR;
}

extern "C" ftmoe_status ftmoe_selftest_wait_timeout(uint64_t timeout_ns, unsigned long long* elapsed_ns,
                                                    void* stream) {
  if (timeout_ns < 1000ull || timeout_ns > 1000000000ull) return FTMOE_INVALID_ARG;
  const cudaError_t e = ftmoe::launch_kernel(ftmoe::wait_timeout_selftest_kernel, dim3(1), dim3(32), 0,
                                             reinterpret_cast<cudaStream_t>(stream), false,
                                             (unsigned long long)timeout_ns, elapsed_ns);
  return e == cudaSuccess ? FTMOE_OK : FTMOE_CUDA_ERROR;
}
