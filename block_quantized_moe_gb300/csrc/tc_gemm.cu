// tcgen05 grouped GEMM (placeholder until the tensor-core kernel lands: reports
// unsupported so the grouped path runs on the streaming kernel).
#include "common.cuh"
#include "internal.h"

namespace ftmoe {

cudaError_t launch_tc_gemm(const TcGemmArgs&, cudaStream_t, int* unsupported) {
  *unsupported = 1;
  return cudaSuccess;
}

FTMOE_DEFINE_ERR_READER(read_err_tc_gemm)

}  // namespace ftmoe
