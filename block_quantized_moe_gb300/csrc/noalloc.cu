// Allocation-free fused forward for callers that cannot obtain device memory themselves.
//
// The intermediate buffers live in one file-scope device array instead of a
// caller-provided workspace. Every GPU that loads the library holds this array until the
// process exits. The array's host-side name is only a stand-in for the symbol, never a
// device address, so the address is fetched with cudaGetSymbolAddress once per device
// (the first call on that device, with it current) and cached. The cached address is that
// of the device's primary context; a context destroyed and recreated (cudaDeviceReset)
// places the array elsewhere, and the library has to be reloaded after it.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace ftmoe {

// Largest workspace the allocation-free forward serves: decode-size shapes (for example
// 8 tokens, top-8, hidden 4096, intermediate 1024 need about 9.2 MiB on the fused decode
// path) fit; larger shapes are refused.
constexpr size_t kNoAllocScratchBytes = 16u << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

static void* noalloc_scratch(int device) {
  constexpr int kMaxDevices = 64;
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  if (device < 0 || device >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[device] = p;
  }
  return addr[device];
}

}  // namespace ftmoe

extern "C" ftmoe_status ftmoe_moe_forward_noalloc(const ftmoe_moe_args* args, void* stream) {
  if (!args) return FTMOE_INVALID_ARG;
  const size_t need = ftmoe_forward_workspace_bytes(&args->shape);
  if (need == 0) return FTMOE_INVALID_ARG;
  if (need > ftmoe::kNoAllocScratchBytes) return FTMOE_WORKSPACE_TOO_SMALL;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return FTMOE_CUDA_ERROR;
  void* scratch = ftmoe::noalloc_scratch(device);
  if (!scratch) return FTMOE_CUDA_ERROR;
  // the forward writes every scratch region before it reads it, so the previous call's
  // contents never leak into this one and nothing needs clearing
  return ftmoe_moe_forward(args, scratch, ftmoe::kNoAllocScratchBytes, stream);
}
