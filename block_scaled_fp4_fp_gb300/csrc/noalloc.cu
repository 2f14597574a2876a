// noalloc.cu -- fp4_amax_global_scale_noalloc: the tensor-amax / global-scale
// entry point for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they need a global scale: code recording into a CUDA stream capture, engines
// that plan every byte of device memory ahead of time and hand kernels a fixed
// arena, and hosts that forbid allocation on their latency-critical path.  The
// regular fp4_amax_global_scale needs caller-provided scratch for its per-block
// partial maxima; this variant keeps that scratch in a fixed file-scope device
// array instead, so the caller passes only the input and the two outputs.
//
// The array lives in every device that loads this library until the process
// exits.  Calls share it: two calls that overlap on the GPU (different streams
// without ordering between them) race on it.  Each call writes every slot it
// later reads, so nothing has to be cleared between calls.
#include <mutex>

#include "../../include/fp4_gb300.h"
#include "common.cuh"
#include "launch.h"

namespace fp4 {
namespace {

constexpr int kNoAllocPartials = 1024;  // 4 KiB of per-block partial maxima
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint32_t g_amax_scratch[kNoAllocPartials];

std::mutex g_mu;
uint32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_amax_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, taken once per device with that device current.
fp4_status scratch_for_current_device(uint32_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP4_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FP4_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_amax_scratch) != cudaSuccess || p == nullptr) return FP4_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<uint32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return FP4_OK;
}

}  // namespace
}  // namespace fp4

extern "C" fp4_status fp4_amax_global_scale_noalloc(const fp4_bf16* x, int64_t n, float* gs_out,
                                                    float* amax_out, cudaStream_t stream) {
  using namespace fp4;
  if (!x || !gs_out || n <= 0) return FP4_ERR_INVALID_ARG;
  if (n > FP4_AMAX_NOALLOC_MAX_ELEMS) return FP4_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(gs_out) & 3) ||
      (amax_out && (reinterpret_cast<uintptr_t>(amax_out) & 3)))
    return FP4_ERR_ALIGNMENT;
  const DevInfo* d = nullptr;  // cached per device: compute capability checked, SM count; allocates nothing
  fp4_status st = (fp4_status)current_device_info(&d);
  if (st != FP4_OK) return st;
  uint32_t* scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != FP4_OK) return st;
  const cudaError_t e = launch_amax(*d, x, n, gs_out, amax_out, scratch, kNoAllocPartials, stream);
  return e == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}
