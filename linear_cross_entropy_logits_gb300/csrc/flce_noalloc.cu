// flce_fwd_bwd_noalloc: the fused forward+backward for callers that cannot hand the
// library a device workspace.
//
// Some callers cannot call cudaMalloc at the point where they need the loss: a framework
// that owns all device memory through its own pool (a raw allocation next to it fails or
// fragments memory), code that must not allocate after start-up because an allocation may
// synchronise the device, or a foreign-function layer that only forwards the inputs and
// outputs of the op. This entry point takes the same arguments as flce_fwd_bwd but uses a
// fixed scratch array compiled into the library instead of a caller-provided workspace.
//
// The scratch is a file-scope __device__ array of FLCE_NOALLOC_SCRATCH_BYTES. Every GPU
// that loads this library holds that much device memory until the process exits. Host code
// cannot use the array's name as a device address, so the first call on each device
// (with that device current) asks the runtime for the address with cudaGetSymbolAddress
// and caches it; make that first call before any stream capture. All calls share the one
// array: calls that overlap on the GPU (different streams, no ordering between them) race
// on it and give wrong results. Nothing in the array needs to start at zero: every call
// rewrites what it reads, and the status word it may hold is cleared by the call itself.
#include <mutex>

#include "flce_internal.cuh"

static __device__ __align__(256) unsigned char g_flce_scratch[FLCE_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {nullptr};

}  // namespace

extern "C" int32_t flce_fwd_bwd_noalloc(const flce_args* args, void* stream) {
  if (!args) return FLCE_ERR_INVALID_ARG;
  if (args->workspace != nullptr || args->workspace_bytes != 0 || args->profile != nullptr)
    return FLCE_ERR_INVALID_ARG;
  if (args->BT <= 0 || args->H <= 0 || args->V <= 0) return FLCE_ERR_INVALID_ARG;
  if (args->in_dtype != FLCE_F32 && args->in_dtype != FLCE_BF16 && args->in_dtype != FLCE_F16)
    return FLCE_ERR_INVALID_ARG;
  // The problem must fit the fixed scratch with at least one 128-row chunk.
  if (flce::plan_rows_for_bytes(args->BT, args->H, args->V, args->in_dtype,
                                FLCE_NOALLOC_SCRATCH_BYTES) <= 0)
    return FLCE_ERR_SCRATCH_LIMIT;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLCE_ERR_CUDA;
  if (dev < 0 || dev >= 64) return FLCE_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_flce_scratch) != cudaSuccess || p == nullptr) return FLCE_ERR_CUDA;
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  flce_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = FLCE_NOALLOC_SCRATCH_BYTES;
  return flce_fwd_bwd(&a, stream);
}
