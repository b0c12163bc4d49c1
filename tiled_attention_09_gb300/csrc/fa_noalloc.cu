// fa_bwd_noalloc: the backward pass with its fp32 workspace (D, LSE*log2e and
// the dQ accumulator) held in a fixed device array that is part of this
// library, for callers that must not allocate device memory themselves.
//
// Who needs it: code that runs inside a host framework's enqueue hook (an
// inference runtime's plugin interface, an extension point of a training
// framework) whose contract forbids allocating on that path, and code whose
// device-memory budget is owned by another allocator, where a stray
// cudaMalloc would fail, fragment the pool or stall the device (it may
// synchronise). Such callers still hand over the inputs and outputs they own;
// only the scratch space comes from here.
//
// The array is device memory of this file's own module. Under lazy module
// loading (the CUDA default) a context gets its copy when the module is loaded
// there, which is the first fa_bwd_noalloc call in that context: that call
// allocates the FA_NOALLOC_SCRATCH_BYTES (64 MiB) through the driver's module
// loader, so it belongs at set-up time, outside the path that must not
// allocate and before any stream capture. Under CUDA_MODULE_LOADING=EAGER every
// context that loads the library gets the copy when the context is created,
// whether or not it ever calls this entry point. Either way the copy lasts as
// long as the context. In host code the array's name is not a device address:
// every call looks up the current device's copy with cudaGetSymbolAddress
// (with that device current), a host-side lookup once the module is loaded.
// Looking it up on every call, rather than caching it per device, keeps the
// address right when a context is re-created (after cudaDeviceReset the module
// is loaded again and the array can sit elsewhere). All calls share the one
// array: two calls whose work can overlap on the GPU (different streams, no
// ordering between them) race on it. Nothing in it has to start at zero: the
// preprocess kernel writes D and LSE*log2e in full and zeroes the dQ
// accumulator on every call.
#include <cuda_runtime.h>

#include <cstddef>

#include "../../include/fa.h"

namespace {

static __device__ __align__(256) unsigned char g_fa_bwd_scratch[FA_NOALLOC_SCRATCH_BYTES];

// Device address of the current device's copy of the scratch array, looked up on every call.
fa_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  if (major != 10 || minor != 3) return FA_ERR_UNSUPPORTED;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_fa_bwd_scratch) != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
  *out = p;
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                    const float* lse, void* dq, void* dk, void* dv, const void* o_lo, int B, int H,
                                    int N, int d, float scale, int causal, fa_dtype dtype, void* stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  if (need == 0) return FA_ERR_UNSUPPORTED;
  if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;  // problem too large for the fixed scratch
  void* ws = nullptr;
  fa_status s = scratch_for_current_device(&ws);
  if (s != FA_OK) return s;
  return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, o_lo, ws, FA_NOALLOC_SCRATCH_BYTES, B, H, N, d, scale, causal, dtype,
                stream);
}
