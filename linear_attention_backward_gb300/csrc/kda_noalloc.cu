// kda_noalloc.cu -- kda_bwd_noalloc: the backward pass with its scratch
// memory (per-chunk states, state gradients and dA_log partials) held in a
// fixed device array that is part of the library image, for callers that
// cannot allocate device memory themselves.
//
// Who needs it: code that runs where cudaMalloc is off limits or unsafe --
// e.g. inside an allocator callback, under a framework whose memory pool
// owns all device memory, in a real-time / pre-allocated-only process, or
// from a plugin host that gives the plugin no allocation API.  kda_bwd asks
// such callers for a workspace buffer they have no way to provide.
//
// How it works: the array below is part of this library's device image, one
// copy per GPU, reserved when the runtime loads the module that holds it --
// under lazy module loading (the CUDA default since 12.2) that is the first
// kda_bwd_noalloc call on a device, under eager loading the creation of the
// context -- and kept until the process exits.  Host code cannot use the
// array's name as a device address (it denotes a host shadow symbol), so
// every call looks the device address up with cudaGetSymbolAddress, with the
// calling thread's current device.  After the first call the lookup only
// reads the runtime's module table; doing it every call (rather than caching
// the pointer) keeps the address right if the context is torn down and the
// module reloaded at another address.
#include <cuda_runtime.h>

#include "kda.h"

namespace {

constexpr size_t kScratchBytes = (size_t)64 << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the current device's copy of the scratch array, or
// nullptr if the runtime cannot give it.
void *scratch_for_current_device() {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
  return p;
}

}  // namespace
extern "C" {

size_t kda_noalloc_scratch_bytes(void) { return kScratchBytes; }

kda_status kda_bwd_noalloc(const kda_shape *shape, const void *q, const void *k, const void *v,
                           const void *g, const void *beta, const float *A_log,
                           const float *dt_bias, const float *h0, const void *dO,
                           const float *dh_T, void *dq, void *dk, void *dv, void *dg,
                           void *dbeta, float *dA_log, float *ddt_bias, float *dh0,
                           kda_stream_t stream) {
  // a bad shape gives need == 0 here and is rejected by kda_bwd itself
  const size_t need = kda_workspace_bytes(shape);
  if (need > kScratchBytes) return KDA_ERR_TOO_LARGE;
  void *ws = scratch_for_current_device();
  if (ws == nullptr) return KDA_ERR_CUDA;
  // The scratch needs no initial content: every part the kernels read is
  // written earlier in the same call.
  return kda_bwd(shape, q, k, v, g, beta, A_log, dt_bias, h0, dO, dh_T, dq, dk, dv, dg, dbeta,
                 dA_log, ddt_bias, dh0, nullptr, ws, kScratchBytes, stream);
}

}  // extern "C"
