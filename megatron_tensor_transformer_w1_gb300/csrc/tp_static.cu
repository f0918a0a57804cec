// tp_static.cu -- a forward pass that allocates no device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run the forward pass: an inference server that reserves all device
// memory up front and forbids allocation while it serves requests, a plugin
// whose host framework owns the allocator and rejects allocations it did not
// make, or a latency-critical loop where an allocation could block.  Such a
// caller passes only its inputs and output; the scratch the forward pass
// needs (the device error word, the hidden activations h^(t) and the fp32
// shard partials y^(t)) comes from the file-scope array below.
//
// The array is static device memory of this file's module.  A device holds
// TPFFN_STATIC_SCRATCH_BYTES of it from the moment the module is loaded on
// that device until the process exits.  Under CUDA's lazy module loading
// (the runtime's default) that moment is the first cudaGetSymbolAddress of
// the array on the device, which is why a call with n_tokens = 0 performs
// exactly that look-up: a caller that must not allocate later makes it at
// start-up, before reserving its memory.
//
// In host code the array's name only stands in for the symbol; the device
// address comes from cudaGetSymbolAddress with the device current, and that
// address is what the kernels receive.  It is looked up on every call (a
// host-side table look-up once the module is loaded), so no address survives
// a device reset or outlives the context it belongs to.
#include <cuda_runtime.h>

#include "tp_internal.h"
#include "tpffn.h"

namespace {

__device__ __align__(256) unsigned char g_static_scratch[TPFFN_STATIC_SCRATCH_BYTES];

// Device address of g_static_scratch on the current device.  Returns nullptr
// (and clears the runtime's error state) when the look-up fails.
void* scratch_address() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return nullptr;
  }
  return p;
}

}  // namespace

extern "C" int tp_ffn_fwd_static_scratch(const tp_ffn_plan* plan, int64_t n_tokens, const void* x,
                                         const void* w13p, const void* w2p, const void* b1, const void* b2,
                                         void* y, tp_stream_t stream) {
  if (!plan || n_tokens < 0) return TP_ERR_INVALID;
  // The standalone shard-sum path: error word + h (no saved activations) +
  // fp32 partials must fit in the static array.
  const size_t need = tp_ffn_workspace_bytes(plan, n_tokens, TP_SUM_STANDALONE);
  if (n_tokens > 0 && (need == 0 || need > TPFFN_STATIC_SCRATCH_BYTES)) return TP_ERR_UNSUPPORTED;
  void* scratch = scratch_address();
  if (!scratch) return TP_ERR_CUDA;
  if (n_tokens == 0) return TP_OK;  // set-up only: the array is now resident on this device
  return tp_ffn_fwd(plan, n_tokens, x, w13p, w2p, b1, b2, y, nullptr, nullptr, scratch,
                    TPFFN_STATIC_SCRATCH_BYTES, TP_SUM_STANDALONE, stream);
}
