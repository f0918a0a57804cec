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
// The array is static device memory of the library's module: every GPU that
// loads the library holds TPFFN_STATIC_SCRATCH_BYTES until the process exits.
// In host code its name only stands in for the symbol; the device address is
// obtained with cudaGetSymbolAddress once per device (with that device
// current) and cached, and that address is what the kernels receive.
#include <cuda_runtime.h>

#include <mutex>

#include "tp_internal.h"
#include "tpffn.h"

namespace {

__device__ __align__(256) unsigned char g_static_scratch[TPFFN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (set-up on the
// first call per device).  Returns nullptr and sets *rc on failure.
void* scratch_address(int* rc) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *rc = TP_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
      *rc = TP_ERR_CUDA;
      return nullptr;
    }
    g_addr[dev] = p;
  }
  return g_addr[dev];
}

}  // namespace

extern "C" int tp_ffn_fwd_static_scratch(const tp_ffn_plan* plan, int64_t n_tokens, const void* x,
                                         const void* w13p, const void* w2p, const void* b1, const void* b2,
                                         void* y, tp_stream_t stream) {
  if (!plan || n_tokens < 0) return TP_ERR_INVALID;
  if (n_tokens == 0) return TP_OK;
  // The standalone shard-sum path: error word + h (no saved activations) +
  // fp32 partials must fit in the static array.
  const size_t need = tp_ffn_workspace_bytes(plan, n_tokens, TP_SUM_STANDALONE);
  if (need == 0 || need > TPFFN_STATIC_SCRATCH_BYTES) return TP_ERR_UNSUPPORTED;
  int rc = TP_OK;
  void* scratch = scratch_address(&rc);
  if (!scratch) return rc;
  return tp_ffn_fwd(plan, n_tokens, x, w13p, w2p, b1, b2, y, nullptr, nullptr, scratch,
                    TPFFN_STATIC_SCRATCH_BYTES, TP_SUM_STANDALONE, stream);
}
