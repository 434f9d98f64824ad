// ds_layer_forward_noalloc: the layer forward for callers that cannot allocate
// device memory.
//
// Some callers of this library cannot call cudaMalloc (or any allocator):
// plugins inside serving frameworks that own and pre-reserve all device
// memory, code that must not trigger the device-wide synchronisation an
// allocation can cause in the middle of a latency-critical loop, and
// real-time or embedded hosts that forbid allocation after start-up.  They
// cannot provide the workspace ds_layer_forward needs, so this entry point
// runs the same region kernels on a workspace that is a file-scope
// __device__ array of this library (kStaticWorkspaceBytes = 16 MiB, held on
// every GPU that loads the library until the process exits).
//
// Host code cannot use the array's name as a device address: its address is
// looked up with cudaGetSymbolAddress once per device, with that device
// current, on the first call made on it (so make the first call before any
// stream capture; the cached address is not valid across cudaDeviceReset).
// Every call shares the array, so calls that overlap on the GPU (other
// streams, other threads) race; each call, once its arguments are accepted,
// clears the status word and counters at the start of the array that must
// start at zero.  ds_noalloc_status reads the status word left by the last
// call on the current device.
#include <mutex>

#include "ds_layer.h"
#include "internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = (size_t)16 << 20;
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_static_mu;
void* g_static_addr[64] = {};

// Device address of the static workspace on the current device (looked up on
// the first use per device); nullptr on failure, with the error recorded.
void* static_workspace(ds_status* s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    ds::set_last_error("cudaGetDevice failed");
    *s = DS_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (g_static_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) {
      ds::set_last_error("cudaGetSymbolAddress of the static workspace failed");
      *s = DS_ERR_CUDA;
      return nullptr;
    }
    g_static_addr[dev] = p;
  }
  *s = DS_OK;
  return g_static_addr[dev];
}

}  // namespace

extern "C" ds_status ds_layer_forward_noalloc(ds_layer* layer, const void* x_in, void* x_out, int batch,
                                              int new_tokens, void* k_cache, void* v_cache, int max_len,
                                              const int32_t* past_len, void* stream) {
  if (layer == nullptr) {
    ds::set_last_error("layer is null");
    return DS_ERR_INVALID_ARG;
  }
  const size_t need = ds_layer_workspace_bytes(layer, batch, new_tokens);
  if (need > kStaticWorkspaceBytes) {
    ds::set_last_error("workspace for this batch shape exceeds the 16 MiB static workspace");
    return DS_ERR_UNSUPPORTED;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != ds::layer_device(layer)) {
    ds::set_last_error("the current device is not the device the layer was created on");
    return DS_ERR_INVALID_ARG;
  }
  ds_status s = DS_OK;
  void* ws = static_workspace(&s);
  if (ws == nullptr) return s;
  size_t zero = 0;
  s = ds::layer_forward_check(layer, x_in, x_out, batch, new_tokens, k_cache, v_cache, max_len, past_len, ws,
                              kStaticWorkspaceBytes, &zero);
  if (s != DS_OK) return s;  // rejected: nothing enqueued, the shared array untouched
  if (cudaMemsetAsync(ws, 0, zero, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    ds::set_last_error("cudaMemsetAsync of the static workspace counters failed");
    return DS_ERR_CUDA;
  }
  return ds::layer_forward_enqueue(layer, x_in, x_out, batch, new_tokens, k_cache, v_cache, max_len, past_len, ws,
                                   stream);
}

extern "C" ds_status ds_noalloc_status(uint32_t* flags_out, void* stream) {
  if (flags_out == nullptr) {
    ds::set_last_error("flags_out is null");
    return DS_ERR_INVALID_ARG;
  }
  ds_status s = DS_OK;
  void* ws = static_workspace(&s);
  if (ws == nullptr) return s;
  return ds_workspace_status(ws, flags_out, stream);
}
