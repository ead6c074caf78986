// noalloc.cu -- an allocation-free variant of the layer forward.
//
// Some callers cannot hand this library a device workspace: plugin hosts whose operator
// interface passes only an op's input and output tensors (no scratch allocator), serving
// loops whose device-memory budget is fixed at start-up and that forbid any allocation on
// the request path, and code that must not call cudaMalloc because it can synchronise the
// device (for example while another stream is being captured in global capture mode).
// For them, moe_layer_forward_static runs the same kernels as moe_layer_forward, with the
// scratch in a file-scope device array instead of a caller buffer.
//
// The array (kStaticScratchBytes, 32 MiB) is part of the library image: every GPU that
// loads the library holds it until the process exits.  In host code `g_scratch` names a
// host-side stand-in, not a device address, so the device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, on the first call
// made on that device.
#include <mutex>

#include "moe_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = (size_t)32 << 20;

__device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

std::mutex g_mu;
void *g_addr[64];
bool g_ready[64];

int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ready[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    g_addr[dev] = p;
    g_ready[dev] = true;
  }
  *out = g_addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" int moe_layer_forward_static(const moe_layer_config *cfg, const void *packed,
                                        const void *x, moe_dtype dtype, int T, float *out,
                                        int32_t *ids, float *w, int32_t *status, void *stream) {
  int r = moe_check_config(cfg);
  if (r) return r;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  size_t need = moe_workspace_bytes(cfg, T);
  if (need == 0) return MOE_ERR_UNSUPPORTED;
  if (need > kStaticScratchBytes) return MOE_ERR_WORKSPACE;  // T too large for the array
  void *ws = nullptr;
  if ((r = scratch_address(&ws))) return r;
  // the forward clears the status word at its start; everything else it reads from the
  // scratch it has written earlier in the same call
  r = moe_layer_forward(cfg, packed, x, dtype, T, out, ids, w, ws, kStaticScratchBytes, stream);
  if (r) return r;
  if (status && cudaMemcpyAsync(status, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                                (cudaStream_t)stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
