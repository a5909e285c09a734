// static_ws.cu -- moe_verify_layer for callers that cannot allocate device
// memory: the layer's scratch lives in a fixed array compiled into this
// library instead of a caller-provided workspace.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it until the process exits.  In host code its name is only a
// stand-in, not a device address; its address on the current device is
// looked up with cudaGetSymbolAddress once per device (the first call on that
// device, which must therefore not happen during a stream capture) and then
// passed to the kernels like any other workspace pointer.
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kStaticWsBytes = size_t(8) << 20;  // 8 MiB: enough for K <= 16 on the largest supported layer
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_static_ws on the current device (set up on first use:
// looked up and zero-filled once).  nullptr on failure.
void* static_ws_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return nullptr;
    if (cudaMemset(p, 0, kStaticWsBytes) != cudaSuccess) return nullptr;
    g_addr[dev] = p;
  }
  return g_addr[dev];
}

}  // namespace

extern "C" moe_status moe_verify_layer_static(const moe_layer* layer, const uint16_t* x_norm, int K,
                                              const uint16_t* residual, uint16_t* y, int32_t* idx_out,
                                              float* w_out, int32_t* group_out, void* stream) {
  const size_t need = moe_verify_layer_workspace_size(layer, K);
  if (need == 0)  // invalid layer or K: the shared checks give the precise status, nothing is enqueued
    return run_layer(layer, x_norm, K, residual, y, idx_out, w_out, group_out, nullptr, 0, stream, true, nullptr);
  if (need > kStaticWsBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  void* ws = static_ws_on_current_device();
  if (!ws) return MOE_ERR_CUDA;
  // the error word of the previous call starts again from zero (the rest of
  // the header, the count of earlier calls, must persist)
  if (cudaMemsetAsync(ws, 0, sizeof(int), static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  return run_layer(layer, x_norm, K, residual, y, idx_out, w_out, group_out, ws, kStaticWsBytes, stream, true,
                   nullptr);
}
