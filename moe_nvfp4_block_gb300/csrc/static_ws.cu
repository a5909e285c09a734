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

// 8 MiB.  Enough for K <= 16 at hidden 2048, 256 experts, top-8,
// intermediate 512 with a shared expert (about 6.8 MB at K = 16); larger
// layers (e.g. 1024 experts at top-32) are refused.
constexpr size_t kStaticWsBytes = size_t(8) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_static_ws on the current device, set up on first use:
// looked up, then zero-filled once on `stream` (the caller's stream, so the
// fill is ordered before the kernel that follows it on that stream, whatever
// kind of stream it is).  nullptr on failure.
void* static_ws_on_current_device(cudaStream_t stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return nullptr;
    if (cudaMemsetAsync(p, 0, kStaticWsBytes, stream) != cudaSuccess) return nullptr;
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
  void* ws = static_ws_on_current_device(static_cast<cudaStream_t>(stream));
  if (!ws) return MOE_ERR_CUDA;
  // (the kernel only ever sets the array's error word, with a compare-and-swap
  // from zero, and never reads it; nothing exposes it, so it is not reset)
  return run_layer(layer, x_norm, K, residual, y, idx_out, w_out, group_out, ws, kStaticWsBytes, stream, true,
                   nullptr);
}
