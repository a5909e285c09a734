// capi.cu -- the C ABI: argument checks, workspace carving, TMA descriptors
// and the launch sequence router -> gate/up -> down on the caller's stream.
//
// The three kernels of a layer are chained with programmatic dependent
// launch: each dependent kernel is scheduled while its predecessor drains and
// waits (griddepcontrol.wait) before reading the predecessor's results.
#include <atomic>
#include <cstring>
#include <mutex>

#include "internal.h"

using namespace moe;

namespace {

std::atomic<uint64_t> g_wait_ns{2000000000ull};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D map over the codes of a projection stack viewed as [n_exp*rows][cols/2]
// bytes; one box = box_rows rows x min(128, cols/2) bytes, swizzled.
bool encode_codes(CUtensorMap* m, const uint8_t* codes, int n_exp, int rows, int cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t rb = (cuuint64_t)cols / 2;
  const cuuint32_t inner = rb >= 128 ? 128 : 64;
  cuuint64_t dims[2] = {rb, (cuuint64_t)n_exp * rows};
  cuuint64_t strides[1] = {rb};
  cuuint32_t box[2] = {inner, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  inner == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_proj(const moe_nvfp4& p) {
  if (!p.codes || !p.scales || !p.tensor_scale) return MOE_ERR_INVALID_ARG;
  if (!aligned16(p.codes) || !aligned16(p.scales) || !aligned16(p.tensor_scale)) return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

moe_status check_layer(const moe_layer* L, int K) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (K < 1 || K > MOE_MAX_ROWS) return MOE_ERR_INVALID_ARG;
  const int H = L->hidden, E = L->n_experts, k = L->top_k, I = L->inter, Is = L->shared_inter;
  if (H <= 0 || E <= 0 || k <= 0 || I <= 0 || Is < 0) return MOE_ERR_INVALID_ARG;
  if (H % 256 != 0 || H > 2048) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!(I == 128 || I == 256 || I == 512)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!(Is == 0 || Is == I)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (k > 32 || k > E || E > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!L->router_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(L->router_w) || !aligned16(L->router_bias)) return MOE_ERR_MISALIGNED;
  moe_status s;
  if ((s = check_proj(L->gate)) != MOE_OK || (s = check_proj(L->up)) != MOE_OK || (s = check_proj(L->down)) != MOE_OK)
    return s;
  if (Is > 0) {
    if ((s = check_proj(L->sh_gate)) != MOE_OK || (s = check_proj(L->sh_up)) != MOE_OK ||
        (s = check_proj(L->sh_down)) != MOE_OK)
      return s;
  }
  return MOE_OK;
}

WsLayout layout_of(const moe_layer* L, int K) {
  return ws_layout(K, L->n_experts, L->top_k, L->hidden, L->inter);
}

RouterArgs router_args(const moe_layer* L, const uint16_t* x, int K, const WsPtrs& wp, int32_t* idx_out,
                       float* w_out, int32_t* group_out) {
  RouterArgs a;
  a.x = x;
  a.router_w = L->router_w;
  a.bias = L->router_bias;
  a.K = K;
  a.H = L->hidden;
  a.E = L->n_experts;
  a.k = L->top_k;
  a.G = group_cap(K, L->n_experts, L->top_k);
  a.has_shared = L->shared_inter > 0;
  a.n_tiles = L->hidden / kDNRows;
  a.ws = wp;
  a.idx_out = idx_out;
  a.w_out = w_out;
  a.group_out = group_out;
  return a;
}

}  // namespace

extern "C" {

size_t moe_group_ints(int K, int n_experts, int top_k) {
  if (K < 1 || n_experts < 1 || top_k < 1) return 0;
  const int G = group_cap(K, n_experts, top_k);
  return (size_t)(2 + 2 * G + K * top_k);
}

size_t moe_verify_layer_workspace_size(const moe_layer* layer, int K) {
  if (check_layer(layer, K) != MOE_OK) return 0;
  return layout_of(layer, K).total;
}

moe_status moe_router_topk(const moe_layer* layer, const uint16_t* x_norm, int K, int32_t* idx, float* w,
                           int32_t* group, void* ws, size_t ws_bytes, void* stream) {
  moe_status s = check_layer(layer, K);
  if (s != MOE_OK) return s;
  if (!x_norm || !idx || !w || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_norm) || !aligned16(ws)) return MOE_ERR_MISALIGNED;
  const WsLayout lay = layout_of(layer, K);
  if (ws_bytes < lay.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const WsPtrs wp = ws_ptrs(ws, lay);
  RouterArgs a = router_args(layer, x_norm, K, wp, idx, w, group);
  if (launch_router(a, static_cast<cudaStream_t>(stream), false) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

static moe_status run_layer(const moe_layer* layer, const uint16_t* x_norm, int K, const uint16_t* residual,
                            uint16_t* y, int32_t* idx_out, float* w_out, int32_t* group_out, void* ws,
                            size_t ws_bytes, void* stream, bool pdl, void* const* events) {
  moe_status s = check_layer(layer, K);
  if (s != MOE_OK) return s;
  if (!x_norm || !y || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_norm) || !aligned16(y) || !aligned16(ws) || !aligned16(residual)) return MOE_ERR_MISALIGNED;
  const WsLayout lay = layout_of(layer, K);
  if (ws_bytes < lay.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const WsPtrs wp = ws_ptrs(ws, lay);
  const int H = layer->hidden, E = layer->n_experts, I = layer->inter;
  const bool has_sh = layer->shared_inter > 0;

  CUtensorMap tg, tu, td, tsg, tsu, tsd;
  if (!encode_codes(&tg, layer->gate.codes, E, I, H, kGURows) ||
      !encode_codes(&tu, layer->up.codes, E, I, H, kGURows) ||
      !encode_codes(&td, layer->down.codes, E, H, I, kDNRows))
    return MOE_ERR_CUDA;
  if (has_sh) {
    if (!encode_codes(&tsg, layer->sh_gate.codes, 1, I, H, kGURows) ||
        !encode_codes(&tsu, layer->sh_up.codes, 1, I, H, kGURows) ||
        !encode_codes(&tsd, layer->sh_down.codes, 1, H, I, kDNRows))
      return MOE_ERR_CUDA;
  } else {
    tsg = tg;
    tsu = tu;
    tsd = td;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint64_t wait_ns = g_wait_ns.load();
  auto mark = [&](int i) {
    return !events || cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st) == cudaSuccess;
  };

  RouterArgs ra = router_args(layer, x_norm, K, wp, idx_out, w_out, group_out);
  if (!mark(0) || launch_router(ra, st, false) != cudaSuccess || !mark(1)) return MOE_ERR_CUDA;

  GateUpArgs ga;
  ga.x = x_norm;
  ga.K = K;
  ga.H = H;
  ga.I = I;
  ga.G = ra.G;
  ga.has_shared = has_sh;
  ga.gate = {layer->gate.scales, layer->gate.tensor_scale};
  ga.up = {layer->up.scales, layer->up.tensor_scale};
  ga.sh_gate = has_sh ? ProjPtrs{layer->sh_gate.scales, layer->sh_gate.tensor_scale} : ga.gate;
  ga.sh_up = has_sh ? ProjPtrs{layer->sh_up.scales, layer->sh_up.tensor_scale} : ga.up;
  ga.ws = wp;
  ga.wait_ns = wait_ns;
  if (launch_gateup(ga, tg, tu, tsg, tsu, st, pdl) != cudaSuccess || !mark(2)) return MOE_ERR_CUDA;

  DownArgs da;
  da.residual = residual;
  da.y = y;
  da.K = K;
  da.H = H;
  da.I = I;
  da.k = layer->top_k;
  da.G = ra.G;
  da.has_shared = has_sh;
  da.routed_scale = layer->routed_scale;
  da.down = {layer->down.scales, layer->down.tensor_scale};
  da.sh_down = has_sh ? ProjPtrs{layer->sh_down.scales, layer->sh_down.tensor_scale} : da.down;
  da.ws = wp;
  da.wait_ns = wait_ns;
  if (launch_down(da, td, tsd, st, pdl) != cudaSuccess || !mark(3)) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_verify_layer(const moe_layer* layer, const uint16_t* x_norm, int K, const uint16_t* residual,
                            uint16_t* y, int32_t* idx_out, float* w_out, int32_t* group_out, void* ws,
                            size_t ws_bytes, void* stream) {
  return run_layer(layer, x_norm, K, residual, y, idx_out, w_out, group_out, ws, ws_bytes, stream, true, nullptr);
}

moe_status moe_verify_layer_profiled(const moe_layer* layer, const uint16_t* x_norm, int K,
                                     const uint16_t* residual, uint16_t* y, void* ws, size_t ws_bytes,
                                     void* stream, void* const* events) {
  return run_layer(layer, x_norm, K, residual, y, nullptr, nullptr, nullptr, ws, ws_bytes, stream, false, events);
}

moe_status verify_accept_prefix(const int32_t* draft, const int32_t* target, int K, int32_t* n_accepted,
                                void* stream) {
  if (!n_accepted || K < 0 || K > 4096 || (K > 0 && (!draft || !target))) return MOE_ERR_INVALID_ARG;
  if (launch_accept(draft, target, K, n_accepted, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

size_t moe_verify_stack_workspace_size(const moe_layer* layers, int n_layers, int K) {
  if (!layers || n_layers < 1) return 0;
  size_t m = 0;
  for (int l = 0; l < n_layers; ++l) {
    if (check_layer(&layers[l], K) != MOE_OK || layers[l].hidden != layers[0].hidden) return 0;
    const size_t b = layout_of(&layers[l], K).total;
    m = b > m ? b : m;
  }
  return m + align256(sizeof(uint16_t) * K * layers[0].hidden);
}

moe_status moe_verify_stack(const moe_layer* layers, int n_layers, uint16_t* x, int K, float eps, void* ws,
                            size_t ws_bytes, void* stream) {
  if (!layers || n_layers < 1 || !x || !ws || !(eps >= 0.f)) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_verify_stack_workspace_size(layers, n_layers, K);
  if (need == 0) {
    for (int l = 0; l < n_layers; ++l) {
      moe_status s = check_layer(&layers[l], K);
      if (s != MOE_OK) return s;
    }
    return MOE_ERR_INVALID_ARG;
  }
  if (ws_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(x) || !aligned16(ws)) return MOE_ERR_MISALIGNED;
  const int H = layers[0].hidden;
  uint16_t* xn = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + need - align256(sizeof(uint16_t) * K * H));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int l = 0; l < n_layers; ++l) {
    if (launch_rmsnorm(x, K, H, eps, xn, st, l > 0) != cudaSuccess) return MOE_ERR_CUDA;
    moe_status s = run_layer(&layers[l], xn, K, x, x, nullptr, nullptr, nullptr, ws, ws_bytes, stream, true, nullptr);
    if (s != MOE_OK) return s;
  }
  return MOE_OK;
}

moe_status moe_rmsnorm(const uint16_t* x, int K, int H, float eps, uint16_t* out, void* stream) {
  if (!x || !out || K < 1 || K > MOE_MAX_ROWS || H < 256 || H % 256 != 0 || !(eps >= 0.f)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out)) return MOE_ERR_MISALIGNED;
  if (launch_rmsnorm(x, K, H, eps, out, static_cast<cudaStream_t>(stream), false) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

size_t moe_lm_head_workspace_size(int K) {
  if (K < 1 || K > MOE_MAX_ROWS) return 0;
  return lmhead_ws_bytes(K);
}

moe_status moe_lm_head_argmax(const uint16_t* x_norm, int K, int H, const uint16_t* W, int V, int32_t* tok,
                              float* best_logit, void* ws, size_t ws_bytes, void* stream) {
  if (!x_norm || !W || !tok || !ws || K < 1 || K > MOE_MAX_ROWS || V < 1) return MOE_ERR_INVALID_ARG;
  if (H < 256 || H % 256 != 0 || H > 2048) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x_norm) || !aligned16(W) || !aligned16(ws)) return MOE_ERR_MISALIGNED;
  if (ws_bytes < lmhead_ws_bytes(K)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  char* b = static_cast<char*>(ws);
  LmHeadArgs a;
  a.x = x_norm;
  a.W = W;
  a.K = K;
  a.H = H;
  a.V = V;
  a.tok = tok;
  a.best = best_logit;
  a.ticket = reinterpret_cast<unsigned*>(b);
  a.part_v = reinterpret_cast<float*>(b + 256);
  a.part_i = reinterpret_cast<int*>(b + 256 + align256(sizeof(float) * kLmMaxGrid * K));
  if (launch_lmhead(a, static_cast<cudaStream_t>(stream), false) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_workspace_error(void* ws, int* code, void* stream) {
  if (!ws || !code) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  *code = v;
  return MOE_OK;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

void moe_debug_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns); }

}  // extern "C"
