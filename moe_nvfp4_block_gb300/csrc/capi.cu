// capi.cu -- the C ABI: argument checks, workspace carving, TMA descriptors
// and the launch sequences on the caller's stream.
//
// A layer call is one launch of the persistent experts kernel (router,
// routing, experts and combine in one grid).  Consecutive kernels of a stack
// or a verify step are chained with programmatic dependent launch: each
// dependent kernel is scheduled while its predecessor drains and waits
// (griddepcontrol.wait) before reading the predecessor's results.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"

using namespace moe;

namespace moe {
unsigned long long* g_trace = nullptr;
}

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

// Map over the codes of a projection stack viewed as rows of cols/2 bytes,
// read as box_rows x (cols/2) tiles laid out in shared memory as
// [line chunk][row][min(128, cols/2) bytes] with the matching swizzle.
// Preferred: one 3-D box per tile (dims: line bytes, rows, line chunks --
// one large request); if the driver refuses that stride order, a 2-D map
// whose box is one line chunk (the kernel then issues one request per chunk).
bool encode_codes(CUtensorMap* m, const uint8_t* codes, int n_exp, int rows, int cols, int box_rows, bool* is3d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t rb = (cuuint64_t)cols / 2;
  const cuuint32_t inner = rb >= 128 ? 128 : 64;
  const CUtensorMapSwizzle sw = inner == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  {
    cuuint64_t dims[3] = {inner, (cuuint64_t)n_exp * rows, rb / inner};
    cuuint64_t strides[2] = {rb, inner};
    cuuint32_t box[3] = {inner, (cuuint32_t)box_rows, (cuuint32_t)(rb / inner)};
    cuuint32_t estr[3] = {1, 1, 1};
    if (fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(codes), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
      *is3d = true;
      return true;
    }
  }
  cuuint64_t dims[2] = {rb, (cuuint64_t)n_exp * rows};
  cuuint64_t strides[1] = {rb};
  cuuint32_t box[2] = {inner, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  *is3d = false;
  return r == CUDA_SUCCESS;
}

// 2-D map over the E4M3 scales of a projection stack viewed as
// [n_exp*rows][cols/16] bytes; one box = box_rows full rows, swizzled by the
// row length (128, 64, 32 bytes) or unswizzled (16 bytes).
bool encode_scales(CUtensorMap* m, const uint8_t* scales, int n_exp, int rows, int cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t rb = (cuuint64_t)cols / 16;
  if (rb < 16 || rb > 128) return false;
  cuuint64_t dims[2] = {rb, (cuuint64_t)n_exp * rows};
  cuuint64_t strides[1] = {rb};
  cuuint32_t box[2] = {(cuuint32_t)rb, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = rb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : rb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                : rb == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                           : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(scales), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

// Map over a KV cache [nkv][C][128] bf16 seen as nkv * C rows of 128 dims,
// 128-byte swizzle, zero fill past the end.  Preferred: 3-D (64 dims, rows,
// 2 dim halves), one 32 KB box = 128 rows x both halves laid out as
// [half][row][64 dims]; else 2-D with a box of one half (64 dims x 128 rows).
bool moe::encode_kv_map(CUtensorMap* m, const uint16_t* cache, int nkv, int C, bool* is3d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  {
    cuuint64_t dims[3] = {64, (cuuint64_t)nkv * (cuuint64_t)C, 2};
    cuuint64_t strides[2] = {256, 128};
    cuuint32_t box[3] = {64, 128, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    if (fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(cache), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
      *is3d = true;
      return true;
    }
  }
  cuuint64_t dims[2] = {128, (cuuint64_t)nkv * (cuuint64_t)C};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  *is3d = false;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(cache), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

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
  if (L->scoring != MOE_SCORE_SOFTMAX && L->scoring != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
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
  a.scoring = L->scoring;
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

// The ten tensor maps of a layer (codes: gate, up, down, shared gate, shared
// up, shared down; scales: gate, up, shared gate, shared up) and whether the
// code maps are 3-D.  False if the driver refuses one.
static bool encode_layer_maps(const moe_layer* layer, CUtensorMap* maps, bool* code3d) {
  const int H = layer->hidden, E = layer->n_experts, I = layer->inter;
  bool d3[6] = {false, false, false, false, false, false};
  if (!encode_codes(&maps[0], layer->gate.codes, E, I, H, kGURows, &d3[0]) ||
      !encode_codes(&maps[1], layer->up.codes, E, I, H, kGURows, &d3[1]) ||
      !encode_codes(&maps[2], layer->down.codes, E, H, I, kDNRows, &d3[2]) ||
      !encode_scales(&maps[6], layer->gate.scales, E, I, H, kGURows) ||
      !encode_scales(&maps[7], layer->up.scales, E, I, H, kGURows))
    return false;
  if (layer->shared_inter > 0) {
    if (!encode_codes(&maps[3], layer->sh_gate.codes, 1, I, H, kGURows, &d3[3]) ||
        !encode_codes(&maps[4], layer->sh_up.codes, 1, I, H, kGURows, &d3[4]) ||
        !encode_codes(&maps[5], layer->sh_down.codes, 1, H, I, kDNRows, &d3[5]) ||
        !encode_scales(&maps[8], layer->sh_gate.scales, 1, I, H, kGURows) ||
        !encode_scales(&maps[9], layer->sh_up.scales, 1, I, H, kGURows))
      return false;
  } else {
    maps[3] = maps[0];
    maps[4] = maps[1];
    maps[5] = maps[2];
    maps[8] = maps[6];
    maps[9] = maps[7];
    d3[3] = d3[0];
    d3[4] = d3[1];
    d3[5] = d3[2];
  }
  *code3d = d3[0] && d3[1] && d3[2] && d3[3] && d3[4] && d3[5];
  return *code3d || !(d3[0] || d3[1] || d3[2] || d3[3] || d3[4] || d3[5]);  // no mixed forms
}

static LayerDesc layer_desc(const moe_layer* layer) {
  LayerDesc d;
  const bool has_sh = layer->shared_inter > 0;
  d.router_w = layer->router_w;
  d.router_bias = layer->router_bias;
  d.gate = {layer->gate.scales, layer->gate.tensor_scale};
  d.up = {layer->up.scales, layer->up.tensor_scale};
  d.down = {layer->down.scales, layer->down.tensor_scale};
  d.sh_gate = has_sh ? ProjPtrs{layer->sh_gate.scales, layer->sh_gate.tensor_scale} : d.gate;
  d.sh_up = has_sh ? ProjPtrs{layer->sh_up.scales, layer->sh_up.tensor_scale} : d.up;
  d.sh_down = has_sh ? ProjPtrs{layer->sh_down.scales, layer->sh_down.tensor_scale} : d.down;
  d.routed_scale = layer->routed_scale;
  d.has_shared = has_sh ? 1 : 0;
  d.scoring = layer->scoring;
  return d;
}

// One launch of the experts kernel for one layer call.
static moe_status launch_layer(const moe_layer* layer, const uint16_t* x, int K, const uint16_t* residual,
                               uint16_t* y, int32_t* idx_out, float* w_out, int32_t* group_out, const WsPtrs& wp,
                               cudaStream_t st, bool pdl, float norm_eps, const L2Prefetch* pf) {
  CUtensorMap maps[kMapsPerLayer];
  bool d3 = false;
  if (!encode_layer_maps(layer, maps, &d3)) return MOE_ERR_CUDA;
  ExpertsCommon c{};
  c.x = x;
  c.residual = residual;
  c.y = y;
  c.K = K;
  c.H = layer->hidden;
  c.I = layer->inter;
  c.E = layer->n_experts;
  c.k = layer->top_k;
  c.G = group_cap(K, layer->n_experts, layer->top_k);
  c.ws = wp;
  c.idx_out = idx_out;
  c.w_out = w_out;
  c.group_out = group_out;
  c.wait_ns = g_wait_ns.load();
  c.trace = g_trace;
  c.code3d = d3 ? 1 : 0;
  c.norm = norm_eps >= 0.f ? 1 : 0;
  c.norm_eps = norm_eps >= 0.f ? norm_eps : 0.f;
  if (pf) c.pf = *pf;
  return launch_experts(c, maps, layer_desc(layer), st, pdl) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

__attribute__((visibility("hidden"))) moe_status run_layer(const moe_layer* layer, const uint16_t* x_norm, int K, const uint16_t* residual,
                            uint16_t* y, int32_t* idx_out, float* w_out, int32_t* group_out, void* ws,
                            size_t ws_bytes, void* stream, bool pdl, void* const* events, float norm_eps,
                            const L2Prefetch* pf) {
  moe_status s = check_layer(layer, K);
  if (s != MOE_OK) return s;
  if (!x_norm || !y || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_norm) || !aligned16(y) || !aligned16(ws) || !aligned16(residual)) return MOE_ERR_MISALIGNED;
  const WsLayout lay = layout_of(layer, K);
  if (ws_bytes < lay.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const WsPtrs wp = ws_ptrs(ws, lay);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (events && cudaStreamIsCapturing(st, &cap) != cudaSuccess) return MOE_ERR_CUDA;
  // inside a graph capture the events become external record nodes, so that
  // their times can be read after a replay
  const unsigned ev_flags = cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
  auto mark = [&](int i) {
    return !events || cudaEventRecordWithFlags(static_cast<cudaEvent_t>(events[i]), st, ev_flags) == cudaSuccess;
  };
  // one launch: the experts kernel computes the router logits itself
  // (events 0 and 1 bracket no work)
  if (!mark(0) || !mark(1)) return MOE_ERR_CUDA;
  // activations in pageable host memory are refused (the device cannot reach
  // it everywhere); rows in page-locked host memory are staged into the
  // workspace by one CTA (every CTA of the layer kernel reads all of them)
  const void* acts[3] = {x_norm, residual, y};
  cudaPointerAttributes pa{};
  for (const void* p : acts) {
    if (!p) continue;
    if (cudaPointerGetAttributes(&pa, p) != cudaSuccess) {
      cudaGetLastError();  // an unknown pointer: not an error of the caller's stream
      continue;
    }
    if (pa.type == cudaMemoryTypeUnregistered) return MOE_ERR_INVALID_ARG;
  }
  if (cudaPointerGetAttributes(&pa, x_norm) != cudaSuccess) {
    cudaGetLastError();
  } else if (pa.type == cudaMemoryTypeHost) {
    uint16_t* xs = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + lay.xs);
    if (launch_stage_rows(x_norm, xs, sizeof(uint16_t) * (size_t)K * layer->hidden, st) != cudaSuccess)
      return MOE_ERR_CUDA;
    x_norm = xs;
  }
  s = launch_layer(layer, x_norm, K, residual, y, idx_out, w_out, group_out, wp, st, pdl, norm_eps, pf);
  if (s != MOE_OK) return s;
  if (!mark(2) || !mark(3)) return MOE_ERR_CUDA;
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
  return m;
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
  // one launch per layer, chained by programmatic dependent launch; each
  // layer kernel applies its RMSNorm to the residual stream x itself
  for (int l = 0; l < n_layers; ++l) {
    moe_status s = run_layer(&layers[l], x, K, x, x, nullptr, nullptr, nullptr, ws, ws_bytes, stream, true, nullptr, eps);
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

// lm_head argmax of x (normalised first, in the kernel, when norm_eps > 0).
static moe_status lm_head_impl(const uint16_t* x_norm, int K, int H, const uint16_t* W, int V, int32_t* tok,
                               float* best_logit, void* ws, size_t ws_bytes, float norm_eps, bool pdl,
                               int* err, void* stream) {
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
  a.err = err ? err : reinterpret_cast<int*>(b);
  a.ticket = reinterpret_cast<unsigned*>(b + 4);
  a.part_v = reinterpret_cast<float*>(b + 256);
  a.part_i = reinterpret_cast<int*>(b + 256 + align256(sizeof(float) * kLmMaxGrid * K));
  a.norm_eps = norm_eps;
  a.wait_ns = g_wait_ns.load();
  cudaError_t e;
  if (lmhead_stream_fits(K, H)) {
    e = launch_lmhead_stream(a, static_cast<cudaStream_t>(stream), pdl);
  } else {
    if (norm_eps > 0.f) return MOE_ERR_UNSUPPORTED_SHAPE;  // the row kernel takes normalised rows
    e = launch_lmhead(a, static_cast<cudaStream_t>(stream), pdl);
  }
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_lm_head_argmax(const uint16_t* x_norm, int K, int H, const uint16_t* W, int V, int32_t* tok,
                              float* best_logit, void* ws, size_t ws_bytes, void* stream) {
  return lm_head_impl(x_norm, K, H, W, V, tok, best_logit, ws, ws_bytes, 0.f, false, nullptr, stream);
}

struct AttnLayout {
  size_t hdr, xn, q, kn, vn, o, part_o, part_ml, total;
};

static AttnLayout attn_layout(int K, int H, int nq, int nkv) {
  AttnLayout L{};
  size_t off = 0;
  auto take = [&](size_t b) {
    size_t r = off;
    off = align256(off + b);
    return r;
  };
  L.hdr = take(256);  // int32 error word first, as in every workspace
  L.xn = take(sizeof(uint16_t) * K * H);
  L.q = take(sizeof(uint16_t) * K * nq * 128);
  L.kn = take(sizeof(uint16_t) * K * nkv * 128);
  L.vn = take(sizeof(uint16_t) * K * nkv * 128);
  L.o = take(sizeof(uint16_t) * K * nq * 128);
  const int tiles = (K * (nq / nkv) + 15) / 16;
  L.part_o = take(sizeof(float) * (size_t)nkv * kAttnMaxSplits * tiles * 16 * 128);
  L.part_ml = take(sizeof(float) * (size_t)nkv * kAttnMaxSplits * tiles * 32);
  L.total = off;
  return L;
}

static moe_status check_attn(int K, int H, int nq, int nkv, int hd, int C) {
  if (K < 1 || K > MOE_MAX_ROWS || nq < 1 || nkv < 1 || C < 0) return MOE_ERR_INVALID_ARG;
  if (hd != 128 || nq % nkv != 0 || K * (nq / nkv) > 16 * kAttnMaxTiles) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (H % 256 != 0 || H > 4096 || nq % 2 != 0 || nq * 128 > 8192 || K * nq > 768 || C % 16 != 0)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

static moe_status check_pos(const moe_attn_pos* p) {
  if (!p) return MOE_OK;
  if (p->window < 0 || (p->window > 0 && p->window < 16)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (p->rotary_dim < 0 || p->rotary_dim > 128 || p->rotary_dim % 2 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (p->rotary_dim > 0 && !(p->rope_theta > 1.f)) return MOE_ERR_INVALID_ARG;
  if (p->rotary_dim > 0 && p->yarn_factor > 1.f && p->yarn_orig_ctx < 1) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// Angle per position of each rotary pair (YaRN-scaled when asked) and the
// logit temperature.
static void rope_freqs(const moe_attn_pos& p, double* f, double* temp) {
  const double two_pi = 6.283185307179586476925286766559;
  const int rd = p.rotary_dim;
  const bool yarn = p.yarn_factor > 1.f;
  for (int i = 0; i < rd / 2; ++i) {
    double fi = std::pow((double)p.rope_theta, -2.0 * i / rd);
    if (yarn) {
      const double r = (double)p.yarn_orig_ctx * fi / two_pi;
      double g = (r - 1.0) / (32.0 - 1.0);
      g = g < 0.0 ? 0.0 : (g > 1.0 ? 1.0 : g);
      fi = (1.0 - g) * fi / (double)p.yarn_factor + g * fi;
    }
    f[i] = fi;
  }
  const double m = yarn ? 0.1 * std::log((double)p.yarn_factor) + 1.0 : 1.0;
  *temp = m * m;
}

size_t moe_attention_workspace_size(int K, int H, int nq, int nkv, int head_dim) {
  if (check_attn(K, H, nq, nkv, head_dim, 0) != MOE_OK) return 0;
  return attn_layout(K, H, nq, nkv).total;
}

// The attention block's launches; `err` receives a failed in-place append
// (the caller's workspace error word).
static moe_status attention_impl(const uint16_t* x, int K, int H, int nq, int nkv, int C, const uint16_t* Wq,
                                 const uint16_t* Wk, const uint16_t* Wv, const uint16_t* Wo, uint16_t* kcache,
                                 uint16_t* vcache, const int32_t* kv_len, const moe_attn_pos* pos, float eps,
                                 uint16_t* x_out,
                                 uint16_t* k_new_out, uint16_t* v_new_out, uint16_t* o_out, char* b,
                                 const AttnLayout& L, int* err, cudaStream_t s) {
  uint16_t* xn = reinterpret_cast<uint16_t*>(b + L.xn);
  uint16_t* q = reinterpret_cast<uint16_t*>(b + L.q);
  uint16_t* kn = k_new_out ? k_new_out : reinterpret_cast<uint16_t*>(b + L.kn);
  uint16_t* vn = v_new_out ? v_new_out : reinterpret_cast<uint16_t*>(b + L.vn);
  uint16_t* o = o_out ? o_out : reinterpret_cast<uint16_t*>(b + L.o);
  GemvArgs g{};
  g.x = x;
  g.K = K;
  g.D = H;
  g.norm_eps = eps;  // the streamed GEMV normalises the rows itself
  g.wait_ns = g_wait_ns.load();
  const bool rope = pos && pos->rotary_dim > 0;
  g.seg[0] = {Wq, q, nullptr, nq * 128, nullptr, nullptr, 0};
  g.seg[1] = {Wk, kn, nullptr, nkv * 128, nullptr, kv_len, C};
  g.seg[2] = {Wv, vn, nullptr, nkv * 128, nullptr, kv_len, C};
  g.nseg = 3;
  g.n_total = (nq + 2 * nkv) * 128;
  g.err = err;
  // the rotary embedding in the streamed projection's epilogue where it
  // takes the shape, else in a kernel of its own after the projection
  double temp = 1.0;
  bool rope_in_gemv = false;
  if (rope) {
    rope_freqs(*pos, g.rope_freq, &temp);
    g.rope_rd = pos->rotary_dim;
    g.rope_len = kv_len;
    g.rope_C = C;
    g.seg[0].rope = g.seg[1].rope = 1;
    rope_in_gemv = gemv_stream_rope_fits(g, num_sms());
    if (!rope_in_gemv) {
      g.rope_rd = 0;
      g.seg[0].rope = g.seg[1].rope = 0;
    }
  }
  // with a device length, the new keys and values also go into the caches
  // in place, at positions *kv_len .. *kv_len + K - 1 (a rotation kernel of
  // its own appends the rotated keys instead)
  if (kv_len && (!rope || rope_in_gemv)) {
    g.seg[1].cache = kcache;
    g.seg[2].cache = vcache;
  }
  if (!gemv_stream_fits(g, num_sms())) {  // the row kernel takes normalised rows
    if (launch_rmsnorm(x, K, H, eps, xn, s, false) != cudaSuccess) return MOE_ERR_CUDA;
    g.x = xn;
    g.norm_eps = 0.f;
  }
  if (launch_gemv(g, s, true) != cudaSuccess) return MOE_ERR_CUDA;
  if (rope && !rope_in_gemv) {
    RopeArgs ra{};
    ra.q = q;
    ra.k = kn;
    ra.v = vn;
    ra.K = K;
    ra.nq = nq;
    ra.nkv = nkv;
    ra.rd = pos->rotary_dim;
    for (int i = 0; i < 64; ++i) ra.freq[i] = g.rope_freq[i];
    ra.len = kv_len;
    ra.C = C;
    ra.kc = kv_len ? kcache : nullptr;
    ra.vc = kv_len ? vcache : nullptr;
    ra.err = err;
    if (launch_rope(ra, s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  AttnArgs a{};
  a.q = q;
  a.kc = kcache;
  a.vc = vcache;
  a.len = kv_len;
  a.k_new = kn;
  a.v_new = vn;
  a.o = o;
  a.K = K;
  a.nq = nq;
  a.nkv = nkv;
  a.C = C;
  a.group = nq / nkv;
  a.tiles = (K * a.group + 15) / 16;
  a.window = pos ? pos->window : 0;
  a.scale_log2 = (float)(1.4426950408889634 * temp / std::sqrt(128.0));
  a.part_o = reinterpret_cast<float*>(b + L.part_o);
  a.part_ml = reinterpret_cast<float*>(b + L.part_ml);
  a.err = err;
  a.wait_ns = g_wait_ns.load();
  AttnStreamArgs sa;
  sa.a = a;
  bool k3 = false, v3 = false;
  if (encode_kv_map(&sa.km, kcache, nkv, C, &k3) && encode_kv_map(&sa.vm, vcache, nkv, C, &v3) && k3 == v3) {
    sa.kv3d = k3 ? 1 : 0;
    if (launch_attention_stream(sa, s, true) != cudaSuccess) return MOE_ERR_CUDA;
  } else if (launch_attention(a, s, true) != cudaSuccess) {
    return MOE_ERR_CUDA;
  }
  GemvArgs go{};
  go.x = o;
  go.K = K;
  go.D = nq * 128;
  go.seg[0] = {Wo, x_out, x, H, nullptr, nullptr, 0};
  go.nseg = 1;
  go.n_total = H;
  go.err = err;
  go.wait_ns = g_wait_ns.load();
  if (launch_gemv(go, s, true) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_attention_block(const uint16_t* x, int K, int H, int nq, int nkv, int head_dim, int C,
                               const uint16_t* Wq, const uint16_t* Wk, const uint16_t* Wv, const uint16_t* Wo,
                               uint16_t* kcache, uint16_t* vcache, const int32_t* kv_len, const moe_attn_pos* pos,
                               float eps, uint16_t* x_out, uint16_t* k_new_out, uint16_t* v_new_out,
                               uint16_t* o_out, void* ws, size_t ws_bytes, void* stream) {
  moe_status st = check_attn(K, H, nq, nkv, head_dim, C);
  if (st != MOE_OK) return st;
  if ((st = check_pos(pos)) != MOE_OK) return st;
  if (!x || !Wq || !Wk || !Wv || !Wo || !x_out || !ws || (C > 0 && (!kcache || !vcache)) || !(eps >= 0.f) ||
      (kv_len && C == 0))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, Wq, Wk, Wv, Wo, kcache, vcache, x_out, k_new_out, v_new_out, o_out, ws};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_MISALIGNED;
  const AttnLayout L = attn_layout(K, H, nq, nkv);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  char* b = static_cast<char*>(ws);
  return attention_impl(x, K, H, nq, nkv, C, Wq, Wk, Wv, Wo, kcache, vcache, kv_len, pos, eps, x_out, k_new_out,
                        v_new_out, o_out, b, L, reinterpret_cast<int*>(b + L.hdr), static_cast<cudaStream_t>(stream));
}

struct MlpLayout {
  size_t hdr, xn, h, total;
};

static MlpLayout mlp_layout(int K, int H, int I) {
  MlpLayout L{};
  size_t off = 0;
  auto take = [&](size_t b) {
    size_t r = off;
    off = align256(off + b);
    return r;
  };
  L.hdr = take(256);
  L.xn = take(sizeof(uint16_t) * K * H);
  L.h = take(sizeof(uint16_t) * K * I);
  L.total = off;
  return L;
}

static moe_status check_mlp(int K, int H, int I) {
  if (K < 1 || K > MOE_MAX_ROWS || I < 1) return MOE_ERR_INVALID_ARG;
  if (H % 256 != 0 || H > 4096 || I % 256 != 0 || K * I > 98304) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

size_t moe_dense_mlp_workspace_size(int K, int H, int I) {
  if (check_mlp(K, H, I) != MOE_OK) return 0;
  return mlp_layout(K, H, I).total;
}

static moe_status dense_mlp_impl(const uint16_t* x, int K, int H, int I, const uint16_t* Wg, const uint16_t* Wu,
                                 const uint16_t* Wd, float eps, uint16_t* x_out, char* b, const MlpLayout& L,
                                 int* err, cudaStream_t s) {
  uint16_t* xn = reinterpret_cast<uint16_t*>(b + L.xn);
  uint16_t* h = reinterpret_cast<uint16_t*>(b + L.h);
  // gate and up in the streamed projection (RMSNorm folded in, SwiGLU in its
  // epilogue) where it takes the shape, else the row kernel on normalised rows
  GemvArgs gu{};
  gu.x = x;
  gu.K = K;
  gu.D = H;
  gu.norm_eps = eps;
  gu.seg[0] = {Wg, h, nullptr, I, nullptr, nullptr, 0};
  gu.seg[1] = {Wu, h, nullptr, I, nullptr, nullptr, 0};
  gu.nseg = 2;
  gu.n_total = 2 * I;
  gu.glu = 1;
  gu.err = err;
  gu.wait_ns = g_wait_ns.load();
  if (gemv_stream_fits(gu, num_sms())) {
    if (launch_gemv_stream(gu, s, true) != cudaSuccess) return MOE_ERR_CUDA;
  } else {
    if (launch_rmsnorm(x, K, H, eps, xn, s, false) != cudaSuccess) return MOE_ERR_CUDA;
    SwigluArgs sa{xn, Wg, Wu, h, K, H, I};
    if (launch_swiglu(sa, s, true) != cudaSuccess) return MOE_ERR_CUDA;
  }
  GemvArgs gd{};
  gd.x = h;
  gd.K = K;
  gd.D = I;
  gd.seg[0] = {Wd, x_out, x, H, nullptr, nullptr, 0};
  gd.nseg = 1;
  gd.n_total = H;
  gd.err = err;
  gd.wait_ns = g_wait_ns.load();
  if (launch_gemv(gd, s, true) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_dense_mlp_block(const uint16_t* x, int K, int H, int I, const uint16_t* Wg, const uint16_t* Wu,
                               const uint16_t* Wd, float eps, uint16_t* x_out, void* ws, size_t ws_bytes,
                               void* stream) {
  moe_status st = check_mlp(K, H, I);
  if (st != MOE_OK) return st;
  if (!x || !Wg || !Wu || !Wd || !x_out || !ws || !(eps >= 0.f)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, Wg, Wu, Wd, x_out, ws};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_MISALIGNED;
  const MlpLayout L = mlp_layout(K, H, I);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return dense_mlp_impl(x, K, H, I, Wg, Wu, Wd, eps, x_out, static_cast<char*>(ws), L,
                        reinterpret_cast<int*>(static_cast<char*>(ws) + L.hdr), static_cast<cudaStream_t>(stream));
}

static int layer_nq(const moe_verify_model* m, const moe_decoder_layer& d) {
  return d.n_q_heads > 0 ? d.n_q_heads : m->n_q_heads;
}

static moe_status check_model(const moe_verify_model* m, int K) {
  if (!m || !m->layers || !m->lm_head || m->n_layers < 1 || m->vocab < 1 || !(m->eps >= 0.f))
    return MOE_ERR_INVALID_ARG;
  moe_status s;
  if (m->hidden > 2048) return MOE_ERR_UNSUPPORTED_SHAPE;  // lm_head and MoE envelope
  if (m->kv_len && m->ctx == 0) return MOE_ERR_INVALID_ARG;
  for (int l = 0; l < m->n_layers; ++l) {
    const moe_decoder_layer& d = m->layers[l];
    if ((s = check_attn(K, m->hidden, layer_nq(m, d), m->n_kv_heads, m->head_dim, m->ctx)) != MOE_OK) return s;
    if ((s = check_pos(&d.pos)) != MOE_OK) return s;
    if (!d.Wq || !d.Wk || !d.Wv || !d.Wo || (m->ctx > 0 && (!d.kcache || !d.vcache))) return MOE_ERR_INVALID_ARG;
    if (d.mlp_gate) {
      if (!d.mlp_up || !d.mlp_down) return MOE_ERR_INVALID_ARG;
      if ((s = check_mlp(K, m->hidden, d.mlp_inter)) != MOE_OK) return s;
    } else {
      if ((s = check_layer(&d.moe, K)) != MOE_OK) return s;
      if (d.moe.hidden != m->hidden) return MOE_ERR_INVALID_ARG;
    }
  }
  return MOE_OK;
}

struct StepLayout {
  size_t moe_ws, attn_ws, mlp_ws, xn, lm_ws, total;
  size_t moe_bytes, attn_bytes, mlp_bytes;
};

static StepLayout step_layout(const moe_verify_model* m, int K) {
  StepLayout L{};
  size_t mb = 256, ab = 0, pb = 0;  // (the MoE workspace's header holds the step's error word)
  for (int l = 0; l < m->n_layers; ++l) {
    const moe_decoder_layer& d = m->layers[l];
    const size_t b = d.mlp_gate ? mlp_layout(K, m->hidden, d.mlp_inter).total : 0;
    pb = b > pb ? b : pb;
    const size_t e = d.mlp_gate ? 0 : layout_of(&d.moe, K).total;
    mb = e > mb ? e : mb;
    const size_t a = attn_layout(K, m->hidden, layer_nq(m, d), m->n_kv_heads).total;
    ab = a > ab ? a : ab;
  }
  size_t off = 0;
  L.moe_ws = off;
  off = align256(off + mb);
  L.attn_ws = off;
  off = align256(off + ab);
  L.mlp_ws = off;
  off = align256(off + pb);
  L.xn = off;
  off = align256(off + sizeof(uint16_t) * K * m->hidden);
  L.lm_ws = off;
  off = align256(off + lmhead_ws_bytes(K));
  L.total = off;
  L.moe_bytes = mb;
  L.attn_bytes = ab;
  L.mlp_bytes = pb;
  return L;
}

size_t moe_verify_step_workspace_size(const moe_verify_model* m, int K) {
  if (check_model(m, K) != MOE_OK) return 0;
  return step_layout(m, K).total;
}

// One target forward over the K rows in x (every layer's attention block and
// MoE block, in place), then the greedy token of every row into `target`.
static moe_status forward_impl(const moe_verify_model* m, uint16_t* x, int K, int32_t* target, char* b,
                               const StepLayout& L, cudaStream_t st) {
  uint16_t* xn = reinterpret_cast<uint16_t*>(b + L.xn);
  const int H = m->hidden;
  int* err = reinterpret_cast<int*>(b + L.moe_ws);  // the step's error word (the MoE workspace header)
  for (int l = 0; l < m->n_layers; ++l) {
    const moe_decoder_layer& d = m->layers[l];
    const int nq = layer_nq(m, d);
    const AttnLayout AL = attn_layout(K, H, nq, m->n_kv_heads);
    moe_status s = attention_impl(x, K, H, nq, m->n_kv_heads, m->ctx, d.Wq, d.Wk, d.Wv, d.Wo, d.kcache, d.vcache,
                                  m->kv_len, &d.pos, m->eps, x, nullptr, nullptr, nullptr, b + L.attn_ws, AL, err, st);
    if (s != MOE_OK) return s;
    if (d.mlp_gate)  // a dense SwiGLU MLP block (Laguna's layer 0)
      s = dense_mlp_impl(x, K, H, d.mlp_inter, d.mlp_gate, d.mlp_up, d.mlp_down, m->eps, x, b + L.mlp_ws,
                         mlp_layout(K, H, d.mlp_inter), err, st);
    else {  // the MoE layer kernel applies its RMSNorm to x itself; from its tail it
            // prefetches the next layer's q/k/v weights into L2
      L2Prefetch pf{};
      if (l + 1 < m->n_layers) {
        const moe_decoder_layer& dn = m->layers[l + 1];
        pf.p[0] = dn.Wq;
        pf.bytes[0] = (uint64_t)layer_nq(m, dn) * 128 * H * 2;
        pf.p[1] = dn.Wk;
        pf.bytes[1] = (uint64_t)m->n_kv_heads * 128 * H * 2;
        pf.p[2] = dn.Wv;
        pf.bytes[2] = pf.bytes[1];
        pf.n = 3;  // (the next layer's KV cache as well was slower: 2.96 against 2.92 ms per step;
                   // its o-projection weights too: 2.70 against 2.68)
      }
      s = run_layer(&d.moe, x, K, x, x, nullptr, nullptr, nullptr, b + L.moe_ws, L.moe_bytes, st, true, nullptr,
                    m->eps, &pf);
    }
    if (s != MOE_OK) return s;
  }
  if (lmhead_stream_fits(K, H))  // the final RMSNorm inside the lm_head kernel
    return lm_head_impl(x, K, H, m->lm_head, m->vocab, target, nullptr, b + L.lm_ws, lmhead_ws_bytes(K), m->eps,
                        true, err, st);
  if (launch_rmsnorm(x, K, H, m->eps, xn, st, false) != cudaSuccess) return MOE_ERR_CUDA;
  return moe_lm_head_argmax(xn, K, H, m->lm_head, m->vocab, target, nullptr, b + L.lm_ws, lmhead_ws_bytes(K), st);
}

moe_status moe_verify_step(const moe_verify_model* m, uint16_t* x, int K, const int32_t* draft, int32_t* target,
                           int32_t* n_accepted, void* ws, size_t ws_bytes, void* stream) {
  moe_status s = check_model(m, K);
  if (s != MOE_OK) return s;
  if (!x || !draft || !target || !n_accepted || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(ws)) return MOE_ERR_MISALIGNED;
  const StepLayout L = step_layout(m, K);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  s = forward_impl(m, x, K, target, static_cast<char*>(ws), L, st);
  if (s != MOE_OK) return s;
  return verify_accept_prefix(draft, target, K, n_accepted, stream);
}

moe_status moe_kv_commit(int32_t* kv_len, const int32_t* n_accepted, int K, int capacity, void* stream) {
  if (!kv_len || !n_accepted || K < 1 || capacity < 0) return MOE_ERR_INVALID_ARG;
  if (launch_kv_commit(kv_len, n_accepted, K, capacity, nullptr, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_synthetic_drafts(const int32_t* target, const uint8_t* coin, const int32_t* alt, int K, int vocab,
                                int32_t* draft, void* stream) {
  if (!target || !coin || !alt || !draft || K < 1 || vocab < 2) return MOE_ERR_INVALID_ARG;
  if (launch_synthetic_drafts(target, coin, alt, K, vocab, draft, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_verify_rounds(const moe_verify_model* m, const uint16_t* x_rounds, int R, int K, const uint8_t* coin,
                             const int32_t* alt, uint16_t* x_work, int32_t* targets, int32_t* drafts,
                             int32_t* n_accepted, void* ws, size_t ws_bytes, void* stream) {
  moe_status s = check_model(m, K);
  if (s != MOE_OK) return s;
  if (!m->kv_len || R < 1 || !x_rounds || !coin || !alt || !x_work || !targets || !drafts || !n_accepted || !ws)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_rounds) || !aligned16(x_work) || !aligned16(ws)) return MOE_ERR_MISALIGNED;
  const StepLayout L = step_layout(m, K);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* b = static_cast<char*>(ws);
  int* err = reinterpret_cast<int*>(b + L.moe_ws);
  const size_t row_bytes = sizeof(uint16_t) * (size_t)K * m->hidden;
  for (int r = 0; r < R; ++r) {
    if (cudaMemcpyAsync(x_work, x_rounds + (size_t)r * K * m->hidden, row_bytes, cudaMemcpyDeviceToDevice, st) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    int32_t* tgt = targets + (size_t)r * K;
    int32_t* dft = drafts + (size_t)r * K;
    s = forward_impl(m, x_work, K, tgt, b, L, st);
    if (s != MOE_OK) return s;
    if (launch_synthetic_drafts(tgt, coin + (size_t)r * K, alt + (size_t)r * K, K, m->vocab, dft, st) != cudaSuccess ||
        launch_accept(dft, tgt, K, n_accepted + r, st) != cudaSuccess ||
        launch_kv_commit(const_cast<int32_t*>(m->kv_len), n_accepted + r, K, m->ctx, err, st) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
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

moe_status moe_host_pointer(const void* host, void** dev) {
  if (!host || !dev) return MOE_ERR_INVALID_ARG;
  // page-locked host memory only: where the device can also reach pageable
  // memory (address translation on a coherent host link), the mapping query
  // succeeds for it as well, so the memory type decides
  cudaPointerAttributes pa{};
  if (cudaPointerGetAttributes(&pa, host) != cudaSuccess || pa.type != cudaMemoryTypeHost || !pa.devicePointer) {
    cudaGetLastError();  // the failed query is not an error of the caller's stream
    return MOE_ERR_INVALID_ARG;
  }
  *dev = pa.devicePointer;
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
    case MOE_ERR_CAPACITY: return "KV cache capacity exceeded";
  }
  return "unknown status";
}

size_t moe_debug_partials_offset(const moe_layer* layer, int K) {
  if (check_layer(layer, K) != MOE_OK) return 0;
  return layout_of(layer, K).dpart;
}

void moe_debug_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns); }

void moe_debug_set_trace(void* buf) { g_trace = static_cast<unsigned long long*>(buf); }

}  // extern "C"
