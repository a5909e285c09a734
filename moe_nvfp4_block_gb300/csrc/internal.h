// internal.h -- shapes, workspace layout and kernel argument blocks shared by
// the C-ABI layer (capi.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_verify.h"

namespace moe {

constexpr int kRouterWarps = 8;          // experts per router CTA
constexpr int kGURows = 16;              // intermediate rows per gate/up item
constexpr int kDNRows = 128;             // hidden rows per down item
constexpr int kMaxStages = 6;            // TMA ring depth limit of the experts kernel

// Bytes of one ring stage: the larger of a gate/up item (codes and scales of
// 16 rows of gate and up) and a down item (128 rows), 1024-aligned.
__host__ __device__ inline int expert_stage_bytes(int H, int I) {
  const int gu = 2 * (kGURows * H / 2) + 2 * (kGURows * H / 16);
  const int dn = kDNRows * I / 2 + kDNRows * I / 16;
  const int m = gu > dn ? gu : dn;
  return (m + 1023) & ~1023;
}

// Byte offsets of the workspace regions (all 256-byte aligned).  The header
// sits at a fixed offset; the other regions' offsets depend on the shape.
// Words exchanged between the CTAs of the experts kernel are tagged: a 32-bit
// payload next to the 32-bit tag of the layer call that wrote it, so stale
// words of earlier calls (or of other shapes) are told apart by the tag and
// nothing is cleared between calls.
struct WsLayout {
  size_t hdr;      // 256 bytes: int32 error word, uint32 router ticket, uint64 experts-kernel CTA exits
  size_t logits;   // float [K][E] (moe_router_topk)
  size_t idx;      // int32 [K][k]
  size_t w;        // float [K][k]
  size_t group;    // int32 [2 + 2G + K*k]
  size_t urow;     // uint32 [G+1]: rows routed to each distinct expert (bitmask)
  size_t slotmap;  // int32 [G+1][K]: slot of the expert in row r's selection, -1 if none
  size_t tlog;     // tagged [K][E]: router logits of the experts kernel
  size_t flags;    // tagged [G+1][I/16][4]: gate/up item done, per duty warp
  size_t h;        // tagged [G+1][K][I/2]: h, two bf16 per word
  size_t dpart;    // tagged [K][k+1][H]: FP32 down partials per (row, slot)
  size_t xs;       // bf16 [K][H]: the rows, staged when the caller's are host memory
  size_t total;
};
inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

inline int group_cap(int K, int E, int k) { return E < K * k ? E : K * k; }

inline WsLayout ws_layout(int K, int E, int k, int H, int I) {
  WsLayout L{};
  const int G = group_cap(K, E, k);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t r = o;
    o = align256(o + bytes);
    return r;
  };
  L.hdr = take(256);
  L.logits = take(sizeof(float) * K * E);
  L.idx = take(sizeof(int32_t) * K * k);
  L.w = take(sizeof(float) * K * k);
  L.group = take(sizeof(int32_t) * (2 + 2 * G + K * k));
  L.urow = take(sizeof(uint32_t) * (G + 1));
  L.slotmap = take(sizeof(int32_t) * (G + 1) * K);
  L.tlog = take(sizeof(uint64_t) * K * E);
  L.flags = take(sizeof(uint64_t) * (size_t)(G + 1) * (I / 16) * 4);
  L.h = take(sizeof(uint64_t) * (size_t)(G + 1) * K * (I / 2));
  L.dpart = take(sizeof(uint64_t) * (size_t)K * (k + 1) * H);
  L.xs = take(sizeof(uint16_t) * (size_t)K * H);
  L.total = o;
  return L;
}

// Pointers into one workspace.
struct WsPtrs {
  int* err;
  unsigned* ticket;
  float* logits;
  int* idx;
  float* w;
  int* group;
  unsigned* urow;
  int* slotmap;
  unsigned long long* exits;  // calls finished by the experts kernel's CTAs (the call index is exits / grid)
  unsigned long long* tlog;
  unsigned long long* flags;
  unsigned long long* h;
  unsigned long long* dpart;
};

inline WsPtrs ws_ptrs(void* ws, const WsLayout& L) {
  char* b = static_cast<char*>(ws);
  WsPtrs p;
  p.err = reinterpret_cast<int*>(b + L.hdr);
  p.ticket = reinterpret_cast<unsigned*>(b + L.hdr + 4);
  p.logits = reinterpret_cast<float*>(b + L.logits);
  p.idx = reinterpret_cast<int*>(b + L.idx);
  p.w = reinterpret_cast<float*>(b + L.w);
  p.group = reinterpret_cast<int*>(b + L.group);
  p.urow = reinterpret_cast<unsigned*>(b + L.urow);
  p.slotmap = reinterpret_cast<int*>(b + L.slotmap);
  p.exits = reinterpret_cast<unsigned long long*>(b + L.hdr + 8);
  p.tlog = reinterpret_cast<unsigned long long*>(b + L.tlog);
  p.flags = reinterpret_cast<unsigned long long*>(b + L.flags);
  p.h = reinterpret_cast<unsigned long long*>(b + L.h);
  p.dpart = reinterpret_cast<unsigned long long*>(b + L.dpart);

  return p;
}

struct RouterArgs {
  const uint16_t* x;        // [K][H]
  const uint16_t* router_w; // [E][H]
  const float* bias;        // [E] or null
  int K, H, E, k, G;
  int has_shared;
  int scoring;              // MOE_SCORE_SOFTMAX or MOE_SCORE_SIGMOID
  WsPtrs ws;
  int32_t* idx_out;         // caller copies (nullable)
  float* w_out;
  int32_t* group_out;
};

// Per-projection pointers the expert kernels need besides the tensor maps.
struct ProjPtrs {
  const uint8_t* scales;
  const float* tscale;
};

// One MoE layer as the experts kernel sees it (everything but the tensor maps).
// Byte ranges a kernel prefetches into L2 for the kernel that follows it,
// once its own stream is issued (each CTA its share); n = 0: none.
struct L2Prefetch {
  const void* p[4];
  uint64_t bytes[4];  // multiples of 16, p 16-byte aligned
  int n;
};

struct LayerDesc {
  const uint16_t* router_w;  // [E][H] bf16
  const float* router_bias;  // [E] or null
  ProjPtrs gate, up, down, sh_gate, sh_up, sh_down;
  float routed_scale;
  int has_shared;
  int scoring;               // MOE_SCORE_SOFTMAX or MOE_SCORE_SIGMOID
};

// Tensor maps of one layer: codes of gate, up, down, shared gate, shared
// up, shared down; E4M3 scales of gate, up, shared gate, shared up.
constexpr int kMapsPerLayer = 10;

// What one launch of the experts kernel runs: one MoE layer call.
struct ExpertsCommon {
  const uint16_t* x;         // [K][H] bf16: the input (normalised, or to normalise when norm)
  const uint16_t* residual;  // [K][H] or null (with norm the residual is x itself)
  uint16_t* y;               // [K][H]
  int K, H, I, E, k, G;
  WsPtrs ws;
  int32_t* idx_out;          // routing copies for the caller (nullable)
  float* w_out;
  int32_t* group_out;
  uint64_t wait_ns;
  unsigned long long* trace;  // [grid][kTraceSlots] milestone timestamps, or null
  int code3d;                 // code maps are 3-D (one request per tile)
  int stages, nred;           // ring depths (set by the launcher)
  int norm;                   // 1: x is the residual stream; the kernel applies the RMSNorm (unit gain)
  float norm_eps;
  L2Prefetch pf;              // the next kernel's first bytes, prefetched once the producer is done
};

struct ExpertsParams {
  CUtensorMap maps[kMapsPerLayer];
  LayerDesc L;
  ExpertsCommon c;
};

constexpr int kTraceSlots = 80;
extern unsigned long long* g_trace;  // debug timeline buffer (null = off)

struct LmHeadArgs {
  const uint16_t* x;  // [K][H] normalised rows (raw rows when norm_eps > 0)
  const uint16_t* W;  // [V][H]
  int K, H, V;
  int32_t* tok;       // [K] out
  float* best;        // [K] out (nullable)
  float* part_v;      // [grid][K]
  int* part_i;        // [grid][K]
  unsigned* ticket;
  float norm_eps;     // streamed kernel: > 0 normalises x while staged
  int rows_per_stage; // streamed kernel (set by its launcher)
  int* err;           // streamed kernel: a ring wait that ran out, or null
  uint64_t wait_ns;
};

constexpr int kLmMaxGrid = 1024;

struct GemvSeg {
  const uint16_t* W;    // [N][D]
  uint16_t* out;        // [K][N]
  const uint16_t* res;  // [K][N] or null
  int N;
  // optional in-place KV append: output (r, n) also goes to
  // cache[n / 128][*len + r][n % 128] of a [N/128][cap][128] cache
  uint16_t* cache;
  const int* len;
  int cap;
  int rope;  // the rotary embedding applies to this matrix's heads (rope_rd > 0)
};

struct GemvArgs {
  const uint16_t* x;  // [K][D]
  int K, D;
  GemvSeg seg[3];
  int nseg, n_total;
  int* err;           // error word (a cache append past its capacity, a wait that ran out), or null
  float norm_eps;     // > 0: x is RMS-normalised first (streamed kernel only)
  uint64_t wait_ns;   // streamed kernel: limit of each ring wait
  // Streamed kernel: the rotary embedding of the rope segments' 128-row
  // heads in the epilogue (0: none): rows i, i + rope_rd/2 (i < rope_rd/2)
  // of a head rotated by the angle (pos0 + r) * rope_freq[i], pos0 =
  // *rope_len or rope_C; rope_rd a multiple of 16.
  int rope_rd;
  const int* rope_len;
  int rope_C;
  double rope_freq[64];
  // Streamed kernel, SwiGLU: seg[0] the gate and seg[1] the up matrix (N
  // rows each, N a multiple of 8, n_total = 2N); the output is
  // h = bf16(silu(gate) * up) into seg[0].out.
  int glu;
};
bool gemv_stream_rope_fits(const GemvArgs& a, int grid);

struct AttnArgs {
  const uint16_t* q;      // [K][nq*128]
  const uint16_t* kc;     // [nkv][C][128]: C positions of capacity
  const uint16_t* vc;
  const int* len;         // valid cached positions (device), or null: all C
  const uint16_t* k_new;  // [K][nkv*128]
  const uint16_t* v_new;
  uint16_t* o;            // [K][nq*128]
  int K, nq, nkv, C, group;
  int tiles;              // 16-row query tiles per KV head: ceil(K * group / 16)
  int window;             // sliding window (positions a row sees, itself included), 0 = all
  float scale_log2;       // log2(e) * temperature / sqrt(128)
  float* part_o;          // [nkv][splits][tiles * 16][128]
  float* part_ml;         // [nkv][splits][tiles * 16][2]
  int* err;               // error word (a ring wait that ran out), or null
  uint64_t wait_ns;       // limit of each ring wait (streamed kernel)
};

// The streamed split kernel's arguments: the caches as bf16 tensor maps over
// [nkv * C rows][128 dims] with the 128-byte swizzle (encode_kv_map).
struct AttnStreamArgs {
  AttnArgs a;
  CUtensorMap km, vm;
  int kv3d;  // the maps are 3-D (one box per chunk) rather than 2-D (one per dim half)
};

constexpr int kAttnMaxSplits = 64;
constexpr int kAttnMaxTiles = 4;  // K * group <= 64 query rows per KV head

// Rotary position embedding of the new rows (in place), at positions
// pos0 + r with pos0 = *len (or C when len is null); optionally the rotated
// keys and the values appended to the caches at those positions.
struct RopeArgs {
  uint16_t* q;            // [K][nq*128]
  uint16_t* k;            // [K][nkv*128]
  const uint16_t* v;      // [K][nkv*128] (for the append)
  int K, nq, nkv, rd;     // rd: rotary dims per head (pairs i, i + rd/2)
  double freq[64];        // angle per position of pair i
  const int* len;
  int C;                  // cache capacity (head stride)
  uint16_t *kc, *vc;      // caches to append to, or null
  int* err;
};
cudaError_t launch_rope(const RopeArgs& a, cudaStream_t s);

// Dense SwiGLU rows: h[r][i] = bf16(silu(x_r . Wg_i) * (x_r . Wu_i)).
struct SwigluArgs {
  const uint16_t* x;   // [K][D]
  const uint16_t* Wg;  // [N][D]
  const uint16_t* Wu;  // [N][D]
  uint16_t* h;         // [K][N]
  int K, D, N;
};
cudaError_t launch_swiglu(const SwigluArgs& a, cudaStream_t s, bool pdl);

cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t s, bool pdl);
// The streamed GEMV (csrc/gemv.cu): whether it takes `a` on `grid` CTAs, and
// its launch.
bool gemv_stream_fits(const GemvArgs& a, int grid);
cudaError_t launch_gemv_stream(const GemvArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_attention_stream(const AttnStreamArgs& p, cudaStream_t s, bool pdl);
cudaError_t launch_attn_combine(const AttnArgs& a, int splits, cudaStream_t s);
int attn_stream_splits(int nkv, int tiles, int C, int window);
bool encode_kv_map(CUtensorMap* m, const uint16_t* cache, int nkv, int C, bool* is3d);
int attn_splits(int nkv, int tiles, int max_chunks);

inline size_t lmhead_ws_bytes(int K) { return 256 + align256(sizeof(float) * kLmMaxGrid * K) + sizeof(int) * kLmMaxGrid * K; }

// Launchers (return cudaGetLastError()).
cudaError_t launch_rmsnorm(const uint16_t* x, int K, int H, float eps, uint16_t* out, cudaStream_t s, bool pdl);
cudaError_t launch_lmhead(const LmHeadArgs& a, cudaStream_t s, bool pdl);
bool lmhead_stream_fits(int K, int H);
cudaError_t launch_lmhead_stream(const LmHeadArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_router(const RouterArgs& a, cudaStream_t s, bool pdl);
// One launch of the experts kernel: maps [kMapsPerLayer].
cudaError_t launch_experts(const ExpertsCommon& c, const CUtensorMap* maps, const LayerDesc& desc, cudaStream_t s,
                           bool pdl);
size_t experts_smem_bytes(int K, int H, int I, int E, int k, int G, int* stages, int* nred);
cudaError_t launch_accept(const int32_t* draft, const int32_t* target, int K, int32_t* out, cudaStream_t s);
cudaError_t launch_kv_commit(int32_t* len, const int32_t* n_accepted, int K, int cap, int* err, cudaStream_t s);
// bytes (a multiple of 16, at most 64 KB) from src to dst in one CTA, with
// programmatic dependent launch: loads before the dependency wait, stores
// after it (accept.cu)
cudaError_t launch_stage_rows(const void* src, void* dst, size_t bytes, cudaStream_t s);
cudaError_t launch_synthetic_drafts(const int32_t* target, const uint8_t* coin, const int32_t* alt, int K, int vocab,
                                    int32_t* draft, cudaStream_t s);

int num_sms();

// Every kernel of the library asks for the same L1/shared-memory split (all
// shared): an SM that runs one kernel's CTAs can then take the next kernel's
// CTAs (programmatic dependent launch) without first draining to change it.
template <typename Kern>
inline cudaError_t max_carveout(Kern kern) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared);
}

}  // namespace moe

// The layer launch sequence behind moe_verify_layer (capi.cu; not exported).
// norm_eps >= 0: x_norm holds the un-normalised rows and the layer kernel
// applies the RMSNorm (unit gain, this eps) itself.
extern "C" __attribute__((visibility("hidden"))) moe_status run_layer(const moe_layer* layer, const uint16_t* x_norm, int K, const uint16_t* residual,
                                uint16_t* y, int32_t* idx_out, float* w_out, int32_t* group_out, void* ws,
                                size_t ws_bytes, void* stream, bool pdl, void* const* events,
                                float norm_eps = -1.f, const moe::L2Prefetch* pf = nullptr);
