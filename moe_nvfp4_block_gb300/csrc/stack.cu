// stack.cu -- the verify step around the MoE layers: RMSNorm between blocks
// and the lm_head greedy argmax over every verify row.
//
// Both use the fixed FP32 order of the router (lane l of a warp owns the
// 16-byte pieces 256*j + 8*l .. +7 of a row and accumulates in element
// order; the 32 partials combine by xor-shuffle rounds 16, 8, 4, 2, 1),
// because their results decide integers: the normalised rows feed the
// router's top-k, and the lm_head logits decide the greedy token of each
// verify row (PR #844, "5. Numerical safety": the verifier takes an argmax
// over every row, not only the last).
#include <cfloat>
#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float warp_sum_xor(float v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

__device__ __forceinline__ bool ranks_before(float la, int a, float lb, int b) {
  return (la > lb) || (la == lb && a < b);
}

}  // namespace

// ------------------------------------------------------------------ RMSNorm
// One warp per row: ss = fixed-order sum of x*x, mean = ss / H,
// inv = 1 / sqrt(mean + eps), out = bf16(x * inv); each step one correctly
// rounded FP32 operation.  The row's pieces are loaded in chunks of 8 per
// lane, each chunk's loads all in flight before its first product, so a row
// of H <= 2048 costs one memory round trip, not one per piece.
__global__ void __launch_bounds__(512) k_rmsnorm(const uint16_t* __restrict__ x, int K, int H, float eps,
                                                 uint16_t* __restrict__ out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  pdl_launch_dependents();
  const int r = blockIdx.x * (blockDim.x >> 5) + warp;
  if (r >= K) return;
  const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)r * H);
  const int nj = H / 256;
  uint4 xv[8];
  auto load_chunk = [&](int j0) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (j0 + u < nj) xv[u] = __ldcg(row + (j0 + u) * 32 + lane);
  };
  float acc = 0.f;
  for (int j0 = 0; j0 < nj; j0 += 8) {
    load_chunk(j0);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (j0 + u >= nj) break;
      const uint32_t q[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const float f = (t & 1) ? bf16_hi(q[t >> 1]) : bf16_lo(q[t >> 1]);
        acc = __fmaf_rn(f, f, acc);
      }
    }
  }
  const float ss = warp_sum_xor(acc);
  const float mean = __fdiv_rn(ss, (float)H);
  const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
  uint4* o = reinterpret_cast<uint4*>(out + (size_t)r * H);
  for (int j0 = 0; j0 < nj; j0 += 8) {
    if (nj > 8) load_chunk(j0);  // (with one chunk the registers still hold it)
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (j0 + u >= nj) break;
      const uint32_t q[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
      uint32_t res[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t lo = float_to_bf16_bits(__fmul_rn(bf16_lo(q[i]), inv));
        const uint32_t hi = float_to_bf16_bits(__fmul_rn(bf16_hi(q[i]), inv));
        res[i] = lo | (hi << 16);
      }
      o[(j0 + u) * 32 + lane] = make_uint4(res[0], res[1], res[2], res[3]);
    }
  }
}

cudaError_t launch_rmsnorm(const uint16_t* x, int K, int H, float eps, uint16_t* out, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32 * K);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  max_carveout(k_rmsnorm);
  return cudaLaunchKernelEx(&cfg, k_rmsnorm, x, K, H, eps, out);
}

// ------------------------------------------------------------------ lm_head argmax
// Persistent: warp w of the grid takes vocab rows w, w + n_warps, ...; the
// next row's 16-byte pieces are loaded before the current row is reduced.
// Each warp keeps, per verify row, the best (logit, index) seen (rows are
// visited in increasing order, so a later equal logit never replaces an
// earlier one).  CTA results go to the workspace; the last CTA (atomic
// ticket) reduces them in CTA order and writes the tokens.
constexpr int kLmWarps = 8;

template <int KR>
__global__ void __launch_bounds__(kLmWarps * 32) k_lmhead_argmax(LmHeadArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ float s_bv[kLmWarps][KR];
  __shared__ int s_bi[kLmWarps][KR];
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = a.K, H = a.H, V = a.V;
  pdl_wait();
  pdl_launch_dependents();
  uint4* xs = reinterpret_cast<uint4*>(smem);
  block_copy_g2s(xs, reinterpret_cast<const uint4*>(a.x), K * H / 8);
  __syncthreads();

  float bv[KR];
  int bi[KR];
#pragma unroll
  for (int r = 0; r < KR; ++r) {
    bv[r] = -INFINITY;
    bi[r] = INT_MAX;
  }
  const int nj = H / 256;  // <= 8
  const int gw = blockIdx.x * kLmWarps + warp, nw = gridDim.x * kLmWarps;
  uint4 cur[8], nxt[8];
  int v = gw;
  if (v < V) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < nj) cur[j] = ldg_nc_v4(reinterpret_cast<const uint4*>(a.W + (size_t)v * H) + j * 32 + lane);
  }
  for (; v < V; v += nw) {
    const int vn = v + nw;
    if (vn < V) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < nj) nxt[j] = ldg_nc_v4(reinterpret_cast<const uint4*>(a.W + (size_t)vn * H) + j * 32 + lane);
    }
    float acc[KR];
#pragma unroll
    for (int r = 0; r < KR; ++r) acc[r] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j >= nj) break;
      const uint32_t wq[4] = {cur[j].x, cur[j].y, cur[j].z, cur[j].w};
#pragma unroll
      for (int r = 0; r < KR; ++r) {
        if (r < K) {
          const uint4 xv = xs[r * (H / 8) + j * 32 + lane];
          const uint32_t xq[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const float xf = (t & 1) ? bf16_hi(xq[t >> 1]) : bf16_lo(xq[t >> 1]);
            const float wf = (t & 1) ? bf16_hi(wq[t >> 1]) : bf16_lo(wq[t >> 1]);
            acc[r] = __fmaf_rn(xf, wf, acc[r]);
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < KR; ++r) {
      if (r < K) {
        const float l = warp_sum_xor(acc[r]);
        if (bi[r] == INT_MAX || l > bv[r]) {  // rows arrive in increasing order
          bv[r] = l;
          bi[r] = v;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
  }
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < KR; ++r) {
      s_bv[warp][r] = bv[r];
      s_bi[warp][r] = bi[r];
    }
  }
  __syncthreads();
  if (threadIdx.x < K) {
    const int r = threadIdx.x;
    float b = -INFINITY;
    int i = INT_MAX;
    for (int w = 0; w < kLmWarps; ++w)
      if (s_bi[w][r] != INT_MAX && (i == INT_MAX || ranks_before(s_bv[w][r], s_bi[w][r], b, i))) {
        b = s_bv[w][r];
        i = s_bi[w][r];
      }
    a.part_v[blockIdx.x * K + r] = b;
    a.part_i[blockIdx.x * K + r] = i;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(a.ticket, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x < K) {
    const int r = threadIdx.x;
    float b = -INFINITY;
    int i = INT_MAX;
    for (int c = 0; c < (int)gridDim.x; ++c) {
      const float cv = __ldcg(a.part_v + c * K + r);
      const int ci = __ldcg(a.part_i + c * K + r);
      if (ci != INT_MAX && (i == INT_MAX || ranks_before(cv, ci, b, i))) {
        b = cv;
        i = ci;
      }
    }
    a.tok[r] = i;
    if (a.best) a.best[r] = b;
  }
  if (threadIdx.x == 0) *a.ticket = 0u;
}

int lmhead_grid() { return 2 * num_sms() < kLmMaxGrid ? 2 * num_sms() : kLmMaxGrid; }

cudaError_t launch_lmhead(const LmHeadArgs& a, cudaStream_t s, bool pdl) {
  const size_t sm = sizeof(uint16_t) * a.K * a.H;
  auto run = [&](auto kern) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e == cudaSuccess) e = max_carveout(kern);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(lmhead_grid());
    cfg.blockDim = dim3(kLmWarps * 32);
    cfg.dynamicSmemBytes = sm;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
  };
  if (a.K <= 4) return run(k_lmhead_argmax<4>);
  if (a.K <= 8) return run(k_lmhead_argmax<8>);
  return run(k_lmhead_argmax<16>);
}

}  // namespace moe
