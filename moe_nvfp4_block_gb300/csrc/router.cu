// router.cu -- router GEMV + softmax + top-k + expert grouping (one launch),
// the moe_router_topk entry point.  (A layer call computes its router
// logits inside the experts kernel, with the same arithmetic.)
//
// Each warp forms the logits of one expert for all K rows: lane l streams the
// 16-byte pieces 256*j + 8*l .. +7 of the expert's bf16 router row and adds
// x*w into one FP32 partial per row in element order; the 32 partials are
// combined by xor-shuffle rounds (distances 16, 8, 4, 2, 1).  This fixed order
// makes the logits -- and so the selected experts -- reproducible bit for bit.
//
// The last CTA to finish (atomic ticket, no spinning) selects the top-k per
// row (larger logit first, lower index on an exact tie), renormalises the
// selected softmax probabilities (PR #844, "4. What I ported": top-k of the
// router scores, renormalised) -- or, with sigmoid scoring, selects by
// score + bias and renormalises the selected scores -- and groups the (row, slot) pairs by expert so
// that each distinct expert is streamed once by the expert kernels (PR #844,
// "8. What I looked at": the stock gather reads an expert once per
// (row, slot)).
#include <cfloat>
#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

__device__ __forceinline__ bool ranks_before(float la, int a, float lb, int b) {
  return (la > lb) || (la == lb && a < b);
}

// Exclusive scan of one int per thread over the block; *total gets the sum.
__device__ int block_exclusive_scan(int v, int* total, int* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int o = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += o;
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int i = 0; i < nw; ++i) {
      int t = scratch[i];
      scratch[i] = run;
      run += t;
    }
    scratch[nw] = run;
  }
  __syncthreads();
  int r = scratch[warp] + inc - v;
  *total = scratch[nw];
  __syncthreads();
  return r;
}

template <int KR>
__global__ void __launch_bounds__(kRouterWarps * 32) k_router(RouterArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_last;
  __shared__ int s_scan[kRouterWarps + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = a.K, H = a.H, E = a.E, k = a.k, G = a.G;

  // The router weights do not depend on earlier kernels: start loading them
  // before the dependency wait.
  const int e = blockIdx.x * kRouterWarps + warp;
  const int nj = H / 256;  // <= 8
  uint4 wv[8];
  if (e < E) {
    const uint4* wrow = reinterpret_cast<const uint4*>(a.router_w + (size_t)e * H);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < nj) wv[j] = ldg_nc_v4(wrow + j * 32 + lane);
  }
  pdl_wait();  // the rows and the workspace are ours from here on
  pdl_launch_dependents();

  // ---------------------------------------------------------------- logits
  {
    uint4* xs = reinterpret_cast<uint4*>(smem);  // [K][H/8]
    const uint4* xg = reinterpret_cast<const uint4*>(a.x);
    block_copy_g2s(xs, xg, K * H / 8);
    __syncthreads();
    if (e < E) {
      float acc[KR];
#pragma unroll
      for (int r = 0; r < KR; ++r) acc[r] = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j >= nj) break;
        const uint32_t wq[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
#pragma unroll
        for (int r = 0; r < KR; ++r) {
          if (r < K) {
            const uint4 xv = xs[r * (H / 8) + j * 32 + lane];
            const uint32_t xq[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const float xf = __uint_as_float((t & 1) ? (xq[t >> 1] & 0xFFFF0000u) : (xq[t >> 1] << 16));
              const float wf = __uint_as_float((t & 1) ? (wq[t >> 1] & 0xFFFF0000u) : (wq[t >> 1] << 16));
              acc[r] = __fmaf_rn(xf, wf, acc[r]);
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < KR; ++r) {
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) acc[r] = __fadd_rn(acc[r], __shfl_xor_sync(0xffffffffu, acc[r], d));
      }
      if (lane == 0) {
        // softmax scoring: logit + bias; sigmoid scoring: the score alone
        // (the bias enters the selection keys below)
        const float b = a.bias ? a.bias[e] : 0.f;
#pragma unroll
        for (int r = 0; r < KR; ++r)
          if (r < K)
            a.ws.logits[(size_t)r * E + e] =
                a.scoring ? sigmoid_score(acc[r]) : (a.bias ? __fadd_rn(acc[r], b) : acc[r]);
      }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned t = atomicAdd(a.ws.ticket, 1u);
      s_last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
  }

  // ---------------------------------------------------------------- top-k (last CTA)
  float* lg = reinterpret_cast<float*>(smem);                    // [K][E]
  unsigned char* taken = smem + sizeof(float) * K * E;           // [K][E]
  size_t off = (sizeof(float) * K * E + K * E + 15) & ~size_t(15);
  float* selv = reinterpret_cast<float*>(smem + off);            // [K][k]
  int* seli = reinterpret_cast<int*>(selv + K * k);              // [K][k]
  unsigned* rowmask = reinterpret_cast<unsigned*>(seli + K * k); // [E]
  int* posmap = reinterpret_cast<int*>(rowmask + E);             // [E]
  unsigned* urow_s = reinterpret_cast<unsigned*>(posmap + E);    // [G+1]

  for (int r = warp; r < K; r += kRouterWarps) {
    float* l = lg + (size_t)r * E;
    unsigned char* tk = taken + (size_t)r * E;
    for (int e = lane; e < E; e += 32) {
      const float v = __ldcg(a.ws.logits + (size_t)r * E + e);
      l[e] = (a.scoring && a.bias) ? __fadd_rn(v, a.bias[e]) : v;  // selection keys
      tk[e] = 0;
    }
    __syncwarp();
    for (int s = 0; s < k; ++s) {
      float bv = -INFINITY;
      int be = INT_MAX;
      for (int e = lane; e < E; e += 32)
        if (!tk[e] && ranks_before(l[e], e, bv, be)) {
          bv = l[e];
          be = e;
        }
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
        const int oe = __shfl_xor_sync(0xffffffffu, be, d);
        if (ranks_before(ov, oe, bv, be)) {
          bv = ov;
          be = oe;
        }
      }
      if (be == INT_MAX) {  // only NaN logits left: take the lowest free index
        int f = INT_MAX;
        for (int e = lane; e < E; e += 32)
          if (!tk[e]) f = min(f, e);
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) f = min(f, __shfl_xor_sync(0xffffffffu, f, d));
        be = f;
        bv = l[be];
      }
      if (lane == 0) {
        tk[be] = 1;
        selv[r * k + s] = bv;
        seli[r * k + s] = be;
      }
      __syncwarp();
    }
    // renormalised softmax over the selected logits (k <= 32); sigmoid
    // scoring: the selected experts' own scores over their sum
    const float m = selv[r * k];
    float ev = 0.f;
    if (lane < k)
      ev = a.scoring ? __ldcg(a.ws.logits + (size_t)r * E + seli[r * k + lane]) : expf(selv[r * k + lane] - m);
    float z = ev;
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
    if (lane < k) {
      const float wv = ev / z;
      const int q = r * k + lane;
      a.ws.idx[q] = seli[q];
      a.ws.w[q] = wv;
      if (a.idx_out) a.idx_out[q] = seli[q];
      if (a.w_out) a.w_out[q] = wv;
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- grouping
  for (int e = threadIdx.x; e < E; e += blockDim.x) rowmask[e] = 0u;
  for (int i = threadIdx.x; i < (G + 1) * K; i += blockDim.x) a.ws.slotmap[i] = -1;
  __syncthreads();
  for (int q = threadIdx.x; q < K * k; q += blockDim.x) atomicOr(&rowmask[seli[q]], 1u << (q / k));
  __syncthreads();

  int* grp = a.ws.group;
  int* gout = a.group_out;
  {
    const int CH = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = threadIdx.x * CH;
    int cnt = 0;
    for (int e = e0; e < min(E, e0 + CH); ++e) cnt += rowmask[e] != 0u;
    int total;
    int u = block_exclusive_scan(cnt, &total, s_scan);
    for (int e = e0; e < min(E, e0 + CH); ++e) {
      if (rowmask[e]) {
        posmap[e] = u;
        urow_s[u] = rowmask[e];
        grp[1 + u] = e;
        if (gout) gout[1 + u] = e;
        ++u;
      }
    }
    if (threadIdx.x == 0) {
      grp[0] = total;
      if (gout) gout[0] = total;
    }
    for (int v = total + threadIdx.x; v < G; v += blockDim.x) {
      grp[1 + v] = -1;
      if (gout) gout[1 + v] = -1;
      urow_s[v] = 0u;
    }
    if (threadIdx.x == 0) urow_s[G] = a.has_shared ? ((K == 32) ? 0xffffffffu : ((1u << K) - 1u)) : 0u;
    __syncthreads();
    for (int v = threadIdx.x; v <= G; v += blockDim.x) a.ws.urow[v] = urow_s[v];
    for (int q = threadIdx.x; q < K * k; q += blockDim.x) a.ws.slotmap[posmap[seli[q]] * K + q / k] = q % k;
    if (a.has_shared)
      for (int r = threadIdx.x; r < K; r += blockDim.x) a.ws.slotmap[G * K + r] = k;

    // offsets and pair lists (routed experts only)
    const int CU = (G + blockDim.x - 1) / blockDim.x;
    const int u0 = threadIdx.x * CU;
    int pc = 0;
    for (int v = u0; v < min(G, u0 + CU); ++v) pc += __popc(urow_s[v]);
    int tot2;
    int o = block_exclusive_scan(pc, &tot2, s_scan);
    for (int v = u0; v < min(G, u0 + CU); ++v) {
      grp[1 + G + v] = o;
      if (gout) gout[1 + G + v] = o;
      const unsigned msk = urow_s[v];
      if (v < total) {
        const int ex = grp[1 + v];
        for (int r = 0; r < K; ++r) {
          if (!((msk >> r) & 1u)) continue;
          int s = 0;
          while (seli[r * k + s] != ex) ++s;
          grp[2 + 2 * G + o] = r * k + s;
          if (gout) gout[2 + 2 * G + o] = r * k + s;
          ++o;
        }
      }
    }
    if (threadIdx.x == 0) {
      grp[1 + 2 * G] = K * k;
      if (gout) gout[1 + 2 * G] = K * k;
    }
  }
  if (threadIdx.x == 0) *a.ws.ticket = 0u;
}

static size_t router_smem(const RouterArgs& a) {
  const size_t x = sizeof(uint16_t) * a.K * a.H;
  size_t t = ((sizeof(float) * a.K * a.E + a.K * a.E + 15) & ~size_t(15)) + sizeof(float) * a.K * a.k +
             sizeof(int) * a.K * a.k + sizeof(unsigned) * a.E + sizeof(int) * a.E + sizeof(unsigned) * (a.G + 1);
  return x > t ? x : t;
}

template <int KR>
static cudaError_t launch_router_t(const RouterArgs& a, cudaStream_t s, bool pdl) {
  const size_t sm = router_smem(a);
  cudaError_t err = cudaFuncSetAttribute(k_router<KR>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (err == cudaSuccess) err = max_carveout(k_router<KR>);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.E + kRouterWarps - 1) / kRouterWarps);
  cfg.blockDim = dim3(kRouterWarps * 32);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_router<KR>, a);
}

cudaError_t launch_router(const RouterArgs& a, cudaStream_t s, bool pdl) {
  if (a.K <= 4) return launch_router_t<4>(a, s, pdl);
  if (a.K <= 8) return launch_router_t<8>(a, s, pdl);
  return launch_router_t<16>(a, s, pdl);
}

}  // namespace moe
