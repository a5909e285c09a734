// lmhead_stream.cu -- the lm_head greedy argmax with the vocab rows streamed
// into shared memory by bulk copies.
//
// Logit (r, v) = fixed-order FP32 dot product of the normalised row x_r with
// vocab row v: lane l of a warp owns elements 256 j + 8 l + i and
// accumulates them in element order, the 32 lane sums are added in xor
// rounds 16, 8, 4, 2, 1.  An exact tie goes to the lower vocab index.  The
// order is the same as the row kernel's in stack.cu, so both give the same
// logits bit for bit.
//
// One CTA per SM owns a contiguous range of vocab rows.  Stages of R rows
// (a 24 or 32 KB slot's worth, at most 8) go through the ring slots; warp
// pair p owns slot p and takes the stages p, p + P, ...; each of its two
// warps reduces R / 2 rows of a stage, so every 16-byte load of x from shared
// memory serves R / 2 rows.  The weights do not depend on the previous
// kernel, so the first stage of every slot is issued before the dependency wait.
// Optionally the rows of x are RMS-normalised while staged (the RMSNorm
// kernel's fixed order and rounding, so bit-identical to normalising first).
#include <cfloat>
#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kLsMaxPairs = 8;
// Bound on waiting for the CTA's own copies before it exits (independent of
// the caller's wait limit, which may be 0 in a test of the give-up path).
constexpr uint64_t kLsDrainNs = 2000000000ull;

__device__ __forceinline__ float lbf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float lbf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float lsum_xor(float v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

__device__ __forceinline__ bool l_before(float la, int a, float lb, int b) {
  return (la > lb) || (la == lb && a < b);
}

struct LsTable {
  uint64_t full[kLsMaxPairs];
  uint64_t empty[kLsMaxPairs];
  int abort;
  int last;
  float inv[16];
  float bv[2 * kLsMaxPairs][16];
  int bi[2 * kLsMaxPairs][16];
};

// Ring shape by K: eight pairs of warps on 24 KB slots while x is small
// (K <= 8; more warps in flight for an issue-bound loop), five pairs on
// 32 KB slots at K = 16 (x takes 64 KB of shared memory).
template <int KR> struct LsShape {
  static constexpr int pairs = KR <= 8 ? 8 : 5;
  static constexpr int slot = KR <= 8 ? 24576 : 32768;
  static constexpr int rpw = KR <= 8 ? 3 : 4;  // vocab rows per warp and stage
  static constexpr bool xf32 = KR <= 4;         // x held as floats (no unpacking per use)
};

}  // namespace

template <int KR>
__global__ void __launch_bounds__(2 * LsShape<KR>::pairs * 32, 1) k_lmhead_stream(const __grid_constant__ LmHeadArgs a) {
  constexpr int kLsPairs = LsShape<KR>::pairs, kLsWarps = 2 * kLsPairs, kLsSlotBytes = LsShape<KR>::slot;
  constexpr int RPW = LsShape<KR>::rpw;
  constexpr bool XF32 = LsShape<KR>::xf32;
  extern __shared__ __align__(128) unsigned char smem[];
  const int K = a.K, H = a.H, V = a.V;
  // x: bf16 rows, or (XF32) floats, the bf16 rows staged in the upper half
  // of the region first
  unsigned char* xreg = smem + kLsPairs * kLsSlotBytes;
  uint4* xs = reinterpret_cast<uint4*>(xreg + (XF32 ? (size_t)K * H * 2 : 0));
  LsTable& T = *reinterpret_cast<LsTable*>(xreg + (size_t)K * H * (XF32 ? 4 : 2));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p = warp >> 1, hw = warp & 1;
  const int R = a.rows_per_stage;
  const int v0 = (int)((long long)blockIdx.x * V / gridDim.x);
  const int v1 = (int)((long long)(blockIdx.x + 1) * V / gridDim.x);
  const int nst = (v1 - v0 + R - 1) / R;
  const uint32_t row_bytes = (uint32_t)H * 2u;
  auto issue = [&](int s, uint64_t pol) {
    const int slot = s % kLsPairs;
    const int vb = v0 + s * R;
    const uint32_t bytes = (uint32_t)min(R, v1 - vb) * row_bytes;
    mbar_arrive_expect_tx(&T.full[slot], bytes);
    bulk_load(smem + (size_t)slot * kLsSlotBytes, a.W + (size_t)vb * H, bytes, &T.full[slot], pol);
  };
  if (threadIdx.x == 0) {
    T.abort = 0;
    for (int i = 0; i < kLsPairs; ++i) {
      mbar_init(&T.full[i], 1);
      mbar_init(&T.empty[i], 2);
    }
    fence_mbar_init();
    const uint64_t pol = policy_evict_first();
    for (int s = 0; s < min(nst, kLsPairs); ++s) issue(s, pol);
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  block_copy_g2s(xs, reinterpret_cast<const uint4*>(a.x), K * H / 8);
  __syncthreads();
  if (a.norm_eps > 0.f) {
    for (int r = warp; r < K; r += kLsWarps) {
      float acc = 0.f;
      for (int j = 0; j < H / 256; ++j) {
        const uint4 xv = xs[r * (H / 8) + j * 32 + lane];
        const uint32_t q[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float f = (i & 1) ? lbf_hi(q[i >> 1]) : lbf_lo(q[i >> 1]);
          acc = __fmaf_rn(f, f, acc);
        }
      }
      acc = lsum_xor(acc);
      const float mean = __fdiv_rn(acc, (float)H);
      if (lane == 0) T.inv[r] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, a.norm_eps)));
    }
    __syncthreads();
    for (int i = threadIdx.x; i < K * H / 8; i += blockDim.x) {
      const float inv = T.inv[i / (H / 8)];
      uint4 v = xs[i];
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t lo = float_to_bf16_bits(__fmul_rn(lbf_lo(w[u]), inv));
        const uint32_t hi = float_to_bf16_bits(__fmul_rn(lbf_hi(w[u]), inv));
        w[u] = lo | (hi << 16);
      }
      xs[i] = v;
    }
    __syncthreads();
  }
  if constexpr (XF32) {
    // the rows to floats (exact), over the region's lower half: every thread
    // holds its pieces before any is overwritten
    const int n16 = K * H / 8;
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = threadIdx.x + u * (int)blockDim.x;
      if (i < n16) v[u] = xs[i];
    }
    __syncthreads();
    // layout [row][piece j][half][lane][4]: lane l's elements 256 j + 8 l + 0..3
    // and + 4..7 are each one float4, lanes of a half consecutive (no bank
    // conflict when a warp reads them)
    float4* xf = reinterpret_cast<float4*>(xreg);
    const int nj8 = H / 256;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = threadIdx.x + u * (int)blockDim.x;
      if (i < n16) {
        const int r = i / (H / 8), c = i - r * (H / 8);  // 16-byte piece c of row r
        const int j = c >> 5, l = c & 31;
        const int b = ((r * nj8 + j) * 2) * 32 + l;
        xf[b] = make_float4(lbf_lo(v[u].x), lbf_hi(v[u].x), lbf_lo(v[u].y), lbf_hi(v[u].y));
        xf[b + 32] = make_float4(lbf_lo(v[u].z), lbf_hi(v[u].z), lbf_lo(v[u].w), lbf_hi(v[u].w));
      }
    }
    __syncthreads();
  }

  float bv[KR];
  int bi[KR];
#pragma unroll
  for (int r = 0; r < KR; ++r) {
    bv[r] = -INFINITY;
    bi[r] = INT_MAX;
  }
  const int nj = H / 256;
  const int rpw = R / 2;  // rows per warp (<= 4)
  volatile int* abort = &T.abort;
  uint64_t pol = 0;
  if (hw == 0 && lane == 0) pol = policy_evict_first();
  int issued = (p < nst) ? 1 : 0;  // this slot's copies (lane 0 of the pair's first warp)
  for (int s = p, k = 0; s < nst; s += kLsPairs, ++k) {
    const uint32_t par = (uint32_t)k & 1u;
    bool ok = !*abort && mbar_wait_bounded(&T.full[p], par, a.wait_ns, abort);
    ok = __all_sync(0xffffffffu, ok);
    const int vb = v0 + s * R;
    const int nr = min(R, v1 - vb);
    float acc[RPW][KR];
#pragma unroll
    for (int q = 0; q < RPW; ++q)
#pragma unroll
      for (int r = 0; r < KR; ++r) acc[q][r] = 0.f;
    if (!ok) {
      *abort = 1;
    } else {
      const uint4* ws = reinterpret_cast<const uint4*>(smem + (size_t)p * kLsSlotBytes);
      const float4* xf4 = reinterpret_cast<const float4*>(xreg);
#pragma unroll
      for (int j = 0; j < 8; ++j) {  // H / 256 <= 8 pieces
        if (j >= nj) break;
        // this lane's 8 weights of each of the warp's rows, as floats
        float wf[RPW][8];
#pragma unroll
        for (int q = 0; q < RPW; ++q) {
          const int row = hw * rpw + q;
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (q < rpw && row < nr) v = ws[row * (H / 8) + j * 32 + lane];
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) wf[q][i] = (i & 1) ? lbf_hi(w4[i >> 1]) : lbf_lo(w4[i >> 1]);
        }
#pragma unroll
        for (int r = 0; r < KR; ++r) {
          if (r < K) {
            float xf[8];
            if constexpr (XF32) {  // x held as floats
              const float4 a0 = xf4[((r * nj + j) * 2) * 32 + lane];
              const float4 a1 = xf4[((r * nj + j) * 2 + 1) * 32 + lane];
              xf[0] = a0.x; xf[1] = a0.y; xf[2] = a0.z; xf[3] = a0.w;
              xf[4] = a1.x; xf[5] = a1.y; xf[6] = a1.z; xf[7] = a1.w;
            } else {
              const uint4 xv = xs[r * (H / 8) + j * 32 + lane];
              const uint32_t xq[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
              for (int i = 0; i < 8; ++i) xf[i] = (i & 1) ? lbf_hi(xq[i >> 1]) : lbf_lo(xq[i >> 1]);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
              for (int q = 0; q < RPW; ++q) acc[q][r] = __fmaf_rn(xf[i], wf[q][i], acc[q][r]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&T.empty[p]);
    if (hw == 0 && lane == 0 && s + kLsPairs < nst) {
      // refill this pair's slot once both warps have read it
      if (!*abort && mbar_wait_bounded(&T.empty[p], par, a.wait_ns, abort)) {
        issue(s + kLsPairs, pol);
        ++issued;
      } else {
        *abort = 1;
      }
    }
    __syncwarp();
    if (ok) {
#pragma unroll
      for (int q = 0; q < RPW; ++q) {
        const int row = hw * rpw + q;
        if (q < rpw && row < nr) {
#pragma unroll
          for (int r = 0; r < KR; ++r) {
            if (r < K) {
              const float l = lsum_xor(acc[q][r]);
              if (bi[r] == INT_MAX || l > bv[r]) {  // this warp's rows arrive in increasing order
                bv[r] = l;
                bi[r] = vb + row;
              }
            }
          }
        }
      }
    }
  }
  __syncthreads();
  if (*abort) {
    // no copy may land in a finished CTA; the ticket is still taken (the
    // tokens of this call are undefined, the next call starts clean)
    if (hw == 0 && lane == 0 && issued > 0) mbar_wait_drain(&T.full[p], (uint32_t)(issued - 1) & 1u, kLsDrainNs);
    if (threadIdx.x == 0 && a.err) atomicCAS(a.err, 0, (int)MOE_ERR_DEVICE_TIMEOUT);
  }
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < KR; ++r) {
      T.bv[warp][r] = bv[r];
      T.bi[warp][r] = bi[r];
    }
  }
  __syncthreads();
  if (threadIdx.x < K) {
    const int r = threadIdx.x;
    float b = -INFINITY;
    int i = INT_MAX;
    for (int w = 0; w < kLsWarps; ++w)
      if (T.bi[w][r] != INT_MAX && (i == INT_MAX || l_before(T.bv[w][r], T.bi[w][r], b, i))) {
        b = T.bv[w][r];
        i = T.bi[w][r];
      }
    a.part_v[blockIdx.x * K + r] = b;
    a.part_i[blockIdx.x * K + r] = i;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) T.last = (atomicAdd(a.ticket, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!T.last) return;
  __threadfence();
  if (threadIdx.x < K) {
    const int r = threadIdx.x;
    float b = -INFINITY;
    int i = INT_MAX;
    for (int c = 0; c < (int)gridDim.x; ++c) {
      const float cv = __ldcg(a.part_v + c * K + r);
      const int ci = __ldcg(a.part_i + c * K + r);
      if (ci != INT_MAX && (i == INT_MAX || l_before(cv, ci, b, i))) {
        b = cv;
        i = ci;
      }
    }
    a.tok[r] = i;
    if (a.best) a.best[r] = b;
  }
  if (threadIdx.x == 0) *a.ticket = 0u;
}

template <int KR>
static size_t lmhead_stream_smem_t(int K, int H) {
  return (size_t)LsShape<KR>::pairs * LsShape<KR>::slot + (size_t)K * H * (LsShape<KR>::xf32 ? 4 : 2) +
         sizeof(LsTable);
}

static size_t lmhead_stream_smem(int K, int H) {
  return K <= 4 ? lmhead_stream_smem_t<4>(K, H) : K <= 8 ? lmhead_stream_smem_t<8>(K, H) : lmhead_stream_smem_t<16>(K, H);
}

bool lmhead_stream_fits(int K, int H) {
  return K <= 16 && H % 256 == 0 && H <= 8192 && lmhead_stream_smem(K, H) <= 227 * 1024;
}

cudaError_t launch_lmhead_stream(const LmHeadArgs& a0, cudaStream_t s, bool pdl) {
  auto run = [&](auto kern, int pairs, int slot, int rpw) {
    LmHeadArgs a = a0;
    a.rows_per_stage = slot / (2 * a.H) < 2 * rpw ? slot / (2 * a.H) : 2 * rpw;
    const size_t sm = lmhead_stream_smem(a.K, a.H);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e == cudaSuccess) e = max_carveout(kern);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms());
    cfg.blockDim = dim3(2 * pairs * 32);
    cfg.dynamicSmemBytes = sm;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
  };
  if (a0.K <= 4) return run(k_lmhead_stream<4>, LsShape<4>::pairs, LsShape<4>::slot, LsShape<4>::rpw);
  if (a0.K <= 8) return run(k_lmhead_stream<8>, LsShape<8>::pairs, LsShape<8>::slot, LsShape<8>::rpw);
  return run(k_lmhead_stream<16>, LsShape<16>::pairs, LsShape<16>::slot, LsShape<16>::rpw);
}

}  // namespace moe
