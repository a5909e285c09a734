// attention.cu -- the GQA attention block of the full verify step.
//
// K verify rows attend over a cache of C positions plus their own K new
// positions (row r sees new positions 0..r), grouped-query with `group` query
// heads per KV head, head dim 128 (README, "Why this challenge exists": all
// layers are GQA with 8 KV heads at head_dim 128).  The block is
//   x_out = bf16( x + bf16(softmax(q k^T / sqrt(128)) v) . Wo^T ),
//   q, k_new, v_new = bf16( rmsnorm(x) . W{q,k,v}^T ).
//
// Kernels:
//  * k_gemv_bf16   -- bf16 GEMV for up to three weight matrices sharing x
//                     (one warp per output row, 16-byte loads, FP32 accumulate,
//                     optional residual add, bf16 output).
//  * k_attn_split  -- flash-decode over the cache: CTA (split, kv head) walks
//                     16-position sub-chunks with tensor-core mma.sync (bf16 in,
//                     FP32 accumulate) for q k^T and p v, online softmax in the
//                     log2 domain, and writes its unnormalised partial
//                     (m, l, o).  The K rows x `group` heads of a KV head form
//                     the 16 query rows of one m16 tile.  Fragments come
//                     straight from global memory with 16-byte loads: the
//                     reduction index (head dim for q k^T, position for p v)
//                     and the output dims are permuted so that each thread's
//                     elements are contiguous in memory.
//  * k_attn_combine-- merges the splits in fixed order with the block-causal
//                     new positions and normalises.
#include <cfloat>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ uint4 ldg_v4(const void* p) { return *reinterpret_cast<const uint4*>(p); }

}  // namespace

// ------------------------------------------------------------------ bf16 GEMV
// One warp per output row; the reduction runs over D in chunks of 2048 (8
// pieces of 256 per lane, 16-byte loads), so D may be any multiple of 256
// that the staged rows fit in shared memory.
template <int KR>
__global__ void __launch_bounds__(256) k_gemv_bf16(GemvArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = a.K, D = a.D, nj = D / 256;
  pdl_wait();
  pdl_launch_dependents();
  uint4* xs = reinterpret_cast<uint4*>(smem);
  block_copy_g2s(xs, reinterpret_cast<const uint4*>(a.x), K * D / 8);
  __syncthreads();
  const int nw = gridDim.x * (blockDim.x >> 5);
  // row n of the concatenated segments: segment and local row
  auto locate = [&](int n, int& sg, int& nl) {
    sg = 0;
    nl = n;
    while (sg + 1 < a.nseg && nl >= a.seg[sg].N) {
      nl -= a.seg[sg].N;
      ++sg;
    }
  };
  for (int n = blockIdx.x * (blockDim.x >> 5) + warp; n < a.n_total; n += nw) {
    int sg, nl;
    locate(n, sg, nl);
    const GemvSeg& S = a.seg[sg];
    const uint4* wrow = reinterpret_cast<const uint4*>(S.W + (size_t)nl * D);
    // lane r < K: row r's residual, issued with the weights
    const float resv = (S.res && lane < K) ? bf_lo(S.res[(size_t)lane * S.N + nl]) : 0.f;
    float acc[KR];
#pragma unroll
    for (int r = 0; r < KR; ++r) acc[r] = 0.f;
    for (int j0 = 0; j0 < nj; j0 += 8) {
      uint4 wv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j0 + j < nj) wv[j] = ldg_nc_v4(wrow + (j0 + j) * 32 + lane);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j0 + j >= nj) break;
        const uint32_t wq[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
#pragma unroll
        for (int r = 0; r < KR; ++r) {
          if (r < K) {
            const uint4 xv = xs[r * (D / 8) + (j0 + j) * 32 + lane];
            const uint32_t xq[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              acc[r] = __fmaf_rn(bf_lo(xq[i]), bf_lo(wq[i]), acc[r]);
              acc[r] = __fmaf_rn(bf_hi(xq[i]), bf_hi(wq[i]), acc[r]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < KR; ++r) {
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], d);
    }
#pragma unroll
    for (int r = 0; r < KR; ++r) {
      if (r < K && lane == r) {
        float v = acc[r];
        if (S.res) v += resv;
        const uint16_t b = float_to_bf16_bits(v);
        S.out[(size_t)r * S.N + nl] = b;
        if (S.cache) {  // in-place KV append at position *len + r
          const int p = *S.len + r;
          if (p < S.cap) S.cache[((size_t)(nl >> 7) * S.cap + p) * 128 + (nl & 127)] = b;
          else if (a.err) atomicCAS(a.err, 0, (int)MOE_ERR_CAPACITY);
        }
      }
    }
  }
}

template <typename Kern, typename Args>
static cudaError_t launch_rows_kernel(Kern kern, const Args& a, size_t sm, cudaStream_t s, bool pdl) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e == cudaSuccess) e = max_carveout(kern);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * num_sms());
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t s, bool pdl) {
  if (gemv_stream_fits(a, num_sms())) return launch_gemv_stream(a, s, pdl);
  if (a.norm_eps > 0.f) return cudaErrorInvalidValue;  // the row kernel takes normalised rows only
  const size_t sm = sizeof(uint16_t) * a.K * a.D;
  if (a.K <= 4) return launch_rows_kernel(k_gemv_bf16<4>, a, sm, s, pdl);
  if (a.K <= 8) return launch_rows_kernel(k_gemv_bf16<8>, a, sm, s, pdl);
  return launch_rows_kernel(k_gemv_bf16<16>, a, sm, s, pdl);
}

// ------------------------------------------------------------------ dense SwiGLU rows
// One warp per intermediate row i: the gate and up rows' dot products with
// every staged row x_r (the GEMV's order), then h = bf16(silu(g) * u).
template <int KR>
__global__ void __launch_bounds__(256) k_swiglu_rows(SwigluArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = a.K, D = a.D, nj = D / 256;
  pdl_wait();
  pdl_launch_dependents();
  uint4* xs = reinterpret_cast<uint4*>(smem);
  block_copy_g2s(xs, reinterpret_cast<const uint4*>(a.x), K * D / 8);
  __syncthreads();
  const int nw = gridDim.x * (blockDim.x >> 5);
  for (int n = blockIdx.x * (blockDim.x >> 5) + warp; n < a.N; n += nw) {
    const uint4* grow = reinterpret_cast<const uint4*>(a.Wg + (size_t)n * D);
    const uint4* urow = reinterpret_cast<const uint4*>(a.Wu + (size_t)n * D);
    float ag[KR], au[KR];
#pragma unroll
    for (int r = 0; r < KR; ++r) ag[r] = au[r] = 0.f;
    for (int j0 = 0; j0 < nj; j0 += 4) {
      uint4 gv[4], uv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j0 + j < nj) {
          gv[j] = ldg_nc_v4(grow + (j0 + j) * 32 + lane);
          uv[j] = ldg_nc_v4(urow + (j0 + j) * 32 + lane);
        }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j0 + j >= nj) break;
        const uint32_t gq[4] = {gv[j].x, gv[j].y, gv[j].z, gv[j].w};
        const uint32_t uq[4] = {uv[j].x, uv[j].y, uv[j].z, uv[j].w};
#pragma unroll
        for (int r = 0; r < KR; ++r) {
          if (r < K) {
            const uint4 xv = xs[r * (D / 8) + (j0 + j) * 32 + lane];
            const uint32_t xq[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              ag[r] = __fmaf_rn(bf_lo(xq[i]), bf_lo(gq[i]), ag[r]);
              ag[r] = __fmaf_rn(bf_hi(xq[i]), bf_hi(gq[i]), ag[r]);
              au[r] = __fmaf_rn(bf_lo(xq[i]), bf_lo(uq[i]), au[r]);
              au[r] = __fmaf_rn(bf_hi(xq[i]), bf_hi(uq[i]), au[r]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < KR; ++r) {
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) {
        ag[r] += __shfl_xor_sync(0xffffffffu, ag[r], d);
        au[r] += __shfl_xor_sync(0xffffffffu, au[r], d);
      }
      if (r < K && lane == r) a.h[(size_t)r * a.N + n] = float_to_bf16_bits(ag[r] * __frcp_rn(1.f + expf(-ag[r])) * au[r]);
    }
  }
}

cudaError_t launch_swiglu(const SwigluArgs& a, cudaStream_t s, bool pdl) {
  const size_t sm = sizeof(uint16_t) * a.K * a.D;
  if (a.K <= 4) return launch_rows_kernel(k_swiglu_rows<4>, a, sm, s, pdl);
  if (a.K <= 8) return launch_rows_kernel(k_swiglu_rows<8>, a, sm, s, pdl);
  return launch_rows_kernel(k_swiglu_rows<16>, a, sm, s, pdl);
}

// ------------------------------------------------------------------ rotary embedding
// For shapes the streamed projection cannot rotate in its epilogue.
// Grid (K, units / 4): CTA (r, j) serves row r.  Its threads first take the
// rd/2 angles (pos0 + r) * freq[i] of that row and their cosines and sines
// (rope_cs, as the projection's epilogue does).  Then each warp takes one unit of the row: a q head, a k
// head or (with caches given) a v head.  For a q or k head, lane l rotates
// the pairs (v[i], v[i + rd/2]) with i = l, l + 32 in FP32 and rounds to
// bf16, in place; a k head's warp then writes its whole rotated head to
// the key cache at position pos0 + r, and a v head's warp copies the value
// head to the value cache (both bounded by the capacity).  No warp reads
// what another one writes.
constexpr int kRopeWarps = 4;

__global__ void __launch_bounds__(kRopeWarps * 32) k_rope(RopeArgs a) {
  __shared__ float s_cos[64], s_sin[64];
  pdl_wait();
  pdl_launch_dependents();
  const int r = blockIdx.x;
  const int half = a.rd / 2;
  const int pos0 = a.len ? *a.len : a.C;
  const int p = pos0 + r;
  for (int i = threadIdx.x; i < half; i += blockDim.x) rope_cs(p, a.freq[i], s_cos[i], s_sin[i]);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.y * kRopeWarps + warp;
  const int nunit = a.nq + a.nkv + (a.kc ? a.nkv : 0);
  if (u >= nunit) return;
  const bool room = p < a.C;
  if (a.kc && !room && u == 0 && lane == 0 && a.err) atomicCAS(a.err, 0, (int)MOE_ERR_CAPACITY);
  if (u >= a.nq + a.nkv) {  // value head: cache append only
    if (!room) return;
    const int kvh = u - a.nq - a.nkv;
    const uint16_t* src = a.v + ((size_t)r * a.nkv + kvh) * 128;
    uint16_t* dst = a.vc + ((size_t)kvh * a.C + p) * 128;
    for (int d = lane; d < 128; d += 32) dst[d] = src[d];
    return;
  }
  const bool isk = u >= a.nq;
  const int kvh = u - a.nq;
  uint16_t* base = isk ? a.k + ((size_t)r * a.nkv + kvh) * 128 : a.q + ((size_t)r * a.nq + u) * 128;
  uint16_t* dst = (isk && a.kc && room) ? a.kc + ((size_t)kvh * a.C + p) * 128 : nullptr;
  for (int i = lane; i < half; i += 32) {
    const float x0 = bf16_bits_to_float(base[i]), x1 = bf16_bits_to_float(base[i + half]);
    const float c = s_cos[i], s = s_sin[i];
    const uint16_t y0 = float_to_bf16_bits(__fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s)));
    const uint16_t y1 = float_to_bf16_bits(__fadd_rn(__fmul_rn(x1, c), __fmul_rn(x0, s)));
    base[i] = y0;
    base[i + half] = y1;
    if (dst) {
      dst[i] = y0;
      dst[i + half] = y1;
    }
  }
  if (dst)  // the dims past the rotary ones, unchanged
    for (int d = a.rd + lane; d < 128; d += 32) dst[d] = base[d];
}

cudaError_t launch_rope(const RopeArgs& a, cudaStream_t s) {
  const int nunit = a.nq + a.nkv + (a.kc ? a.nkv : 0);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.K, (nunit + kRopeWarps - 1) / kRopeWarps);
  cfg.blockDim = dim3(kRopeWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  max_carveout(k_rope);
  return cudaLaunchKernelEx(&cfg, k_rope, a);
}

// ------------------------------------------------------------------ split-KV attention
// Query row i of the m16 tile = r * group + hh (r < K, hh < group); rows
// past K * group are zero.  Physical layout of a 16-position sub-chunk as
// seen by the fragments: logical position 2t+b <-> physical 4t+b and
// 2t+8+b <-> 4t+2+b (b = 0, 1), so each thread's four positions of the
// p v step are consecutive; logical output dim (n-block nb, column c) <->
// physical dim 16*c + nb, so each thread's V columns are 16 consecutive dims.
constexpr int kAttnWarps = 4;

__global__ void __launch_bounds__(kAttnWarps * 32) k_attn_split(AttnArgs a) {
  __shared__ float s_m[kAttnWarps][16], s_l[kAttnWarps][16];
  __shared__ float s_o[kAttnWarps][16][129];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int kvh = blockIdx.y, split = blockIdx.x, tile = blockIdx.z;
  const int HD = 128;
  pdl_wait();
  pdl_launch_dependents();

  // Q fragments: thread t holds head dims [32t, 32t+32) of the tile's rows g
  // and g+8 (query rows 16 tile + g, + 8 of the KV head)
  uint32_t qa[8][4];
  const int nrow = a.K * a.group;
  {
    uint4 rg[4], rh[4];
#pragma unroll
    for (int hrow = 0; hrow < 2; ++hrow) {
      const int i = 16 * tile + g + 8 * hrow;
      uint4* dst = hrow ? rh : rg;
      if (i < nrow) {
        const int r = i / a.group, hh = i % a.group;
        const uint16_t* src = a.q + (size_t)r * a.nq * HD + (size_t)(kvh * a.group + hh) * HD + 32 * t;
#pragma unroll
        for (int u = 0; u < 4; ++u) dst[u] = ldg_v4(src + 8 * u);
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) dst[u] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t* wg = reinterpret_cast<const uint32_t*>(&rg[ks >> 1]);
      const uint32_t* wh = reinterpret_cast<const uint32_t*>(&rh[ks >> 1]);
      const int w0 = (ks & 1) * 2;
      qa[ks][0] = wg[w0];
      qa[ks][1] = wh[w0];
      qa[ks][2] = wg[w0 + 1];
      qa[ks][3] = wh[w0 + 1];
    }
  }

  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int nb = 0; nb < 16; ++nb)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[nb][c] = 0.f;

  // Cv valid positions of a cache of a.C (the head stride); a partial last
  // 16-position sub-chunk is masked (its keys and values read as zero, its
  // scores as -inf).  With a window W, query row i (verify row r = i / group,
  // at position Cv + r) sees the cached positions from Cv + r - W + 1 on:
  // the splits walk the sub-chunks from the lowest row's start, and scores
  // before a row's own start are masked.
  const int Cv = a.len ? min(*a.len, a.C) : a.C;
  const int n16 = (Cv + 15) / 16;
  const int lo = a.window > 0 ? max(0, Cv - a.window + 1) : 0;
  const int s16 = lo / 16;
  const int c0 = s16 + (int)(((long long)split * (n16 - s16)) / gridDim.x);
  const int c1 = s16 + (int)(((long long)(split + 1) * (n16 - s16)) / gridDim.x);
  // the window start of this thread's two score rows (g and g + 8 of the tile)
  int rs[2] = {0, 0};
  if (a.window > 0) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = 16 * tile + g + 8 * hr;
      rs[hr] = Cv + (i < nrow ? i / a.group : 0) - a.window + 1;
    }
  }
  const int rs_max = max(rs[0], rs[1]);
  const uint16_t* kbase = a.kc + (size_t)kvh * a.C * HD;
  const uint16_t* vbase = a.vc + (size_t)kvh * a.C * HD;
  const int pk0 = 4 * (g >> 1) + (g & 1);  // physical row of logical column g (n-block 0); +2 for n-block 1

  for (int sc = c0 + warp; sc < c1; sc += kAttnWarps) {
    const uint16_t* kb = kbase + (size_t)sc * 16 * HD;
    const uint16_t* vb = vbase + (size_t)sc * 16 * HD;
    const int rem = Cv - sc * 16;  // valid positions of this sub-chunk (16 unless it is the last)
    uint4 kr[2][4], vr[4][2];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        kr[nb][u] = pk0 + 2 * nb < rem ? ldg_nc_v4(kb + (size_t)(pk0 + 2 * nb) * HD + 32 * t + 8 * u)
                                       : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
      for (int u = 0; u < 2; ++u)
        vr[p][u] = 4 * t + p < rem ? ldg_nc_v4(vb + (size_t)(4 * t + p) * HD + 16 * g + 8 * u)
                                   : make_uint4(0, 0, 0, 0);

    float s[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
      for (int c = 0; c < 4; ++c) s[nb][c] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(&kr[nb][ks >> 1]);
        const int w0 = (ks & 1) * 2;
        mma_bf16(s[nb], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], w[w0], w[w0 + 1]);
      }
    }
    if (rem < 16 || sc * 16 < rs_max) {
      // score (row g + 8 (c >> 1), logical column 8 nb + 2t + b) sits at
      // physical position 4t + 2nb + b
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int pp = 4 * t + 2 * nb + (c & 1);
          if (pp >= rem || sc * 16 + pp < rs[c >> 1]) s[nb][c] = -INFINITY;
        }
    }
    // online softmax (log2 domain); row 0 = query g, row 1 = query g+8
    float mx[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      float v = -INFINITY;
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        s[nb][2 * hr] *= a.scale_log2;
        s[nb][2 * hr + 1] *= a.scale_log2;
        v = fmaxf(v, fmaxf(s[nb][2 * hr], s[nb][2 * hr + 1]));
      }
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
      mx[hr] = fmaxf(m[hr], v);
      const float alpha = exp2f(m[hr] - mx[hr]);
      m[hr] = mx[hr];
      l[hr] *= alpha;
#pragma unroll
      for (int nb = 0; nb < 16; ++nb) {
        o[nb][2 * hr] *= alpha;
        o[nb][2 * hr + 1] *= alpha;
      }
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        s[nb][2 * hr] = exp2f(s[nb][2 * hr] - mx[hr]);
        s[nb][2 * hr + 1] = exp2f(s[nb][2 * hr + 1] - mx[hr]);
        l[hr] += s[nb][2 * hr] + s[nb][2 * hr + 1];
      }
    }
    // P as the A operand (k = 16 logical positions)
    const uint32_t pa0 = pack_bf16x2(s[0][0], s[0][1]);
    const uint32_t pa1 = pack_bf16x2(s[0][2], s[0][3]);
    const uint32_t pa2 = pack_bf16x2(s[1][0], s[1][1]);
    const uint32_t pa3 = pack_bf16x2(s[1][2], s[1][3]);
    // V as B: k = logical positions (2t, 2t+1 | 2t+8, 2t+9) = physical rows
    // 4t, 4t+1 | 4t+2, 4t+3; n = logical dim (nb, g) = physical dim 16g + nb
    const uint32_t* v0 = reinterpret_cast<const uint32_t*>(vr[0]);
    const uint32_t* v1 = reinterpret_cast<const uint32_t*>(vr[1]);
    const uint32_t* v2 = reinterpret_cast<const uint32_t*>(vr[2]);
    const uint32_t* v3 = reinterpret_cast<const uint32_t*>(vr[3]);
#pragma unroll
    for (int nb = 0; nb < 16; ++nb) {
      const int wi = nb >> 1;
      const uint32_t sel = (nb & 1) ? 0x7632u : 0x5410u;  // high or low halves
      const uint32_t b0 = __byte_perm(v0[wi], v1[wi], sel);
      const uint32_t b1 = __byte_perm(v2[wi], v3[wi], sel);
      mma_bf16(o[nb], pa0, pa1, pa2, pa3, b0, b1);
    }
  }

  // per-warp row sums, then merge the warps in fixed order
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 1);
    l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 2);
  }
  if (t == 0) {
    s_m[warp][g] = m[0];
    s_m[warp][g + 8] = m[1];
    s_l[warp][g] = l[0];
    s_l[warp][g + 8] = l[1];
  }
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) {
    s_o[warp][g][16 * (2 * t) + nb] = o[nb][0];
    s_o[warp][g][16 * (2 * t + 1) + nb] = o[nb][1];
    s_o[warp][g + 8][16 * (2 * t) + nb] = o[nb][2];
    s_o[warp][g + 8][16 * (2 * t + 1) + nb] = o[nb][3];
  }
  __syncthreads();
  const int d = threadIdx.x;  // 128 threads = head dims
  const int TR = a.tiles * 16;  // query rows per KV head in the partial buffers
  float* po = a.part_o + ((size_t)(kvh * gridDim.x + split) * TR + 16 * tile) * HD;
  float* pml = a.part_ml + ((size_t)(kvh * gridDim.x + split) * TR + 16 * tile) * 2;
  for (int i = 0; i < 16; ++i) {
    float M = -INFINITY;
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, s_m[w][i]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kAttnWarps; ++w) {
        const float f = exp2f(s_m[w][i] - M);
        L += s_l[w][i] * f;
        O += s_o[w][i][d] * f;
      }
    }
    po[i * HD + d] = O;
    if (d == 0) {
      pml[2 * i] = M;
      pml[2 * i + 1] = L;
    }
  }
}

// One CTA per (query head h, row r); 128 threads = head dims.  Merges the
// splits of KV head h/group in split order with the row's visible new
// positions 0..r and writes o = bf16(O / L).  Every global load is issued up
// front (every warp: the splits' maxima and sums; every thread: its dim of
// the splits' outputs, q and the new keys and values).  Every warp forms the
// split weights exp2(m_s - Ms) with shuffles and each thread accumulates its
// dim over the splits at once (so the loads are consumed as they land); the
// new positions then join with the usual rescaling to the row's maximum.
// The dependent kernel (the o-projection, which reads only its weights
// before its own wait) is released at once.
template <int MAXS>
__global__ void __launch_bounds__(128) k_attn_combine(AttnArgs a, int splits) {
  __shared__ float s_red[4][16];
  const int h = blockIdx.x, r = blockIdx.y, d = threadIdx.x;
  const int warp = d >> 5, lane = d & 31;
  const int HD = 128, kvh = h / a.group, hh = h % a.group;
  const int i = r * a.group + hh;
  pdl_launch_dependents();
  pdl_wait();
  const int TR = a.tiles * 16;
  const float* pml = a.part_ml + (size_t)kvh * splits * TR * 2 + 2 * i;
  const float* po = a.part_o + ((size_t)kvh * splits * TR + i) * HD + d;
  // every load first: lane s of every warp the (m, l) of splits s and s + 32,
  // every thread its dim of the splits' outputs, q, the new keys and values
  float ms[2] = {-INFINITY, -INFINITY}, ls[2] = {0.f, 0.f};
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int sp = lane + 32 * u;
    if (sp < splits) {
      ms[u] = __ldcg(pml + (size_t)sp * TR * 2);
      ls[u] = __ldcg(pml + (size_t)sp * TR * 2 + 1);
    }
  }
  float ov[MAXS / 32][32];  // this thread's split outputs (splits <= MAXS)
#pragma unroll
  for (int c = 0; c < MAXS / 32; ++c)
#pragma unroll
    for (int u = 0; u < 32; ++u) ov[c][u] = 32 * c + u < splits ? __ldcg(po + (size_t)(32 * c + u) * TR * HD) : 0.f;
  const float qd = bf_lo(a.q[(size_t)r * a.nq * HD + (size_t)h * HD + d]);
  float kd[16], vd[16];  // the new positions j <= r (r < K <= 16)
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    kd[j] = vd[j] = 0.f;
    if (j <= r) {
      kd[j] = bf_lo(a.k_new[(size_t)j * a.nkv * HD + (size_t)kvh * HD + d]);
      vd[j] = bf_lo(a.v_new[(size_t)j * a.nkv * HD + (size_t)kvh * HD + d]);
    }
  }
  // the splits, in every warp alike: Ms = max m_s (xor rounds), weights
  // f_s = exp2(m_s - Ms) (0 for an empty split), Ls = sum l_s f_s (xor
  // rounds), and this thread's Os = sum over s in order of f_s O_s
  float Ms = fmaxf(ms[0], ms[1]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) Ms = fmaxf(Ms, __shfl_xor_sync(0xffffffffu, Ms, o));
  float f[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) f[u] = ms[u] == -INFINITY ? 0.f : exp2f(ms[u] - Ms);
  float Ls = f[0] * ls[0] + f[1] * ls[1];
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
  float Os = 0.f;
#pragma unroll
  for (int c = 0; c < MAXS / 32; ++c)
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const int s = 32 * c + u;
      const float fs = __shfl_sync(0xffffffffu, f[c < 2 ? c : 1], u);
      if (s < splits) Os += ov[c][u] * fs;
    }
  // scores of the new positions (log2 domain): per warp a xor sum, then the
  // four warps in a fixed order
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j > r) break;
    float p = qd * kd[j];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
    if (lane == 0) s_red[warp][j] = p;
  }
  __syncthreads();
  float sc[16];
  float M = Ms;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    sc[j] = -INFINITY;
    if (j <= r) {
      sc[j] = ((s_red[0][j] + s_red[1][j]) + (s_red[2][j] + s_red[3][j])) * a.scale_log2;
      M = fmaxf(M, sc[j]);
    }
  }
  // the splits' sums rescaled to the row's maximum, then the new positions
  // in order 0..r
  const float cs = Ms == -INFINITY ? 0.f : exp2f(Ms - M);
  float O = Os * cs, L = Ls * cs;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j > r) break;
    const float fj = exp2f(sc[j] - M);
    L += fj;
    O += fj * vd[j];
  }
  a.o[(size_t)r * a.nq * HD + (size_t)h * HD + d] = float_to_bf16_bits(O / L);
}

// Splits per (KV head, tile): about two CTAs per SM in all, no more than
// there are 16-position sub-chunks to walk.
int attn_splits(int nkv, int tiles, int max_chunks) {
  int s = (2 * num_sms() + nkv * tiles - 1) / (nkv * tiles);
  if (s > max_chunks) s = max_chunks;
  return s < 1 ? 1 : (s > kAttnMaxSplits ? kAttnMaxSplits : s);
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s, bool pdl) {
  const int chunks = (a.window > 0 ? (a.window + 31) / 16 : (a.C + 15) / 16);
  const int splits = attn_splits(a.nkv, a.tiles, chunks);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(splits, a.nkv, a.tiles);
  cfg.blockDim = dim3(kAttnWarps * 32);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  max_carveout(k_attn_split);
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_attn_split, a);
  if (e != cudaSuccess) return e;
  return launch_attn_combine(a, splits, s);
}

cudaError_t launch_attn_combine(const AttnArgs& a, int splits, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nq, a.K);
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // at most 32 splits: a smaller register footprint, so a merge CTA fits on
  // an SM beside the attention and the o-projection CTAs
  if (splits <= 32) {
    max_carveout(k_attn_combine<32>);
    return cudaLaunchKernelEx(&cfg, k_attn_combine<32>, a, splits);
  }
  max_carveout(k_attn_combine<64>);
  return cudaLaunchKernelEx(&cfg, k_attn_combine<64>, a, splits);
}

}  // namespace moe
