// gemv.cu -- streamed bf16 GEMV for the projections around attention:
//   out[r][n] = bf16( sum_c x[r][c] * W[n][c]  (+ res[r][n]) ),   r < K <= 16,
// for up to three weight matrices that share x (q, k, v), laid end to end
// as one list of output rows; optionally x is first RMS-normalised.
//
// One CTA per SM.  CTA b owns a contiguous range of output rows and streams
// exactly those weight rows -- each byte once -- through a ring of shared-
// memory stages filled by bulk copies.  The weights do not depend on the
// previous kernel, so the first ring-full is issued before the dependency
// wait and lands while that kernel finishes.
//
// The CTA's rows are cut into groups of up to 8 consecutive rows of one
// matrix, and each group into D / 2048 column blocks: a stage holds one
// block of one group (8 x 4 KB; rows 4160 bytes apart in shared memory, so
// that a warp's reads of the 8 rows fall on all 32 banks).  The 16 warps
// split the reduction dimension: warp w owns columns [128 w, 128 w + 128)
// of every block and keeps its fragments of x in registers for the whole
// kernel.  Per stage and 16-column step a warp issues one mma.sync m16n8k16
// (A = the K rows of x, B = the group's rows as the n dimension, FP32
// accumulate) into the group's accumulators.  After the last stage the 16
// warps' partial sums of each output are added in warp order.
//
// Column order inside a warp's 32-column pieces: thread t of a quad reads
// the 8 consecutive columns [8t, 8t+8).  Its first four are its logical
// k = 2t, 2t+1, 2t+8, 2t+9 of the piece's even 16-column step, the last four
// those of the odd step.  x and W use the same order, so every product is
// x[r][c] * W[n][c]; only the order of the FP32 sum differs from a plain
// dot product.
//
// Two epilogues pair rows that the walk keeps in one CTA (rows split in
// units of 16, two 8-row groups each): the rotary embedding of the q and k
// heads (rows i and i + rd/2 of a head) and SwiGLU (gate row n and up row
// n), both formed from the two groups' outputs before anything is stored.
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kGsWarps = 16;
constexpr int kGsStages = 6;
constexpr int kGsRows = 8;                 // rows per group (the mma's n dimension)
constexpr int kGsCols = 2048;              // columns per block: 4 KB of a row
constexpr int kGsPitch = kGsCols * 2 + 64; // bytes between a stage's rows
constexpr int kGsStageBytes = kGsRows * kGsPitch;
constexpr int kGsMaxGroups = 16;  // row groups per CTA (one accumulator set each), at most
constexpr int kGsTail = 1024;     // barriers and the group table after the ring
// Bound on waiting for the CTA's own copies before it exits (independent of
// the caller's wait limit, which may be 0 in a test of the give-up path).
constexpr uint64_t kGsDrainNs = 2000000000ull;
// Accumulator sets (row groups) of an instantiation: x's fragments take
// KPW * 2 * KH registers, so the narrow ones have room for more sets.
constexpr int gs_max_groups(int kpw, int kh) {
  return kpw * kh <= 8 ? 16 : (kpw * kh <= 16 ? 12 : (kpw <= 16 ? 8 : 4));
}

__device__ __forceinline__ float bfl(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bfh(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void mma_bf16_gs(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16(x * inv) of both halves of a bf16 pair.
__device__ __forceinline__ uint32_t scale_pair(uint32_t w, float inv) {
  const uint32_t lo = float_to_bf16_bits(__fmul_rn(bfl(w), inv));
  const uint32_t hi = float_to_bf16_bits(__fmul_rn(bfh(w), inv));
  return lo | (hi << 16);
}

struct GsTable {
  uint64_t full[kGsStages];
  uint64_t empty[kGsStages];
  int seg[kGsMaxGroups], row[kGsMaxGroups], n[kGsMaxGroups];
  int pair[kGsMaxGroups];  // rotary embedding: 1 the first rows of a pair (the next group the second), 2 the second
  int ng;
  int abort;
  float inv[16];
};
static_assert(sizeof(GsTable) <= kGsTail, "group table");
// the partial sums of every group fit the ring once it is free
static_assert(kGsMaxGroups * kGsWarps * 128 * 4 <= kGsStages * kGsStageBytes, "reduction area");
static_assert(kGsPitch % 16 == 0 && kGsStageBytes % 16 == 0, "bulk copy alignment");

}  // namespace

template <int KPW, int KH, int NG>
__global__ void __launch_bounds__(kGsWarps * 32, 1) k_gemv_stream(const __grid_constant__ GemvArgs a) {
  static_assert(NG <= kGsMaxGroups && KPW % 8 == 0, "accumulator sets, column blocks");
  constexpr int NCB = KPW / 8;  // column blocks of 2048
  extern __shared__ __align__(1024) unsigned char smem[];
  GsTable& T = *reinterpret_cast<GsTable*>(smem + kGsStages * kGsStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int D = a.D, K = a.K;
  int issued = 0;  // warp 0: stages whose copies were issued
  uint64_t pol = 0;

  // stage s = block s % NCB of group s / NCB, issued by warp 0: lane 0 posts
  // the stage's bytes, then lane i copies row i (4 KB)
  auto issue = [&](int s) {
    const int slot = s % kGsStages, gr = s / NCB, cb = s - gr * NCB;
    const int nr = T.n[gr];
    if (lane == 0) mbar_arrive_expect_tx(&T.full[slot], (uint32_t)nr * (kGsCols * 2));
    __syncwarp();
    if (lane < nr)
      bulk_load(smem + (size_t)slot * kGsStageBytes + (size_t)lane * kGsPitch,
                a.seg[T.seg[gr]].W + (size_t)(T.row[gr] + lane) * D + (size_t)cb * kGsCols, kGsCols * 2,
                &T.full[slot], pol);
  };

  if (threadIdx.x == 0) {
    // this CTA's output rows [r0, r1), cut into groups at matrix ends.  With
    // the rotary embedding the rows are split in units of 16 and a rope
    // matrix's head is walked in the order 0-7, h-(h+7), 8-15, (h+8)-(h+15),
    // ... (h = rope_rd / 2), then the rows past rope_rd: the two groups of a
    // rotation pair are consecutive in one CTA.
    const int unit = (a.rope_rd || a.glu) ? 16 : 1, nu = a.n_total / unit;
    const int r0 = (int)((long long)blockIdx.x * nu / gridDim.x) * unit;
    const int r1 = (int)((long long)(blockIdx.x + 1) * nu / gridDim.x) * unit;
    int ng = 0, cur = r0, base = 0, sg = 0;
    T.abort = 0;
    while (cur < r1) {
      if (ng == NG) {  // more groups than accumulator sets: refused by the launcher
        T.abort = 1;
        break;
      }
      if (a.glu) {  // unit u: gate rows 8u .. 8u + 7, then the same up rows
        const int up = (cur >> 3) & 1;
        T.seg[ng] = up;
        T.row[ng] = (cur >> 4) * 8;
        T.n[ng] = kGsRows;
        T.pair[ng] = 1 + up;
        ++ng;
        cur += kGsRows;
        continue;
      }
      while (cur >= base + a.seg[sg].N) base += a.seg[sg++].N;
      const int nr = min(kGsRows, min(r1, base + a.seg[sg].N) - cur);
      int row = cur - base, pair = 0;
      if (a.rope_rd && a.seg[sg].rope) {
        const int v = row & 127;
        if (v < a.rope_rd) {
          pair = 1 + ((v >> 3) & 1);
          row = row - v + (pair == 2 ? a.rope_rd / 2 : 0) + 8 * (v >> 4);
        }
      }
      T.seg[ng] = sg;
      T.row[ng] = row;
      T.n[ng] = nr;
      T.pair[ng] = pair;
      ++ng;
      cur += nr;
    }
    T.ng = T.abort ? 0 : ng;
    for (int i = 0; i < kGsStages; ++i) {
      mbar_init(&T.full[i], 1);
      mbar_init(&T.empty[i], kGsWarps);
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    __syncwarp();
    pol = policy_evict_first();
    const int first = min(T.ng * NCB, kGsStages);
    for (; issued < first; ++issued) issue(issued);
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  if (T.abort && threadIdx.x == 0 && a.err) atomicCAS(a.err, 0, (int)MOE_ERR_UNSUPPORTED_SHAPE);

  // x fragments of this warp's columns, piece p (32 columns) at column
  // 2048 (p / 4) + 128 warp + 32 (p % 4) + 8t: xa[2p], xa[2p + 1] hold
  // [0], [1] = a0, a2 (row g) and [2], [3] = a1, a3 (row g + 8)
  const int cw = warp * 128 + 8 * t;
  uint32_t xa[KPW][2 * KH];
#pragma unroll
  for (int p = 0; p < KPW / 2; ++p)
#pragma unroll
    for (int h = 0; h < KH; ++h) {
      const int r = g + 8 * h;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < K) v = *reinterpret_cast<const uint4*>(a.x + (size_t)r * D + (p >> 2) * kGsCols + cw + 32 * (p & 3));
      xa[2 * p][2 * h] = v.x;
      xa[2 * p][2 * h + 1] = v.y;
      xa[2 * p + 1][2 * h] = v.z;
      xa[2 * p + 1][2 * h + 1] = v.w;
    }
  if (a.norm_eps > 0.f) {
    // RMSNorm of row `warp` in the fixed order of the RMSNorm kernel: lane l
    // owns elements 256 j + 8 l + i, each squared and accumulated in element
    // order, the 32 lane sums added in xor rounds 16, 8, 4, 2, 1
    if (warp < K) {
      const uint4* row = reinterpret_cast<const uint4*>(a.x + (size_t)warp * D);
      float acc = 0.f;
      for (int j0 = 0; j0 < D / 256; j0 += 8) {
        uint4 xv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (j0 + u < D / 256) xv[u] = __ldcg(row + (j0 + u) * 32 + lane);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (j0 + u >= D / 256) break;
          const uint32_t q[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float f = (i & 1) ? bfh(q[i >> 1]) : bfl(q[i >> 1]);
            acc = __fmaf_rn(f, f, acc);
          }
        }
      }
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, d));
      const float mean = __fdiv_rn(acc, (float)D);
      if (lane == 0) T.inv[warp] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, a.norm_eps)));
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < KH; ++h) {
      const int r = g + 8 * h;
      if (r < K) {
        const float inv = T.inv[r];
#pragma unroll
        for (int k = 0; k < KPW; ++k) {
          xa[k][2 * h] = scale_pair(xa[k][2 * h], inv);
          xa[k][2 * h + 1] = scale_pair(xa[k][2 * h + 1], inv);
        }
      }
    }
  }

  float acc[NG][4];
#pragma unroll
  for (int gr = 0; gr < NG; ++gr)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[gr][c] = 0.f;
  const int ng = T.ng, nst = T.ng * NCB;
  volatile int* abort = &T.abort;
#pragma unroll
  for (int gr = 0; gr < NG; ++gr) {
    if (gr >= ng) break;
    // lanes of rows past the group's own (a short group) read nothing:
    // their n columns are zero and unused
    const bool live = g < T.n[gr];
#pragma unroll
    for (int cb = 0; cb < NCB; ++cb) {
      const int s = gr * NCB + cb;
      const int slot = s % kGsStages;
      const uint32_t par = (uint32_t)(s / kGsStages) & 1u;
      bool ok = !*abort && mbar_wait_bounded(&T.full[slot], par, a.wait_ns, abort);
      ok = __all_sync(0xffffffffu, ok);  // converged for mma.sync; one outcome per warp
      if (!ok) {
        *abort = 1;
      } else {
        const unsigned char* wp = smem + (size_t)slot * kGsStageBytes + (size_t)(live ? g : 0) * kGsPitch + cw * 2;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int p = 4 * cb + q;
          const uint4 w = live ? *reinterpret_cast<const uint4*>(wp + 64 * q) : make_uint4(0, 0, 0, 0);
          if constexpr (KH > 1) {
            mma_bf16_gs(acc[gr], xa[2 * p][0], xa[2 * p][2], xa[2 * p][1], xa[2 * p][3], w.x, w.y);
            mma_bf16_gs(acc[gr], xa[2 * p + 1][0], xa[2 * p + 1][2], xa[2 * p + 1][1], xa[2 * p + 1][3], w.z, w.w);
          } else {
            mma_bf16_gs(acc[gr], xa[2 * p][0], 0u, xa[2 * p][1], 0u, w.x, w.y);
            mma_bf16_gs(acc[gr], xa[2 * p + 1][0], 0u, xa[2 * p + 1][1], 0u, w.z, w.w);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&T.empty[slot]);
      if (warp == 0 && issued < nst && issued == s + kGsStages) {
        // refill this slot once every warp has read it
        bool go = false;
        if (lane == 0) {
          go = !*abort && mbar_wait_bounded(&T.empty[slot], par, a.wait_ns, abort);
          if (!go) *abort = 1;
        }
        if (__shfl_sync(0xffffffffu, go, 0)) {
          issue(issued);
          ++issued;
        }
      }
      __syncwarp();
    }
  }
  __syncthreads();  // every warp is done with the ring
  if (*abort) {
    if (threadIdx.x == 0) {
      if (a.err) atomicCAS(a.err, 0, (int)MOE_ERR_DEVICE_TIMEOUT);
      // no copy may land in the shared memory of a finished CTA
      for (int s = max(0, issued - kGsStages); s < issued; ++s)
        mbar_wait_drain(&T.full[s % kGsStages], (uint32_t)(s / kGsStages) & 1u, kGsDrainNs);
    }
    return;
  }

  // partial sums to the (now free) ring: red[gr][w][m][n], m < 16, n < 8
  float* red = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int gr = 0; gr < NG; ++gr) {
    if (gr >= ng) break;
    float* p = red + ((size_t)gr * kGsWarps + warp) * 128;
    p[g * 8 + 2 * t] = acc[gr][0];
    p[g * 8 + 2 * t + 1] = acc[gr][1];
    p[(g + 8) * 8 + 2 * t] = acc[gr][2];
    p[(g + 8) * 8 + 2 * t + 1] = acc[gr][3];
  }
  __syncthreads();
  // output (m, nl) of segment S: the row, and with a cache its in-place
  // KV append at position *len + m
  auto store = [&](const GemvSeg& S, int m, int nl, uint16_t b) {
    S.out[(size_t)m * S.N + nl] = b;
    if (S.cache) {
      const int p = *S.len + m;
      if (p < S.cap) S.cache[((size_t)(nl >> 7) * S.cap + p) * 128 + (nl & 127)] = b;
      else if (a.err) atomicCAS(a.err, 0, (int)MOE_ERR_CAPACITY);
    }
  };
  for (int idx = threadIdx.x; idx < ng * 128; idx += blockDim.x) {
    const int gr = idx >> 7, m = (idx >> 3) & 15, n = idx & 7;
    if (m >= K || n >= T.n[gr] || T.pair[gr] == 2) continue;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kGsWarps; ++w) v += red[((size_t)gr * kGsWarps + w) * 128 + m * 8 + n];
    const GemvSeg& S = a.seg[T.seg[gr]];
    const int nl = T.row[gr] + n;
    if (T.pair[gr] == 1 && a.glu) {
      // gate row nl and up row nl: h = bf16(silu(g) * u), the FP32 sums unrounded
      float u = 0.f;
#pragma unroll
      for (int w = 0; w < kGsWarps; ++w) u += red[((size_t)(gr + 1) * kGsWarps + w) * 128 + m * 8 + n];
      store(S, m, nl, float_to_bf16_bits(v * __frcp_rn(1.f + expf(-v)) * u));
      continue;
    }
    if (T.pair[gr] == 1) {
      // rows i = nl % 128 and i + rope_rd/2 of the head: each rounded to
      // bf16, rotated in FP32 by the row's angle, rounded again
      float v1 = 0.f;
#pragma unroll
      for (int w = 0; w < kGsWarps; ++w) v1 += red[((size_t)(gr + 1) * kGsWarps + w) * 128 + m * 8 + n];
      const float x0 = bfl(float_to_bf16_bits(v)), x1 = bfl(float_to_bf16_bits(v1));
      float c, sn;
      rope_cs((a.rope_len ? *a.rope_len : a.rope_C) + m, a.rope_freq[nl & 127], c, sn);
      store(S, m, nl, float_to_bf16_bits(__fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, sn))));
      store(S, m, T.row[gr + 1] + n, float_to_bf16_bits(__fadd_rn(__fmul_rn(x1, c), __fmul_rn(x0, sn))));
      continue;
    }
    if (S.res) v += bfl(S.res[(size_t)m * S.N + nl]);
    store(S, m, nl, float_to_bf16_bits(v));
  }
}

// Row groups a CTA of the grid needs (at most): its rows in groups of 8,
// plus one per matrix end inside its range.
static int gemv_stream_groups(const GemvArgs& a, int grid) {
  if (a.rope_rd || a.glu) {  // units of 16 rows, matrix ends on unit boundaries
    const int nu = a.n_total / 16;
    return 2 * ((nu + grid - 1) / grid);
  }
  const int rows_max = (a.n_total + grid - 1) / grid;
  return (rows_max + kGsRows - 1) / kGsRows + (a.nseg - 1);
}

// Whether the streamed kernel takes this GEMV: D a whole number of column
// blocks, x's fragments within the registers, and no CTA needing more row
// groups than an instantiation has accumulator sets.
bool gemv_stream_fits(const GemvArgs& a, int grid) {
  if (a.K < 1 || a.K > 16 || a.D % kGsCols != 0) return false;
  const int kpw = a.D / 256;
  if (kpw != 8 && kpw != 16 && kpw != 24 && kpw != 32) return false;
  if (a.K > 8 && kpw > 16) return false;
  return gemv_stream_groups(a, grid) <= gs_max_groups(kpw, a.K > 8 ? 2 : 1);
}

// Whether the streamed kernel can apply the rotary embedding in its
// epilogue: rope_rd a multiple of 16 up to 128, every matrix whole heads.
bool gemv_stream_rope_fits(const GemvArgs& a, int grid) {
  if (a.rope_rd < 16 || a.rope_rd > 128 || a.rope_rd % 16 != 0) return false;
  for (int i = 0; i < a.nseg; ++i)
    if (a.seg[i].N % 128 != 0) return false;
  return gemv_stream_fits(a, grid);
}

cudaError_t launch_gemv_stream(const GemvArgs& a, cudaStream_t s, bool pdl) {
  const int kpw = a.D / 256;
  const bool two = a.K > 8;
  const int ng = gemv_stream_groups(a, num_sms());
  void (*kern)(GemvArgs) = nullptr;
  // the smallest set count that suffices (fewer accumulator registers)
  if (kpw == 8 && ng > 12 && !two) kern = k_gemv_stream<8, 1, 16>;
  else if (kpw == 8 && ng > 8) kern = two ? k_gemv_stream<8, 2, 12> : k_gemv_stream<8, 1, 12>;
  else if (kpw == 8) kern = two ? k_gemv_stream<8, 2, 8> : k_gemv_stream<8, 1, 8>;
  else if (kpw == 16 && ng > 8 && !two) kern = k_gemv_stream<16, 1, 12>;
  else if (kpw == 16 && ng <= 4) kern = two ? k_gemv_stream<16, 2, 4> : k_gemv_stream<16, 1, 4>;
  else if (kpw == 16 && ng <= 8) kern = two ? k_gemv_stream<16, 2, 8> : k_gemv_stream<16, 1, 8>;
  else if (kpw == 24 && !two) kern = ng <= 2 ? k_gemv_stream<24, 1, 2> : k_gemv_stream<24, 1, 4>;
  else if (kpw == 32 && !two) kern = ng <= 2 ? k_gemv_stream<32, 1, 2> : k_gemv_stream<32, 1, 4>;
  if (!kern) return cudaErrorInvalidValue;
  const size_t sm = (size_t)kGsStages * kGsStageBytes + kGsTail;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e == cudaSuccess) e = max_carveout(kern);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(kGsWarps * 32);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace moe
