// gemv.cu -- streamed bf16 GEMV for the projections around attention:
//   out[r][n] = bf16( sum_c x[r][c] * W[n][c]  (+ res[r][n]) ),   r < K <= 16,
// for up to three weight matrices that share x (q, k, v), laid end to end
// as one list of output rows; optionally x is first RMS-normalised.
//
// One CTA per SM.  CTA b owns a contiguous range of output rows and streams
// exactly those weight rows -- each byte once -- through a ring of shared-
// memory stages filled by bulk copies.  The weights do not depend on the
// previous kernel, so the first ring-full is issued before the dependency
// wait and lands while that kernel finishes.  A stage holds up to
// R = min(8, 16384 / D) consecutive rows of one matrix (at most 32 KB).
//
// The 16 warps split the reduction dimension: warp w owns columns
// [w D/16, (w+1) D/16) and keeps its fragments of x in registers for the
// whole kernel.  Per stage and 16-column step a warp issues one
// mma.sync m16n8k16 (A = the K rows of x, B = the stage's rows as the n
// dimension, FP32 accumulate).  After the last stage the 16 warps' partial
// sums of each output are added in warp order.
//
// Column order inside a warp's 32-column blocks: thread t of a quad reads
// the 8 consecutive columns [8t, 8t+8).  Its first four are its logical
// k = 2t, 2t+1, 2t+8, 2t+9 of the block's even 16-column step, the last four
// those of the odd step.  x and W use the same order, so every product is
// x[r][c] * W[n][c]; only the order of the FP32 sum differs from a plain
// dot product.
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kGsWarps = 16;
constexpr int kGsStages = 6;
constexpr int kGsStageBytes = 32768;
constexpr int kGsMaxBlocks = 12;  // stages per CTA (one accumulator set each), at most
// Accumulator sets: 8, or 12 where x's fragments (KPW * 2 * KH registers)
// leave room; the 8-set form runs whenever it suffices.
constexpr int gs_max_sets(int kpw, int kh) { return kpw * kh <= 16 ? 12 : 8; }
constexpr int kGsTail = 1024;    // barriers and the stage table after the ring
// Bound on waiting for the CTA's own copies before it exits (independent of
// the caller's wait limit, which may be 0 in a test of the give-up path).
constexpr uint64_t kGsDrainNs = 2000000000ull;

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
  int seg[kGsMaxBlocks], row[kGsMaxBlocks], n[kGsMaxBlocks];
  int nst;
  int abort;
  float inv[16];
};
static_assert(sizeof(GsTable) <= kGsTail, "stage table");
// the partial sums of every set fit the ring once it is free
static_assert(kGsMaxBlocks * kGsWarps * 128 * 4 <= kGsStages * kGsStageBytes, "reduction area");

}  // namespace

template <int KPW, int KH, int NB>
__global__ void __launch_bounds__(kGsWarps * 32, 1) k_gemv_stream(const __grid_constant__ GemvArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  GsTable& T = *reinterpret_cast<GsTable*>(smem + kGsStages * kGsStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int D = a.D, K = a.K;
  int issued = 0;  // thread 0: stages whose copy was issued
  uint64_t pol = 0;

  static_assert(NB <= kGsMaxBlocks, "accumulator sets");
  auto issue = [&](int s) {
    const int slot = s % kGsStages;
    const uint32_t bytes = (uint32_t)T.n[s] * (uint32_t)D * 2u;
    mbar_arrive_expect_tx(&T.full[slot], bytes);
    bulk_load(smem + (size_t)slot * kGsStageBytes, a.seg[T.seg[s]].W + (size_t)T.row[s] * D, bytes,
              &T.full[slot], pol);
  };

  if (threadIdx.x == 0) {
    // this CTA's output rows [r0, r1), cut into stages at matrix ends
    const int r0 = (int)((long long)blockIdx.x * a.n_total / gridDim.x);
    const int r1 = (int)((long long)(blockIdx.x + 1) * a.n_total / gridDim.x);
    int ns = 0, cur = r0, base = 0, sg = 0;
    T.abort = 0;
    while (cur < r1) {
      while (cur >= base + a.seg[sg].N) base += a.seg[sg++].N;
      if (ns == NB) {  // more stages than accumulator sets: refused by the launcher
        T.abort = 1;
        break;
      }
      const int nr = min(a.rows_per_stage, min(r1, base + a.seg[sg].N) - cur);
      T.seg[ns] = sg;
      T.row[ns] = cur - base;
      T.n[ns] = nr;
      ++ns;
      cur += nr;
    }
    T.nst = T.abort ? 0 : ns;
    for (int i = 0; i < kGsStages; ++i) {
      mbar_init(&T.full[i], 1);
      mbar_init(&T.empty[i], kGsWarps);
    }
    fence_mbar_init();
    pol = policy_evict_first();
    for (; issued < min(T.nst, kGsStages); ++issued) issue(issued);
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  if (T.abort && threadIdx.x == 0 && a.err) atomicCAS(a.err, 0, (int)MOE_ERR_UNSUPPORTED_SHAPE);

  // x fragments of this warp's columns: xa[k][0], xa[k][1] = a0, a2 (row g);
  // xa[k][2], xa[k][3] = a1, a3 (row g + 8)
  const int cb = warp * (D / kGsWarps) + 8 * t;
  uint32_t xa[KPW][2 * KH];
#pragma unroll
  for (int kp = 0; kp < KPW / 2; ++kp)
#pragma unroll
    for (int h = 0; h < KH; ++h) {
      const int r = g + 8 * h;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < K) v = *reinterpret_cast<const uint4*>(a.x + (size_t)r * D + cb + 32 * kp);
      xa[2 * kp][2 * h] = v.x;
      xa[2 * kp][2 * h + 1] = v.y;
      xa[2 * kp + 1][2 * h] = v.z;
      xa[2 * kp + 1][2 * h + 1] = v.w;
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

  float acc[NB][4];
#pragma unroll
  for (int s = 0; s < NB; ++s)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[s][c] = 0.f;
  const int ns = T.nst;
  volatile int* abort = &T.abort;
#pragma unroll
  for (int s = 0; s < NB; ++s) {
    if (s >= ns) break;
    const int slot = s % kGsStages;
    const uint32_t par = (uint32_t)(s / kGsStages) & 1u;
    bool ok = !*abort && mbar_wait_bounded(&T.full[slot], par, a.wait_ns, abort);
    ok = __all_sync(0xffffffffu, ok);  // converged for mma.sync; one verdict per warp
    if (!ok) {
      *abort = 1;
    } else {
      // lanes of rows past the stage's own (R < 8, or a short last stage)
      // read nothing: their n columns are zero and unused
      const bool live = g < T.n[s];
      const unsigned char* wp = smem + (size_t)slot * kGsStageBytes + ((size_t)(live ? g : 0) * D + cb) * 2;
#pragma unroll
      for (int kp = 0; kp < KPW / 2; ++kp) {
        const uint4 w = live ? *reinterpret_cast<const uint4*>(wp + 64 * kp) : make_uint4(0, 0, 0, 0);
        if constexpr (KH > 1) {
          mma_bf16_gs(acc[s], xa[2 * kp][0], xa[2 * kp][2], xa[2 * kp][1], xa[2 * kp][3], w.x, w.y);
          mma_bf16_gs(acc[s], xa[2 * kp + 1][0], xa[2 * kp + 1][2], xa[2 * kp + 1][1], xa[2 * kp + 1][3], w.z, w.w);
        } else {
          mma_bf16_gs(acc[s], xa[2 * kp][0], 0u, xa[2 * kp][1], 0u, w.x, w.y);
          mma_bf16_gs(acc[s], xa[2 * kp + 1][0], 0u, xa[2 * kp + 1][1], 0u, w.z, w.w);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&T.empty[slot]);
    if (threadIdx.x == 0 && issued < ns && issued == s + kGsStages) {
      // refill this slot once every warp has read it
      if (!*abort && mbar_wait_bounded(&T.empty[slot], par, a.wait_ns, abort)) {
        issue(issued);
        ++issued;
      } else {
        *abort = 1;
      }
    }
    __syncwarp();
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

  // partial sums to the (now free) ring: red[s][w][m][n], m < 16, n < 8
  float* red = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int s = 0; s < NB; ++s) {
    if (s >= ns) break;
    float* p = red + ((size_t)s * kGsWarps + warp) * 128;
    p[g * 8 + 2 * t] = acc[s][0];
    p[g * 8 + 2 * t + 1] = acc[s][1];
    p[(g + 8) * 8 + 2 * t] = acc[s][2];
    p[(g + 8) * 8 + 2 * t + 1] = acc[s][3];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < ns * 128; idx += blockDim.x) {
    const int s = idx >> 7, m = (idx >> 3) & 15, n = idx & 7;
    if (m >= K || n >= T.n[s]) continue;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kGsWarps; ++w) v += red[((size_t)s * kGsWarps + w) * 128 + m * 8 + n];
    const GemvSeg& S = a.seg[T.seg[s]];
    const int nl = T.row[s] + n;
    if (S.res) v += bfl(S.res[(size_t)m * S.N + nl]);
    const uint16_t b = float_to_bf16_bits(v);
    S.out[(size_t)m * S.N + nl] = b;
    if (S.cache) {  // in-place KV append at position *len + m
      const int p = *S.len + m;
      if (p < S.cap) S.cache[((size_t)(nl >> 7) * S.cap + p) * 128 + (nl & 127)] = b;
      else if (a.err) atomicCAS(a.err, 0, (int)MOE_ERR_CAPACITY);
    }
  }
}

int gemv_rows_per_stage(int D) { return kGsStageBytes / (2 * D) < 8 ? kGsStageBytes / (2 * D) : 8; }

// Whether the streamed kernel takes this GEMV: x's fragments must fit the
// registers and no CTA may need more stages than it has accumulator sets.
static int gemv_stream_sets(const GemvArgs& a, int grid) {
  const int R = gemv_rows_per_stage(a.D);
  const int rows_max = (a.n_total + grid - 1) / grid;
  return (rows_max + R - 1) / R + (a.nseg - 1);
}

bool gemv_stream_fits(const GemvArgs& a, int grid) {
  if (a.K < 1 || a.K > 16 || a.D % 512 != 0) return false;
  const int kpw = a.D / 256;
  if (kpw != 8 && kpw != 16 && kpw != 24 && kpw != 32) return false;
  if (a.K > 8 && kpw > 16) return false;
  return gemv_stream_sets(a, grid) <= gs_max_sets(kpw, a.K > 8 ? 2 : 1);
}

cudaError_t launch_gemv_stream(const GemvArgs& a, cudaStream_t s, bool pdl) {
  const int kpw = a.D / 256;
  const bool two = a.K > 8;
  const bool wide = gemv_stream_sets(a, num_sms()) > 8;
  void (*kern)(GemvArgs) = nullptr;
  if (kpw == 8 && wide) kern = two ? k_gemv_stream<8, 2, 12> : k_gemv_stream<8, 1, 12>;
  else if (kpw == 8) kern = two ? k_gemv_stream<8, 2, 8> : k_gemv_stream<8, 1, 8>;
  else if (kpw == 16 && wide && !two) kern = k_gemv_stream<16, 1, 12>;
  else if (kpw == 16 && !wide) kern = two ? k_gemv_stream<16, 2, 8> : k_gemv_stream<16, 1, 8>;
  else if (kpw == 24 && !two && !wide) kern = k_gemv_stream<24, 1, 8>;
  else if (kpw == 32 && !two && !wide) kern = k_gemv_stream<32, 1, 8>;
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
