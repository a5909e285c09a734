// attn_stream.cu -- the split-KV attention over the cache, with the cached
// keys and values streamed into shared memory by TMA.
//
// CTA (split, KV head, query tile) walks a contiguous range of 128-position
// chunks of its KV head.  A chunk's keys and its values are each one 32 KB
// box (128 rows x head dims 0-63 and 64-127, 128-byte swizzled), in a ring of
// three 64 KB stages.
// The cache below the valid length does not depend on the previous kernel
// (the new rows' projection), so the first ring-full is issued before the
// dependency wait.  Warp w takes positions [16w, 16w + 16) of every chunk:
// S = Q K^T with the query tile's 16 rows as the m16 dimension (K fragments
// by ldmatrix from the swizzled rows), online softmax in the log2 domain,
// O += P V (V fragments by transposing ldmatrix).  The 8 warps' (m, l, O)
// are merged in warp order into the split's partial, which the merge kernel
// (k_attn_combine) combines with the block-causal new positions.
//
// Query row i of a tile = verify row i / group, head i % group of the KV
// head; rows past K * group are zero.  Masked: positions at or past the
// valid length (their keys and values may be stale or in flight; the values
// are zeroed in registers so that 0 * garbage cannot give NaN) and, with a
// sliding window, positions before a row's window start.
#include <cfloat>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kAsWarps = 8;
constexpr int kAsPos = 128;                     // positions per chunk
constexpr int kAsHalf = kAsPos * 128;           // one box: 128 rows x 64 dims x 2 B
constexpr int kAsStageBytes = 4 * kAsHalf;      // K lo, K hi, V lo, V hi
constexpr int kAsStages = 3;
// Bound on waiting for the CTA's own copies before it exits (independent of
// the caller's wait limit, which may be 0 in a test of the give-up path).
constexpr uint64_t kAsDrainNs = 2000000000ull;

struct AsTable {
  uint64_t full[kAsStages];
  uint64_t empty[kAsStages];
  int abort;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_as(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2_as(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Shared-memory address of the 16-byte piece holding dims [d0, d0 + 8) of
// chunk row `row` in a stage's key (v = 0) or value (v = 1) boxes.
__device__ __forceinline__ uint32_t piece(uint32_t stage, int v, int row, int d0) {
  const int half = d0 >> 6, c = (d0 & 63) >> 3;
  return stage + (uint32_t)((2 * v + half) * kAsHalf + row * 128 + ((c ^ (row & 7)) << 4));
}

}  // namespace

__global__ void __launch_bounds__(kAsWarps * 32, 1) k_attn_stream(const __grid_constant__ AttnStreamArgs P) {
  const AttnArgs& a = P.a;
  extern __shared__ __align__(1024) unsigned char smem[];
  AsTable& T = *reinterpret_cast<AsTable*>(smem + kAsStages * kAsStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int kvh = blockIdx.y, split = blockIdx.x, tile = blockIdx.z;

  // The valid length and the cached rows below it were written by kernels
  // that completed before the previous kernel passed its own dependency
  // wait, so they are read before this kernel's.
  const int Cv = a.len ? min(*a.len, a.C) : a.C;
  const int lo = a.window > 0 ? max(0, Cv - a.window + 1) : 0;
  const int s0 = lo / kAsPos, nch = (Cv + kAsPos - 1) / kAsPos;
  const int c0 = s0 + (int)(((long long)split * (nch - s0)) / gridDim.x);
  const int c1 = s0 + (int)(((long long)(split + 1) * (nch - s0)) / gridDim.x);
  const int nst = c1 - c0;
  int issued = 0;  // thread 0
  uint64_t pol = 0;
  auto issue = [&](int s) {
    const int slot = s % kAsStages;
    unsigned char* st = smem + (size_t)slot * kAsStageBytes;
    const int row = kvh * a.C + (c0 + s) * kAsPos;
    mbar_arrive_expect_tx(&T.full[slot], kAsStageBytes);
    if (P.kv3d) {  // one box per chunk: [half][row][64 dims]
      tma_load_3d(st, &P.km, 0, row, 0, &T.full[slot], pol);
      tma_load_3d(st + 2 * kAsHalf, &P.vm, 0, row, 0, &T.full[slot], pol);
    } else {
      tma_load_2d(st, &P.km, 0, row, &T.full[slot], pol);
      tma_load_2d(st + kAsHalf, &P.km, 64, row, &T.full[slot], pol);
      tma_load_2d(st + 2 * kAsHalf, &P.vm, 0, row, &T.full[slot], pol);
      tma_load_2d(st + 3 * kAsHalf, &P.vm, 64, row, &T.full[slot], pol);
    }
  };
  if (threadIdx.x == 0) {
    T.abort = 0;
    for (int i = 0; i < kAsStages; ++i) {
      mbar_init(&T.full[i], 1);
      mbar_init(&T.empty[i], kAsWarps);
    }
    fence_mbar_init();
    prefetch_tensormap(&P.km);
    prefetch_tensormap(&P.vm);
    pol = policy_evict_first();
    for (; issued < min(nst, kAsStages); ++issued) issue(issued);
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();

  // Q fragments (A operand, 8 k-steps of 16 head dims): rows g and g + 8
  const int nrow = a.K * a.group;
  uint32_t qa[8][4];
  int rs[2] = {0, 0};  // window start of rows g, g + 8
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int i = 16 * tile + g + 8 * hr;
    const uint32_t* qrow = nullptr;
    if (i < nrow) {
      const int r = i / a.group, hh = i - r * a.group;
      qrow = reinterpret_cast<const uint32_t*>(a.q + (size_t)r * a.nq * 128 + (size_t)(kvh * a.group + hh) * 128);
      if (a.window > 0) rs[hr] = Cv + r - a.window + 1;
    }
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qa[ks][hr] = qrow ? qrow[8 * ks + t] : 0u;          // dims 16 ks + 2t, +1
      qa[ks][2 + hr] = qrow ? qrow[8 * ks + 4 + t] : 0u;  // dims 16 ks + 8 + 2t, +1
    }
  }
  const int rs_max = max(rs[0], rs[1]);

  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int nb = 0; nb < 16; ++nb)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[nb][c] = 0.f;

  volatile int* abort = &T.abort;
  const int lj = lane >> 3, lr = lane & 7;  // ldmatrix: this lane's matrix and row
  for (int s = 0; s < nst; ++s) {
    const int slot = s % kAsStages;
    const uint32_t par = (uint32_t)(s / kAsStages) & 1u;
    bool ok = !*abort && mbar_wait_bounded(&T.full[slot], par, a.wait_ns, abort);
    ok = __all_sync(0xffffffffu, ok);
    const int pos0 = (c0 + s) * kAsPos + 16 * warp;  // this warp's first position
    const int rem = Cv - pos0;                       // valid positions from pos0
    if (!ok) {
      *abort = 1;
    } else if (rem > 0 && pos0 + 16 > lo) {
      const uint32_t st = smem_addr(smem + (size_t)slot * kAsStageBytes);
      float sc[2][4];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int c = 0; c < 4; ++c) sc[nb][c] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        // matrices: (positions 0-7 | 8-15) x (dims lo | hi of the k-step)
        uint32_t kb[4];
        ldsm_x4(piece(st, 0, 16 * warp + 8 * (lj >> 1) + lr, 16 * ks + 8 * (lj & 1)), kb);
        mma_bf16_as(sc[0], qa[ks], kb[0], kb[1]);
        mma_bf16_as(sc[1], qa[ks], kb[2], kb[3]);
      }
      if (rem < 16 || pos0 < rs_max) {
        // score (row g + 8 (c >> 1), position 8 nb + 2t + (c & 1))
#pragma unroll
        for (int nb = 0; nb < 2; ++nb)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int pp = 8 * nb + 2 * t + (c & 1);
            if (pp >= rem || pos0 + pp < rs[c >> 1]) sc[nb][c] = -INFINITY;
          }
      }
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        float v = -INFINITY;
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
          sc[nb][2 * hr] *= a.scale_log2;
          sc[nb][2 * hr + 1] *= a.scale_log2;
          v = fmaxf(v, fmaxf(sc[nb][2 * hr], sc[nb][2 * hr + 1]));
        }
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
        const float mx = fmaxf(m[hr], v);
        const float ref = mx == -INFINITY ? 0.f : mx;  // a row with nothing visible yet
        const float alpha = exp2f(m[hr] - ref);
        m[hr] = mx;
        l[hr] *= alpha;
#pragma unroll
        for (int nb = 0; nb < 16; ++nb) {
          o[nb][2 * hr] *= alpha;
          o[nb][2 * hr + 1] *= alpha;
        }
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
          sc[nb][2 * hr] = exp2f(sc[nb][2 * hr] - ref);
          sc[nb][2 * hr + 1] = exp2f(sc[nb][2 * hr + 1] - ref);
          l[hr] += sc[nb][2 * hr] + sc[nb][2 * hr + 1];
        }
      }
      const uint32_t pa[4] = {pack_bf16x2_as(sc[0][0], sc[0][1]), pack_bf16x2_as(sc[0][2], sc[0][3]),
                              pack_bf16x2_as(sc[1][0], sc[1][1]), pack_bf16x2_as(sc[1][2], sc[1][3])};
      // the positions of this thread's V halves: 2t, 2t + 1 (b0) and 2t + 8, 2t + 9 (b1)
      const uint32_t keep0 = (2 * t < rem ? 0x0000FFFFu : 0u) | (2 * t + 1 < rem ? 0xFFFF0000u : 0u);
      const uint32_t keep1 = (2 * t + 8 < rem ? 0x0000FFFFu : 0u) | (2 * t + 9 < rem ? 0xFFFF0000u : 0u);
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        // matrices: (positions 0-7 | 8-15) x (dims 16 np + 0-7 | 8-15), transposed
        uint32_t vb[4];
        ldsm_x4_t(piece(st, 1, 16 * warp + 8 * (lj & 1) + lr, 16 * np + 8 * (lj >> 1)), vb);
        if (rem < 16) {
          vb[0] &= keep0;
          vb[1] &= keep1;
          vb[2] &= keep0;
          vb[3] &= keep1;
        }
        mma_bf16_as(o[2 * np], pa, vb[0], vb[1]);
        mma_bf16_as(o[2 * np + 1], pa, vb[2], vb[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&T.empty[slot]);
    if (threadIdx.x == 0 && issued < nst && issued == s + kAsStages) {
      if (!*abort && mbar_wait_bounded(&T.empty[slot], par, a.wait_ns, abort)) {
        issue(issued);
        ++issued;
      } else {
        *abort = 1;
      }
    }
    __syncwarp();
  }
  __syncthreads();  // the ring is free
  if (*abort) {
    if (threadIdx.x == 0) {
      if (a.err) atomicCAS(a.err, 0, (int)MOE_ERR_DEVICE_TIMEOUT);
      for (int s = max(0, issued - kAsStages); s < issued; ++s)
        mbar_wait_drain(&T.full[s % kAsStages], (uint32_t)(s / kAsStages) & 1u, kAsDrainNs);
    }
    return;
  }

  // merge the warps in warp order (in the ring's memory)
  float* s_m = reinterpret_cast<float*>(smem);         // [8][16]
  float* s_l = s_m + kAsWarps * 16;                    // [8][16]
  float* s_o = s_l + kAsWarps * 16;                    // [8][16][129]
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 1);
    l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 2);
  }
  if (t == 0) {
    s_m[warp * 16 + g] = m[0];
    s_m[warp * 16 + g + 8] = m[1];
    s_l[warp * 16 + g] = l[0];
    s_l[warp * 16 + g + 8] = l[1];
  }
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) {
    float* r0 = s_o + (warp * 16 + g) * 129 + 8 * nb + 2 * t;
    float* r1 = s_o + (warp * 16 + g + 8) * 129 + 8 * nb + 2 * t;
    r0[0] = o[nb][0];
    r0[1] = o[nb][1];
    r1[0] = o[nb][2];
    r1[1] = o[nb][3];
  }
  __syncthreads();
  const int d = threadIdx.x & 127;
  const int TR = a.tiles * 16;
  float* po = a.part_o + ((size_t)(kvh * gridDim.x + split) * TR + 16 * tile) * 128;
  float* pml = a.part_ml + ((size_t)(kvh * gridDim.x + split) * TR + 16 * tile) * 2;
  for (int i = threadIdx.x >> 7; i < 16; i += kAsWarps * 32 / 128) {
    float M = -INFINITY;
    for (int w = 0; w < kAsWarps; ++w) M = fmaxf(M, s_m[w * 16 + i]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kAsWarps; ++w) {
        const float f = exp2f(s_m[w * 16 + i] - M);
        L += s_l[w * 16 + i] * f;
        O += s_o[(w * 16 + i) * 129 + d] * f;
      }
    }
    po[i * 128 + d] = O;
    if (d == 0) {
      pml[2 * i] = M;
      pml[2 * i + 1] = L;
    }
  }
}

size_t attn_stream_smem() { return (size_t)kAsStages * kAsStageBytes + 256; }

// Splits per (KV head, tile): about one CTA per SM in all, no more than
// there are chunks to walk.
int attn_stream_splits(int nkv, int tiles, int C, int window) {
  const int chunks = window > 0 ? (window + kAsPos - 1) / kAsPos + 1 : (C + kAsPos - 1) / kAsPos;
  int s = num_sms() / (nkv * tiles);
  if (s > chunks) s = chunks;
  return s < 1 ? 1 : (s > kAttnMaxSplits ? kAttnMaxSplits : s);
}

cudaError_t launch_attention_stream(const AttnStreamArgs& P, cudaStream_t s, bool pdl) {
  const AttnArgs& a = P.a;
  const int splits = attn_stream_splits(a.nkv, a.tiles, a.C, a.window);
  const size_t sm = attn_stream_smem();
  cudaError_t e = cudaFuncSetAttribute(k_attn_stream, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e == cudaSuccess) e = max_carveout(k_attn_stream);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(splits, a.nkv, a.tiles);
  cfg.blockDim = dim3(kAsWarps * 32);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_attn_stream, P);
  if (e != cudaSuccess) return e;
  return launch_attn_combine(a, splits, s);
}

}  // namespace moe
