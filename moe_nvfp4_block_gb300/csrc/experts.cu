// experts.cu -- the experts of one MoE verify-layer call in one persistent kernel.
//
// One CTA per SM: a producer warp streams weight tiles into a ring of shared
// memory stages with TMA (2-D tiled copies with swizzle for the 4-bit codes
// and the gate/up E4M3 scales, 1-D bulk copies for the down scales) and eight
// consumer warps decode and multiply.  The CTA's work is a fixed sequence of
// items: its shared-expert gate/up items, its routed gate/up items, then its
// down items.  Every distinct expert is streamed exactly once per call
// however many rows chose it (PR #844, "8. What I looked at": the stock gather
// re-reads an expert once per (row, slot)).
//
// Overlap: before the programmatic-launch wait the producer already streams
// the shared expert's first tiles (they do not depend on the routing) and the
// consumers stage the activations.  After it, every CTA reads the router
// logits and computes the same routing (top-k with lower-index tie-break,
// renormalised softmax weights, grouping) on its own -- no serial hand-off.
// A down item of expert u waits (bounded) until all gate/up items of u have
// published h; its weight tiles are already in flight by then.
//
// Decode: ldmatrix pulls 32 bits of codes per thread and row; the hardware
// FP4 -> FP16 convert turns 8 codes into four f16x2, and one f16x2 multiply
// by the block's E4M3 scale gives the exact element (e2m1 * e4m3 has at most
// 6 significant bits and lies in [2^-10, 2688]).  mma.sync m16n8k16 then
// multiplies 16 weight rows by the verify rows (n = 8 or 16 columns) with
// FP32 accumulation; the tensor scale is applied to the accumulator.  The k
// index of an mma step is a permutation of the physical k (any order is a
// valid dot product): thread t's elements are its own 8 consecutive codes.
// Activations enter as FP16 after an exact per-row power-of-two rescaling
// (max |value| into [2^14, 2^15)), undone in FP32.
//
// Combine: per-(row, slot) FP32 partials; the CTA that completes the last
// item of a 64-row hidden tile (atomic count, no waiting) forms
// y = bf16(routed_scale * sum_s w_s d_s + d_shared + residual) in slot order
// (PR #844, "4. What I ported": weighted sum, routed scale, shared add,
// residual add in one pass).
#include <cfloat>
#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kConsumerThreads = 256;
constexpr int kThreads = kConsumerThreads + 32;
constexpr uint64_t kDrainNs = 2000000000ull;  // bound on waiting for our own copies before exit

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ void set_error(int* err, int code) { atomicCAS(err, 0, code); }

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned atom_acq_rel_add(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Power-of-two shift that maps max |x| into [2^14, 2^15).
__device__ __forceinline__ int row_shift(unsigned amax_bits) {
  const float amax = __uint_as_float(amax_bits);
  if (!(amax > 0.f)) return 0;
  int e = (int)((amax_bits >> 23) & 0xFF) - 127;
  if (e < -126) e = -126;
  int s = 14 - e;
  return s > 126 ? 126 : (s < -126 ? -126 : s);
}

__device__ __forceinline__ float pow2f(int s) { return __int_as_float((s + 127) << 23); }

// 8 bf16 (one uint4) * scale -> 4 f16x2.
__device__ __forceinline__ void bf16x8_to_f16x8(const uint4 v, float scale, uint32_t* out) {
  const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    out[i] = pack_f16x2(__uint_as_float(q[i] << 16) * scale, __uint_as_float(q[i] & 0xFFFF0000u) * scale);
}

__device__ __forceinline__ bool ranks_before(float la, int a, float lb, int b) {
  return (la > lb) || (la == lb && a < b);
}

// Selection keys: a logit and its expert index packed into one integer that
// orders exactly like "larger logit first, lower index on an exact tie":
// the float's bits mapped to an unsigned order in the high word, the
// complement of the index in the low word.  Larger key = ranks first.
__device__ __forceinline__ unsigned long long sel_key(float v, int e) {
  const unsigned b = __float_as_uint(v);
  const unsigned o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)o << 32) | (unsigned)(0xFFFFFFFFu - (unsigned)e);
}

__device__ __forceinline__ int key_index(unsigned long long k) { return (int)(0xFFFFFFFFu - (unsigned)k); }

__device__ __forceinline__ float key_value(unsigned long long k) {
  const unsigned o = (unsigned)(k >> 32);
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

__device__ __forceinline__ void kx(unsigned long long& a, unsigned long long& b) {  // a <- larger
  const unsigned long long hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}

// The 8 largest keys of a warp's 256 candidates (8 per lane), in descending
// order, on every lane: lane-local bitonic sort, then five xor rounds that
// keep the largest 8 of two sorted lists (the elementwise max of a[j] and
// b[7-j] is their top 8 as a bitonic sequence, sorted by a 3-stage merge).
__device__ __forceinline__ void warp_top8(unsigned long long (&v)[8]) {
#pragma unroll
  for (int size = 2; size <= 8; size <<= 1)
#pragma unroll
    for (int d = size >> 1; d >= 1; d >>= 1)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = i ^ d;
        if (j > i) {
          if ((i & size) == 0) kx(v[i], v[j]);
          else kx(v[j], v[i]);
        }
      }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
    unsigned long long p[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) p[j] = __shfl_xor_sync(0xffffffffu, v[j], d);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = v[j] > p[7 - j] ? v[j] : p[7 - j];
#pragma unroll
    for (int dd = 4; dd >= 1; dd >>= 1)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = i ^ dd;
        if (j > i) kx(v[i], v[j]);
      }
  }
}

// Geometry of one projection's codes tile: `chunks` TMA boxes of
// [rows][inner bytes], box c at c * rows * inner.
struct TileGeo {
  int inner;   // 128 or 64 bytes
  int mask;    // swizzle mask: 7 (128B) or 3 (64B)
  int units;   // 16-byte units per line
};

__device__ __forceinline__ TileGeo tile_geo(int cols) {
  TileGeo g;
  const int rb = cols / 2;
  g.inner = rb >= 128 ? 128 : 64;
  g.mask = g.inner == 128 ? 7 : 3;
  g.units = g.inner / 16;
  return g;
}

// The 4 E4M3 scales thread t needs for one k-unit (128 k) of one row, from
// the 8 bytes [8 ku, 8 ku + 8) of the row's scales: blocks 2q + t/2, q = 0..3;
// returned as four f16x2 each holding one scale twice.
__device__ __forceinline__ void unit_scales(uint2 s8, int t, uint32_t (&out)[4]) {
  const uint32_t four = __byte_perm(s8.x, s8.y, (t >> 1) ? 0x7531u : 0x6420u);
  uint32_t lo, hi;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"(static_cast<uint16_t>(four & 0xFFFF)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"(static_cast<uint16_t>(four >> 16)));
  out[0] = __byte_perm(lo, lo, 0x1010);
  out[1] = __byte_perm(lo, lo, 0x3232);
  out[2] = __byte_perm(hi, hi, 0x1010);
  out[3] = __byte_perm(hi, hi, 0x3232);
}

// One k-unit (128 k) of a 16-row m-tile against NB n-blocks of B.
//   tile: shared address of the codes tile (box_rows rows per box)
//   sg, sh: the row-g and row-(g+8) scales of this k-unit (unit_scales)
template <int NB>
__device__ __forceinline__ void kunit_mma(uint32_t tile, const TileGeo& geo, int box_rows, int row0, int ku,
                                          const uint32_t (&sg)[4], const uint32_t (&sh)[4],
                                          const uint32_t (&b)[NB][16], float (&acc0)[NB][4],
                                          float (&acc1)[NB][4], int lane) {
  const int q0 = (ku * 4) % geo.units;
  const int c = (ku * 4) / geo.units;
  const int mi = lane >> 3, rr = lane & 7;
  const int lrow = row0 + rr + 8 * (mi & 1);
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const int unit = q0 + 2 * p + (mi >> 1);
    const uint32_t off = swizzle_off((uint32_t)((c * box_rows + lrow) * geo.inner + unit * 16), geo.mask);
    uint32_t r0, r1, r2, r3;
    ldmatrix_x4(tile + off, r0, r1, r2, r3);
    // r0: row g unit q, r1: row g+8 unit q, r2: row g unit q+1, r3: row g+8 unit q+1
    const uint32_t rq[2][2] = {{r0, r1}, {r2, r3}};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int q = 2 * p + h;
      uint32_t dg[4], dh[4];
      e2m1x8_to_f16x8(rq[h][0], dg);
      e2m1x8_to_f16x8(rq[h][1], dh);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        dg[i] = hmul2(dg[i], sg[q]);
        dh[i] = hmul2(dh[i], sh[q]);
      }
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {  // two independent accumulation chains
        mma_f16(acc0[nb], dg[0], dh[0], dg[1], dh[1], b[nb][q * 4 + 0], b[nb][q * 4 + 1]);
        mma_f16(acc1[nb], dg[2], dh[2], dg[3], dh[3], b[nb][q * 4 + 2], b[nb][q * 4 + 3]);
      }
    }
  }
}

// Item kinds of a CTA's sequence.
constexpr int kShGU = 0, kRtGU = 1, kDN = 2;

struct Item {
  int kind;
  int slot;  // u (routed) or G (shared)
  int tile;  // m-tile (gate/up, 16 rows) or hidden tile (down, 64 rows)
};

// The CTA's work: n_shb shared gate/up items (round-robin over CTAs), a
// contiguous range of routed gate/up items balanced against them, then a
// contiguous range of down items.
struct Plan {
  int n_shb, gu0, gu1, dn0, dn1;
};

__device__ __forceinline__ int shared_before(int b, int n_sh, int grid) {
  return (n_sh / grid) * b + min(b, n_sh % grid);
}

__device__ Plan make_plan(int n_sh, int n_rgu, int n_dn) {
  const int grid = gridDim.x, b = blockIdx.x;
  Plan p;
  p.n_shb = shared_before(b + 1, n_sh, grid) - shared_before(b, n_sh, grid);
  const long long T = n_sh + n_rgu;
  // routed items before CTA c: its share of all gate/up items minus the
  // shared items already placed on CTAs < c.  When every CTA's share is at
  // least its shared items this is monotone in c; otherwise take the running
  // maximum (small workloads only).
  auto R0 = [&](int c) {
    long long v = (long long)c * T / grid - shared_before(c, n_sh, grid);
    return v < 0 ? 0LL : (v > n_rgu ? (long long)n_rgu : v);
  };
  auto R = [&](int c) {
    if (T >= (long long)grid * ((n_sh + grid - 1) / grid + 1)) return (int)R0(c);
    long long best = 0;
    for (int d = 0; d <= c; ++d) best = max(best, R0(d));
    return (int)best;
  };
  p.gu0 = R(b);
  p.gu1 = (b + 1 == grid) ? n_rgu : R(b + 1);
  p.dn0 = (int)(((long long)b * n_dn) / grid);
  p.dn1 = (int)(((long long)(b + 1) * n_dn) / grid);
  return p;
}

__device__ __forceinline__ int plan_len(const Plan& p) { return p.n_shb + (p.gu1 - p.gu0) + (p.dn1 - p.dn0); }

__device__ __forceinline__ Item plan_item(const Plan& p, int l, int mt_per, int n_tiles, int has_sh, int G,
                                          int n_sh, int grid) {
  Item it;
  if (l < p.n_shb) {
    it.kind = kShGU;
    it.slot = G;
    it.tile = blockIdx.x + l * grid;  // shared items are round-robin
    (void)n_sh;
    return it;
  }
  l -= p.n_shb;
  if (l < p.gu1 - p.gu0) {
    const int v = p.gu0 + l;
    it.kind = kRtGU;
    it.slot = v / mt_per;
    it.tile = v % mt_per;
    return it;
  }
  l -= p.gu1 - p.gu0;
  const int v = p.dn0 + l;
  const int si = v / n_tiles;
  it.kind = kDN;
  it.tile = v % n_tiles;
  it.slot = (has_sh && si == 0) ? G : si - has_sh;
  return it;
}

}  // namespace

template <int NB, int KUG, int KUD>
__global__ void __launch_bounds__(kThreads, 1)
    k_moe_experts(const __grid_constant__ CUtensorMap tm_gate, const __grid_constant__ CUtensorMap tm_up,
                  const __grid_constant__ CUtensorMap tm_down, const __grid_constant__ CUtensorMap tm_sgate,
                  const __grid_constant__ CUtensorMap tm_sup, const __grid_constant__ CUtensorMap tm_sdown,
                  const __grid_constant__ CUtensorMap tm_gate_s, const __grid_constant__ CUtensorMap tm_up_s,
                  const __grid_constant__ CUtensorMap tm_sgate_s, const __grid_constant__ CUtensorMap tm_sup_s,
                  ExpertsArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kExpStages], empty_bar[kExpStages];
  __shared__ unsigned s_xamax[16];
  __shared__ int s_abort, s_nu;
  __shared__ float s_hinv[16];

  const int H = a.H, I = a.I, K = a.K, G = a.G, E = a.E, k = a.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const TileGeo ggu = tile_geo(H), gdn = tile_geo(I);
  const int gu_code = kGURows * H / 2, gu_scale = kGURows * H / 16;
  const int dn_code = kDNRows * I / 2, dn_scale = kDNRows * I / 16;
  const int stage_bytes = expert_stage_bytes(H, I);
  const int mt_per = I / kGURows, n_tiles = H / kDNRows;
  const int n_sh = a.has_shared ? I / kGURows : 0;
  const int grid = gridDim.x;
  const int smask = (H / 16 >= 128) ? 7 : (H / 16 == 64 ? 3 : (H / 16 == 32 ? 1 : 0));

  float* red = reinterpret_cast<float*>(smem + kExpStages * stage_bytes);  // [2][8][2][NB][128]
  unsigned char* rsm = reinterpret_cast<unsigned char*>(red + 2 * 8 * 2 * NB * 128);
  // routing state (shared by all warps after the routing step)
  float* s_w = reinterpret_cast<float*>(rsm);                // [K][k]
  int* s_idx = reinterpret_cast<int*>(s_w + K * k);          // [K][k]
  unsigned* s_rowmask = reinterpret_cast<unsigned*>(s_idx + K * k);  // [E]
  int* s_pos = reinterpret_cast<int*>(s_rowmask + E);        // [E]
  int* s_uexp = s_pos + E;                                   // [G+1]
  float* s_tse = reinterpret_cast<float*>(s_uexp + G + 1);  // [E+1][3] tensor scales per expert (E = shared)
  signed char* s_slot = reinterpret_cast<signed char*>(s_tse + 3 * (E + 1));  // [(G+1)*K]

  if (threadIdx.x == 0) {
    for (int s = 0; s < kExpStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kExpWarps);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < 16) s_xamax[threadIdx.x] = 0u;
  __syncthreads();

  // optional timeline: globaltimer stamps of this CTA's milestones
  unsigned long long* trace = a.trace ? a.trace + (size_t)blockIdx.x * kTraceSlots : nullptr;
  auto stamp = [&](int m) {
    if (trace) trace[m] = global_timer_ns();
  };
  if (threadIdx.x == 0) stamp(0);
  const uint64_t pol = policy_evict_first();
  // Producer: issue the TMA copies of item l of `p` into its stage.
  auto issue = [&](const Plan& p, int l, const Item& it) {
    const int st = l % kExpStages;
    unsigned char* stg = smem + st * stage_bytes;
    if (it.kind != kDN) {
      const bool sh = it.kind == kShGU;
      const int e = sh ? 0 : s_uexp[it.slot];
      const int row0 = e * I + it.tile * kGURows;
      const CUtensorMap* mg = sh ? &tm_sgate : &tm_gate;
      const CUtensorMap* mu = sh ? &tm_sup : &tm_up;
      const CUtensorMap* msg = sh ? &tm_sgate_s : &tm_gate_s;
      const CUtensorMap* msu = sh ? &tm_sup_s : &tm_up_s;
      const int chunks = (H / 2) / ggu.inner;
      if (lane == 0) mbar_arrive_expect_tx(&full_bar[st], 2 * gu_code + 2 * gu_scale);
      __syncwarp();
      if (a.code3d) {  // one request per projection tile
        if (lane == 0) tma_load_3d(stg, mg, 0, row0, 0, &full_bar[st], pol);
        else if (lane == 1) tma_load_3d(stg + gu_code, mu, 0, row0, 0, &full_bar[st], pol);
      } else if (lane < chunks)
        tma_load_2d(stg + lane * kGURows * ggu.inner, mg, lane * ggu.inner, row0, &full_bar[st], pol);
      else if (lane >= 16 && lane < 16 + chunks)
        tma_load_2d(stg + gu_code + (lane - 16) * kGURows * ggu.inner, mu, (lane - 16) * ggu.inner, row0,
                    &full_bar[st], pol);
      if (lane == 30)
        tma_load_2d(stg + 2 * gu_code, msg, 0, row0, &full_bar[st], pol);
      else if (lane == 31)
        tma_load_2d(stg + 2 * gu_code + gu_scale, msu, 0, row0, &full_bar[st], pol);
    } else {
      const bool sh = it.slot == G;
      const int e = sh ? 0 : s_uexp[it.slot];
      const int row0 = e * H + it.tile * kDNRows;
      const CUtensorMap* m = sh ? &tm_sdown : &tm_down;
      const unsigned char* sp = sh ? a.sh_down.scales : a.down.scales;
      const int chunks = (I / 2) / gdn.inner;
      if (lane == 0) mbar_arrive_expect_tx(&full_bar[st], dn_code + dn_scale);
      __syncwarp();
      if (a.code3d) {
        if (lane == 0) tma_load_3d(stg, m, 0, row0, 0, &full_bar[st], pol);
      } else if (lane < chunks)
        tma_load_2d(stg + lane * kDNRows * gdn.inner, m, lane * gdn.inner, row0, &full_bar[st], pol);
      if (lane == 31)
        bulk_load(stg + dn_code, sp + (size_t)row0 * (I / 16), dn_scale, &full_bar[st], pol);
    }
    __syncwarp();
  };

  // ---------------------------------------------------------------- before the dependency wait
  // The shared items of this CTA come first in its sequence and need no routing.
  Plan pre;
  pre.n_shb = shared_before(blockIdx.x + 1, n_sh, grid) - shared_before(blockIdx.x, n_sh, grid);
  pre.gu0 = pre.gu1 = pre.dn0 = pre.dn1 = 0;
  int issued = 0;
  if (warp == kExpWarps) {
    if (lane == 0) {
      prefetch_tensormap(&tm_gate);
      prefetch_tensormap(&tm_up);
      prefetch_tensormap(&tm_down);
    }
    for (; issued < pre.n_shb && issued < kExpStages; ++issued)
      issue(pre, issued, plan_item(pre, issued, mt_per, n_tiles, a.has_shared, G, n_sh, grid));
  }

  // activations (the block input is complete before the router kernel started)
  uint32_t bx[KUG][NB][16];
  if (warp < kExpWarps) {
    for (int e = threadIdx.x; e < E; e += kConsumerThreads) s_rowmask[e] = 0u;
    for (int i = threadIdx.x; i < (G + 1) * K; i += kConsumerThreads) s_slot[i] = -1;
    for (int e = threadIdx.x; e <= E; e += kConsumerThreads) {  // tensor scales, slot E = shared
      const bool shx = e == E;
      if (shx && !a.has_shared) continue;
      s_tse[3 * e + 0] = shx ? a.sh_gate.tscale[0] : a.gate.tscale[e];
      s_tse[3 * e + 1] = shx ? a.sh_up.tscale[0] : a.up.tscale[e];
      s_tse[3 * e + 2] = shx ? a.sh_down.tscale[0] : a.down.tscale[e];
    }
    uint4 raw[KUG][NB][4];
    const int KU = H / 128;
#pragma unroll
    for (int j = 0; j < KUG; ++j) {
      const int ku = warp + kExpWarps * j;
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const int n = nb * 8 + g;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (ku < KU && n < K) v = *reinterpret_cast<const uint4*>(a.x + (size_t)n * H + ku * 128 + q * 32 + 8 * t);
          raw[j][nb][q] = v;
        }
      }
    }
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      unsigned mx = 0;
#pragma unroll
      for (int j = 0; j < KUG; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t w4[4] = {raw[j][nb][q].x, raw[j][nb][q].y, raw[j][nb][q].z, raw[j][nb][q].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            mx = max(mx, (w4[i] << 16) & 0x7FFFFFFFu);
            mx = max(mx, w4[i] & 0x7FFF0000u);
          }
        }
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const int n = nb * 8 + g;
      if (t == 0 && n < K) atomicMax(&s_xamax[n], mx);
    }
    consumer_bar();
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int n = nb * 8 + g;
      const float sc = (n < K) ? pow2f(row_shift(s_xamax[n])) : 1.f;
#pragma unroll
      for (int j = 0; j < KUG; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) bf16x8_to_f16x8(raw[j][nb][q], sc, &bx[j][nb][q * 4]);
    }
  }

  if (threadIdx.x == 0) stamp(1);
  pdl_wait();  // router logits complete; per-call counters cleared
  if (threadIdx.x == 0) stamp(2);

  // ---------------------------------------------------------------- routing (every CTA, identical)
  if (warp < kExpWarps) {
    const bool fast = E <= 256 && k <= 8;
    for (int r = warp; r < K; r += kExpWarps) {
      if (fast) {
        unsigned long long v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int e = lane + 32 * i;
          v[i] = (e < E) ? sel_key(__ldcg(a.logits + (size_t)r * E + e), e) : 0ull;
        }
        if (threadIdx.x == 0) stamp(10);
        warp_top8(v);
        if (threadIdx.x == 0) stamp(11);
        if (lane == 0) {
#pragma unroll
          for (int s = 0; s < 8; ++s)
            if (s < k) {
              s_idx[r * k + s] = key_index(v[s]);
              s_w[r * k + s] = key_value(v[s]);  // logit for now
            }
        }
      } else {
        float lv[32];
        unsigned taken = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = lane + 32 * i;
          lv[i] = (e < E) ? __ldcg(a.logits + (size_t)r * E + e) : -INFINITY;
        }
        for (int s = 0; s < k; ++s) {
          float bv = -INFINITY;
          int be = INT_MAX;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && ranks_before(lv[i], e, bv, be)) {
              bv = lv[i];
              be = e;
            }
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
          if (be == INT_MAX) {  // only NaN logits left: lowest free index
            int f = INT_MAX;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (lane + 32 * i < E && !((taken >> i) & 1u)) f = min(f, lane + 32 * i);
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) f = min(f, __shfl_xor_sync(0xffffffffu, f, d));
            be = f;
            float mine = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (lane + 32 * i == be) mine = lv[i];
            bv = __shfl_sync(0xffffffffu, mine, be & 31);
          }
          if ((be & 31) == lane) taken |= 1u << (be >> 5);
          if (lane == 0) {
            s_idx[r * k + s] = be;
            s_w[r * k + s] = bv;  // logit for now
          }
        }
      }
      __syncwarp();
      const float m = s_w[r * k];
      const float ev = (lane < k) ? expf(s_w[r * k + lane] - m) : 0.f;
      float z = ev;
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
      __syncwarp();
      if (lane < k) {
        s_w[r * k + lane] = ev / z;
        atomicOr(&s_rowmask[s_idx[r * k + lane]], 1u << r);
      }
    }
    if (threadIdx.x == 0) stamp(12);
    // grouping: distinct experts ascending, (row, slot) per expert
    consumer_bar();
    if (threadIdx.x == 0) stamp(13);
    if (warp == 0) {  // one warp: lane l owns experts [l*CH, l*CH + CH), scan in lane order
      const int CH = (E + 31) / 32;
      const int e0 = lane * CH;
      int cnt = 0;
      for (int e = e0; e < min(E, e0 + CH); ++e) cnt += s_rowmask[e] != 0u;
      int inc = cnt;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += o;
      }
      int u = inc - cnt;
      for (int e = e0; e < min(E, e0 + CH); ++e)
        if (s_rowmask[e]) {
          s_pos[e] = u;
          s_uexp[u] = e;
          ++u;
        }
      if (lane == 31) s_nu = inc;
    }
    consumer_bar();
    for (int q = threadIdx.x; q < K * k; q += kConsumerThreads)
      s_slot[s_pos[s_idx[q]] * K + q / k] = (signed char)(q % k);
    if (a.has_shared)
      for (int r = threadIdx.x; r < K; r += kConsumerThreads) s_slot[G * K + r] = (signed char)k;
    if (threadIdx.x < 1) s_uexp[G] = E;  // the shared expert's scales sit at index E
    if (threadIdx.x == 0) stamp(14);
    consumer_bar();
    if (threadIdx.x == 0) stamp(15);
    // the routing outputs of the call (one CTA writes them)
    if (blockIdx.x == 0) {
      for (int q = threadIdx.x; q < K * k; q += kConsumerThreads) {
        if (a.idx_out) a.idx_out[q] = s_idx[q];
        if (a.w_out) a.w_out[q] = s_w[q];
      }
      if (a.group_out) {
        const int nu = s_nu;
        int* go = a.group_out;
        if (threadIdx.x == 0) {
          go[0] = nu;
          go[1 + 2 * G] = K * k;
        }
        for (int v = threadIdx.x; v < G; v += kConsumerThreads) {
          go[1 + v] = v < nu ? s_uexp[v] : -1;
          int o = 0;  // pairs of the experts before v
          for (int u = 0; u < v && u < nu; ++u) o += __popc(s_rowmask[s_uexp[u]]);
          go[1 + G + v] = o;
          if (v < nu) {
            const int ex = s_uexp[v];
            for (int r = 0; r < K; ++r) {
              if (!((s_rowmask[ex] >> r) & 1u)) continue;
              go[2 + 2 * G + o] = r * k + s_slot[v * K + r];
              ++o;
            }
          }
        }
      }
    }
  }
  __syncthreads();
  pdl_launch_dependents();
  if (threadIdx.x == 0) stamp(3);

  const int n_u = s_nu;
  const int n_slots = n_u + (a.has_shared ? 1 : 0);
  const Plan plan = make_plan(n_sh, n_u * mt_per, n_slots * n_tiles);
  const int L = plan_len(plan);

  if (warp == kExpWarps) {
    // ------------------------------------------------------------ producer
    for (int l = issued; l < L; ++l) {
      const int st = l % kExpStages;
      int ok = 1;
      if (lane == 0 && l >= kExpStages) {
        if (!mbar_wait_bounded(&empty_bar[st], ((l / kExpStages) - 1) & 1, a.wait_ns, &s_abort)) {
          ok = 0;
          s_abort = 1;
          set_error(a.ws.err, MOE_ERR_DEVICE_TIMEOUT);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok || s_abort) break;
      issue(plan, l, plan_item(plan, l, mt_per, n_tiles, a.has_shared, G, n_sh, grid));
      issued = l + 1;
    }
    if (lane == 0 && trace) trace[9] = global_timer_ns();
    if (lane == 0) {
      for (int j = (issued > kExpStages ? issued - kExpStages : 0); j < issued; ++j)
        mbar_wait_bounded(&full_bar[j % kExpStages], (j / kExpStages) & 1, kDrainNs, &s_abort);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int KUgu = H / 128, KUdn = I / 128;
  // gate/up items publish per epilogue warp (4 * NB of them), down items
  // count per consumer warp (8), so neither needs a second CTA barrier
  const unsigned gu_target = (unsigned)(mt_per * 4 * NB);
  int pub_slot = -1;      // slot whose finished gate/up items are not yet published
  unsigned pub_count = 0;  // how many of them (this warp's share of each)
  uint32_t bh[KUD][NB][16];
  int cur_slot = -1;
  const int mt = warp & 3, kh = warp >> 2;  // down: m-tile of 16 rows, k-half
  const int L_gu = plan.n_shb + (plan.gu1 - plan.gu0);  // all gate/up items precede the down items
  for (int l = 0; l < L_gu; ++l) {
    const Item it = plan_item(plan, l, mt_per, n_tiles, a.has_shared, G, n_sh, grid);
    const int st = l % kExpStages;
    unsigned char* stg = smem + st * stage_bytes;
    float* rb = red + (size_t)(l & 1) * (8 * 2 * NB * 128);
    {
      // ------------------------------------------------ gate/up item
      const bool ok = mbar_wait_bounded(&full_bar[st], (l / kExpStages) & 1, a.wait_ns, &s_abort);
      if (threadIdx.x == 0 && l < 11) stamp(16 + 4 * l);
      if (!ok && lane == 0) {
        s_abort = 1;
        set_error(a.ws.err, MOE_ERR_DEVICE_TIMEOUT);
      }
      float ag[NB][4], au[NB][4], ag1[NB][4], au1[NB][4];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) ag[nb][i] = au[nb][i] = ag1[nb][i] = au1[nb][i] = 0.f;
      if (ok) {
        const uint32_t tg = smem_addr(stg), tu = smem_addr(stg + gu_code);
        const unsigned char* sgt = stg + 2 * gu_code;
        const unsigned char* sut = stg + 2 * gu_code + gu_scale;
        const int sstride = H / 16;
#pragma unroll
        for (int j = 0; j < KUG; ++j) {
          const int ku = warp + kExpWarps * j;
          if (ku < KUgu) {
            uint32_t s0[4], s1[4], u0[4], u1[4];
            const uint32_t o0 = swizzle_off((uint32_t)(g * sstride + 8 * ku), smask);
            const uint32_t o1 = swizzle_off((uint32_t)((g + 8) * sstride + 8 * ku), smask);
            unit_scales(*reinterpret_cast<const uint2*>(sgt + o0), t, s0);
            unit_scales(*reinterpret_cast<const uint2*>(sgt + o1), t, s1);
            unit_scales(*reinterpret_cast<const uint2*>(sut + o0), t, u0);
            unit_scales(*reinterpret_cast<const uint2*>(sut + o1), t, u1);
            kunit_mma<NB>(tg, ggu, kGURows, 0, ku, s0, s1, bx[j], ag, ag1, lane);
            kunit_mma<NB>(tu, ggu, kGURows, 0, ku, u0, u1, bx[j], au, au1, lane);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[st]);
      if (threadIdx.x == 0 && l < 11) stamp(17 + 4 * l);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        *reinterpret_cast<float4*>(rb + ((warp * 2 + 0) * NB + nb) * 128 + lane * 4) =
            make_float4(ag[nb][0] + ag1[nb][0], ag[nb][1] + ag1[nb][1], ag[nb][2] + ag1[nb][2],
                        ag[nb][3] + ag1[nb][3]);
        *reinterpret_cast<float4*>(rb + ((warp * 2 + 1) * NB + nb) * 128 + lane * 4) =
            make_float4(au[nb][0] + au1[nb][0], au[nb][1] + au1[nb][1], au[nb][2] + au1[nb][2],
                        au[nb][3] + au1[nb][3]);
      }
      consumer_bar();
      if (threadIdx.x == 0 && l < 11) stamp(18 + 4 * l);
      if (s_abort) break;
      // epilogue: 128 * NB threads; with NB = 1 the two halves of the warps
      // take turns, so each warp's epilogue overlaps the other half's compute
      const int etid = (NB == 1) ? (int)threadIdx.x - 128 * (l & 1) : (int)threadIdx.x;
      if (etid >= 0 && etid < 128 * NB) {
        const int nb = etid >> 7, o = etid & 127;
        const int i = o >> 3, c = o & 7;
        const int n = nb * 8 + c;
        if (n < K) {
          const int fl = (i & 7) * 4 + (c >> 1), fe = (i >> 3) * 2 + (c & 1);
          float gs = 0.f, us = 0.f;
#pragma unroll
          for (int w = 0; w < kExpWarps; ++w) {
            gs += rb[((w * 2 + 0) * NB + nb) * 128 + fl * 4 + fe];
            us += rb[((w * 2 + 1) * NB + nb) * 128 + fl * 4 + fe];
          }
          const float inv = pow2f(-row_shift(s_xamax[n]));
          const int ex = s_uexp[it.slot];
          const float gv = gs * inv * s_tse[3 * ex + 0];
          const float uv = us * inv * s_tse[3 * ex + 1];
          const float hv = gv / (1.f + expf(-gv)) * uv;
          const uint16_t hb = float_to_bf16_bits(hv);
          a.ws.h[((size_t)it.slot * K + n) * I + it.tile * kGURows + i] = hb;
          atomicMax(&a.ws.hamax[it.slot * K + n], (unsigned)(hb & 0x7FFFu));
        }
        pub_slot = it.slot;
        ++pub_count;
      }
      // publish finished items once per slot: at the last item of a slot
      // every warp with items of that slot releases its count (the warp sync
      // makes the release cover every lane's h writes)
      const bool boundary =
          l + 1 == L_gu || plan_item(plan, l + 1, mt_per, n_tiles, a.has_shared, G, n_sh, grid).slot != it.slot;
      if (boundary && pub_count) {
        __syncwarp();
        if (lane == 0) red_release_add(&a.ws.done[pub_slot], pub_count);
        pub_count = 0;
      }
      if (threadIdx.x == 0) stamp(4);
      if (threadIdx.x == 0 && l < 11) stamp(19 + 4 * l);
    }
  }
  for (int l = L_gu; l < L && !s_abort; ++l) {
    const Item it = plan_item(plan, l, mt_per, n_tiles, a.has_shared, G, n_sh, grid);
    const int st = l % kExpStages;
    unsigned char* stg = smem + st * stage_bytes;
    float* rb = red + (size_t)(l & 1) * (8 * 2 * NB * 128);
    {
      // ------------------------------------------------ down item
      if (it.slot != cur_slot) {
        cur_slot = it.slot;
        if (threadIdx.x == 0) {
          const uint64_t t0 = global_timer_ns();
          bool ready = false;
          while (!(ready = ld_acquire(&a.ws.done[it.slot]) >= gu_target)) {
            if (s_abort || a.wait_ns == 0 || global_timer_ns() - t0 > a.wait_ns) break;
          }
          if (!ready) {
            s_abort = 1;
            set_error(a.ws.err, MOE_ERR_DEVICE_TIMEOUT);
          }
          if (trace && trace[5] == 0) {
            trace[5] = t0;
            trace[6] = global_timer_ns();
          }
        }
        consumer_bar();
        if (s_abort) break;
        if (threadIdx.x < K)
          s_hinv[threadIdx.x] = pow2f(-row_shift(__ldcg(a.ws.hamax + it.slot * K + threadIdx.x) << 16));
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const int n = nb * 8 + g;
          const float sc = (n < K) ? pow2f(row_shift(__ldcg(a.ws.hamax + it.slot * K + n) << 16)) : 1.f;
#pragma unroll
          for (int j = 0; j < KUD; ++j) {
            const int ku = kh + 2 * j;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 v = make_uint4(0, 0, 0, 0);
              if (ku < KUdn && n < K)
                v = __ldcg(reinterpret_cast<const uint4*>(a.ws.h + ((size_t)it.slot * K + n) * I + ku * 128 +
                                                          q * 32 + 8 * t));
              bf16x8_to_f16x8(v, sc, &bh[j][nb][q * 4]);
            }
          }
        }
      }
      const bool ok = mbar_wait_bounded(&full_bar[st], (l / kExpStages) & 1, a.wait_ns, &s_abort);
      if (!ok && lane == 0) {
        s_abort = 1;
        set_error(a.ws.err, MOE_ERR_DEVICE_TIMEOUT);
      }
      float acc[NB][4], acc1[NB][4];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nb][i] = acc1[nb][i] = 0.f;
      if (ok) {
        const uint32_t tc = smem_addr(stg);
        const unsigned char* srow = stg + dn_code + (mt * 16 + g) * (I / 16);
#pragma unroll
        for (int j = 0; j < KUD; ++j) {
          const int ku = kh + 2 * j;
          if (ku < KUdn) {
            uint32_t s0[4], s1[4];
            unit_scales(*reinterpret_cast<const uint2*>(srow + 8 * ku), t, s0);
            unit_scales(*reinterpret_cast<const uint2*>(srow + 8 * (I / 16) + 8 * ku), t, s1);
            kunit_mma<NB>(tc, gdn, kDNRows, mt * 16, ku, s0, s1, bh[j], acc, acc1, lane);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[st]);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
        *reinterpret_cast<float4*>(rb + (warp * NB + nb) * 128 + lane * 4) =
            make_float4(acc[nb][0] + acc1[nb][0], acc[nb][1] + acc1[nb][1], acc[nb][2] + acc1[nb][2],
                        acc[nb][3] + acc1[nb][3]);
      consumer_bar();
      if (s_abort) break;
      const float ts = s_tse[3 * s_uexp[it.slot] + 2];
      for (int o = threadIdx.x; o < 4 * NB * 128; o += kConsumerThreads) {
        const int m = o / (NB * 128), rem = o % (NB * 128);
        const int nb = rem >> 7, oo = rem & 127;
        const int i = oo >> 3, c = oo & 7;
        const int n = nb * 8 + c;
        if (n >= K) continue;
        const int s = s_slot[it.slot * K + n];
        if (s < 0) continue;
        const int fl = (i & 7) * 4 + (c >> 1), fe = (i >> 3) * 2 + (c & 1);
        const float v = rb[(m * NB + nb) * 128 + fl * 4 + fe] + rb[((m + 4) * NB + nb) * 128 + fl * 4 + fe];
        a.ws.dpart[((size_t)n * (k + 1) + s) * H + it.tile * kDNRows + m * 16 + i] = v * s_hinv[n] * ts;
      }
    }
  }
  // every CTA's partials are written: grid-wide barrier (the launch is
  // cooperative, all CTAs are resident; the wait is bounded), then CTA b
  // combines hidden tiles b, b + grid, ... :
  //   y = bf16(routed_scale * sum_s w_s d_s + d_shared + residual), slots in order
  consumer_bar();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(a.ws.gridbar, 1u);
    const uint64_t t0 = global_timer_ns();
    while (ld_acquire(a.ws.gridbar) < (unsigned)grid) {
      if (s_abort || a.wait_ns == 0 || global_timer_ns() - t0 > a.wait_ns) {
        s_abort = 1;
        set_error(a.ws.err, MOE_ERR_DEVICE_TIMEOUT);
        break;
      }
    }
    if (trace) trace[60] = global_timer_ns();
  }
  consumer_bar();
  if (!s_abort) {
    for (int tile = blockIdx.x; tile < n_tiles; tile += grid) {
      for (int o = threadIdx.x; o < K * kDNRows; o += kConsumerThreads) {
        const int n = o / kDNRows, j = tile * kDNRows + o % kDNRows;
        float acc2 = 0.f;
        for (int s = 0; s < k; ++s)
          acc2 = __fmaf_rn(s_w[n * k + s], __ldcg(a.ws.dpart + ((size_t)n * (k + 1) + s) * H + j), acc2);
        float v = a.routed_scale * acc2;
        if (a.has_shared) v += __ldcg(a.ws.dpart + ((size_t)n * (k + 1) + k) * H + j);
        if (a.residual) v += bf16_bits_to_float(a.residual[(size_t)n * H + j]);
        a.y[(size_t)n * H + j] = float_to_bf16_bits(v);
      }
    }
  }
  if (threadIdx.x == 0) {
    stamp(7);
    if (trace) trace[8] = (unsigned long long)L | ((unsigned long long)plan.n_shb << 16) |
                          ((unsigned long long)(plan.gu1 - plan.gu0) << 24) |
                          ((unsigned long long)(plan.dn1 - plan.dn0) << 40);
  }
}

// =====================================================================
// launcher
// =====================================================================

static int g_num_sms = 0;

int num_sms() {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 1;
  }
  return g_num_sms;
}

size_t experts_smem_bytes(int K, int H, int I, int E, int k, int G) {
  const int NB = K > 8 ? 2 : 1;
  size_t s = 1024 + (size_t)kExpStages * expert_stage_bytes(H, I) + sizeof(float) * 2 * 8 * 2 * NB * 128;
  s += sizeof(float) * K * k + sizeof(int) * K * k + sizeof(unsigned) * E + sizeof(int) * E + sizeof(int) * (G + 1) +
       sizeof(float) * 3 * (G + 1) + sizeof(float) * 3 * (E + 1) + (size_t)(G + 1) * K;
  return s;
}

template <int NB, int KUG, int KUD>
static cudaError_t launch_experts_t(const ExpertsArgs& a, const CUtensorMap* maps, cudaStream_t s, bool pdl) {
  auto kern = k_moe_experts<NB, KUG, KUD>;
  const size_t smem = experts_smem_bytes(a.K, a.H, a.I, a.E, a.k, a.G);
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  err = cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7],
                           maps[8], maps[9], a);
  if (err != cudaSuccess && pdl) {  // fall back to a cooperative launch without overlap
    cudaGetLastError();
    attr[0].val.programmaticStreamSerializationAllowed = 0;
    err = cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7],
                             maps[8], maps[9], a);
  }
  return err;
}

cudaError_t launch_experts(const ExpertsArgs& a, const CUtensorMap* maps, cudaStream_t s, bool pdl) {
  const bool nb2 = a.K > 8;
  const bool kug2 = a.H > 1024;
  const bool kud2 = a.I > 256;
  if (!nb2) {
    if (kug2) return kud2 ? launch_experts_t<1, 2, 2>(a, maps, s, pdl) : launch_experts_t<1, 2, 1>(a, maps, s, pdl);
    return kud2 ? launch_experts_t<1, 1, 2>(a, maps, s, pdl) : launch_experts_t<1, 1, 1>(a, maps, s, pdl);
  }
  if (kug2) return kud2 ? launch_experts_t<2, 2, 2>(a, maps, s, pdl) : launch_experts_t<2, 2, 1>(a, maps, s, pdl);
  return kud2 ? launch_experts_t<2, 1, 2>(a, maps, s, pdl) : launch_experts_t<2, 1, 1>(a, maps, s, pdl);
}

}  // namespace moe
