// experts.cu -- NVFP4 expert GEMVs over the distinct experts of a verify call.
//
// Both kernels are persistent (one CTA per SM): a producer warp streams the
// weight tiles of consecutive work items into a ring of shared-memory stages
// with TMA (2-D tiled copies, 128-byte swizzle, for the 4-bit codes; 1-D bulk
// copies for the E4M3 scales), and eight consumer warps decode and multiply.
//
// Decode: ldmatrix pulls 32 bits of codes per thread and row; the hardware
// FP4 -> FP16 convert turns 8 codes into four f16x2, and one f16x2 multiply
// by the block's E4M3 scale (converted to FP16) gives the exact element
// (e2m1 * e4m3 has at most 6 significant bits and lies in [2^-10, 2688]).
// The tensor-core mma.sync m16n8k16 then multiplies 16 weight rows by the
// verify rows (the n = 8 or 16 columns), accumulating in FP32; the FP32
// tensor scale is applied to the accumulator.  Because a dot product may sum
// over k in any order, the k index of an mma step is a permutation of the
// physical k: thread t's fragment elements come from its own 8 consecutive
// codes (one 32-bit word), which keeps every load 32-bit and bank-conflict
// free and gives each thread a single scale per 16-byte unit.
//
// Activations enter as FP16 after an exact per-row power-of-two rescaling
// (max |value| mapped into [2^14, 2^15)), which keeps any bf16 row inside
// FP16 range without rounding; the inverse power of two is applied in FP32.
//
// Work items: gate/up -- (expert, 16 intermediate rows), both projections;
// down -- (expert, 64 hidden rows).  Each CTA takes a contiguous range of
// items, so consecutive items mostly share an expert.  Every distinct expert
// is read exactly once per call however many rows chose it (PR #844,
// "8. What I looked at": the stock gather re-reads an expert per (row, slot)).
//
// Combine (down kernel): per-(row, slot) FP32 partials, then the CTA that
// completes the last item of a 64-row hidden tile (atomic count, no waiting)
// forms y = bf16(routed_scale * sum_s w_s d_s + d_shared + residual) in slot
// order (PR #844, "4. What I ported": weighted sum, x2.5 routed scale,
// shared add, residual add -- one pass, fixed order).
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

// 8 bf16 (one uint4) * 2^shift -> 4 f16x2.
__device__ __forceinline__ void bf16x8_to_f16x8(const uint4 v, float scale, uint32_t* out) {
  const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    out[i] = pack_f16x2(__uint_as_float(q[i] << 16) * scale, __uint_as_float(q[i] & 0xFFFF0000u) * scale);
}

// Tile geometry of one projection's codes in shared memory: `chunks` TMA
// boxes of [box_rows][inner bytes], box c at c * box_rows * inner.
struct TileGeo {
  int inner;   // 128 or 64 bytes
  int mask;    // swizzle mask: 7 (128B) or 3 (64B)
  int units;   // 16-byte units per line = inner / 16
  int chunks;  // row bytes / inner
};

__device__ __forceinline__ TileGeo tile_geo(int cols) {
  TileGeo g;
  const int rb = cols / 2;
  g.inner = rb >= 128 ? 128 : 64;
  g.mask = g.inner == 128 ? 7 : 3;
  g.units = g.inner / 16;
  g.chunks = rb / g.inner;
  return g;
}

// One k-unit (128 k) of a 16-row m-tile against NB n-blocks of resident B.
//   tile:   shared address of the codes tile, box_rows rows per box
//   srow_g: shared pointer to row g's scales (row stride `sstride` bytes)
//   b:      B fragments of this k-unit, [NB][4 units][4 regs]
template <int NB>
__device__ __forceinline__ void kunit_mma(uint32_t tile, const TileGeo& geo, int box_rows, int row0, int ku,
                                          const unsigned char* srow_g, int sstride, const uint32_t (&b)[NB][16],
                                          float (&acc)[NB][4], int lane) {
  const int t = lane & 3;
  const int q0 = (ku * 4) % geo.units;
  const int c = (ku * 4) / geo.units;
  const int mi = lane >> 3, rr = lane & 7;
  const int lrow = row0 + rr + 8 * (mi & 1);
  // scales of rows g and g+8 for the 4 units: block = c*inner/8 + 2q + t/2
  const int blk0 = c * geo.inner / 8 + 2 * q0 + (t >> 1);
  uint32_t sg[4], sh[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    sg[q] = e4m3_to_f16x2_dup(srow_g[blk0 + 2 * q]);
    sh[q] = e4m3_to_f16x2_dup(srow_g[8 * sstride + blk0 + 2 * q]);
  }
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
      for (int nb = 0; nb < NB; ++nb) {
        mma_f16(acc[nb], dg[0], dh[0], dg[1], dh[1], b[nb][q * 4 + 0], b[nb][q * 4 + 1]);
        mma_f16(acc[nb], dg[2], dh[2], dg[3], dh[3], b[nb][q * 4 + 2], b[nb][q * 4 + 3]);
      }
    }
  }
}

struct Range {
  int begin, end;
};

__device__ __forceinline__ Range cta_range(int n_items) {
  Range r;
  r.begin = (int)(((long long)blockIdx.x * n_items) / gridDim.x);
  r.end = (int)(((long long)(blockIdx.x + 1) * n_items) / gridDim.x);
  return r;
}

}  // namespace

// =====================================================================
// gate/up + SwiGLU
// =====================================================================
//
// Item i < n_sh: shared expert rows [16 i, 16 i + 16); then routed items
// (u, mt) for the n_u distinct experts.  Output: h[slot][row n][I] (bf16) for
// all K rows, slot = u (routed) or G (shared), and hamax[slot][n].
template <int NB, int KUW>
__global__ void __launch_bounds__(kThreads, 1)
    k_gateup(const __grid_constant__ CUtensorMap tm_gate, const __grid_constant__ CUtensorMap tm_up,
             const __grid_constant__ CUtensorMap tm_sgate, const __grid_constant__ CUtensorMap tm_sup,
             GateUpArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kGUStages], empty_bar[kGUStages];
  __shared__ unsigned s_xamax[16];
  __shared__ int s_abort;

  const int H = a.H, I = a.I, K = a.K, G = a.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TileGeo geo = tile_geo(H);
  const int code_bytes = kGURows * H / 2;  // one projection's codes per item
  const int scale_bytes = kGURows * H / 16;
  const int stage_bytes = ((2 * code_bytes + 2 * scale_bytes) + 1023) & ~1023;
  float* red = reinterpret_cast<float*>(smem + kGUStages * stage_bytes);  // [2][8][2][NB][32][4]

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGUStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kGUWarps);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < 16) s_xamax[threadIdx.x] = 0u;
  __syncthreads();

  pdl_wait();  // routing of this call is complete and visible
  pdl_launch_dependents();

  const int n_sh = a.has_shared ? I / kGURows : 0;
  const int n_u = __ldcg(a.ws.group);
  const int mt_per = I / kGURows;
  const int n_items = n_sh + n_u * mt_per;
  const Range rg = cta_range(n_items);

  if (warp == kGUWarps) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
      prefetch_tensormap(&tm_gate);
      prefetch_tensormap(&tm_up);
    }
    int issued = 0;
    for (int it = rg.begin; it < rg.end; ++it, ++issued) {
      const int st = issued % kGUStages;
      int ok = 1;
      if (lane == 0 && issued >= kGUStages) {
        if (!mbar_wait_bounded(&empty_bar[st], ((issued / kGUStages) - 1) & 1, a.wait_ns, &s_abort)) {
          ok = 0;
          s_abort = 1;
          set_error(a.ws.err, MOE_ERR_DEVICE_TIMEOUT);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok || s_abort) break;
      const bool sh = it < n_sh;
      int row0;
      const CUtensorMap *mg, *mu;
      const unsigned char *sgp, *sup;
      if (sh) {
        row0 = it * kGURows;
        mg = &tm_sgate;
        mu = &tm_sup;
        sgp = a.sh_gate.scales;
        sup = a.sh_up.scales;
      } else {
        const int v = it - n_sh;
        const int e = __ldcg(a.ws.group + 1 + v / mt_per);
        row0 = e * I + (v % mt_per) * kGURows;
        mg = &tm_gate;
        mu = &tm_up;
        sgp = a.gate.scales;
        sup = a.up.scales;
      }
      unsigned char* stg = smem + st * stage_bytes;
      if (lane == 0) mbar_arrive_expect_tx(&full_bar[st], 2 * code_bytes + 2 * scale_bytes);
      __syncwarp();
      if (lane < geo.chunks)
        tma_load_2d(stg + lane * kGURows * geo.inner, mg, lane * geo.inner, row0, &full_bar[st], pol);
      else if (lane >= 16 && lane < 16 + geo.chunks)
        tma_load_2d(stg + code_bytes + (lane - 16) * kGURows * geo.inner, mu, (lane - 16) * geo.inner, row0,
                    &full_bar[st], pol);
      else if (lane == 30)
        bulk_load(stg + 2 * code_bytes, sgp + (size_t)row0 * (H / 16), scale_bytes, &full_bar[st], pol);
      else if (lane == 31)
        bulk_load(stg + 2 * code_bytes + scale_bytes, sup + (size_t)row0 * (H / 16), scale_bytes, &full_bar[st],
                  pol);
      __syncwarp();
    }
    // drain: our copies must land before the CTA exits
    if (lane == 0) {
      for (int j = (issued > kGUStages ? issued - kGUStages : 0); j < issued; ++j)
        mbar_wait_bounded(&full_bar[j % kGUStages], (j / kGUStages) & 1, kDrainNs, &s_abort);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  const int KU = H / 128;
  // resident activations: B fragments of this warp's k-units
  uint32_t bx[KUW][NB][16];
  {
    uint4 raw[KUW][NB][4];
    unsigned mx = 0;
#pragma unroll
    for (int j = 0; j < KUW; ++j) {
      const int ku = warp + kGUWarps * j;
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
    // per-row max |x| (rows n = nb*8+g): thread partial -> shuffle over t -> smem
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      mx = 0;
#pragma unroll
      for (int j = 0; j < KUW; ++j)
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
      const int sft = (n < K) ? row_shift(s_xamax[n]) : 0;
      const float sc = pow2f(sft);
#pragma unroll
      for (int j = 0; j < KUW; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) bf16x8_to_f16x8(raw[j][nb][q], sc, &bx[j][nb][q * 4]);
    }
  }

  const int sstride = H / 16;
  int local = 0;
  for (int it = rg.begin; it < rg.end; ++it, ++local) {
    const int st = local % kGUStages;
    const bool ok = mbar_wait_bounded(&full_bar[st], (local / kGUStages) & 1, a.wait_ns, &s_abort);
    if (!ok && lane == 0) {
      s_abort = 1;
      set_error(a.ws.err, MOE_ERR_DEVICE_TIMEOUT);
    }
    float ag[NB][4], au[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i) ag[nb][i] = au[nb][i] = 0.f;
    if (ok) {
      unsigned char* stg = smem + st * stage_bytes;
      const uint32_t tg = smem_addr(stg), tu = smem_addr(stg + code_bytes);
      const unsigned char* sg_row = stg + 2 * code_bytes + g * sstride;
      const unsigned char* su_row = stg + 2 * code_bytes + scale_bytes + g * sstride;
#pragma unroll
      for (int j = 0; j < KUW; ++j) {
        const int ku = warp + kGUWarps * j;
        if (ku < KU) {
          kunit_mma<NB>(tg, geo, kGURows, 0, ku, sg_row, sstride, bx[j], ag, lane);
          kunit_mma<NB>(tu, geo, kGURows, 0, ku, su_row, sstride, bx[j], au, lane);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[st]);
    // cross-warp reduction (fixed order over warps)
    float* rb = red + (size_t)(local & 1) * (kGUWarps * 2 * NB * 128);
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      *reinterpret_cast<float4*>(rb + ((warp * 2 + 0) * NB + nb) * 128 + lane * 4) =
          make_float4(ag[nb][0], ag[nb][1], ag[nb][2], ag[nb][3]);
      *reinterpret_cast<float4*>(rb + ((warp * 2 + 1) * NB + nb) * 128 + lane * 4) =
          make_float4(au[nb][0], au[nb][1], au[nb][2], au[nb][3]);
    }
    consumer_bar();
    if (s_abort) break;
    const int tid = threadIdx.x;
    if (tid < 128 * NB) {
      const int nb = tid >> 7, o = tid & 127;
      const int i = o >> 3, c = o & 7;
      const int n = nb * 8 + c;
      if (n < K) {
        const int fl = (i & 7) * 4 + (c >> 1), fe = (i >> 3) * 2 + (c & 1);
        float gs = 0.f, us = 0.f;
#pragma unroll
        for (int w = 0; w < kGUWarps; ++w) {
          gs += rb[((w * 2 + 0) * NB + nb) * 128 + fl * 4 + fe];
          us += rb[((w * 2 + 1) * NB + nb) * 128 + fl * 4 + fe];
        }
        const bool sh = it < n_sh;
        int slot, mt;
        float tsg, tsu;
        if (sh) {
          slot = G;
          mt = it;
          tsg = a.sh_gate.tscale[0];
          tsu = a.sh_up.tscale[0];
        } else {
          const int v = it - n_sh;
          slot = v / mt_per;
          mt = v % mt_per;
          const int e = __ldcg(a.ws.group + 1 + slot);
          tsg = a.gate.tscale[e];
          tsu = a.up.tscale[e];
        }
        const float inv = pow2f(-row_shift(s_xamax[n]));
        const float gv = gs * inv * tsg;
        const float uv = us * inv * tsu;
        const float hv = gv / (1.f + expf(-gv)) * uv;
        const uint16_t hb = float_to_bf16_bits(hv);
        a.ws.h[((size_t)slot * K + n) * I + mt * kGURows + i] = hb;
        atomicMax(&a.ws.hamax[slot * K + n], (unsigned)(hb & 0x7FFFu));
      }
    }
  }
}

// =====================================================================
// down + combine
// =====================================================================
//
// Items: (slot index si, hidden tile); si < n_u routed, si == n_u shared.
// dpart[n][s][H]: FP32 partial of row n's slot s (s = k: shared expert).
template <int NB, int KUW>
__global__ void __launch_bounds__(kThreads, 1)
    k_down(const __grid_constant__ CUtensorMap tm_down, const __grid_constant__ CUtensorMap tm_sdown, DownArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kDNStages], empty_bar[kDNStages];
  __shared__ int s_abort, s_combine;

  const int H = a.H, I = a.I, K = a.K, G = a.G, k = a.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TileGeo geo = tile_geo(I);
  const int code_bytes = kDNRows * I / 2;
  const int scale_bytes = kDNRows * I / 16;
  const int stage_bytes = ((code_bytes + scale_bytes) + 1023) & ~1023;
  float* red = reinterpret_cast<float*>(smem + kDNStages * stage_bytes);  // [2][8][NB][32][4]

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDNStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kDNWarps);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  pdl_wait();
  pdl_launch_dependents();

  const int n_u = __ldcg(a.ws.group);
  const int n_tiles = H / kDNRows;
  const int n_slots = n_u + (a.has_shared ? 1 : 0);
  const int n_items = n_slots * n_tiles;
  const Range rg = cta_range(n_items);

  if (warp == kDNWarps) {
    const uint64_t pol = policy_evict_first();
    if (lane == 0) prefetch_tensormap(&tm_down);
    int issued = 0;
    for (int it = rg.begin; it < rg.end; ++it, ++issued) {
      const int st = issued % kDNStages;
      int ok = 1;
      if (lane == 0 && issued >= kDNStages) {
        if (!mbar_wait_bounded(&empty_bar[st], ((issued / kDNStages) - 1) & 1, a.wait_ns, &s_abort)) {
          ok = 0;
          s_abort = 1;
          set_error(a.ws.err, MOE_ERR_DEVICE_TIMEOUT);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok || s_abort) break;
      const int si = it / n_tiles, tile = it % n_tiles;
      const bool sh = si == n_u;
      const int e = sh ? 0 : __ldcg(a.ws.group + 1 + si);
      const int row0 = e * H + tile * kDNRows;
      const CUtensorMap* m = sh ? &tm_sdown : &tm_down;
      const unsigned char* sp = sh ? a.sh_down.scales : a.down.scales;
      unsigned char* stg = smem + st * stage_bytes;
      if (lane == 0) mbar_arrive_expect_tx(&full_bar[st], code_bytes + scale_bytes);
      __syncwarp();
      if (lane < geo.chunks)
        tma_load_2d(stg + lane * kDNRows * geo.inner, m, lane * geo.inner, row0, &full_bar[st], pol);
      else if (lane == 31)
        bulk_load(stg + code_bytes, sp + (size_t)row0 * (I / 16), scale_bytes, &full_bar[st], pol);
      __syncwarp();
    }
    if (lane == 0) {
      for (int j = (issued > kDNStages ? issued - kDNStages : 0); j < issued; ++j)
        mbar_wait_bounded(&full_bar[j % kDNStages], (j / kDNStages) & 1, kDrainNs, &s_abort);
    }
    return;
  }

  const int g = lane >> 2, t = lane & 3;
  const int KU = I / 128;
  const int mt = warp & 3;         // m-tile of 16 rows inside the 64-row item
  const int kh = warp >> 2;        // k-units kh, kh+2, ...
  const int sstride = I / 16;
  uint32_t bh[KUW][NB][16];
  int cur_si = -1;
  int local = 0;
  for (int it = rg.begin; it < rg.end; ++it, ++local) {
    const int si = it / n_tiles, tile = it % n_tiles;
    const bool sh = si == n_u;
    const int slot = sh ? G : si;
    if (si != cur_si) {  // load this expert's h rows as FP16 B fragments
      cur_si = si;
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const int n = nb * 8 + g;
        const float sc = (n < K) ? pow2f(row_shift(__ldcg(a.ws.hamax + slot * K + n) << 16)) : 1.f;
#pragma unroll
        for (int j = 0; j < KUW; ++j) {
          const int ku = kh + 2 * j;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (ku < KU && n < K)
              v = __ldcg(reinterpret_cast<const uint4*>(a.ws.h + ((size_t)slot * K + n) * I + ku * 128 + q * 32 + 8 * t));
            bf16x8_to_f16x8(v, sc, &bh[j][nb][q * 4]);
          }
        }
      }
    }
    const int st = local % kDNStages;
    const bool ok = mbar_wait_bounded(&full_bar[st], (local / kDNStages) & 1, a.wait_ns, &s_abort);
    if (!ok && lane == 0) {
      s_abort = 1;
      set_error(a.ws.err, MOE_ERR_DEVICE_TIMEOUT);
    }
    float acc[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nb][i] = 0.f;
    if (ok) {
      unsigned char* stg = smem + st * stage_bytes;
      const uint32_t tc = smem_addr(stg);
      const unsigned char* s_row = stg + code_bytes + (mt * 16 + g) * sstride;
#pragma unroll
      for (int j = 0; j < KUW; ++j) {
        const int ku = kh + 2 * j;
        if (ku < KU) kunit_mma<NB>(tc, geo, kDNRows, mt * 16, ku, s_row, sstride, bh[j], acc, lane);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[st]);
    float* rb = red + (size_t)(local & 1) * (kDNWarps * NB * 128);
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
      *reinterpret_cast<float4*>(rb + (warp * NB + nb) * 128 + lane * 4) =
          make_float4(acc[nb][0], acc[nb][1], acc[nb][2], acc[nb][3]);
    consumer_bar();
    if (s_abort) break;
    // 4 m-tiles x NB n-blocks x 128 outputs; warps (m, m+4) hold the two halves of k
    const float ts = sh ? a.sh_down.tscale[0] : a.down.tscale[__ldcg(a.ws.group + 1 + si)];
    for (int o = threadIdx.x; o < 4 * NB * 128; o += kConsumerThreads) {
      const int m = o / (NB * 128), rem = o % (NB * 128);
      const int nb = rem >> 7, oo = rem & 127;
      const int i = oo >> 3, c = oo & 7;
      const int n = nb * 8 + c;
      if (n >= K) continue;
      const int s = __ldcg(a.ws.slotmap + slot * K + n);
      if (s < 0) continue;
      const int fl = (i & 7) * 4 + (c >> 1), fe = (i >> 3) * 2 + (c & 1);
      const float v = rb[(m * NB + nb) * 128 + fl * 4 + fe] + rb[((m + 4) * NB + nb) * 128 + fl * 4 + fe];
      const float inv = pow2f(-row_shift(__ldcg(a.ws.hamax + slot * K + n) << 16));
      a.ws.dpart[((size_t)n * (k + 1) + s) * H + tile * kDNRows + m * 16 + i] = v * inv * ts;
    }
    __threadfence();
    consumer_bar();
    if (threadIdx.x == 0) {
      const unsigned done = atomicAdd(&a.ws.tilecnt[tile], 1u);
      s_combine = (done == (unsigned)(n_slots - 1));
    }
    consumer_bar();
    if (s_combine) {
      __threadfence();
      for (int o = threadIdx.x; o < K * kDNRows; o += kConsumerThreads) {
        const int n = o / kDNRows, j = tile * kDNRows + o % kDNRows;
        float acc2 = 0.f;
        for (int s = 0; s < k; ++s)
          acc2 = __fmaf_rn(__ldcg(a.ws.w + n * k + s), __ldcg(a.ws.dpart + ((size_t)n * (k + 1) + s) * H + j), acc2);
        float v = a.routed_scale * acc2;
        if (a.has_shared) v += __ldcg(a.ws.dpart + ((size_t)n * (k + 1) + k) * H + j);
        if (a.residual) v += bf16_bits_to_float(a.residual[(size_t)n * H + j]);
        a.y[(size_t)n * H + j] = float_to_bf16_bits(v);
      }
      if (threadIdx.x == 0) a.ws.tilecnt[tile] = 0u;
    }
  }
}

// =====================================================================
// launchers
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

template <typename Kern, typename... Args>
static cudaError_t launch_persistent(Kern kern, size_t smem, cudaStream_t s, bool pdl, Args... args) {
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

cudaError_t launch_gateup(const GateUpArgs& a, const CUtensorMap& gate, const CUtensorMap& up,
                          const CUtensorMap& sh_gate, const CUtensorMap& sh_up, cudaStream_t s, bool pdl) {
  const int stage = ((2 * kGURows * a.H / 2 + 2 * kGURows * a.H / 16) + 1023) & ~1023;
  const int NB = a.K > 8 ? 2 : 1;
  const size_t smem = 1024 + (size_t)kGUStages * stage + sizeof(float) * 2 * kGUWarps * 2 * NB * 128;
  const bool kuw2 = a.H > 1024;
  if (NB == 1)
    return kuw2 ? launch_persistent(k_gateup<1, 2>, smem, s, pdl, gate, up, sh_gate, sh_up, a)
                : launch_persistent(k_gateup<1, 1>, smem, s, pdl, gate, up, sh_gate, sh_up, a);
  return kuw2 ? launch_persistent(k_gateup<2, 2>, smem, s, pdl, gate, up, sh_gate, sh_up, a)
              : launch_persistent(k_gateup<2, 1>, smem, s, pdl, gate, up, sh_gate, sh_up, a);
}

cudaError_t launch_down(const DownArgs& a, const CUtensorMap& down, const CUtensorMap& sh_down, cudaStream_t s,
                        bool pdl) {
  const int stage = ((kDNRows * a.I / 2 + kDNRows * a.I / 16) + 1023) & ~1023;
  const int NB = a.K > 8 ? 2 : 1;
  const size_t smem = 1024 + (size_t)kDNStages * stage + sizeof(float) * 2 * kDNWarps * NB * 128;
  const bool kuw2 = a.I > 256;
  if (NB == 1)
    return kuw2 ? launch_persistent(k_down<1, 2>, smem, s, pdl, down, sh_down, a)
                : launch_persistent(k_down<1, 1>, smem, s, pdl, down, sh_down, a);
  return kuw2 ? launch_persistent(k_down<2, 2>, smem, s, pdl, down, sh_down, a)
              : launch_persistent(k_down<2, 1>, smem, s, pdl, down, sh_down, a);
}

}  // namespace moe
