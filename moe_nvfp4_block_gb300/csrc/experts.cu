// experts.cu -- one MoE verify-layer call in one persistent kernel: router
// logits, top-k routing and grouping, the NVFP4 experts, and the combine.
//
// One CTA per SM: a producer warp streams weight tiles into a ring of shared
// memory stages with TMA (tiled copies with swizzle for the 4-bit codes
// and the gate/up E4M3 scales, 1-D bulk copies for the down scales) and
// sixteen compute warps decode and multiply.  The CTA's work is a fixed
// sequence of items: its shared-expert gate/up items, its routed gate/up
// items, then its down items.  Every distinct expert is streamed exactly once
// per call however many rows chose it (PR #844, "8. What I looked at": the
// stock gather re-reads an expert once per (row, slot)).
//
// Router: the CTAs share the K x E logits (each forms those of its own
// experts, in the fixed order of the router GEMV, and publishes them as
// tagged words), then every CTA reads all of them and computes the same
// routing (top-k with lower-index tie-break, renormalised softmax weights,
// grouping) on its own -- no second kernel, no serial hand-off.  Before the
// programmatic-launch wait the producer already streams the shared expert's
// first tiles and the compute warps hold their router rows.
//
// Exchange between CTAs: h (gate/up -> down), the down partials (down ->
// combine) and the logits are tagged 64-bit words (the call's tag next to a
// 32-bit payload), so a reader validates each word itself: no fences, no
// grid barrier, no per-call clearing.  Relaxed counters, cleared a call
// ahead, only tell readers when to look.
//
// Decode: ldmatrix pulls 32 bits of codes per thread and row; the hardware
// FP4 -> FP16 convert turns 8 codes into four f16x2, and one f16x2 multiply
// by the block's E4M3 scale gives the exact element (e2m1 * e4m3 has at most
// 6 significant bits and lies in [2^-10, 2688]).  mma.sync m16n8k16 then
// multiplies 16 weight rows by the verify rows (n = 8 or 16 columns) with
// FP32 accumulation; the tensor scale is applied to the accumulator.  The k
// index of an mma step is a permutation of the physical k (any order is a
// valid dot product): thread t's elements are its own 8 consecutive codes.
// Activations enter as FP16 after an exact power-of-two rescaling (per row;
// h per row and 128-wide k-unit), undone in FP32.
//
// Combine: per-(row, slot) FP32 partials; the outputs are shared by the CTAs,
// y = bf16(routed_scale * sum_s w_s d_s + d_shared + residual) in slot order,
// every FP32 operation rounded on its own
// (PR #844, "4. What I ported": weighted sum, routed scale, shared add,
// residual add in one pass).
#include <cfloat>
#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

// Warp roles: kCompWarps compute warps (warp w decodes and multiplies
// k-unit w, 128 wide, of every item, so H <= 2048, and reduces its share of
// every item's outputs) and one producer warp that issues the TMA copies.
constexpr int kCompWarps = 16;
constexpr int kCompThreads = kCompWarps * 32;
constexpr int kProducerWarp = kCompWarps;
constexpr int kThreads = kCompThreads + 32;
constexpr uint64_t kDrainNs = 2000000000ull;  // bound on waiting for our own copies before exit

// named barrier 1: the compute warps
__device__ __forceinline__ void comp_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kCompThreads) : "memory"); }

__device__ __forceinline__ void set_error(int* err, int code) { atomicCAS(err, 0, code); }

// Tagged words: a 32-bit payload in the low half and the call's tag in the
// high half, written and read as one naturally aligned 64-bit access, which
// is single-copy atomic.  A reader that sees this call's tag sees the payload
// written with it, so the words need no fence and no flag, and stale words
// of earlier calls (older tags) need no clearing.  Counters only tell a
// reader when to look.
__device__ __forceinline__ unsigned long long tagged(unsigned tag, unsigned v) {
  return ((unsigned long long)tag << 32) | v;
}
__device__ __forceinline__ bool has_tag(unsigned long long w, unsigned tag) { return (unsigned)(w >> 32) == tag; }

__device__ __forceinline__ void st_tagged(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// The same by an atomic exchange, for words every CTA waits on at once (the
// router logits): plain stores from some SMs reached readers on other SMs
// microseconds late on this two-die part, while atomics, performed where the
// line lives, were visible at the next read.
__device__ __forceinline__ void xchg_tagged(unsigned long long* p, unsigned long long v) {
  unsigned long long prev;
  asm volatile("atom.relaxed.gpu.global.exch.b64 %0, [%1], %2;" : "=l"(prev) : "l"(p), "l"(v) : "memory");
  (void)prev;
}

__device__ __forceinline__ unsigned long long ld_tagged(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Two consecutive tagged words (16-byte aligned); each element is one
// 64-bit access.
__device__ __forceinline__ void ld_tagged2(const unsigned long long* p, unsigned long long& a, unsigned long long& b) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
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
// order: lane s (< 8) gets the s-th into `mine`, every lane the first into
// `first`.  A lane-local bitonic sort puts each lane's best first, then 8
// rounds of a warp arg-max, each two redux.sync max steps (the high word,
// then the low word among the lanes holding the high word's maximum; the low
// word encodes the expert index, so the maximum key is unique) after which
// its lane drops it.
__device__ __forceinline__ void warp_top8(unsigned long long (&v)[8], int lane, unsigned long long& mine,
                                          unsigned long long& first) {
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
  mine = 0ull;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const unsigned hi = (unsigned)(v[0] >> 32), lo = (unsigned)v[0];
    const unsigned mh = __reduce_max_sync(0xffffffffu, hi);
    const unsigned ml = __reduce_max_sync(0xffffffffu, hi == mh ? lo : 0u);
    const unsigned long long key = ((unsigned long long)mh << 32) | ml;
    if (s == 0) first = key;
    if (lane == s) mine = key;
    if (hi == mh && lo == ml) {
#pragma unroll
      for (int i = 0; i < 7; ++i) v[i] = v[i + 1];
      v[7] = 0ull;
    }
  }
}

// Whether a warp's bounded wait that began at t0 gives up now (the abort
// flag is set, or the limit has passed): lane 0 decides for the warp.
__device__ __forceinline__ bool warp_gives_up(uint64_t t0, uint64_t wait_ns, const int* abort_flag, int lane) {
  int stop = 0;
  if (lane == 0)
    stop = *reinterpret_cast<const volatile int*>(abort_flag) != 0 || wait_ns == 0 || global_timer_ns() - t0 > wait_ns;
  return __shfl_sync(0xffffffffu, stop, 0) != 0;
}

// Top-k of one row of E tagged logits for any E <= 1024, k <= 32 (lane l
// holds experts l + 32 i), read once every word carries `tag` (a bounded
// wait; false if it gave up): k rounds of a warp arg-max, larger logit first
// and lower index on ties; NaN logits rank last, lowest index first.  Lane 0
// writes the selected experts and their keys.  With `sel_bias` (sigmoid
// scoring) the words hold scores and the keys are score + bias.
__device__ __noinline__ bool topk_general(const unsigned long long* row, unsigned tag, uint64_t wait_ns,
                                          const int* abort_flag, int E, int k, int* idx, float* w,
                                          const float* sel_bias, int lane) {
  float lv[32];
  unsigned taken = 0;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    bool mine = true;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int e = lane + 32 * i;
      float v = -INFINITY;
      if (e < E) {
        const unsigned long long wv = ld_tagged(row + e);
        mine &= has_tag(wv, tag);
        v = __uint_as_float((unsigned)wv);
        if (sel_bias) v = __fadd_rn(v, sel_bias[e]);  // sigmoid scoring: selection key = score + bias
      }
      lv[i] = v;
    }
    if (__all_sync(0xffffffffu, mine)) break;
    if (warp_gives_up(t0, wait_ns, abort_flag, lane)) return false;
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
      idx[s] = be;
      w[s] = bv;  // logit for now
    }
  }
  return true;
}

// Routing of row r when E <= 256 and k <= 8 (one warp, in its own function
// so that its registers do not weigh on the item loops): waits (bounded)
// until the row's tagged logits all carry `tag`, selects the top k, and
// writes the renormalised weights, the experts and the row's bits of the
// expert masks.  Softmax scoring: the words are logits (bias included), the
// weights the softmax over the selection.  Sigmoid scoring: the words are
// scores, the keys score + bias, the weights the selected scores over their
// sum.  On giving up it writes experts 0 .. k-1 (in range for the tables)
// and returns false.
__device__ __noinline__ bool route_row_fast(const unsigned long long* row, unsigned tag, int E, int k, int r,
                                            uint64_t wait_ns, const int* abort_flag, int* s_idx, float* s_w,
                                            unsigned* s_rowmask, unsigned* s_used, int scoring,
                                            const float* sel_bias, int lane) {
  bool got = true;
  unsigned long long v[8];
  float sc[8];  // sigmoid scoring: the raw scores of this lane's experts
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    bool mine = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      v[i] = 0ull;
      sc[i] = 0.f;
      if (e < E) {
        const unsigned long long wv = ld_tagged(row + e);
        mine &= has_tag(wv, tag);
        const float val = __uint_as_float((unsigned)wv);
        sc[i] = val;
        v[i] = sel_key(scoring && sel_bias ? __fadd_rn(val, sel_bias[e]) : val, e);
      }
    }
    if (__all_sync(0xffffffffu, mine)) break;
    if (warp_gives_up(t0, wait_ns, abort_flag, lane)) {
      got = false;
      break;
    }
  }
  unsigned long long sel, first;  // lane s < k takes selection s
  warp_top8(v, lane, sel, first);
  const int sel_e = got ? key_index(sel) : lane;
  float ev;
  if (scoring) {
    // the selected expert's own score (not its key) from the lane holding it
    float mys = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float t = __shfl_sync(0xffffffffu, sc[i], sel_e & 31);
      if (i == (sel_e >> 5)) mys = t;
    }
    ev = (lane < k && got) ? mys : 0.f;
  } else {
    // renormalised softmax over the selected logits (selections live in
    // lanes < k; the others add exact zeros to the sum)
    const float top = key_value(first);
    ev = (lane < k && got) ? expf(key_value(sel) - top) : 0.f;
  }
  float z = ev;
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
  if (lane < k) {
    s_idx[r * k + lane] = sel_e;
    s_w[r * k + lane] = got ? ev / z : 0.f;
    atomicOr(&s_rowmask[sel_e], 1u << r);
    atomicOr(&s_used[sel_e >> 5], 1u << (sel_e & 31));
  }
  return got;
}

// The grouping of one call for the caller (one warp): the distinct experts,
// the (row, slot) pairs before each, and each expert's pairs r * k + slot in
// row order.
__device__ __noinline__ void write_groups(int* go, int nu, int G, int K, int k, const int* uexp,
                                         const unsigned* rowmask, const signed char* slot, int lane) {
  if (lane == 0) {
    go[0] = nu;
    go[1 + 2 * G] = K * k;
  }
  int before = 0;
  for (int v0 = 0; v0 < G; v0 += 32) {
    const int v = v0 + lane;
    const unsigned rm = v < nu ? rowmask[uexp[v]] : 0u;
    const int c = __popc(rm);
    int inc = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, inc, d);
      if (lane >= d) inc += o;
    }
    int o = before + inc - c;
    if (v < G) {
      go[1 + v] = v < nu ? uexp[v] : -1;
      go[1 + G + v] = o;
    }
    for (int r = 0; r < K; ++r)
      if ((rm >> r) & 1u) go[2 + 2 * G + o++] = r * k + slot[v * K + r];
    before += __shfl_sync(0xffffffffu, inc, 31);
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

// The two ldmatrix offsets (swizzled, bytes from the tile start) a lane uses
// for k-unit `ku` of a tile whose m-tile starts at row0: they depend only on
// the warp's k-unit and the lane, so a warp computes them once.
__device__ __forceinline__ void kunit_offsets(const TileGeo& geo, int box_rows, int row0, int ku, int lane,
                                              uint32_t (&off)[2]) {
  const int q0 = (ku * 4) % geo.units;
  const int c = (ku * 4) / geo.units;
  const int mi = lane >> 3, rr = lane & 7;
  const int lrow = row0 + rr + 8 * (mi & 1);
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const int unit = q0 + 2 * p + (mi >> 1);
    off[p] = swizzle_off((uint32_t)((c * box_rows + lrow) * geo.inner + unit * 16), geo.mask);
  }
}

// The codes of one k-unit for this lane (kunit_offsets): a[p][0..3] are
// row g unit q, row g+8 unit q, row g unit q+1, row g+8 unit q+1 (q = 2p).
__device__ __forceinline__ void kunit_load(uint32_t tile, const uint32_t (&off)[2], uint32_t (&a)[2][4]) {
#pragma unroll
  for (int p = 0; p < 2; ++p) ldmatrix_x4(tile + off[p], a[p][0], a[p][1], a[p][2], a[p][3]);
}

// One k-unit (128 k) of a 16-row m-tile against NB n-blocks of B, from the
// codes of kunit_load and the scales of unit_scales (rows g and g+8).
template <int NB>
__device__ __forceinline__ void kunit_mma_regs(const uint32_t (&a)[2][4], const uint32_t (&sg)[4],
                                               const uint32_t (&sh)[4], const uint32_t (&b)[NB][16],
                                               float (&acc0)[NB][4], float (&acc1)[NB][4]) {
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const uint32_t rq[2][2] = {{a[p][0], a[p][1]}, {a[p][2], a[p][3]}};
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
        mma_f16(acc0[nb], dg[0], dh[0], dg[1], dh[1], b[nb][q * 4 + 0], b[nb][q * 4 + 1]);
        mma_f16(acc1[nb], dg[2], dh[2], dg[3], dh[3], b[nb][q * 4 + 2], b[nb][q * 4 + 3]);
      }
    }
  }
}

// kunit_mma_regs straight from shared memory.
template <int NB>
__device__ __forceinline__ void kunit_mma_at(uint32_t tile, const uint32_t (&off)[2], const uint32_t (&sg)[4],
                                             const uint32_t (&sh)[4], const uint32_t (&b)[NB][16],
                                             float (&acc0)[NB][4], float (&acc1)[NB][4]) {
  uint32_t a[2][4];
  kunit_load(tile, off, a);
  kunit_mma_regs<NB>(a, sg, sh, b, acc0, acc1);
}

// Item kinds of a CTA's sequence (in this order).
constexpr int kShGU = 0, kRtGU = 1, kDN = 2, kEnd = 4;  // kind 3: the second down range

struct Item {
  int kind;
  int slot;  // u (routed) or G (shared)
  int tile;  // m-tile (gate/up, 16 rows) or hidden tile (down, 64 rows)
};

// Items before part c when n items are dealt to `parts` parts as evenly as
// possible, the low parts taking one more.
__device__ __forceinline__ int split_before(int c, int n, int parts) { return c * (n / parts) + min(c, n % parts); }

// The CTA's work: its gate/up items, dealt round-robin in the global order
// (shared items first, then the routed ones slot-major), so every slot's
// items finish in one early round across the CTAs and the down items of a
// slot rarely wait; then two contiguous ranges of the down items: [dn0, dn1)
// in the first half of the slot-major down list (slots that finish early,
// dealt to the CTAs in order) and [dn2, dn3) in the second half (dealt in
// reverse order), so every CTA starts its down work on early slots.
// Gate/up item V of the global order goes to CTA V mod grid: CTA b holds
// n_shb shared items (V = b, b + grid, ...) then rt_count routed ones, the
// first being routed item rt_first, the next ones grid apart.
struct Plan {
  int n_shb, rt_first, rt_count, dn0, dn1, dn2, dn3;
};

__device__ __forceinline__ Plan make_plan(int n_sh, int n_rgu, int n_dn) {
  const int grid = gridDim.x, b = blockIdx.x;
  const int T = n_sh + n_rgu;
  Plan p;
  p.n_shb = split_before(b + 1, n_sh, grid) - split_before(b, n_sh, grid);
  p.rt_count = split_before(b + 1, T, grid) - split_before(b, T, grid) - p.n_shb;
  p.rt_first = b + p.n_shb * grid - n_sh;
  const int h1 = n_dn / 2, h2 = n_dn - h1;
  p.dn0 = split_before(b, h1, grid);
  p.dn1 = split_before(b + 1, h1, grid);
  p.dn2 = h1 + split_before(grid - 1 - b, h2, grid);
  p.dn3 = h1 + split_before(grid - b, h2, grid);
  return p;
}

__device__ __forceinline__ int plan_len(const Plan& p) { return p.n_shb + p.rt_count + (p.dn1 - p.dn0) + (p.dn3 - p.dn2); }

// Walks a CTA's items in order with no division per item.  Routed gate/up
// item v is tile v % mt_per of slot v / mt_per (mt_per a power of two); down
// items are slot-major with the shared slot first.
struct Seq {
  Plan p;
  int mt_per, lg_mt, n_tiles, G, has_sh;
  int dn_slot, dn_tile, dn2_slot, dn2_tile;  // first item of each down range
};

__device__ __forceinline__ Seq make_seq(const Plan& p, int mt_per, int n_tiles, int G, int has_sh) {
  Seq s;
  s.p = p;
  s.mt_per = mt_per;
  s.n_tiles = n_tiles;
  s.G = G;
  s.has_sh = has_sh;
  s.lg_mt = __ffs(mt_per) - 1;
  const int si = p.dn0 / n_tiles;
  s.dn_tile = p.dn0 - si * n_tiles;
  s.dn_slot = has_sh ? (si == 0 ? G : si - 1) : si;
  const int si2 = p.dn2 / n_tiles;
  s.dn2_tile = p.dn2 - si2 * n_tiles;
  s.dn2_slot = has_sh ? (si2 == 0 ? G : si2 - 1) : si2;
  return s;
}

struct Cursor {
  Item it;
  int left;  // items left in the current phase, this one included
  int v;     // routed gate/up item index (routed phase)
};

__device__ __forceinline__ void seq_phase(Cursor& c, const Seq& s, int kind) {
  for (; kind < kEnd; ++kind) {
    if (kind == kShGU) {
      c.left = s.p.n_shb;
      c.it.slot = s.G;
      c.it.tile = blockIdx.x;
    } else if (kind == kRtGU) {
      c.left = s.p.rt_count;
      c.v = s.p.rt_first;
      c.it.slot = c.v >> s.lg_mt;
      c.it.tile = c.v & (s.mt_per - 1);
    } else if (kind == kDN) {
      c.left = s.p.dn1 - s.p.dn0;
      c.it.slot = s.dn_slot;
      c.it.tile = s.dn_tile;
    } else {
      c.left = s.p.dn3 - s.p.dn2;
      c.it.slot = s.dn2_slot;
      c.it.tile = s.dn2_tile;
    }
    c.it.kind = kind;
    if (c.left > 0) return;
  }
  c.it.kind = kEnd;
  c.left = 0;
}

__device__ __forceinline__ Cursor seq_begin(const Seq& s) {
  Cursor c;
  seq_phase(c, s, kShGU);
  return c;
}

__device__ __forceinline__ void seq_next(Cursor& c, const Seq& s) {
  if (--c.left > 0) {
    if (c.it.kind == kShGU) {
      c.it.tile += gridDim.x;
    } else if (c.it.kind == kRtGU) {
      c.v += gridDim.x;
      c.it.slot = c.v >> s.lg_mt;
      c.it.tile = c.v & (s.mt_per - 1);
    } else if (++c.it.tile == s.n_tiles) {
      c.it.tile = 0;
      c.it.slot = (c.it.slot == s.G) ? 0 : c.it.slot + 1;
    }
    return;
  }
  if (c.it.kind < kEnd) seq_phase(c, s, c.it.kind + 1);
}

// Everything the producer needs to issue an item's copies.
struct IssueCtx {
  const CUtensorMap *gate, *up, *down, *sgate, *sup, *sdown, *gate_s, *up_s, *sgate_s, *sup_s;
  const unsigned char *down_scales, *sh_down_scales;
  const int* uexp;  // distinct experts (shared memory)
  int H, I, G, code3d;
  uint64_t pol;
};

// Issue the TMA copies of one item into stage `stg`, completion on `bar`
// (called by the whole producer warp).
__device__ __forceinline__ void issue_item(const IssueCtx& c, const Item it, unsigned char* stg, uint64_t* bar,
                                        int lane) {
  const int H = c.H, I = c.I;
  if (it.kind < kDN) {  // gate/up
    const TileGeo geo = tile_geo(H);
    const int code = kGURows * H / 2, scale = kGURows * H / 16;
    const bool sh = it.kind == kShGU;
    const int e = sh ? 0 : c.uexp[it.slot];
    const int row0 = e * I + it.tile * kGURows;
    const CUtensorMap* mg = sh ? c.sgate : c.gate;
    const CUtensorMap* mu = sh ? c.sup : c.up;
    const CUtensorMap* msg = sh ? c.sgate_s : c.gate_s;
    const CUtensorMap* msu = sh ? c.sup_s : c.up_s;
    const int chunks = (H / 2) / geo.inner;
    if (lane == 0) mbar_arrive_expect_tx(bar, 2 * code + 2 * scale);
    __syncwarp();
    if (c.code3d) {  // one request per projection tile: lane 0 gate, lane 1 up, in one instruction
      if (lane < 2) tma_load_3d(stg + lane * code, lane ? mu : mg, 0, row0, 0, bar, c.pol);
    } else if (lane < chunks)
      tma_load_2d(stg + lane * kGURows * geo.inner, mg, lane * geo.inner, row0, bar, c.pol);
    else if (lane >= 16 && lane < 16 + chunks)
      tma_load_2d(stg + code + (lane - 16) * kGURows * geo.inner, mu, (lane - 16) * geo.inner, row0, bar, c.pol);
    if (lane >= 30)  // the two scale tiles
      tma_load_2d(stg + 2 * code + (lane - 30) * scale, lane == 31 ? msu : msg, 0, row0, bar, c.pol);
  } else {
    const TileGeo geo = tile_geo(I);
    const int code = kDNRows * I / 2, scale = kDNRows * I / 16;
    const bool sh = it.slot == c.G;
    const int e = sh ? 0 : c.uexp[it.slot];
    const int row0 = e * H + it.tile * kDNRows;
    const CUtensorMap* m = sh ? c.sdown : c.down;
    const unsigned char* sp = sh ? c.sh_down_scales : c.down_scales;
    const int chunks = (I / 2) / geo.inner;
    if (lane == 0) mbar_arrive_expect_tx(bar, code + scale);
    __syncwarp();
    if (c.code3d) {
      if (lane == 0) tma_load_3d(stg, m, 0, row0, 0, bar, c.pol);
    } else if (lane < chunks)
      tma_load_2d(stg + lane * kDNRows * geo.inner, m, lane * geo.inner, row0, bar, c.pol);
    if (lane == 31) bulk_load(stg + code, sp + (size_t)row0 * (I / 16), scale, bar, c.pol);
  }
  __syncwarp();
}


// Tag of the words a layer call writes: the call's index plus one (never 0,
// the value of a zero-filled workspace).
__device__ __forceinline__ unsigned call_tag(unsigned long long call) {
  return (unsigned)(call % 0xFFFFFFFFull) + 1u;
}

}  // namespace

// The experts kernel: one MoE layer call in one persistent launch.  Every CTA
// stages the K input rows, normalises them when asked, forms its share of the
// router logits and publishes them, routes every row, streams its items of
// the layer's distinct experts, and combines its share of the outputs.
template <int NB>
__global__ void __launch_bounds__(kThreads, 1) k_moe_experts(const __grid_constant__ ExpertsParams P) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
  __shared__ unsigned s_xamax[16];
  __shared__ unsigned s_used[32];  // bitmask of the experts any row selected
  __shared__ int s_abort, s_nu;
  __shared__ unsigned long long s_call;

  const ExpertsCommon& a = P.c;
  const int H = a.H, I = a.I, K = a.K, G = a.G, E = a.E, k = a.k;
  const int S = a.stages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int stage_bytes = expert_stage_bytes(H, I);
  const int mt_per = I / kGURows, n_tiles = H / kDNRows;
  const int grid = gridDim.x;

  // reduction slots (two, alternating by item): the compute warps' FP32
  // partials, then the inverse h scales of down items ([k-unit][row], 4 x 16).  Warp w's block
  // starts at w * kWarpStride + red_skew(w): the skew puts the partials that
  // the 4 lanes of an epilogue quad read (warps 4j + 0..3) in distinct banks.
  constexpr int kWarpStride = 2 * NB * 128 + 32;
  constexpr int kRedPart = kCompWarps * kWarpStride;
  constexpr int kRedFloats = kRedPart + 64;
  auto red_at = [](int w) { return w * kWarpStride + 2 * (w & 1) + 16 * ((w >> 1) & 1); };
  float* red = reinterpret_cast<float*>(smem + (size_t)S * stage_bytes);
  unsigned char* rsm = reinterpret_cast<unsigned char*>(red + 2 * kRedFloats);
  // routing state (shared by all warps after the routing step)
  float* s_w = reinterpret_cast<float*>(rsm);                         // [K][k]
  int* s_idx = reinterpret_cast<int*>(s_w + K * k);                   // [K][k]
  unsigned* s_rowmask = reinterpret_cast<unsigned*>(s_idx + K * k);   // [E] rows that chose expert e
  int* s_uexp = reinterpret_cast<int*>(s_rowmask + E);                // [G+1] distinct experts, ascending
  float* s_tse = reinterpret_cast<float*>(s_uexp + G + 1);            // [E+1][3] tensor scales (E = shared)
  float* s_bias = s_tse + 3 * (E + 1);                                // [E] router bias (0 if none)
  signed char* s_slot = reinterpret_cast<signed char*>(s_bias + E);   // [(G+1)*K]
  // the K input rows, staged once per CTA and layer in the reduction slots
  // (idle until the layer's first item)
  uint4* xs = reinterpret_cast<uint4*>(red);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kCompWarps);
    }
    s_abort = 0;
    s_call = 0ull;
    fence_mbar_init();
  }
  __syncthreads();
  // optional timeline: globaltimer stamps of this CTA's milestones
  unsigned long long* trace = a.trace ? a.trace + (size_t)blockIdx.x * kTraceSlots : nullptr;
  auto stamp = [&](int m) {
    if (trace) trace[m] = global_timer_ns();
  };
  if (threadIdx.x == 0) stamp(0);
  auto fail = [&]() {
    s_abort = 1;
    set_error(a.ws.err, MOE_ERR_DEVICE_TIMEOUT);
  };
  auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&s_abort) != 0; };
  // a bounded wait whose outcome is the same on every lane of the warp
  auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, a.wait_ns, &s_abort));
    if (!ok && lane == 0) fail();
    return ok;
  };
  const LayerDesc& D = P.L;
  // shared-expert gate/up items (CTA b holds b, b + grid, ...)
  const int n_sh = D.has_shared ? mt_per : 0;
  const int n_shb = split_before(blockIdx.x + 1, n_sh, grid) - split_before(blockIdx.x, n_sh, grid);
  // The CTA's item sequence, from the distinct-expert count.
  auto make_cta_seq = [&]() {
    const int n_u = *reinterpret_cast<volatile int*>(&s_nu);
    const int n_slots = n_u + (D.has_shared ? 1 : 0);
    return make_seq(make_plan(n_sh, n_u * mt_per, n_slots * n_tiles), mt_per, n_tiles, G, D.has_shared);
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // The CTA's shared-expert gate/up items (no routing needed: issued
    // before the dependency wait), then, once warp 0 has listed the distinct
    // experts, its routed gate/up and down items.  Item j goes to stage j % S
    // on pass j / S.
    const uint64_t pol = policy_evict_first();
    int issued = 0, st = 0, pass = 0;
    bool live = true;
    auto issue_next = [&](const IssueCtx& ic, const Item& it, int li) {
      int ok = 1;
      if (lane == 0 && pass > 0 && !mbar_wait_bounded(&empty_bar[st], (pass - 1) & 1, a.wait_ns, &s_abort)) {
        ok = 0;
        fail();
      }
      if (__shfl_sync(0xffffffffu, ok, 0) == 0) return false;
      if (lane == 0 && trace && li < 24) trace[40 + li] = global_timer_ns();  // item li issued
      issue_item(ic, it, smem + (size_t)st * stage_bytes, &full_bar[st], lane);
      ++issued;
      if (++st == S) {
        st = 0;
        ++pass;
      }
      return true;
    };
    do {
      const CUtensorMap* mp = P.maps;
      IssueCtx ic;
      ic.gate = mp + 0;
      ic.up = mp + 1;
      ic.down = mp + 2;
      ic.sgate = mp + 3;
      ic.sup = mp + 4;
      ic.sdown = mp + 5;
      ic.gate_s = mp + 6;
      ic.up_s = mp + 7;
      ic.sgate_s = mp + 8;
      ic.sup_s = mp + 9;
      ic.down_scales = D.down.scales;
      ic.sh_down_scales = D.sh_down.scales;
      ic.uexp = s_uexp;
      ic.H = H;
      ic.I = I;
      ic.G = G;
      ic.code3d = a.code3d;
      ic.pol = pol;
      if (lane < kMapsPerLayer) prefetch_tensormap(mp + lane);
      Item it;
      it.kind = kShGU;
      it.slot = G;
      it.tile = blockIdx.x;
      for (int j = 0; j < n_shb && live; ++j, it.tile += grid) live = issue_next(ic, it, j);
      if (!live) break;
      asm volatile("bar.sync 2, 64;" ::: "memory");  // the distinct experts are listed
      if (lane == 0) stamp(3);
      const Seq seq = make_cta_seq();
      const int L = plan_len(seq.p);
      Cursor cur = seq_begin(seq);
      for (int j = 0; j < n_shb; ++j) seq_next(cur, seq);
      for (int j = n_shb; j < L && live; ++j, seq_next(cur, seq)) live = issue_next(ic, cur.it, j);
    } while (false);
    if (lane == 0 && trace) trace[9] = global_timer_ns();
    if (lane == 0 && live) l2_prefetch_list(a.pf, blockIdx.x, grid);  // the next kernel's first bytes
    if (lane == 0) {
      // every copy of the last S items has landed before the CTA may exit
      // (a stage is reissued only after the compute warps saw its previous
      // copy complete, so older copies have landed)
      for (int j = (issued > S ? issued - S : 0); j < issued; ++j)
        mbar_wait_drain(&full_bar[j % S], (j / S) & 1, kDrainNs);
    }
    return;
  }

  // -------------------------------------------------------------- compute warps
  const int tid = threadIdx.x;
  // Per-layer preparation that needs no layer input: routing tables cleared,
  // the router bias to shared memory, the tensor scales (slot E = shared) of
  // this thread's first expert to registers (stored to shared memory after
  // the router step, so their DRAM latency is hidden; the rest, for E >= 512,
  // at once), and the warp's first router row to registers.
  const int M = (E + grid - 1) / grid;  // router experts per CTA: b + grid m, m < M
  const int n_pairs = M * K;            // (expert, row) pairs: p = warp, warp + 16, ...: m = p % M, row p / M

  // activations as FP16 B fragments: compute warp w holds k-unit w of every
  // row (from the staged rows)
  auto load_x = [&](uint4 (&raw)[NB][4]) {
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int n = nb * 8 + g;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (warp < H / 128 && n < K) v = xs[n * (H / 8) + warp * 16 + q * 4 + t];
        raw[nb][q] = v;
      }
    }
  };
  const int KUgu = H / 128, KUdn = I / 128;
  const TileGeo ggu = tile_geo(H), gdn = tile_geo(I);
  const int gu_code = kGURows * H / 2, gu_scale = kGURows * H / 16;
  const int dn_code = kDNRows * I / 2;
  const int smask = (H / 16 >= 128) ? 7 : (H / 16 == 64 ? 3 : (H / 16 == 32 ? 1 : 0));
  const int sstride = H / 16;
  const bool gu_active = warp < KUgu;
  const uint32_t so0 = swizzle_off((uint32_t)(g * sstride + 8 * warp), smask);
  const uint32_t so1 = swizzle_off((uint32_t)((g + 8) * sstride + 8 * warp), smask);
  uint32_t goff[2];  // this lane's ldmatrix offsets in a gate/up codes tile
  kunit_offsets(ggu, kGURows, 0, gu_active ? warp : 0, lane, goff);
  const int mA = warp & 3, kq = warp >> 2;
  const bool dn_active = kq < KUdn;
  uint32_t doffA[2], doffB[2];  // this lane's ldmatrix offsets in a down codes tile
  kunit_offsets(gdn, kDNRows, mA * 16, dn_active ? kq : 0, lane, doffA);
  kunit_offsets(gdn, kDNRows, (mA + 4) * 16, dn_active ? kq : 0, lane, doffB);
  const int lg_mt = __ffs(mt_per) - 1;
  int st = 0, fp = 0;  // ring position of the next item: stage st, pass fp
  auto advance = [&]() {
    if (++st == S) {
      st = 0;
      ++fp;
    }
  };

  {
    // Preparation that needs no layer input, before the dependency wait:
    // routing tables cleared, the router bias to shared memory, the
    // tensor scales (slot E = shared) of this thread's expert to registers
    // (stored to shared memory after the router step, so their DRAM latency
    // is hidden; the rest, for E >= 512, at once), and the warp's first
    // router row to registers (lane l holds pieces 256 j + 8 l .. + 7).
    uint4 lw[8];
    int lw_e = -1;
    float tse0[3] = {0.f, 0.f, 0.f};
    {
      for (int e = tid; e < E; e += kCompThreads) {
        s_rowmask[e] = 0u;
        s_bias[e] = D.router_bias ? D.router_bias[e] : 0.f;
      }
      for (int i = tid; i < (G + 1) * K; i += kCompThreads) s_slot[i] = -1;
      if (tid < 16) s_xamax[tid] = 0u;
      if (tid < 32) s_used[tid] = 0u;
      auto tse_of = [&](int e, int j) {
        const float* ts = j == 0 ? (e == E ? D.sh_gate.tscale : D.gate.tscale)
                                 : (j == 1 ? (e == E ? D.sh_up.tscale : D.up.tscale)
                                           : (e == E ? D.sh_down.tscale : D.down.tscale));
        return ts[e == E ? 0 : e];
      };
      if (tid < E || (tid == E && D.has_shared))
        for (int j = 0; j < 3; ++j) tse0[j] = tse_of(tid, j);
      for (int e = tid + kCompThreads; e <= E; e += kCompThreads)
        if (e < E || D.has_shared)
          for (int j = 0; j < 3; ++j) s_tse[3 * e + j] = tse_of(e, j);
#pragma unroll
      for (int j = 0; j < 8; ++j) lw[j] = make_uint4(0, 0, 0, 0);
      if (warp < n_pairs) {
        const int e = (int)blockIdx.x + grid * (warp % M);
        if (e < E) {
          const uint4* wrow = reinterpret_cast<const uint4*>(D.router_w + (size_t)e * H);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (j < H / 256) lw[j] = ldg_nc_v4(wrow + j * 32 + lane);
          lw_e = e;
        }
      }
    }
    if (tid == 0) stamp(1);
    pdl_wait();  // the block input (and the workspace) are complete from here on
    if (tid == 0) stamp(2);
    // The call's index: the calls finished by the CTAs of all earlier
    // launches over the grid (every CTA adds one as its last act, after this
    // read, so the quotient is the same for every CTA).
    // (the read overlaps the copy of the rows below; the barrier after the
    // copy publishes it)
    if (tid == 0) s_call = __ldcg(a.ws.exits) / (unsigned long long)grid;

    // ---------------------------------------------------------------- input rows
    // [K][H] bf16 into xs, then, when asked, warp r normalises row r with
    // the RMSNorm kernel's arithmetic (a fixed-order FP32 sum of squares,
    // then each step one correctly rounded operation), so the rows are bit
    // for bit that kernel's output.  Every CTA has staged its rows before it
    // publishes its logits, and no CTA writes y before it has read all
    // logits, so y may be the input itself.
    {
      // the compute threads copy x, eight 16-byte loads in flight each
      const uint4* xg = reinterpret_cast<const uint4*>(a.x);
      const int n16 = K * H / 8;
      for (int i0 = tid; i0 < n16; i0 += 8 * kCompThreads) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (i0 + u * kCompThreads < n16) v[u] = __ldcg(xg + i0 + u * kCompThreads);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (i0 + u * kCompThreads < n16) xs[i0 + u * kCompThreads] = v[u];
      }
    }
    comp_bar();  // the rows staged, s_call written, the tables cleared
    const unsigned long long call = *reinterpret_cast<volatile unsigned long long*>(&s_call);
    const unsigned tag = call_tag(call);
    if (a.norm) {
      for (int r = warp; r < K; r += kCompWarps) {
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < H / 256) v[j] = xs[r * (H / 8) + j * 32 + lane];
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j >= H / 256) break;
          const uint32_t q[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float f = __uint_as_float((u & 1) ? (q[u >> 1] & 0xFFFF0000u) : (q[u >> 1] << 16));
            ss = __fmaf_rn(f, f, ss);
          }
        }
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, d));
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)H), a.norm_eps)));
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j >= H / 256) break;
          uint32_t q[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t lo = float_to_bf16_bits(__fmul_rn(__uint_as_float(q[i] << 16), inv));
            const uint32_t hi = float_to_bf16_bits(__fmul_rn(__uint_as_float(q[i] & 0xFFFF0000u), inv));
            q[i] = lo | (hi << 16);
          }
          xs[r * (H / 8) + j * 32 + lane] = make_uint4(q[0], q[1], q[2], q[3]);
        }
      }
      comp_bar();  // the rows are normalised
    }
    if (tid == 0) stamp(15);

    // ---------------------------------------------------------------- router logits
    // This CTA's share: per lane, products in element order over the pieces
    // j, then xor rounds 16 .. 1 (the router GEMV's fixed order, so the
    // logits are the same bits), published as tagged words the moment they
    // are formed.  Softmax scoring publishes logit + bias, sigmoid scoring the
    // score (the bias only enters the selection keys).
    for (int p = warp; p < n_pairs; p += kCompWarps) {
      const int e = (int)blockIdx.x + grid * (p % M), r = p / M;
      if (e >= E) continue;
      if (e != lw_e) {
        const uint4* wrow = reinterpret_cast<const uint4*>(D.router_w + (size_t)e * H);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < H / 256) lw[j] = ldg_nc_v4(wrow + j * 32 + lane);
        lw_e = e;
      }
      uint4 xv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < H / 256) xv[j] = xs[r * (H / 8) + j * 32 + lane];
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j >= H / 256) break;
        const uint32_t xq[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
        const uint32_t wq[4] = {lw[j].x, lw[j].y, lw[j].z, lw[j].w};
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float xf = __uint_as_float((u & 1) ? (xq[u >> 1] & 0xFFFF0000u) : (xq[u >> 1] << 16));
          const float wf = __uint_as_float((u & 1) ? (wq[u >> 1] & 0xFFFF0000u) : (wq[u >> 1] << 16));
          acc = __fmaf_rn(xf, wf, acc);
        }
      }
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, d));
      if (lane == 0) {
        const float lg = D.scoring ? sigmoid_score(acc) : (D.router_bias ? __fadd_rn(acc, s_bias[e]) : acc);
        xchg_tagged(a.ws.tlog + (size_t)r * E + e, tagged(tag, __float_as_uint(lg)));
      }
    }
    if (tid == 0) stamp(14);
    {
      uint4 raw[NB][4];
      load_x(raw);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        unsigned mx = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t w4[4] = {raw[nb][q].x, raw[nb][q].y, raw[nb][q].z, raw[nb][q].w};
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
    }
    if (tid <= E)
      for (int j = 0; j < 3; ++j) s_tse[3 * tid + j] = tse0[j];

    // ---------------------------------------------------------------- routing (every CTA, identical)
    {
      const bool fast = E <= 256 && k <= 8;
      for (int r = warp; r < K; r += kCompWarps) {
        // row r's logits, once every word of it carries this call's tag (a
        // bounded wait; on giving up, experts 0 .. k-1 keep the tables in
        // range and the abort flag stops the work)
        const unsigned long long* row = a.ws.tlog + (size_t)r * E;
        bool got;
        const float* sel_bias = (D.scoring && D.router_bias) ? s_bias : nullptr;
        if (fast) {
          got = route_row_fast(row, tag, E, k, r, a.wait_ns, &s_abort, s_idx, s_w, s_rowmask, s_used, D.scoring,
                               sel_bias, lane);
        } else {
          got = topk_general(row, tag, a.wait_ns, &s_abort, E, k, s_idx + r * k, s_w + r * k, sel_bias, lane);
          __syncwarp();
          const int sel_e = got ? (lane < k ? s_idx[r * k + lane] : 0) : lane;
          const float sel_l = got ? (lane < k ? s_w[r * k + lane] : 0.f) : 0.f;
          const float top = got ? s_w[r * k] : 0.f;
          __syncwarp();
          // softmax over the selected logits; sigmoid scoring: the selected
          // experts' own scores (their words already carry this call's tag)
          const float ev = (lane < k) ? (D.scoring ? (got ? __uint_as_float((unsigned)ld_tagged(row + sel_e)) : 0.f)
                                                   : expf(sel_l - top))
                                      : 0.f;
          float z = ev;
#pragma unroll
          for (int d = 16; d >= 1; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
          if (lane < k) {
            s_idx[r * k + lane] = sel_e;
            s_w[r * k + lane] = ev / z;
            atomicOr(&s_rowmask[sel_e], 1u << r);
            atomicOr(&s_used[sel_e >> 5], 1u << (sel_e & 31));
          }
        }
        if (!got && lane == 0) fail();
      }
      comp_bar();
      if (tid == 0) stamp(13);
      // grouping: the distinct experts in ascending order are the set bits of
      // s_used; an expert's position is the number of set bits before it
      // (every warp forms the per-word prefix itself: no further barrier)
      const int n_words = (E + 31) >> 5;
      const unsigned used = lane < n_words ? s_used[lane] : 0u;
      const int cnt = __popc(used);
      int inc = cnt;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += o;
      }
      const int excl = inc - cnt;
      if (warp == 0) {
        int u = excl;
        for (unsigned m = used; m; m &= m - 1) s_uexp[u++] = lane * 32 + __ffs(m) - 1;
        if (lane == 31) s_nu = inc;
        if (lane == 0) s_uexp[G] = E;  // the shared expert's scales sit at index E
        // the producer needs only the distinct experts and their count: hand
        // them over now (named barrier 2: this warp arrives, the producer
        // waits; warp 0 arrives once per layer whatever happened)
        __syncwarp();
        asm volatile("bar.arrive 2, 64;" ::: "memory");
      }
      for (int base = 0; base < K * k; base += kCompThreads) {
        const int q = base + tid;
        const int e = q < K * k ? s_idx[q] : 0;
        const int pre_w = __shfl_sync(0xffffffffu, excl, (e >> 5) & 31);
        const unsigned uw = __shfl_sync(0xffffffffu, used, (e >> 5) & 31);
        if (q < K * k) {
          const int u = pre_w + __popc(uw & ((1u << (e & 31)) - 1u));
          s_slot[u * K + q / k] = (signed char)(q % k);
        }
      }
      if (D.has_shared)
        for (int r = tid; r < K; r += kCompThreads) s_slot[G * K + r] = (signed char)k;
      comp_bar();  // the (row, slot) map is complete
    }
    pdl_launch_dependents();

    // ---------------------------------------------------------------- items
    // Warp w owns k-unit w (128 k) of every gate/up item, and m-tile w % 4,
    // k-unit w / 4 of every down item.  Per item: codes and scales to
    // registers, the stage back to the producer, the MMAs, the FP32 partials
    // to the item's reduction slot, one barrier of the compute warps, then
    // each warp reduces its share of the item's outputs.  No wait ever leaves
    // this loop early (a failed wait sets the abort flag and the remaining
    // items run without work), so every compute warp meets every barrier.
    uint32_t bx[NB][16];
    {
      uint4 raw[NB][4];
      load_x(raw);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const int n = nb * 8 + g;
        const float sc = (n < K) ? pow2f(row_shift(s_xamax[n])) : 1.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) bf16x8_to_f16x8(raw[nb][q], sc, &bx[nb][q * 4]);
      }
    }
    comp_bar();  // every warp is done with the staged rows before partials overwrite them
    int L_gu, L_all;
    {
      const Plan p0 = make_cta_seq().p;
      L_gu = p0.n_shb + p0.rt_count;
      L_all = plan_len(p0);
      if (tid == 0 && trace) {  // (counts, not times: for reading the item stamps)
        trace[66] = (unsigned long long)L_gu;
        trace[67] = (unsigned long long)L_all;
      }
    }
    // this CTA's gate/up items: global items V = b + i * grid, shared tile V
    // for V < n_sh, else routed v = V - n_sh (slot v / mt_per, tile
    // v % mt_per; mt_per is a power of two)
    for (int li = 0; li < L_gu; ++li, advance()) {
      unsigned char* stg = smem + (size_t)st * stage_bytes;
      float* rb = red + (size_t)(li & 1) * kRedFloats;
      const bool ok = warp_wait(&full_bar[st], fp & 1);
      if (tid == 0 && li < 24) stamp(16 + li);  // item li landed
      // this warp's codes and scales to registers, then the stage goes back
      uint32_t ag[2][4], au[2][4];
      uint2 sr[4];
      if (ok && gu_active) {
        const uint32_t tg = smem_addr(stg);
        kunit_load(tg, goff, ag);
        kunit_load(tg + gu_code, goff, au);
        const unsigned char* sgt = stg + 2 * gu_code;
        sr[0] = *reinterpret_cast<const uint2*>(sgt + so0);
        sr[1] = *reinterpret_cast<const uint2*>(sgt + so1);
        sr[2] = *reinterpret_cast<const uint2*>(sgt + gu_scale + so0);
        sr[3] = *reinterpret_cast<const uint2*>(sgt + gu_scale + so1);
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(&empty_bar[st]);  // only a stage whose copy landed goes back
      if (ok && gu_active) {
        // gate and up inline: two independent chains
        uint32_t s0[4], s1[4], u0[4], u1[4];
        unit_scales(sr[0], t, s0);
        unit_scales(sr[1], t, s1);
        unit_scales(sr[2], t, u0);
        unit_scales(sr[3], t, u1);
        float cg[NB][4], cu[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int i = 0; i < 4; ++i) cg[nb][i] = cu[nb][i] = 0.f;
        kunit_mma_regs<NB>(ag, s0, s1, bx, cg, cg);
        kunit_mma_regs<NB>(au, u0, u1, bx, cu, cu);
        float* wb = rb + red_at(warp) + lane * 4;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          float* pg = wb + (0 * NB + nb) * 128;
          float* pu = wb + (1 * NB + nb) * 128;
          *reinterpret_cast<float2*>(pg) = make_float2(cg[nb][0], cg[nb][1]);
          *reinterpret_cast<float2*>(pg + 2) = make_float2(cg[nb][2], cg[nb][3]);
          *reinterpret_cast<float2*>(pu) = make_float2(cu[nb][0], cu[nb][1]);
          *reinterpret_cast<float2*>(pu + 2) = make_float2(cu[nb][2], cu[nb][3]);
        }
      }
      comp_bar();
      // epilogue, by the 4 warps of group li % 4 (the others move on to the
      // next item): thread o of the group owns output o (row o / 8 of the
      // item's 16, column o % 8 of each n-block) and sums its 16 k-unit
      // partials in k-unit order
      const bool live = !__any_sync(0xffffffffu, aborted());
      if ((warp >> 2) == (li & 3) && live) {
        const int Vg = (int)blockIdx.x + li * grid;
        const int slot = Vg < n_sh ? G : (Vg - n_sh) >> lg_mt;
        const int tile = Vg < n_sh ? Vg : ((Vg - n_sh) & (mt_per - 1));
        const int ex = s_uexp[slot];
        const float tg = s_tse[3 * ex + 0], tu = s_tse[3 * ex + 1];
        const int o = (warp & 3) * 32 + lane;
        const int i = o >> 3, c = o & 7;
        const int f0 = ((i & 7) * 4 + (c >> 1)) * 4 + (i >> 3) * 2 + (c & 1);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const int n = nb * 8 + c;
          const int f = nb * 128 + f0;
          float gs = 0.f, us = 0.f;
#pragma unroll
          for (int w = 0; w < kCompWarps; ++w) {
            if (w < KUgu) {
              gs += rb[red_at(w) + f];
              us += rb[red_at(w) + NB * 128 + f];
            }
          }
          // (rows n >= K have zero activations, so h = 0 there)
          const float inv = pow2f(-row_shift(s_xamax[n]));
          const float gv = gs * inv * tg;
          const float uv = us * inv * tu;
          const float hv = gv * __frcp_rn(1.f + expf(-gv)) * uv;
          const unsigned hb = float_to_bf16_bits(hv);
          // h rows i and i + 1 (lanes o and o + 8 of this warp) share a word
          const unsigned hn = __shfl_down_sync(0xffffffffu, hb, 8);
          if (n < K && (i & 1) == 0)
            st_tagged(a.ws.h + ((size_t)slot * K + n) * (I / 2) + ((tile * kGURows + i) >> 1),
                      tagged(tag, hb | (hn << 16)));
        }
        // this duty warp's h words are written: its done flag (the flag only
        // tells readers when to look; the tags make the h words themselves
        // safe to read)
        __syncwarp();
        if (lane == 0) st_tagged(a.ws.flags + ((size_t)slot * mt_per + tile) * 4 + (warp & 3), tagged(tag, 1u));
      }
    }
    // down items: 8 m-tiles of 16 rows x I/128 k-units; warp w takes k-unit
    // w / 4 of m-tiles w % 4 and w % 4 + 4 (one set of h fragments for both)
    {
      const Seq seq = make_cta_seq();
      uint32_t bh[NB][16];
      float hinv = 1.f, hinv1 = 1.f;  // inverse h scales of rows g and 8 + g
      int cur_slot = -1;
      Cursor dc;
      seq_phase(dc, seq, kDN);
      for (int li = L_gu; li < L_all; ++li, seq_next(dc, seq), advance()) {
        const Item it = dc.it;
        unsigned char* stg = smem + (size_t)st * stage_bytes;
        float* rb = red + (size_t)(li & 1) * kRedFloats;
        bool ok = !__any_sync(0xffffffffu, aborted());
        if (ok && it.slot != cur_slot) {
          // h of this slot, k-unit kq, as B fragments: every warp reads its
          // words at once (they usually carry this call's tag already: one
          // round trip); if some do not, it waits (bounded, no CTA barrier)
          // until the 32 done flags of the 8 gate/up items that produce its
          // k-unit carry the tag -- one word per lane and attempt -- and
          // reads the words again, after a pause in the rare case that one
          // is not visible yet; each k-unit takes its own per-row
          // power-of-two scale
          cur_slot = it.slot;
          unsigned mx[NB];
          if (ok) {
            const unsigned long long* hs = a.ws.h + (size_t)it.slot * K * (I / 2) + kq * 64 + 4 * t;
            const unsigned long long* fl = a.ws.flags + (size_t)it.slot * mt_per * 4 + 32 * kq + lane;
            const uint64_t t0 = global_timer_ns();
            bool flagged = false;
            for (;;) {
              bool mine = true;
#pragma unroll
              for (int nb = 0; nb < NB; ++nb) {
                const int n = nb * 8 + g;
                mx[nb] = 0u;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  unsigned long long w0 = 0ull, w1 = 0ull, w2 = 0ull, w3 = 0ull;
                  if (dn_active && n < K) {
                    ld_tagged2(hs + (size_t)n * (I / 2) + q * 16, w0, w1);
                    ld_tagged2(hs + (size_t)n * (I / 2) + q * 16 + 2, w2, w3);
                    mine &= has_tag(w0, tag) & has_tag(w1, tag) & has_tag(w2, tag) & has_tag(w3, tag);
                  }
                  const uint32_t hw[4] = {(uint32_t)w0, (uint32_t)w1, (uint32_t)w2, (uint32_t)w3};
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    bh[nb][q * 4 + j] = hw[j];  // bf16 pairs for now
                    mx[nb] = max(mx[nb], (hw[j] << 16) & 0x7FFFFFFFu);
                    mx[nb] = max(mx[nb], hw[j] & 0x7FFF0000u);
                  }
                }
              }
              if (__all_sync(0xffffffffu, mine)) break;
              if (warp_gives_up(t0, a.wait_ns, &s_abort, lane)) {
                ok = false;
                break;
              }
              if (!flagged) {  // not all there yet: the done flags first
                flagged = true;
                for (;;) {
                  if (__all_sync(0xffffffffu, has_tag(ld_tagged(fl), tag))) break;
                  if (warp_gives_up(t0, a.wait_ns, &s_abort, lane)) {
                    ok = false;
                    break;
                  }
                }
                if (!ok) break;
              }
            }
          }
          if (!ok && lane == 0) fail();
          if (ok) {
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              mx[nb] = max(mx[nb], __shfl_xor_sync(0xffffffffu, mx[nb], 1));
              mx[nb] = max(mx[nb], __shfl_xor_sync(0xffffffffu, mx[nb], 2));
              const int n = nb * 8 + g;
              const int sh = (n < K) ? row_shift(mx[nb]) : 0;
              const float sc = pow2f(sh);
              if (nb == 0) hinv = pow2f(-sh);
              else hinv1 = pow2f(-sh);
#pragma unroll
              for (int q = 0; q < 4; ++q)
                bf16x8_to_f16x8(make_uint4(bh[nb][q * 4 + 0], bh[nb][q * 4 + 1], bh[nb][q * 4 + 2], bh[nb][q * 4 + 3]),
                                sc, &bh[nb][q * 4]);
            }
          }
          if (tid == 0 && li == L_gu) stamp(65);  // the first down item's h is in
        }
        const bool landed = warp_wait(&full_bar[st], fp & 1);
        if (tid == 0 && li < 24) stamp(16 + li);  // item li landed
        ok = landed && ok;
        uint32_t adA[2][4], adB[2][4];
        uint2 sr[4];
        if (ok && dn_active) {
          const uint32_t tc = smem_addr(stg);
          kunit_load(tc, doffA, adA);
          kunit_load(tc, doffB, adB);
          const unsigned char* srA = stg + dn_code + (mA * 16 + g) * (I / 16) + 8 * kq;
          const unsigned char* srB = srA + 64 * (I / 16);  // 4 m-tiles further
          sr[0] = *reinterpret_cast<const uint2*>(srA);
          sr[1] = *reinterpret_cast<const uint2*>(srA + 8 * (I / 16));
          sr[2] = *reinterpret_cast<const uint2*>(srB);
          sr[3] = *reinterpret_cast<const uint2*>(srB + 8 * (I / 16));
        }
        __syncwarp();
        if (landed && lane == 0) mbar_arrive(&empty_bar[st]);  // only a stage whose copy landed goes back
        if (ok && dn_active) {
          float cA[NB][4], cB[NB][4];
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int i = 0; i < 4; ++i) cA[nb][i] = cB[nb][i] = 0.f;
          uint32_t s0[4], s1[4], u0[4], u1[4];
          unit_scales(sr[0], t, s0);
          unit_scales(sr[1], t, s1);
          unit_scales(sr[2], t, u0);
          unit_scales(sr[3], t, u1);
          kunit_mma_regs<NB>(adA, s0, s1, bh, cA, cA);
          kunit_mma_regs<NB>(adB, u0, u1, bh, cB, cB);
          float* wb = rb + red_at(warp) + lane * 4;
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            float* pa = wb + (0 * NB + nb) * 128;
            float* pb = wb + (1 * NB + nb) * 128;
            *reinterpret_cast<float2*>(pa) = make_float2(cA[nb][0], cA[nb][1]);
            *reinterpret_cast<float2*>(pa + 2) = make_float2(cA[nb][2], cA[nb][3]);
            *reinterpret_cast<float2*>(pb) = make_float2(cB[nb][0], cB[nb][1]);
            *reinterpret_cast<float2*>(pb + 2) = make_float2(cB[nb][2], cB[nb][3]);
          }
        }
        if (mA == 0 && dn_active && t == 0) {  // the inverse h scales of k-unit kq
          rb[kRedPart + kq * 16 + g] = hinv;
          if (NB == 2) rb[kRedPart + kq * 16 + 8 + g] = hinv1;
        }
        comp_bar();
        // epilogue, by the 4 warps of group li % 4 (the others move on to the
        // next item): thread o of the group owns output (i, c) of m-tiles
        // M = 0..7 in each n-block; the k-unit partials of m-tile M sit at
        // warps M % 4 + 4 q, in their first (M < 4) or second half
        const bool live = !__any_sync(0xffffffffu, aborted());
        if ((warp >> 2) == (li & 3) && live) {
          const float ts = s_tse[3 * s_uexp[it.slot] + 2];
          const int o = (warp & 3) * 32 + lane;
          const int i = o >> 3, c = o & 7;
          const int f0 = ((i & 7) * 4 + (c >> 1)) * 4 + (i >> 3) * 2 + (c & 1);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            const int n = nb * 8 + c;
            if (n >= K) continue;
            const int s = s_slot[it.slot * K + n];
            if (s < 0) continue;
            float iq[4];  // inverse h scale of each k-unit (exact powers of two)
#pragma unroll
            for (int q = 0; q < 4; ++q) iq[q] = q < KUdn ? rb[kRedPart + q * 16 + n] : 0.f;
            unsigned long long* dst = a.ws.dpart + ((size_t)n * (k + 1) + s) * H + it.tile * kDNRows + i;
#pragma unroll
            for (int Mi = 0; Mi < 8; ++Mi) {
              const int f = ((Mi >> 2) * NB + nb) * 128 + f0;
              float v4[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) v4[q] = q < KUdn ? rb[red_at(q * 4 + (Mi & 3)) + f] * iq[q] : 0.f;
              const float v = ((v4[0] + v4[1]) + v4[2]) + v4[3];  // k-units in order
              st_tagged(dst + Mi * 16, tagged(tag, __float_as_uint(v * ts)));
            }
          }
        }
      }
    }

    // ---------------------------------------------------------------- combine
    // The outputs, shared by the CTAs (no grid barrier): each thread takes
    // pairs of outputs (j, j + 1) of a row and polls their tagged partials
    // (bounded; a pause between attempts), then
    //   y = bf16(((routed_scale * sum_s w_s d_s) + d_shared) + residual),
    // slots in order, each FP32 operation rounded on its own.  The residual
    // of a call that normalises its input is that input, else the caller's.
    if (tid == 0) stamp(64);
    if (!__any_sync(0xffffffffu, aborted())) {
      const int hs = D.has_shared;
      const int ns = k + (hs ? 1 : 0);  // partials per output
      const int HP = H / 2;
      const uint16_t* res = a.norm ? a.x : a.residual;
      // output pairs dealt evenly over the CTAs (each takes a contiguous run)
      const int o_end = split_before(blockIdx.x + 1, K * HP, grid);
      for (int o = split_before(blockIdx.x, K * HP, grid) + tid; o < o_end; o += kCompThreads) {
        const int n = o / HP, j = 2 * (o - n * HP);
        const unsigned long long* dp = a.ws.dpart + (size_t)n * (k + 1) * H + j;
        float rv0 = 0.f, rv1 = 0.f;
        if (res) {
          const unsigned u = *reinterpret_cast<const unsigned*>(res + (size_t)n * H + j);
          rv0 = __uint_as_float(u << 16);
          rv1 = __uint_as_float(u & 0xFFFF0000u);
        }
        float acc0 = 0.f, acc1 = 0.f, sh0 = 0.f, sh1 = 0.f;
        bool good = true;
        constexpr int kChunk = 12;  // top-8 and the shared expert: one round
        for (int s0 = 0; s0 < ns && good; s0 += kChunk) {
          unsigned long long pw[kChunk][2];
          const uint64_t t0 = global_timer_ns();
          for (;;) {  // every load of the chunk in flight at once
            bool all = true;
#pragma unroll
            for (int u = 0; u < kChunk; ++u) {
              pw[u][0] = pw[u][1] = 0ull;
              if (s0 + u < ns) {
                ld_tagged2(dp + (size_t)(s0 + u) * H, pw[u][0], pw[u][1]);
                all &= has_tag(pw[u][0], tag) & has_tag(pw[u][1], tag);
              }
            }
            if (all) break;
            if (aborted() || a.wait_ns == 0 || global_timer_ns() - t0 > a.wait_ns) {
              good = false;
              break;
            }
          }
#pragma unroll
          for (int u = 0; u < kChunk; ++u) {
            const int s = s0 + u;
            const float p0 = __uint_as_float((unsigned)pw[u][0]), p1 = __uint_as_float((unsigned)pw[u][1]);
            if (s < k) {
              const float wv = s_w[n * k + s];
              acc0 = __fadd_rn(acc0, __fmul_rn(wv, p0));
              acc1 = __fadd_rn(acc1, __fmul_rn(wv, p1));
            } else if (s == k) {
              sh0 = p0;
              sh1 = p1;
            }
          }
        }
        if (!__all_sync(__activemask(), good)) {
          if (!good) fail();
          break;
        }
        float v0 = __fmul_rn(D.routed_scale, acc0), v1 = __fmul_rn(D.routed_scale, acc1);
        if (hs) {
          v0 = __fadd_rn(v0, sh0);
          v1 = __fadd_rn(v1, sh1);
        }
        if (res) {
          v0 = __fadd_rn(v0, rv0);
          v1 = __fadd_rn(v1, rv1);
        }
        const unsigned pair = float_to_bf16_bits(v0) | ((unsigned)float_to_bf16_bits(v1) << 16);
        *reinterpret_cast<unsigned*>(a.y + (size_t)n * H + j) = pair;
      }
    }
  }
  // the routing outputs of the call (one CTA writes them, off the critical path)
  if (blockIdx.x == 0) {
    for (int q = tid; q < K * k; q += kCompThreads) {
      if (a.idx_out) a.idx_out[q] = s_idx[q];
      if (a.w_out) a.w_out[q] = s_w[q];
    }
    if (a.group_out && warp == 0) write_groups(a.group_out, s_nu, G, K, k, s_uexp, s_rowmask, s_slot, lane);
  }
  // one exit per CTA and call, whatever happened: the next call's index
  comp_bar();
  if (tid == 0) {
    atomicAdd(a.ws.exits, 1ull);
    stamp(7);
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

// Dynamic shared memory of the experts kernel: the TMA ring, the reduction
// slots and the routing arrays.  The ring takes as many stages as fit the
// opt-in limit (at most kMaxStages).
static size_t routing_smem_bytes(int K, int E, int k, int G) {
  return sizeof(float) * K * k + sizeof(int) * K * k + sizeof(unsigned) * E + sizeof(int) * (G + 1) +
         sizeof(float) * 3 * (E + 1) + sizeof(float) * E + (size_t)(G + 1) * K + 16;
}

static size_t red_slot_bytes(int NB) { return sizeof(float) * ((size_t)kCompWarps * (2 * NB * 128 + 32) + 64); }

size_t experts_smem_bytes(int K, int H, int I, int E, int k, int G, int* stages, int* nred) {
  const int NB = K > 8 ? 2 : 1;
  const int nr = 2;
  const size_t fixed = 1024 + routing_smem_bytes(K, E, k, G) + nr * red_slot_bytes(NB);
  const size_t limit = 232448 - 2048;  // opt-in maximum less the static shared memory
  const size_t sb = expert_stage_bytes(H, I);
  int st = fixed < limit ? (int)((limit - fixed) / sb) : 0;
  if (st > kMaxStages) st = kMaxStages;
  if (stages) *stages = st;
  if (nred) *nred = nr;
  return fixed + (size_t)st * sb;
}

template <int NB>
static cudaError_t launch_experts_t(const ExpertsCommon& c, const CUtensorMap* maps, const LayerDesc& desc,
                                    cudaStream_t s, bool pdl) {
  auto kern = k_moe_experts<NB>;
  int stages = 0, nred = 0;
  const size_t smem = experts_smem_bytes(c.K, c.H, c.I, c.E, c.k, c.G, &stages, &nred);
  const int grid = num_sms();
  if (stages < 2 || c.H > 128 * kCompWarps || c.I > 128 * 4 ||
      sizeof(uint16_t) * (size_t)c.K * c.H > 2 * red_slot_bytes(NB))  // the staged rows fit the reduction slots
    return cudaErrorInvalidValue;
  ExpertsParams p;
  p.c = c;
  p.c.stages = stages;
  p.c.nred = nred;
  for (int j = 0; j < kMapsPerLayer; ++j) p.maps[j] = maps[j];
  p.L = desc;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err == cudaSuccess) err = max_carveout(kern);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  // The CTAs wait on one another, so all of them must be resident: one CTA
  // per SM (the shared memory allows no more, the grid has no more), which
  // holds whenever nothing else occupies an SM for long; every such wait is
  // bounded and reports MOE_ERR_DEVICE_TIMEOUT otherwise.  The launch is
  // not cooperative: a cooperative grid is placed only once all of it fits,
  // i.e. after every CTA of the previous kernel has exited, while a plain
  // launch with programmatic overlap lets each CTA start (and load its
  // router rows and tensor scales) as soon as its SM is free (measured:
  // 0.6-1.1 us per layer call).
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess || per_sm < 1)
    return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, kern, p);
  if (err != cudaSuccess && pdl) {  // fall back to a launch without overlap
    cudaGetLastError();
    attr[0].val.programmaticStreamSerializationAllowed = 0;
    err = cudaLaunchKernelEx(&cfg, kern, p);
  }
  return err;
}

cudaError_t launch_experts(const ExpertsCommon& c, const CUtensorMap* maps, const LayerDesc& desc, cudaStream_t s,
                           bool pdl) {
  return c.K > 8 ? launch_experts_t<2>(c, maps, desc, s, pdl) : launch_experts_t<1>(c, maps, desc, s, pdl);
}

}  // namespace moe
