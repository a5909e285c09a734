// ptx.cuh -- thin inline-PTX wrappers used by the sm_103a kernels:
// mbarriers with bounded waits, TMA (cp.async.bulk / cp.async.bulk.tensor),
// ldmatrix, mma.sync, FP4/FP8 -> FP16 conversions, PDL controls.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: the thread sleeps in hardware until the
// phase completes or about `hint_ns` pass, so a waiting warp takes no issue
// slots from the warps that work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// The waiting part of mbar_wait_bounded, kept out of line (one copy).
static __device__ __noinline__ bool mbar_wait_loop(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                                   const volatile int* abort) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// Waits (bounded by `limit_ns`, never cut short by an abort flag) for the
// copies that complete phase `parity` of `bar`: a CTA must not exit while
// its own bulk copies may still write its shared memory.
static __device__ __noinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait_sleep(bar, parity, 20000u))
    if (global_timer_ns() - t0 > limit_ns) return false;
  return true;
}

// Waits for phase `parity` of `bar` to complete.  Gives up (returns false)
// after `limit_ns` nanoseconds, or at once when *abort is set by another
// warp; limit_ns == 0 gives up immediately.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                                  const volatile int* abort) {
  if (limit_ns == 0) return false;
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_loop(bar, parity, limit_ns, abort);
}

// ---------------------------------------------------------------- TMA

// 2-D tiled tensor load into shared memory, completion counted on `bar`.
// c0 is the inner (byte) coordinate and must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// 3-D tiled tensor load (the code tiles: 128-byte lines, rows, line chunks).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Contiguous global -> shared bulk copy (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Bulk prefetch of [p, p + bytes) into L2 (p 16-byte aligned, bytes a
// multiple of 16), issued in pieces of at most 64 KB.
__device__ __forceinline__ void l2_prefetch_span(const void* p, uint64_t bytes) {
  const char* c = static_cast<const char*>(p);
  while (bytes > 0) {
    const uint32_t n = bytes > 65536u ? 65536u : (uint32_t)bytes;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c), "r"(n) : "memory");
    c += n;
    bytes -= n;
  }
}

// Share `part` of `nparts` of every range of a prefetch list (each range cut
// at 16-byte boundaries into nparts slices).
template <typename List>
__device__ __forceinline__ void l2_prefetch_list(const List& pf, int part, int nparts) {
  for (int i = 0; i < pf.n; ++i) {
    const uint64_t total = pf.bytes[i];
    const uint64_t a = (total * (uint64_t)part / (uint64_t)nparts) & ~(uint64_t)15;
    const uint64_t b = part + 1 == nparts ? total : (total * (uint64_t)(part + 1) / (uint64_t)nparts) & ~(uint64_t)15;
    if (b > a) l2_prefetch_span(static_cast<const char*>(pf.p[i]) + a, b - a);
  }
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// L2 policy for data read once (weights stream through).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- PDL

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// ---------------------------------------------------------------- tensor-core fragments

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A(16x16, f16, row) * B(16x8, f16, col), FP32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Eight E2M1 codes (one 32-bit word, element j in nibble j) -> four f16x2;
// d[i] holds elements 2i (low half) and 2i+1 (high half).
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&d)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(w));
}

// One E4M3 code -> f16x2 holding the value twice.
__device__ __forceinline__ uint32_t e4m3_to_f16x2_dup(uint32_t code) {
  uint32_t d;
  uint16_t pair = static_cast<uint16_t>(code | (code << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(pair));
  return d;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Two floats -> f16x2 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) { return __uint_as_float(b16 << 16); }

// Cosine and sine of the rotary angle p * f (p a position, f the pair's angle
// per position).  The product and its reduction by 2 pi are taken in double
// (Cody and Waite's two-constant reduction, "Software Manual for the
// Elementary Functions", 1980: 2 pi = C1 + C2, C1 the double nearest 2 pi);
// the sine and cosine of the reduced angle (|r| <= pi) in FP32.  Positions
// reach the cache length, where an FP32 product would lose the angle; the
// reduction keeps the FP64 work to five operations per angle.
__device__ __forceinline__ void rope_cs(int p, double f, float& c, float& s) {
  const double th = (double)p * f;
  const double k = rint(th * 0.15915494309189535);  // 1 / (2 pi)
  double r = fma(-k, 6.283185307179586, th);        // C1
  r = fma(-k, 2.4492935982947064e-16, r);           // C2 = 2 pi - C1
  sincosf((float)r, &s, &c);
}

// Router score of the sigmoid-scored router (MOE_SCORE_SIGMOID): the logistic
// function as one fixed sequence of correctly rounded FP32 operations, so any
// implementation of the same sequence selects the same experts.  exp(-l) by
// Cody and Waite's argument reduction -- n = rint(-l log2 e), r = -l - n ln2
// with ln 2 split into a 16-bit head (n * head exact) and a tail -- and the
// degree-7 Taylor polynomial of e^r (|r| <= ln2/2: truncation below 1e-8),
// scaled by 2^n (exact: the clamp keeps |n| <= 116); then 1 / (1 + e).
__device__ __forceinline__ float sigmoid_score(float l) {
  if (l < -80.f) l = -80.f;
  if (l > 80.f) l = 80.f;
  const float t = -l;
  const float n = rintf(__fmul_rn(t, 0x1.715476p+0f));  // log2(e)
  float r = __fmaf_rn(-n, 0x1.62e4p-1f, t);            // ln 2, head: 45426 / 2^16
  r = __fmaf_rn(-n, 0x1.7f7d1cp-20f, r);                // ln 2, tail
  float p = 0x1.a01a02p-13f;                            // 1/7!
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);                 // 1/6!
  p = __fmaf_rn(p, r, 0x1.111112p-7f);                  // 1/5!
  p = __fmaf_rn(p, r, 0x1.555556p-5f);                  // 1/4!
  p = __fmaf_rn(p, r, 0x1.555556p-3f);                  // 1/3!
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  const float e = __fmul_rn(p, __int_as_float(((int)n + 127) << 23));
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, e));
}

// Round a float to bf16 (nearest even), returning the bit pattern.
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

// 128-bit read-only load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Copies n 16-byte words from global to shared memory with the whole block.
// Each thread puts up to 8 loads in flight before it stores them: a plain
// strided copy loop waits for every load before it issues the next, so its
// time grows with n in whole L2 round trips.
__device__ __forceinline__ void block_copy_g2s(uint4* dst, const uint4* src, int n) {
  for (int i0 = threadIdx.x; i0 < n; i0 += 8 * (int)blockDim.x) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * (int)blockDim.x;
      if (i < n) v[u] = __ldcg(src + i);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * (int)blockDim.x;
      if (i < n) dst[i] = v[u];
    }
  }
}

// Byte offset of a 16-byte unit inside a TMA tile written with the 128-byte
// (mask 7) or 64-byte (mask 3) swizzle: bits [6:4] (or [5:4]) of the address
// are XORed with bits [9:7] (or [8:7]).  `off` is relative to a tile base
// aligned to 1024 bytes.
__device__ __forceinline__ uint32_t swizzle_off(uint32_t off, uint32_t mask) {
  return off ^ (((off >> 7) & mask) << 4);
}

}  // namespace moe
