// accept.cu -- longest accepted prefix of a drafted block: the first row
// whose draft token differs from the target's greedy token, or K (README of
// mlxfast Laguna XS 2.1 (DFlash), opening section: decode advances by the
// longest correct prefix).  One warp scans 32 rows per step with a ballot.
// Also the small kernels around it: the cache-length commit of the verify
// loop, the synthetic drafter, and the staging of a layer call's host rows.
#include "internal.h"
#include "ptx.cuh"

namespace moe {

__global__ void __launch_bounds__(32) k_accept(const int32_t* __restrict__ draft,
                                               const int32_t* __restrict__ target, int K, int32_t* out) {
  const int lane = threadIdx.x;
  int n = K;
  for (int base = 0; base < K; base += 32) {
    const int i = base + lane;
    const bool miss = (i < K) && (draft[i] != target[i]);
    const unsigned m = __ballot_sync(0xffffffffu, miss);
    if (m) {
      n = base + __ffs(m) - 1;
      break;
    }
  }
  if (lane == 0) *out = n;
}

cudaError_t launch_accept(const int32_t* draft, const int32_t* target, int K, int32_t* out, cudaStream_t s) {
  max_carveout(k_accept);
  k_accept<<<1, 32, 0, s>>>(draft, target, K, out);
  return cudaGetLastError();
}

// After a verify round with n accepted drafts the rows 0 .. min(n + 1, K) - 1
// hold valid tokens (row 0 is the last committed token, row i + 1 the draft
// the target confirmed at row i): their keys and values, already written in
// place at positions len .. len + K - 1, become part of the cache, and the
// rest are dropped simply by not counting them -- no replay forward, no copy
// (PR #844, "8. What I looked at", items 1 and 2; "10. Next step").
__global__ void k_kv_commit(int32_t* len, const int32_t* n_accepted, int K, int cap, int* err) {
  const int n = *n_accepted;
  const int c = n + 1 < K ? n + 1 : K;
  const int nl = *len + c;
  if (nl > cap) {
    if (err) atomicCAS(err, 0, (int)MOE_ERR_CAPACITY);
    *len = cap;
  } else {
    *len = nl;
  }
}

cudaError_t launch_kv_commit(int32_t* len, const int32_t* n_accepted, int K, int cap, int* err, cudaStream_t s) {
  max_carveout(k_kv_commit);
  k_kv_commit<<<1, 1, 0, s>>>(len, n_accepted, K, cap, err);
  return cudaGetLastError();
}

// A drafter with a controlled acceptance rate, for benchmarks and tests (no
// draft model is involved): row r's draft is the target's own token where
// coin[r] != 0, else a different token, (target_r + 1 + alt_r) mod vocab with
// 0 <= alt_r < vocab - 1.  The coins are the caller's seeded draws.
__global__ void k_synthetic_drafts(const int32_t* target, const uint8_t* coin, const int32_t* alt, int K, int vocab,
                                   int32_t* draft) {
  for (int r = threadIdx.x; r < K; r += blockDim.x) {
    const long long t = target[r];
    draft[r] = coin[r] ? (int32_t)t : (int32_t)((t + 1 + (long long)alt[r]) % vocab);
  }
}

cudaError_t launch_synthetic_drafts(const int32_t* target, const uint8_t* coin, const int32_t* alt, int K, int vocab,
                                    int32_t* draft, cudaStream_t s) {
  max_carveout(k_synthetic_drafts);
  k_synthetic_drafts<<<1, 32, 0, s>>>(target, coin, alt, K, vocab, draft);
  return cudaGetLastError();
}

// A layer call's rows in page-locked host memory, staged into the workspace
// once, so that the layer kernel's CTAs read them from L2 rather than each
// across the host link.  The loads do not depend on the previous kernel and
// are issued before the dependency wait; the stores, into memory that the
// previous call may still use, after it.
constexpr int kStageThreads = 512;
constexpr int kStageVecs = 8;  // 16-byte pieces per thread: K * H * 2 <= 64 KB

__global__ void __launch_bounds__(kStageThreads) k_stage_rows(const uint4* src, uint4* dst, int n16) {
  pdl_launch_dependents();
  uint4 v[kStageVecs];
#pragma unroll
  for (int u = 0; u < kStageVecs; ++u) {
    const int i = threadIdx.x + u * kStageThreads;
    if (i < n16) v[u] = src[i];
  }
  pdl_wait();
#pragma unroll
  for (int u = 0; u < kStageVecs; ++u) {
    const int i = threadIdx.x + u * kStageThreads;
    if (i < n16) dst[i] = v[u];
  }
}

cudaError_t launch_stage_rows(const void* src, void* dst, size_t bytes, cudaStream_t s) {
  const size_t n16 = bytes / 16;
  if (bytes % 16 != 0 || n16 > (size_t)kStageThreads * kStageVecs) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kStageThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  max_carveout(k_stage_rows);
  return cudaLaunchKernelEx(&cfg, k_stage_rows, static_cast<const uint4*>(src), static_cast<uint4*>(dst), (int)n16);
}

}  // namespace moe
