// accept.cu -- longest accepted prefix of a drafted block: the first row
// whose draft token differs from the target's greedy token, or K (README of
// mlxfast Laguna XS 2.1 (DFlash), opening section: decode advances by the
// longest correct prefix).  One warp scans 32 rows per step with a ballot.
#include "internal.h"

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
  k_accept<<<1, 32, 0, s>>>(draft, target, K, out);
  return cudaGetLastError();
}

}  // namespace moe
