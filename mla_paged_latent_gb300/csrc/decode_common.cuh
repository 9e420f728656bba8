// Device helpers shared by the decode kernels: the unit schedule of a
// split-KV partition and the base-2 exponential.
#pragma once
#include <cstdint>

#include "mla_kernels.h"

namespace mla {

__device__ __forceinline__ int num_blocks(const DecodeParams& P, int r) {
  const int K = P.topk > 0 ? P.topk : P.seqlens[r];
  const int nb = (K + kBlockRows - 1) / kBlockRows;
  return nb < 1 ? 1 : nb;
}

// Segments (request, block range, split index) of one partition, in order.
template <typename F>
__device__ __forceinline__ void for_each_unit(const DecodeParams& P, int part, F&& f) {
  const int* s = P.sched + 8 * part;
  const int b0 = s[0], k0 = s[1], b1 = s[2], k1 = s[3], fs = s[4];
  for (int r = b0; r < P.batch && (r < b1 || (r == b1 && k1 > 0)); ++r) {
    const int nb = num_blocks(P, r);
    const int lo = (r == b0) ? k0 : 0;
    const int hi = (r == b1) ? (k1 < nb ? k1 : nb) : nb;
    if (hi <= lo) continue;
    f(r, lo, hi, (r == b0) ? fs : 0);
  }
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace mla
