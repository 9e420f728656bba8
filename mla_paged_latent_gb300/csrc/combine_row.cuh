// The merge of one query row's split-KV partials, shared by the combine kernel and the
// fused combine + value up-projection so that both write the same merged rows.
#pragma once
#include <cstdint>

#include "ptx_sm103.cuh"

namespace mla {

// Warp-wide, one query row `row` of a request with ns >= 2 partials starting at split s0:
// lse = ln sum_s e^(lse_s); out = sum_s e^(lse_s - lse) o_s ("mla_attention.py ·
// tduncan/Nvidia-Optimization-Stack-VLLM", Chunked Prefill: merge_attn_states; an empty
// partial has lse = -inf and weight 0), then the sink factor 1 / (1 + e^(sink - lse))
// ("MLA" API page of HALOps, mla_output_proj: the split-KV LSE combine receives attn_sink).
// acc[4 k + i] receives element 4 (32 k + lane) + i; the return value is lse (-inf, with
// acc = 0, when every partial is empty).
__device__ __forceinline__ float merge_row(const float* __restrict__ part_out, const float* __restrict__ part_lse,
                                           int s0, int ns, int R, int row, int lane, const float* __restrict__ sink,
                                           int head, float (&acc)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  float lse_tot;
  if (ns <= 4) {
    // up to 4 splits (the common case): every load first, in one round trip to memory
    float ls[4];
    float4 v[4][4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      ls[s] = -INFINITY;
      if (s < ns) {
        ls[s] = part_lse[(int64_t)(s0 + s) * R + row];
        const float4* src = reinterpret_cast<const float4*>(part_out + ((int64_t)(s0 + s) * R + row) * 512);
#pragma unroll
        for (int k = 0; k < 4; ++k) v[s][k] = src[k * 32 + lane];
      }
    }
    const float mx = fmaxf(fmaxf(ls[0], ls[1]), fmaxf(ls[2], ls[3]));
    if (mx == -INFINITY) return -INFINITY;
    float tot = 0.f;
#pragma unroll
    for (int s = 0; s < 4; ++s)
      if (s < ns) tot += expf(ls[s] - mx);
    lse_tot = mx + logf(tot);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      if (s >= ns || ls[s] == -INFINITY) continue;
      const float w = expf(ls[s] - lse_tot);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[4 * k + 0] += w * v[s][k].x;
        acc[4 * k + 1] += w * v[s][k].y;
        acc[4 * k + 2] += w * v[s][k].z;
        acc[4 * k + 3] += w * v[s][k].w;
      }
    }
  } else {
    float mx = -INFINITY;
    for (int s = lane; s < ns; s += 32) mx = fmaxf(mx, part_lse[(int64_t)(s0 + s) * R + row]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (mx == -INFINITY) return -INFINITY;
    float tot = 0.f;
    for (int s = lane; s < ns; s += 32) tot += expf(part_lse[(int64_t)(s0 + s) * R + row] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    lse_tot = mx + logf(tot);
    for (int s = 0; s < ns; ++s) {
      const float ls = part_lse[(int64_t)(s0 + s) * R + row];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - lse_tot);
      const float4* src = reinterpret_cast<const float4*>(part_out + ((int64_t)(s0 + s) * R + row) * 512);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 v = src[k * 32 + lane];
        acc[4 * k + 0] += w * v.x;
        acc[4 * k + 1] += w * v.y;
        acc[4 * k + 2] += w * v.z;
        acc[4 * k + 3] += w * v.w;
      }
    }
  }
  float f = 1.f;
  if (sink != nullptr) f = 1.f / (1.f + expf(sink[head] - lse_tot));
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] *= f;
  return lse_tot;
}

// Round a merged row to bf16 and store it (dst = the row's 512 elements), rounding acc in place.
__device__ __forceinline__ void store_row_bf16(uint16_t* dst, int lane, float (&acc)[16]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t lo = f32x2_to_bf16x2(acc[4 * k], acc[4 * k + 1]);
    const uint32_t hi = f32x2_to_bf16x2(acc[4 * k + 2], acc[4 * k + 3]);
    *reinterpret_cast<uint2*>(dst + (k * 32 + lane) * 4) = make_uint2(lo, hi);
    acc[4 * k] = __uint_as_float(lo << 16);
    acc[4 * k + 1] = __uint_as_float(lo & 0xFFFF0000u);
    acc[4 * k + 2] = __uint_as_float(hi << 16);
    acc[4 * k + 3] = __uint_as_float(hi & 0xFFFF0000u);
  }
}

}  // namespace mla
