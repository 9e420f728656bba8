// Split combine, KV-row write and page gather kernels for sm_103a.
#include <cstdint>
#include <cuda_runtime.h>

#include "combine_row.cuh"
#include "mla_kernels.h"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
  return static_cast<uint16_t>(f32x2_to_bf16x2(x, 0.f) & 0xFFFFu);
}
__device__ __forceinline__ float bf16_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// ----------------------------------------------------------------------------- combine
// One warp per query row of a request that the plan split into >= 2 pieces (the merge
// itself is merge_row in combine_row.cuh).
__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ part_out,
                                                      const float* __restrict__ part_lse,
                                                      const int32_t* __restrict__ num_splits, int R, int heads,
                                                      const float* __restrict__ sink, uint16_t* __restrict__ out,
                                                      float* __restrict__ lse, const float* __restrict__ part_max,
                                                      float* __restrict__ max_logits) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y;
  const int s0 = num_splits[b];
  const int ns = num_splits[b + 1] - s0;
  if (ns < 2) return;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= R) return;
  const int lane = threadIdx.x & 31;
  const int64_t orow = (int64_t)b * R + row;
  float acc[16];
  const float lse_tot = merge_row(part_out, part_lse, s0, ns, R, row, lane, sink, row % heads, acc);
  store_row_bf16(out + orow * 512, lane, acc);
  if (lane == 0) lse[orow] = lse_tot;
  if (max_logits != nullptr) {  // the largest scaled score: the largest over the splits
    float m = -INFINITY;
    for (int s = lane; s < ns; s += 32) m = fmaxf(m, part_max[(int64_t)(s0 + s) * R + row]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) max_logits[orow] = m;
  }
}

// One warp per query row: the merged (split) or decode-written (unsplit) row, with the
// inverse RoPE applied to elements [rope0, rope0 + 64): pair i = (u, v) -> (u c + v s,
// v c - u s), (c, s) = freqs[pos, 2i], freqs[pos, 2i + 1] ("MLA" API page of HALOps,
// mla_output_proj: the split-KV partials merged by LSE, then the RoPE of O undone). Written
// back to out.
__global__ void __launch_bounds__(256) combine_inv_rope_kernel(
    const float* __restrict__ part_out, const float* __restrict__ part_lse, const int32_t* __restrict__ num_splits,
    int R, int sq, int heads, const float* __restrict__ sink, const int32_t* __restrict__ positions,
    const float* __restrict__ freqs, int max_pos, int rope0, uint16_t* __restrict__ out, float* __restrict__ lse) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= R) return;
  const int lane = threadIdx.x & 31;
  const int64_t orow = (int64_t)b * R + row;
  const int s0 = num_splits[b];
  const int ns = num_splits[b + 1] - s0;
  float acc[16];
  if (ns >= 2 && part_out != nullptr) {  // no partials given: every row is taken as written
    const float lse_tot = merge_row(part_out, part_lse, s0, ns, R, row, lane, sink, row % heads, acc);
    store_row_bf16(out + orow * 512, lane, acc);  // acc now holds the bf16 values
    if (lane == 0) lse[orow] = lse_tot;
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint2 v = *reinterpret_cast<const uint2*>(out + orow * 512 + (k * 32 + lane) * 4);
      acc[4 * k] = __uint_as_float(v.x << 16);
      acc[4 * k + 1] = __uint_as_float(v.x & 0xFFFF0000u);
      acc[4 * k + 2] = __uint_as_float(v.y << 16);
      acc[4 * k + 3] = __uint_as_float(v.y & 0xFFFF0000u);
    }
  }
  const int pos = positions[b * sq + row / heads];
  if (pos < 0 || pos >= max_pos) return;  // no table row: left as merged
  const float* f = freqs + (int64_t)pos * 64;
  // lane holds elements d = 4 (32 k + lane) .. +3, i.e. pairs (d, d + 1) and (d + 2, d + 3)
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int d = (k * 32 + lane) * 4;
    if (d < rope0 || d >= rope0 + 64) continue;
    const int i = (d - rope0) >> 1;
    float y[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float c = f[2 * (i + h)], sn = f[2 * (i + h) + 1];
      const float u = acc[4 * k + 2 * h], v = acc[4 * k + 2 * h + 1];
      y[2 * h] = u * c + v * sn;
      y[2 * h + 1] = v * c - u * sn;
    }
    *reinterpret_cast<uint2*>(out + orow * 512 + d) = make_uint2(f32x2_to_bf16x2(y[0], y[1]), f32x2_to_bf16x2(y[2], y[3]));
  }
}

// ----------------------------------------------------------------------------- window runs
// One warp per token: compress its window (kv_indices[t, 0 .. len), len = topk_lengths[t]
// clamped to [0, topk], or topk) into at most two runs of consecutive cache slots ("MLA" API
// page of HALOps, mla_attention_plan). A run continues while the next slot is the previous
// one plus kv_run_step and lies on the same page; a window of more than two runs is cut to
// its first row. Each run is stored from its lowest slot upwards (attention does not depend
// on the order of its rows): row g < len0 is slot slot0 + g, row g >= len0 slot1 + g - len0.
// The lanes read 32 window entries at a time and find the run breaks with one ballot.
__global__ void __launch_bounds__(128) swa_plan_kernel(const int32_t* __restrict__ idx,
                                                       const int32_t* __restrict__ lens, int T, int topk,
                                                       int log2_ps, int step, int4* __restrict__ runs) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int len = lens ? lens[t] : topk;
  len = len < 0 ? 0 : (len > topk ? topk : len);
  if (len == 0) {
    if (lane == 0) runs[t] = make_int4(0, 0, 0, 0);
    return;
  }
  const int32_t* w = idx + (int64_t)t * topk;
  const int first = w[0];
  int nb = 0, b1 = len, s1 = 0;  // breaks found; row and slot of the first break
  int carry = first;
  for (int base = 0; base < len && nb < 2; base += 32) {
    const int g = base + lane;
    const bool valid = g < len;
    const int cur = valid ? w[g] : 0;
    int prev = __shfl_up_sync(0xffffffffu, cur, 1);
    if (lane == 0) prev = carry;
    const bool brk = valid && g > 0 && (cur != prev + step || (cur >> log2_ps) != (prev >> log2_ps));
    unsigned m = __ballot_sync(0xffffffffu, brk);
    while (m != 0u && nb < 2) {
      const int l = __ffs(m) - 1;
      const int v = __shfl_sync(0xffffffffu, cur, l);
      if (nb == 0) {
        b1 = base + l;
        s1 = v;
      }
      ++nb;
      m &= m - 1u;
    }
    carry = __shfl_sync(0xffffffffu, cur, 31);
  }
  if (lane != 0) return;
  if (nb >= 2) {
    runs[t] = make_int4(first, 1, first, 1);
    return;
  }
  const int c0 = b1;  // len when the window is one run
  const int lo0 = step > 0 ? first : first - (c0 - 1);
  const int lo1 = nb == 1 ? (step > 0 ? s1 : s1 - (len - b1 - 1)) : lo0 + c0;
  runs[t] = make_int4(lo0, c0, lo1, len);
}

// ----------------------------------------------------------------------------- kv write
// 448 * 2^e as fp32 (exact; +inf once it exceeds the fp32 range).
__device__ __forceinline__ float pow2x448(int e) {
  const int E = e + 8 + 127;  // 448 = 1.75 * 2^8
  if (E >= 255) return __uint_as_float(0x7F800000u);
  if (E <= 0) return 0.f;
  return __uint_as_float((static_cast<uint32_t>(E) << 23) | 0x600000u);
}
// Smallest e with 448 * 2^e >= a (a >= 1e-10), clamped to [-127, 127]; decided by
// exact comparisons of powers of two.
__device__ __forceinline__ int group_exponent(float a) {
  if (!(a <= 3.4028235e38f)) return 127;
  int e = static_cast<int>((__float_as_uint(a) >> 23) & 0xFFu) - 127 - 8;
  while (e < 127 && !(pow2x448(e) >= a)) ++e;
  while (e > -127 && pow2x448(e - 1) >= a) --e;
  return e;
}
// 2^-e as fp32 (exact for e in [-127, 126]).
__device__ __forceinline__ float pow2neg(int e) {
  const int E = 127 - e;
  if (E >= 255) return __uint_as_float(0x7F800000u);
  if (E <= 0) return __uint_as_float(0x00400000u >> (-E));
  return __uint_as_float(static_cast<uint32_t>(E) << 23);
}

// Write one bf16 row (generic pointer x, 16-byte aligned, row_elems values) into its
// page slot; all 32 lanes of the warp take part ("MLA" API page of HALOps,
// mla_attention: KV cache write of the RMSNorm'd row; kv_cache parameter for the layout).
__device__ __forceinline__ void write_row(const uint16_t* x, int lane, uint8_t* __restrict__ kv, int layout,
                                          int64_t page, int off, int page_size, int64_t page_bytes) {
  if (layout == 0) {
    const uint4* src = reinterpret_cast<const uint4*>(x);
    uint4* dst = reinterpret_cast<uint4*>(kv + page * page_bytes + (int64_t)off * 1152);
    for (int c = lane; c < 72; c += 32) dst[c] = src[c];
    return;
  }
  const int nope = layout == 1 ? 448 : 512;
  const int row_bytes = layout == 1 ? 576 : 640;
  uint8_t* dst = kv + page * page_bytes + (int64_t)off * row_bytes;
  // lane l holds elements [16 l, 16 l + 16), loaded at once; NoPE group g is lanes 4g .. 4g+3
  // (in the 512-wide DSV4 row, lanes 28-31 hold the RoPE part)
  float v[16];
  {
    const uint4 a = reinterpret_cast<const uint4*>(x)[2 * lane];
    const uint4 b = reinterpret_cast<const uint4*>(x)[2 * lane + 1];
    const uint32_t h[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[2 * k] = bf16_to_f32(h[k] & 0xFFFFu);
      v[2 * k + 1] = bf16_to_f32(h[k] >> 16);
    }
  }
  const bool in_nope = lane * 16 < nope;
  float a = 0.f;  // fmaxf returns the number when one operand is NaN: NaN elements do not count
#pragma unroll
  for (int k = 0; k < 16; ++k) a = fmaxf(a, fabsf(v[k]));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
  a = fmaxf(a, 1e-10f);
  const int e = group_exponent(a);
  if (in_nope) {
    const float sc = pow2neg(e);
    uint32_t w4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint16_t c0, c1;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c0) : "f"(v[4 * k + 1] * sc), "f"(v[4 * k] * sc));
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c1) : "f"(v[4 * k + 3] * sc), "f"(v[4 * k + 2] * sc));
      w4[k] = static_cast<uint32_t>(c0) | (static_cast<uint32_t>(c1) << 16);
      // a NaN element (left out of the amax above) is stored as the NaN code 0x7F, whatever its sign
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (v[4 * k + b] != v[4 * k + b]) w4[k] = (w4[k] & ~(0xFFu << (8 * b))) | (0x7Fu << (8 * b));
    }
    reinterpret_cast<uint4*>(dst)[lane] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
  } else {
    // DSV4 row: its 64 RoPE elements stay bf16, after the 448 code bytes
    const uint4* src = reinterpret_cast<const uint4*>(x) + 2 * lane;
    uint4* d2 = reinterpret_cast<uint4*>(dst + nope + (lane * 16 - nope) * 2);
    d2[0] = src[0];
    d2[1] = src[1];
  }
  // scale bytes: group g's exponent sits in lane 4g; lane 0 assembles the 8-byte slot
  uint32_t sbytes[2] = {0u, 0u};
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const int eg = __shfl_sync(0xffffffffu, e, 4 * g);
    if (g < nope / 64) sbytes[g >> 2] |= static_cast<uint32_t>(eg + 127) << (8 * (g & 3));
  }
  // the 576-wide row's RoPE part: 64 bf16 copied
  if (layout != 1 && lane < 8)
    reinterpret_cast<uint4*>(dst + nope)[lane] = reinterpret_cast<const uint4*>(x + nope)[lane];
  if (lane == 0) {
    uint2* sp = reinterpret_cast<uint2*>(kv + page * page_bytes + (int64_t)page_size * row_bytes + off * 8);
    *sp = make_uint2(sbytes[0], sbytes[1]);
  }
}

// One warp per new row, already normalised.
__global__ void __launch_bounds__(128) kv_write_kernel(const uint16_t* __restrict__ rows,
                                                       const int32_t* __restrict__ slots, int n,
                                                       uint8_t* __restrict__ kv, int layout, int64_t num_pages,
                                                       int page_size, int64_t page_bytes, uint32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= n) return;
  const int64_t slot = slots[r];
  if (slot < 0) return;
  const int64_t page = slot / page_size;
  if (page >= num_pages) {  // reported, not written
    if (lane == 0 && status != nullptr) atomicOr(status, 4u);
    return;
  }
  const int row_elems = layout == 1 ? 512 : 576;
  write_row(rows + (int64_t)r * row_elems, lane, kv, layout, page, static_cast<int>(slot % page_size), page_size,
            page_bytes);
}

// One warp per raw row: RMSNorm of the 512 latent elements and RoPE of the 64 RoPE
// elements in fp32 ("MLA" API page of HALOps, mla_attention: its normalise-and-rotate
// step before the cache write, kv_norm_weight / kv_eps / positions / freqs_real), the row
// rounded to bf16 in shared memory, then written as write_row writes it. Lane l
// holds latent elements [16 l, 16 l + 16) and RoPE pair l of the 576-wide layouts.
__global__ void __launch_bounds__(128) kv_write_norm_rope_kernel(
    const uint16_t* __restrict__ raw, const int32_t* __restrict__ slots, const int32_t* __restrict__ positions,
    const uint16_t* __restrict__ w, float eps, const float* __restrict__ freqs, int max_pos, int n,
    uint8_t* __restrict__ kv, int layout, int64_t num_pages, int page_size, int64_t page_bytes, uint32_t* status) {
  pdl_trigger();
  pdl_wait();
  __shared__ __align__(16) uint16_t srow[4][576];
  const int wi = threadIdx.x >> 5;
  const int r = blockIdx.x * 4 + wi;
  const int lane = threadIdx.x & 31;
  if (r >= n) return;
  const int64_t slot = slots[r];
  if (slot < 0) return;
  const int64_t page = slot / page_size;
  const int pos = positions[r];
  const uint32_t bad = (page >= num_pages ? 4u : 0u) | (pos < 0 || pos >= max_pos ? 8u : 0u);
  if (bad != 0u) {  // reported, not written
    if (lane == 0 && status != nullptr) atomicOr(status, bad);
    return;
  }
  const int row_elems = layout == 1 ? 512 : 576;
  const uint16_t* x = raw + (int64_t)r * row_elems;
  const float* f = freqs + (int64_t)pos * 64;
  float v[16];
  {
    const uint4 a = reinterpret_cast<const uint4*>(x)[2 * lane];
    const uint4 b = reinterpret_cast<const uint4*>(x)[2 * lane + 1];
    const uint32_t h[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[2 * k] = bf16_to_f32(h[k] & 0xFFFFu);
      v[2 * k + 1] = bf16_to_f32(h[k] >> 16);
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) ss = fmaf(v[k], v[k], ss);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float rinv = 1.0f / sqrtf(ss * (1.0f / 512.0f) + eps);
  {
    const uint4 a = reinterpret_cast<const uint4*>(w)[2 * lane];
    const uint4 b = reinterpret_cast<const uint4*>(w)[2 * lane + 1];
    const uint32_t h[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[2 * k] = v[2 * k] * rinv * bf16_to_f32(h[k] & 0xFFFFu);
      v[2 * k + 1] = v[2 * k + 1] * rinv * bf16_to_f32(h[k] >> 16);
    }
  }
  if (layout == 1 && lane >= 28) {
    // DSV4 row: elements 448..511 (lanes 28-31) are the RoPE part, rotated after the norm
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = 8 * (lane - 28) + k;
      const float c = f[2 * i], s = f[2 * i + 1];
      const float x0 = v[2 * k], x1 = v[2 * k + 1];
      v[2 * k] = x0 * c - x1 * s;
      v[2 * k + 1] = x0 * s + x1 * c;
    }
  }
  uint32_t o[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) o[k] = f32x2_to_bf16x2(v[2 * k], v[2 * k + 1]);
  reinterpret_cast<uint4*>(srow[wi])[2 * lane] = make_uint4(o[0], o[1], o[2], o[3]);
  reinterpret_cast<uint4*>(srow[wi])[2 * lane + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  if (layout != 1) {
    // k_pe (elements 512..575) is rotated as it comes, without the norm
    const uint32_t two = reinterpret_cast<const uint32_t*>(x + 512)[lane];
    const float x0 = bf16_to_f32(two & 0xFFFFu), x1 = bf16_to_f32(two >> 16);
    const float c = f[2 * lane], s = f[2 * lane + 1];
    reinterpret_cast<uint32_t*>(srow[wi] + 512)[lane] = f32x2_to_bf16x2(x0 * c - x1 * s, x0 * s + x1 * c);
  }
  __syncwarp();
  write_row(srow[wi], lane, kv, layout, page, static_cast<int>(slot % page_size), page_size, page_bytes);
}

// ----------------------------------------------------------------------------- gather
__global__ void __launch_bounds__(128) kv_gather_kernel(const uint8_t* __restrict__ kv, int layout,
                                                        int64_t num_pages, int page_size, int64_t page_bytes,
                                                        const int32_t* __restrict__ bt_row, int max_pages,
                                                        int length, float* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int j = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (j >= length) return;
  const int dqk = layout == 1 ? 512 : 576;
  float* o = out + (int64_t)j * dqk;
  const int pi = j / page_size;
  const int64_t page = pi < max_pages ? bt_row[pi] : -1;
  if (page < 0 || page >= num_pages) {
    for (int d = lane; d < dqk; d += 32) o[d] = __uint_as_float(0x7FC00000u);
    return;
  }
  const int off = j % page_size;
  if (layout == 0) {
    const uint16_t* src = reinterpret_cast<const uint16_t*>(kv + page * page_bytes + (int64_t)off * 1152);
    for (int d = lane; d < 576; d += 32) o[d] = bf16_to_f32(src[d]);
    return;
  }
  const int nope = layout == 1 ? 448 : 512;
  const int row_bytes = layout == 1 ? 576 : 640;
  const uint8_t* src = kv + page * page_bytes + (int64_t)off * row_bytes;
  const uint8_t* sc = kv + page * page_bytes + (int64_t)page_size * row_bytes + off * 8;
  for (int d = 2 * lane; d < nope; d += 64) {
    const uint32_t two = *reinterpret_cast<const uint16_t*>(src + d);
    const float2 v = e4m3x2_to_f32x2(two);
    const float s = ue8m0_to_f32(sc[d >> 6]);
    o[d] = v.x * s;
    o[d + 1] = v.y * s;
  }
  const uint16_t* rope = reinterpret_cast<const uint16_t*>(src + nope);
  for (int d = lane; d < 64; d += 32) o[nope + d] = bf16_to_f32(rope[d]);
}

}  // namespace

cudaError_t launch_combine(const float* part_out, const float* part_lse, const int32_t* num_splits, int batch,
                           int rows_per_req, int heads, const float* sink, uint16_t* out, float* lse,
                           const float* part_max, float* max_logits, cudaStream_t stream) {
  if (batch <= 0 || rows_per_req <= 0) return cudaSuccess;
  // one warp per row, four rows per 128-thread block (96 registers a thread: five blocks
  // per SM, against two of 256 threads)
  dim3 grid((rows_per_req + 3) / 4, batch);
  return launch_pdl(combine_kernel, grid, dim3(128), 0, stream, part_out, part_lse, num_splits, rows_per_req, heads,
                    sink, out, lse, part_max, max_logits);
}

cudaError_t launch_swa_plan(const int32_t* kv_indices, const int32_t* topk_lengths, int num_tokens, int topk,
                            int page_size, int kv_run_step, int32_t* runs, cudaStream_t stream) {
  int lg = 0;
  while ((1 << lg) < page_size) ++lg;
  return launch_pdl(swa_plan_kernel, dim3((num_tokens + 3) / 4), dim3(128), 0, stream, kv_indices, topk_lengths,
                    num_tokens, topk, lg, kv_run_step, reinterpret_cast<int4*>(runs));
}

cudaError_t launch_combine_inv_rope(const float* part_out, const float* part_lse, const int32_t* num_splits, int batch,
                                    int sq, int heads, const float* sink, const int32_t* positions, const float* freqs,
                                    int max_pos, int rope0, uint16_t* out, float* lse, cudaStream_t stream) {
  const int R = sq * heads;
  dim3 grid((R + 7) / 8, batch);
  return launch_pdl(combine_inv_rope_kernel, grid, dim3(256), 0, stream, part_out, part_lse, num_splits, R, sq, heads,
                    sink, positions, freqs, max_pos, rope0, out, lse);
}

cudaError_t launch_kv_write(const uint16_t* rows, const int32_t* slots, int n, uint8_t* kv, int layout,
                            int64_t num_pages, int page_size, int64_t page_bytes, uint32_t* status,
                            cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  return launch_pdl(kv_write_kernel, dim3((n + 3) / 4), dim3(128), 0, stream, rows, slots, n, kv, layout, num_pages,
                    page_size, page_bytes, status);
}

cudaError_t launch_kv_write_norm_rope(const uint16_t* raw, const int32_t* slots, const int32_t* positions,
                                     const uint16_t* norm_weight, float eps, const float* freqs, int max_pos, int n,
                                     uint8_t* kv, int layout, int64_t num_pages, int page_size, int64_t page_bytes,
                                     uint32_t* status, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  return launch_pdl(kv_write_norm_rope_kernel, dim3((n + 3) / 4), dim3(128), 0, stream, raw, slots, positions,
                    norm_weight, eps, freqs, max_pos, n, kv, layout, num_pages, page_size, page_bytes, status);
}

cudaError_t launch_kv_gather(const uint8_t* kv, int layout, int64_t num_pages, int page_size, int64_t page_bytes,
                             const int32_t* bt_row, int max_pages, int length, float* out, cudaStream_t stream) {
  if (length <= 0) return cudaSuccess;
  return launch_pdl(kv_gather_kernel, dim3((length + 3) / 4), dim3(128), 0, stream, kv, layout, num_pages, page_size,
                    page_bytes, bt_row, max_pages, length, out);
}

}  // namespace mla
