// Value up-projection of the latent attention output, fused with the split combine.
//
// In the absorbed form the decode returns, per query row (token t, head n), the
// attention-weighted latent x = sum_j p_j kv_c_j (512 wide). The head's value is
// o_v = x W_UV[n] with W_UV [N, 512, dv] ("mla_attention.py ·
// tduncan/Nvidia-Optimization-Stack-VLLM": _v_up_proj multiplies (N, B, L) by
// W_UV (N, L, V)). Split requests are merged first, by log-sum-exp of their
// partials with the sink applied once, exactly as mla_combine does; the merged
// latent row is rounded to bf16 (what mla_combine writes) and multiplied in that
// precision.
//
// One CTA per head: W_UV[n] (512 x 128 bf16, 128 KB) is loaded once by TMA; token
// blocks of 64 rows are merged or read by sixteen warps into a K-major shared tile
// X [64 x 512]; one thread issues D^T = W^T X^T as 32 tcgen05 MMAs (M = 128 value
// dims, N = 64 tokens, K = 16) into TMEM; warps 0-3 write o_v. The merge is
// merge_row (combine_row.cuh), so the merged rows equal mla_combine's bit for bit.
#include <cstdint>
#include <cuda_runtime.h>

#include "combine_row.cuh"
#include "mla_kernels.h"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

constexpr int kVupThreads = 512;  // 16 warps: 4 latent rows each per 64-token block
constexpr uint32_t kWBytes = 512 * 128 * 2;      // W_UV[n]: 2 slabs (64 value dims each) of 512 x 128 B
constexpr uint32_t kWSlab = 512 * 128;           // 64 KB
constexpr uint32_t kXSlab = 64 * 128;            // 64 token rows x 64 latent elements
constexpr uint32_t kXBytes = 8 * kXSlab;         // 64 KB
constexpr uint32_t kVupSmem = kWBytes + kXBytes + 1024 + 64;

struct VupParams {
  const float* part_out;      // [S, R, 512] or null when no request is split
  const float* part_lse;      // [S, R]
  const int32_t* num_splits;  // [B + 1]
  const float* sink;          // [N] or null
  uint16_t* out;              // latent out bf16 [T, N, 512]: read (unsplit rows), written (split rows)
  float* lse;                 // [T, N]: written for split rows
  uint16_t* o_v;              // bf16 [T, N, 128]
  unsigned int* status;       // optional status word (bit 0: a bounded wait ran out)
  int32_t batch, sq, heads, rows_per_req, tokens;
};

__device__ __forceinline__ uint16_t to_bf16(float x) { return static_cast<uint16_t>(f32x2_to_bf16x2(x, 0.f) & 0xFFFFu); }

__device__ bool wait_bounded(uint32_t bar, uint32_t parity, unsigned int* status) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > 2000000000ull) {
      if (status) atomicOr(status, 1u);
      return false;
    }
  }
  return true;
}

__global__ void __launch_bounds__(kVupThreads, 1)
    vup_kernel(const __grid_constant__ VupParams P, const __grid_constant__ CUtensorMap w_map) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_addr(smem);
  const uint32_t w_s = sb, x_s = sb + kWBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWBytes + kXBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4);
  volatile int* fail_flag = reinterpret_cast<volatile int*>(bars + 5);
  const uint32_t bar_w = smem_addr(&bars[0]), bar_d = smem_addr(&bars[1]);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = blockIdx.x;

  if (tid == 0) {
    mbar_init(bar_w, 1);
    mbar_init(bar_d, 1);
    *fail_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(tmem_slot), 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();
  pdl_wait();
  const uint32_t tmem = *tmem_slot;
  if (tid == 0) {
    tma_prefetch_desc(&w_map);
    mbar_arrive_expect_tx(bar_w, kWBytes);
    for (int h = 0; h < 2; ++h)
      for (int lb = 0; lb < 8; ++lb) tma_load_3d(w_s + h * kWSlab + lb * 64 * 128, &w_map, 64 * h, 64 * lb, n, bar_w);
  }
  const int R = P.rows_per_req;
  const int nblk = (P.tokens + 63) / 64;
  for (int tb = 0; tb < nblk; ++tb) {
    // ---- X: the merged (or decode-written) latent rows of this head, bf16, K-major SW128.
    // Each warp first asks L2 for all of its rows (partials or decode output), so that only
    // its first row waits for HBM.
    if (lane == 0) {
      for (int rr = warp; rr < 64; rr += kVupThreads / 32) {
        const int t = tb * 64 + rr;
        if (t >= P.tokens) break;
        const int b = t / P.sq;
        const int row = (t % P.sq) * P.heads + n;
        const int s0 = P.num_splits[b];
        const int ns = P.num_splits[b + 1] - s0;
        if (ns >= 2 && P.part_out != nullptr) {
          for (int s = 0; s < ns; ++s)
            prefetch_l2_bulk(P.part_out + ((int64_t)(s0 + s) * R + row) * 512, 2048);
        } else {
          prefetch_l2_bulk(P.out + ((int64_t)b * R + row) * 512, 1024);
        }
      }
    }
    for (int rr = warp; rr < 64; rr += kVupThreads / 32) {
      const int t = tb * 64 + rr;
      float acc[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] = 0.f;
      if (t < P.tokens) {
        const int b = t / P.sq;
        const int row = (t % P.sq) * P.heads + n;  // row within the request
        const int64_t orow = (int64_t)b * R + row;
        const int s0 = P.num_splits[b];
        const int ns = P.num_splits[b + 1] - s0;
        if (ns >= 2 && P.part_out != nullptr) {
          // merged exactly as the combine kernel merges it, and written back the same way
          const float lse_tot = merge_row(P.part_out, P.part_lse, s0, ns, R, row, lane, P.sink, n, acc);
          store_row_bf16(P.out + orow * 512, lane, acc);
          if (lane == 0) P.lse[orow] = lse_tot;
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint2 v = *reinterpret_cast<const uint2*>(P.out + orow * 512 + (k * 32 + lane) * 4);
            acc[4 * k] = __uint_as_float(v.x << 16);
            acc[4 * k + 1] = __uint_as_float(v.x & 0xFFFF0000u);
            acc[4 * k + 2] = __uint_as_float(v.y << 16);
            acc[4 * k + 3] = __uint_as_float(v.y & 0xFFFF0000u);
          }
        }
      }
      // lane holds latent elements d = 4 (32 k + lane) .. +3; 8-byte pieces stay inside a 16-B chunk
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int d = (k * 32 + lane) * 4;
        const uint32_t lo = f32x2_to_bf16x2(acc[4 * k], acc[4 * k + 1]);
        const uint32_t hi = f32x2_to_bf16x2(acc[4 * k + 2], acc[4 * k + 3]);
        const uint32_t a = x_s + (d >> 6) * kXSlab + sw128_offset(rr, d & 63);
        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(a), "r"(lo), "r"(hi) : "memory");
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- D^T [128 value dims x 64 tokens] = W^T X^T, K = 512
    if (tid == 0) {
      bool ok = tb > 0 || wait_bounded(bar_w, 0, P.status);
      if (ok) {
        constexpr uint32_t idesc = idesc_bf16_f32(128, 64, 1, 0);
        const uint64_t wdesc = sdesc_sw128(0, kWSlab, 1024) | (w_s >> 4);  // MN-major: value dims in 2 slabs
        const uint64_t xdesc = sdesc_sw128(0, 16, 1024) | (x_s >> 4);      // K-major token rows
#pragma unroll 1
        for (int j = 0; j < 32; ++j)
          mma_bf16_ss(tmem, wdesc + j * (2048 >> 4), xdesc + (j >> 2) * (kXSlab >> 4) + (j & 3) * 2, idesc,
                      j ? 1u : 0u);
        mma_commit(bar_d);
      } else {
        *fail_flag = 1;
      }
    }
    __syncthreads();
    if (*fail_flag) break;
    // ---- o_v[t, n, v] = bf16(D^T[v, t]); warp w reaches TMEM lanes 32 w .. 32 w + 31
    if (warp < 4) {
      const bool ok = wait_bounded(bar_d, tb & 1, P.status);
      if (ok) {
        tc_fence_after();
        const int v = warp * 32 + lane;
        for (int c = 0; c < 64; c += 16) {
          uint32_t r16[16];
          tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c, r16);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int t = tb * 64 + c + i;
            if (t < P.tokens) P.o_v[((int64_t)t * P.heads + n) * 128 + v] = to_bf16(__uint_as_float(r16[i]));
          }
        }
      } else {
        *fail_flag = 1;
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*fail_flag) break;
  }
  // copies or MMAs that may still be in flight after a failed wait: give them time to land
  if (tid == 0 && *fail_flag) {
    wait_bounded(bar_w, 0, nullptr);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64);
}

}  // namespace

cudaError_t launch_combine_v_up(const float* part_out, const float* part_lse, const int32_t* num_splits, int batch,
                                int sq, int heads, const float* sink, uint16_t* out, float* lse, uint16_t* o_v,
                                unsigned int* status, const CUtensorMap& w_map, cudaStream_t stream) {
  VupParams p;
  p.part_out = part_out;
  p.part_lse = part_lse;
  p.num_splits = num_splits;
  p.sink = sink;
  p.out = out;
  p.lse = lse;
  p.o_v = o_v;
  p.status = status;
  p.batch = batch;
  p.sq = sq;
  p.heads = heads;
  p.rows_per_req = sq * heads;
  p.tokens = batch * sq;
  cudaError_t e = cudaFuncSetAttribute(vup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kVupSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(vup_kernel, dim3(heads), dim3(kVupThreads), kVupSmem, stream, p, w_map);
}

}  // namespace mla
