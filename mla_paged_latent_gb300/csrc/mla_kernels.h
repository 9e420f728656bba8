// Internal interface between the C-ABI layer (api.cpp) and the CUDA kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <vector>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mla {

constexpr int kBlockRows = 64;    // KV rows per tile
constexpr int kGroupRows = 64;    // query rows per work item
constexpr int kDecodeThreads = 512;

struct DecodeParams {
  const uint16_t* q;              // bf16 [T, heads, dqk] (L2 prefetch; loads use the tensor map)
  const uint8_t* kv;              // paged cache (converter path and L2 prefetch)
  const int32_t* block_table;     // [batch, max_pages]; null: positions are rows of one unpaged run
  const int32_t* seqlens;         // [batch]; null: every request has uniform_len rows
  const float* sink;              // [heads] or null
  const int32_t* indices;         // [T, topk] or null
  const int32_t* runs;            // [T, 4] (slot0, len0, slot1, rows) or null: run-window mode
  const int32_t* sched;           // [num_partitions, 8]
  const int32_t* num_splits;      // [batch + 1]
  uint16_t* out;                  // bf16 [T, heads, 512]
  float* lse;                     // [T, heads]
  float* part_out;                // [total_splits, R, 512]
  float* part_lse;                // [total_splits, R]
  float* max_logits;              // [T, heads] or null: the largest scaled score of each row
  float* part_max;                // [total_splits, R]: its split partials (with max_logits)
  unsigned int* status;           // device status word
  int64_t num_pages;
  int64_t page_bytes;
  int32_t row_bytes;
  int32_t page_size;
  int32_t log2_ps;
  int32_t max_pages;
  int32_t batch;
  int32_t sq;
  int32_t heads;
  int32_t rows_per_req;           // R = sq * heads
  int32_t groups;                 // ceil(R / 64)
  int32_t qbox_rows;              // rows of one Q TMA box = min(64, R)
  int32_t topk;
  int32_t causal;
  int32_t num_partitions;
  int32_t num_work;               // num_partitions * groups
  float scale_log2;               // sm_scale * log2(e)
  int32_t test_withhold_signal;   // MLA_DECODE_TEST_WITHHOLD_SIGNAL: skip the first S-complete commit
  int32_t uniform_len;            // rows of every request when seqlens is null
};

// Tensor maps that move whole 64-row blocks in one copy (a tensor copy costs about the same
// issue time whatever its size, so few large copies beat many 8-KiB slabs): q9 = 64 query
// rows x the 9 dim slabs of a bf16 576-wide row, landing slab-major; kv3 / kv2 = 3 / 2 dim
// slabs of one 64-row page block. Only encoded (valid) when page_size >= 64 and the
// request has >= 64 query rows.
struct WideMaps {
  CUtensorMap q9;
  CUtensorMap kv3;
  CUtensorMap kv2;
  int valid;
};

// Kernel variants: layout 0 with TMA page loads (dense), layout 0 gathered by
// the converter warps (sparse), layouts 1 and 2 (fp8, dense or sparse).
enum class DecodeVariant { kBf16Tma = 0, kBf16Gather = 1, kFp8_448 = 2, kFp8_512 = 3 };

size_t decode_smem_bytes(DecodeVariant v);

// The CTA-pair kernel (decode_pair_sm103.cu): bf16 rows loaded by TMA, query rows in
// groups of 128 (rows_per_req % 128 == 0); `clusters` pairs of CTAs.
size_t decode_pair_smem_bytes();
cudaError_t launch_decode_pair(const DecodeParams& p, const CUtensorMap& q_map, const CUtensorMap& kv_map,
                               const WideMaps& wide, int clusters, cudaStream_t stream);
cudaError_t decode_pair_max_clusters(int* clusters);
cudaError_t launch_decode(DecodeVariant v, const DecodeParams& p, const CUtensorMap& q_map,
                          const CUtensorMap& kv_map, int grid, cudaStream_t stream);

cudaError_t launch_combine(const float* part_out, const float* part_lse, const int32_t* num_splits, int batch,
                           int rows_per_req, int heads, const float* sink, uint16_t* out, float* lse,
                           const float* part_max, float* max_logits, cudaStream_t stream);

cudaError_t launch_kv_write(const uint16_t* rows, const int32_t* slots, int n, uint8_t* kv, int layout,
                            int64_t num_pages, int page_size, int64_t page_bytes, uint32_t* status,
                            cudaStream_t stream);

cudaError_t launch_kv_write_norm_rope(const uint16_t* raw, const int32_t* slots, const int32_t* positions,
                                     const uint16_t* norm_weight, float eps, const float* freqs, int max_pos, int n,
                                     uint8_t* kv, int layout, int64_t num_pages, int page_size, int64_t page_bytes,
                                     uint32_t* status, cudaStream_t stream);

cudaError_t launch_swa_plan(const int32_t* kv_indices, const int32_t* topk_lengths, int num_tokens, int topk,
                            int page_size, int kv_run_step, int32_t* runs, cudaStream_t stream);

cudaError_t launch_combine_inv_rope(const float* part_out, const float* part_lse, const int32_t* num_splits, int batch,
                                    int sq, int heads, const float* sink, const int32_t* positions, const float* freqs,
                                    int max_pos, int rope0, uint16_t* out, float* lse, cudaStream_t stream);

cudaError_t launch_combine_v_up(const float* part_out, const float* part_lse, const int32_t* num_splits, int batch,
                                int sq, int heads, const float* sink, uint16_t* out, float* lse, uint16_t* o_v,
                                unsigned int* status, const CUtensorMap& w_map, cudaStream_t stream);

cudaError_t launch_kv_gather(const uint8_t* kv, int layout, int64_t num_pages, int page_size, int64_t page_bytes,
                             const int32_t* bt_row, int max_pages, int length, float* out, cudaStream_t stream);

// Host split-KV plan (rule documented on mla_decode_plan in include/mla_decode.h).
struct PlanResult {
  std::vector<int32_t> sched;        // [partitions * 8]
  std::vector<int32_t> num_splits;   // [batch + 1]
  int partitions = 0;
  int groups = 0;
  int total_splits = 0;
  int max_splits = 0;
};
#ifdef __CUDACC__
// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel on `stream` drains (hiding the launch gap); every
// kernel of this library calls pdl_wait() before it reads its inputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}
#endif

// Workspace bytes of a decode with `total_splits` splits of `rows_per_req` query rows:
// the status header, the split partial lse (padded to 256 B) and the partial outputs.
size_t workspace_bytes_for(int64_t total_splits, int64_t rows_per_req);

// Rows of request r: its cache length, or the one length of all requests (sparse prefill).
__host__ __device__ inline int request_len(const DecodeParams& P, int r) {
  return P.seqlens != nullptr ? P.seqlens[r] : P.uniform_len;
}

PlanResult make_plan(const int32_t* seqlens, int batch, int sq, int heads, int topk, int min_splits, int num_sms);

}  // namespace mla
