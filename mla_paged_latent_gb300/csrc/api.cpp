// C ABI of the paged-latent MLA decode library: argument validation, error
// strings, TMA tensor-map encoding and kernel launches. Declarations and the
// meaning of every argument are in include/mla_decode.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "mla_decode.h"
#include "mla_kernels.h"

namespace {

thread_local std::string g_last_error = "no error";

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(MLA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int log2i(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

int layout_geometry(int layout, int page_size, int64_t* row_bytes, int64_t* page_bytes, int* dqk) {
  switch (layout) {
    case MLA_KV_BF16_576:
      *row_bytes = 1152;
      *page_bytes = static_cast<int64_t>(page_size) * 1152;
      *dqk = 576;
      return 0;
    case MLA_KV_FP8_448_UE8M0:
      *row_bytes = 576;
      *page_bytes = ((static_cast<int64_t>(page_size) * 584 + 575) / 576) * 576;
      *dqk = 512;
      return 0;
    case MLA_KV_FP8_512_UE8M0:
      *row_bytes = 640;
      *page_bytes = ((static_cast<int64_t>(page_size) * 648 + 639) / 640) * 640;
      *dqk = 576;
      return 0;
    default:
      return -1;
  }
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

namespace mla {
size_t workspace_bytes_for(int64_t total_splits, int64_t rows_per_req) {
  // status header, partial lse (padded to 256 B), partial out, partial max logits (padded)
  const size_t n = static_cast<size_t>(total_splits) * static_cast<size_t>(rows_per_req);
  return MLA_WORKSPACE_HEADER + align256(n * sizeof(float)) + n * MLA_DV * sizeof(float) + align256(n * sizeof(float));
}
}  // namespace mla

namespace {
using mla::workspace_bytes_for;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn(int* err) {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  static int status = 0;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || p == nullptr) status = 1;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  *err = status;
  return fn;
}

// Most 2-CTA clusters of the pair decode kernel resident at once on the current device
// (looked up once per device).
int pair_cluster_capacity(int* n) {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return fail(MLA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  if (cache[dev] == 0) {
    int c = 0;
    e = mla::decode_pair_max_clusters(&c);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveClusters (pair decode kernel)");
    if (c < 1) return fail(MLA_ERR_UNSUPPORTED, "no 2-CTA cluster of the pair decode kernel fits on this device");
    cache[dev] = c;
  }
  *n = cache[dev];
  return 0;
}

int current_sm_count(int* n) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
  return 0;
}

}  // namespace

namespace mla {
// Lets other translation units of the library report a failure through mla_last_error().
int set_last_error(int code, const char* msg) {
  g_last_error = msg;
  return code;
}
}  // namespace mla

extern "C" {

const char* mla_last_error(void) { return g_last_error.c_str(); }

int mla_page_bytes(mla_kv_layout layout, int32_t page_size, int64_t* page_bytes) {
  if (page_bytes == nullptr) return fail(MLA_ERR_INVALID_ARG, "mla_page_bytes: page_bytes is NULL");
  if (!pow2(page_size)) return fail(MLA_ERR_INVALID_ARG, "page_size %d is not a power of two", page_size);
  int64_t rb;
  int dqk;
  if (layout_geometry(layout, page_size, &rb, page_bytes, &dqk) != 0)
    return fail(MLA_ERR_INVALID_ARG, "unknown layout %d", static_cast<int>(layout));
  return MLA_OK;
}

int mla_decode_plan(const int32_t* cache_seqlens, int32_t batch, int32_t q_tokens_per_req, int32_t num_heads,
                    int32_t topk, int32_t min_splits, int32_t num_sms, int32_t* sched, int32_t sched_capacity,
                    int32_t* num_splits, mla_plan_info* info) {
  if (cache_seqlens == nullptr || info == nullptr) return fail(MLA_ERR_INVALID_ARG, "mla_decode_plan: NULL argument");
  if (batch < 1 || q_tokens_per_req < 1 || num_heads < 1 || topk < 0 || min_splits < 1 || num_sms < 1)
    return fail(MLA_ERR_INVALID_ARG,
                "mla_decode_plan: batch=%d q_tokens=%d heads=%d topk=%d min_splits=%d num_sms=%d out of range", batch,
                q_tokens_per_req, num_heads, topk, min_splits, num_sms);
  for (int b = 0; b < batch; ++b)
    if (cache_seqlens[b] < 0) return fail(MLA_ERR_INVALID_ARG, "cache_seqlens[%d] = %d < 0", b, cache_seqlens[b]);
  const mla::PlanResult p =
      mla::make_plan(cache_seqlens, batch, q_tokens_per_req, num_heads, topk, min_splits, num_sms);
  info->num_partitions = p.partitions;
  info->groups = p.groups;
  info->total_splits = p.total_splits;
  info->max_splits = p.max_splits;
  info->workspace_bytes = workspace_bytes_for(p.total_splits, static_cast<int64_t>(q_tokens_per_req) * num_heads);
  if (sched == nullptr) return MLA_OK;
  if (num_splits == nullptr) return fail(MLA_ERR_INVALID_ARG, "mla_decode_plan: num_splits is NULL");
  if (sched_capacity < p.partitions)
    return fail(MLA_ERR_CAPACITY, "mla_decode_plan: sched needs %d rows, capacity %d", p.partitions, sched_capacity);
  std::memcpy(sched, p.sched.data(), p.sched.size() * sizeof(int32_t));
  std::memcpy(num_splits, p.num_splits.data(), p.num_splits.size() * sizeof(int32_t));
  return MLA_OK;
}

}  // extern "C"

namespace {
// Shared body of mla_decode and mla_decode_runs. runs != NULL selects the run-window mode:
// candidates are the rows of each token's (at most two) slot runs, topk is the window, and
// block_table / cache_seqlens are not used.
int decode_impl(const void* q, const void* kv_cache, mla_kv_layout layout, int64_t num_pages, int32_t page_size,
                const int32_t* block_table, int32_t max_pages, const int32_t* cache_seqlens, int32_t batch,
                int32_t q_tokens_per_req, int32_t num_heads, float sm_scale, const float* sink,
                const int32_t* indices, const int32_t* runs, int32_t topk, int32_t causal, const int32_t* sched,
                const int32_t* num_splits, int32_t num_partitions, int32_t total_splits, void* workspace,
                size_t workspace_bytes, void* out, float* lse, uint32_t flags, void* stream, int32_t uniform_len = 0,
                float* max_logits = nullptr) {
  if (!q || !kv_cache || !sched || !num_splits || !workspace || !out || !lse)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: NULL pointer argument");
  // block_table and cache_seqlens are required except for run windows and for the unpaged
  // run of sparse prefill (uniform_len > 0)
  if (runs == nullptr && uniform_len == 0 && (!block_table || !cache_seqlens))
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: NULL pointer argument");
  if (runs != nullptr) {
    if (indices != nullptr || topk < 1 || causal)
      return fail(MLA_ERR_INVALID_ARG, "mla_decode_runs: window must be >= 1, with no indices and no causal mask");
    max_pages = 1;
  }
  int64_t row_bytes, page_bytes;
  int dqk;
  if (layout_geometry(layout, page_size, &row_bytes, &page_bytes, &dqk) != 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: unknown layout %d", static_cast<int>(layout));
  if (!pow2(page_size) || page_size < 8)
    return fail(MLA_ERR_UNSUPPORTED, "mla_decode: page_size %d must be a power of two >= 8", page_size);
  if (batch < 1 || q_tokens_per_req < 1 || num_heads < 1 || num_pages < 1 || max_pages < 1 || num_partitions < 1)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: batch/q_tokens/heads/num_pages/max_pages/num_partitions must be >= 1");
  const int64_t R = static_cast<int64_t>(q_tokens_per_req) * num_heads;
  if (R > 4096) return fail(MLA_ERR_UNSUPPORTED, "mla_decode: q_tokens_per_req * num_heads = %lld > 4096", (long long)R);
  if (static_cast<int64_t>(batch) * R >= (1ll << 31))
    return fail(MLA_ERR_UNSUPPORTED, "mla_decode: too many query rows");
  if (runs == nullptr && (indices != nullptr) != (topk > 0))
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: indices must be given exactly when topk > 0 (topk=%d)", topk);
  if ((indices != nullptr || runs != nullptr) && q_tokens_per_req > 1 && num_heads % mla::kGroupRows != 0)
    return fail(MLA_ERR_UNSUPPORTED, "mla_decode: sparse decode with several tokens needs heads %% 64 == 0");
  if (total_splits < batch) return fail(MLA_ERR_INVALID_ARG, "mla_decode: total_splits %d < batch %d", total_splits, batch);
  if (!(sm_scale > 0.f) || !(sm_scale < 1e30f))
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: sm_scale must be a positive finite number");
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out))
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: q, kv_cache and out must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: workspace must be 256-byte aligned");
  const size_t need = workspace_bytes_for(total_splits, R);
  if (workspace_bytes < need)
    return fail(MLA_ERR_WORKSPACE_TOO_SMALL, "mla_decode: workspace %zu bytes < %zu needed", workspace_bytes, need);

  int enc_err = 0;
  EncodeTiledFn encode = get_encode_fn(&enc_err);
  if (enc_err) return fail(MLA_ERR_CUDA, "mla_decode: cuTensorMapEncodeTiled is unavailable");
  int num_sms = 0;
  if (int rc = current_sm_count(&num_sms)) return rc;

  const int groups = static_cast<int>((R + mla::kGroupRows - 1) / mla::kGroupRows);
  const int qbox = static_cast<int>(R < mla::kGroupRows ? R : mla::kGroupRows);
  CUtensorMap q_map, kv_map;
  std::memset(&q_map, 0, sizeof q_map);
  std::memset(&kv_map, 0, sizeof kv_map);
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(dqk), static_cast<cuuint64_t>(batch) * R};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(dqk) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(qbox)};
    const cuuint32_t es[2] = {1, 1};
    CUresult r = encode(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MLA_ERR_CUDA, "mla_decode: encoding the q tensor map failed (%d)", (int)r);
  }
  const bool tma_kv = (layout == MLA_KV_BF16_576) && indices == nullptr && runs == nullptr;
  if (tma_kv) {
    const cuuint64_t dims[3] = {576, static_cast<cuuint64_t>(page_size), static_cast<cuuint64_t>(num_pages)};
    const cuuint64_t strides[2] = {1152, static_cast<cuuint64_t>(page_bytes)};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(page_size < 64 ? page_size : 64), 1};
    const cuuint32_t es[3] = {1, 1, 1};
    CUresult r = encode(&kv_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(kv_cache), dims, strides, box,
                        es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MLA_ERR_CUDA, "mla_decode: encoding the KV tensor map failed (%d)", (int)r);
  }

  // whole 64-row blocks in few copies: Q rows x 9 dim slabs, and 3 or 2 dim slabs of a page block
  mla::WideMaps wide;
  std::memset(&wide, 0, sizeof wide);
  if (tma_kv && page_size >= 64 && qbox == 64) {
    const cuuint32_t es[4] = {1, 1, 1, 1};
    const cuuint64_t qd[3] = {64, static_cast<cuuint64_t>(batch) * R, 9};
    const cuuint64_t qs[2] = {1152, 128};
    const cuuint32_t qb[3] = {64, 64, 9};
    CUresult r = encode(&wide.q9, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), qd, qs, qb, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MLA_ERR_CUDA, "mla_decode: encoding the wide q tensor map failed (%d)", (int)r);
    const cuuint64_t kd[4] = {64, static_cast<cuuint64_t>(page_size), 9, static_cast<cuuint64_t>(num_pages)};
    const cuuint64_t ks[3] = {1152, 128, static_cast<cuuint64_t>(page_bytes)};
    const cuuint32_t kb3[4] = {64, 64, 3, 1};
    const cuuint32_t kb2[4] = {64, 64, 2, 1};
    r = encode(&wide.kv3, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(kv_cache), kd, ks, kb3, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MLA_ERR_CUDA, "mla_decode: encoding the wide KV tensor map failed (%d)", (int)r);
    r = encode(&wide.kv2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(kv_cache), kd, ks, kb2, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MLA_ERR_CUDA, "mla_decode: encoding the wide KV tensor map failed (%d)", (int)r);
    wide.valid = 1;
  }

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t nrows = static_cast<size_t>(total_splits) * static_cast<size_t>(R);
  mla::DecodeParams p;
  std::memset(&p, 0, sizeof p);
  p.q = static_cast<const uint16_t*>(q);
  p.kv = static_cast<const uint8_t*>(kv_cache);
  p.block_table = block_table;
  p.seqlens = cache_seqlens;
  p.sink = sink;
  p.indices = indices;
  p.runs = runs;
  p.sched = sched;
  p.num_splits = num_splits;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.status = reinterpret_cast<unsigned int*>(ws);
  p.part_lse = reinterpret_cast<float*>(ws + MLA_WORKSPACE_HEADER);
  p.part_out = reinterpret_cast<float*>(ws + MLA_WORKSPACE_HEADER + align256(nrows * sizeof(float)));
  p.part_max = reinterpret_cast<float*>(ws + MLA_WORKSPACE_HEADER + align256(nrows * sizeof(float)) +
                                        nrows * MLA_DV * sizeof(float));
  p.max_logits = max_logits;
  p.uniform_len = uniform_len;
  p.num_pages = num_pages;
  p.page_bytes = page_bytes;
  p.row_bytes = static_cast<int32_t>(row_bytes);
  p.page_size = page_size;
  p.log2_ps = log2i(page_size);
  p.max_pages = max_pages;
  p.batch = batch;
  p.sq = q_tokens_per_req;
  p.heads = num_heads;
  p.rows_per_req = static_cast<int32_t>(R);
  p.groups = groups;
  p.qbox_rows = qbox;
  p.topk = topk;
  p.causal = causal ? 1 : 0;
  p.num_partitions = num_partitions;
  p.num_work = num_partitions * groups;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.test_withhold_signal = (flags & MLA_DECODE_TEST_WITHHOLD_SIGNAL) ? 1 : 0;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (tma_kv && R % 128 == 0 && !(flags & MLA_DECODE_SINGLE_SM)) {
    // query rows in groups of 128: one CTA pair per (partition, group of 128 rows)
    int cap = 0;
    if (int rc = pair_cluster_capacity(&cap)) return rc;
    const int work = num_partitions * static_cast<int>(R / 128);
    e = mla::launch_decode_pair(p, q_map, kv_map, wide, work < cap ? work : cap, s);
    if (e != cudaSuccess) return cuda_fail(e, "mla_decode: pair decode launch");
  } else {
    mla::DecodeVariant v;
    if (layout == MLA_KV_BF16_576) v = tma_kv ? mla::DecodeVariant::kBf16Tma : mla::DecodeVariant::kBf16Gather;
    else if (layout == MLA_KV_FP8_448_UE8M0) v = mla::DecodeVariant::kFp8_448;
    else v = mla::DecodeVariant::kFp8_512;
    const int grid = p.num_work < num_sms ? p.num_work : num_sms;
    e = mla::launch_decode(v, p, q_map, kv_map, grid, s);
    if (e != cudaSuccess) return cuda_fail(e, "mla_decode: decode launch");
  }
  if (total_splits > batch && !(flags & MLA_DECODE_SKIP_COMBINE)) {
    e = mla::launch_combine(p.part_out, p.part_lse, num_splits, batch, static_cast<int>(R), num_heads, sink, p.out,
                            lse, p.part_max, max_logits, s);
    if (e != cudaSuccess) return cuda_fail(e, "mla_decode: combine launch");
  }
  return MLA_OK;
}
}  // namespace

extern "C" {

int mla_decode(const void* q, const void* kv_cache, mla_kv_layout layout, int64_t num_pages, int32_t page_size,
               const int32_t* block_table, int32_t max_pages, const int32_t* cache_seqlens, int32_t batch,
               int32_t q_tokens_per_req, int32_t num_heads, float sm_scale, const float* sink,
               const int32_t* indices, int32_t topk, int32_t causal, const int32_t* sched,
               const int32_t* num_splits, int32_t num_partitions, int32_t total_splits, void* workspace,
               size_t workspace_bytes, void* out, float* lse, uint32_t flags, void* stream) {
  return decode_impl(q, kv_cache, layout, num_pages, page_size, block_table, max_pages, cache_seqlens, batch,
                     q_tokens_per_req, num_heads, sm_scale, sink, indices, nullptr, topk, causal, sched, num_splits,
                     num_partitions, total_splits, workspace, workspace_bytes, out, lse, flags, stream);
}

int mla_decode_runs(const void* q, const void* kv_cache, mla_kv_layout layout, int64_t num_pages, int32_t page_size,
                    const int32_t* runs, int32_t window, int32_t batch, int32_t q_tokens_per_req, int32_t num_heads,
                    float sm_scale, const float* sink, const int32_t* sched, const int32_t* num_splits,
                    int32_t num_partitions, int32_t total_splits, void* workspace, size_t workspace_bytes, void* out,
                    float* lse, uint32_t flags, void* stream) {
  if (runs == nullptr) return fail(MLA_ERR_INVALID_ARG, "mla_decode_runs: runs is NULL");
  if (reinterpret_cast<uintptr_t>(runs) & 15u)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode_runs: runs must be 16-byte aligned");
  return decode_impl(q, kv_cache, layout, num_pages, page_size, nullptr, 1, nullptr, batch, q_tokens_per_req,
                     num_heads, sm_scale, sink, nullptr, runs, window, 0, sched, num_splits, num_partitions,
                     total_splits, workspace, workspace_bytes, out, lse, flags, stream);
}

int mla_sparse_prefill(const void* q, const void* kv, int32_t s_kv, const int32_t* indices, int32_t topk,
                       int32_t num_tokens, int32_t num_heads, float sm_scale, const int32_t* sched,
                       const int32_t* num_splits, int32_t num_partitions, int32_t total_splits, void* workspace,
                       size_t workspace_bytes, void* out, float* max_logits, float* lse, uint32_t flags,
                       void* stream) {
  if (!indices || !max_logits) return fail(MLA_ERR_INVALID_ARG, "mla_sparse_prefill: NULL pointer argument");
  if (flags & MLA_DECODE_SKIP_COMBINE)
    return fail(MLA_ERR_INVALID_ARG, "mla_sparse_prefill: MLA_DECODE_SKIP_COMBINE is not accepted");
  if (s_kv < 1 || topk < 1 || num_tokens < 1)
    return fail(MLA_ERR_INVALID_ARG, "mla_sparse_prefill: s_kv, topk and num_tokens must be >= 1");
  if (reinterpret_cast<uintptr_t>(max_logits) & 3u)
    return fail(MLA_ERR_INVALID_ARG, "mla_sparse_prefill: max_logits must be 4-byte aligned");
  // kv as 64-row pages of one unpaged run; token t is a request of one query token whose
  // candidates are its index list (positions of the run), every request s_kv rows long
  const int64_t num_pages = (static_cast<int64_t>(s_kv) + 63) / 64;
  return decode_impl(q, kv, MLA_KV_BF16_576, num_pages, 64, nullptr, 1, nullptr, num_tokens, 1, num_heads, sm_scale,
                     nullptr, indices, nullptr, topk, 0, sched, num_splits, num_partitions, total_splits, workspace,
                     workspace_bytes, out, lse, flags & ~static_cast<uint32_t>(MLA_DECODE_TEST_WITHHOLD_SIGNAL), stream,
                     s_kv, max_logits);
}

int mla_swa_plan(const int32_t* kv_indices, const int32_t* topk_lengths, int32_t num_tokens, int32_t topk,
                 int32_t page_size, int32_t kv_run_step, int32_t* runs, void* stream) {
  if (!kv_indices || !runs) return fail(MLA_ERR_INVALID_ARG, "mla_swa_plan: NULL pointer argument");
  if (num_tokens < 1 || topk < 1) return fail(MLA_ERR_INVALID_ARG, "mla_swa_plan: num_tokens and topk must be >= 1");
  if (!pow2(page_size)) return fail(MLA_ERR_INVALID_ARG, "mla_swa_plan: page_size %d not a power of two", page_size);
  if (reinterpret_cast<uintptr_t>(runs) & 15u) return fail(MLA_ERR_INVALID_ARG, "mla_swa_plan: runs must be 16-byte aligned");
  if (kv_run_step != 1 && kv_run_step != -1)
    return fail(MLA_ERR_INVALID_ARG, "mla_swa_plan: kv_run_step must be 1 or -1 (got %d)", kv_run_step);
  cudaError_t e = mla::launch_swa_plan(kv_indices, topk_lengths, num_tokens, topk, page_size, kv_run_step, runs,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_swa_plan: launch");
  return MLA_OK;
}

int mla_combine(const float* part_out, const float* part_lse, const int32_t* num_splits, int32_t batch,
                int32_t rows_per_req, int32_t num_heads, const float* sink, void* out, float* lse, void* stream) {
  if (!part_out || !part_lse || !num_splits || !out || !lse) return fail(MLA_ERR_INVALID_ARG, "mla_combine: NULL pointer");
  if (batch < 1 || rows_per_req < 1 || num_heads < 1 || rows_per_req % num_heads != 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_combine: bad sizes batch=%d rows=%d heads=%d", batch, rows_per_req, num_heads);
  if (!aligned16(part_out) || (reinterpret_cast<uintptr_t>(out) & 7u) != 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_combine: part_out must be 16-byte and out 8-byte aligned");
  cudaError_t e = mla::launch_combine(part_out, part_lse, num_splits, batch, rows_per_req, num_heads, sink,
                                      static_cast<uint16_t*>(out), lse, nullptr, nullptr,
                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_combine: launch");
  return MLA_OK;
}

int mla_kv_write(const void* rows, const int32_t* slots, int32_t n, void* kv_cache, mla_kv_layout layout,
                 int64_t num_pages, int32_t page_size, uint32_t* status, void* stream) {
  if (n < 0) return fail(MLA_ERR_INVALID_ARG, "mla_kv_write: n < 0");
  if (n == 0) return MLA_OK;
  if (!rows || !slots || !kv_cache) return fail(MLA_ERR_INVALID_ARG, "mla_kv_write: NULL pointer");
  int64_t rb, pb;
  int dqk;
  if (layout_geometry(layout, page_size, &rb, &pb, &dqk) != 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_kv_write: unknown layout %d", static_cast<int>(layout));
  if (!pow2(page_size)) return fail(MLA_ERR_INVALID_ARG, "mla_kv_write: page_size %d not a power of two", page_size);
  if (num_pages < 1) return fail(MLA_ERR_INVALID_ARG, "mla_kv_write: num_pages < 1");
  if (!aligned16(rows) || !aligned16(kv_cache))
    return fail(MLA_ERR_INVALID_ARG, "mla_kv_write: rows and kv_cache must be 16-byte aligned");
  cudaError_t e = mla::launch_kv_write(static_cast<const uint16_t*>(rows), slots, n, static_cast<uint8_t*>(kv_cache),
                                       static_cast<int>(layout), num_pages, page_size, pb, status,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_kv_write: launch");
  return MLA_OK;
}

int mla_combine_inv_rope(const float* part_out, const float* part_lse, const int32_t* num_splits, int32_t batch,
                         int32_t q_tokens_per_req, int32_t num_heads, const float* sink, const int32_t* positions,
                         const float* freqs, int32_t max_pos, int32_t rope0, void* out, float* lse, void* stream) {
  if (!num_splits || !positions || !freqs || !out || !lse)
    return fail(MLA_ERR_INVALID_ARG, "mla_combine_inv_rope: NULL pointer argument");
  if (batch < 1 || q_tokens_per_req < 1 || num_heads < 1 || max_pos < 1)
    return fail(MLA_ERR_INVALID_ARG, "mla_combine_inv_rope: batch, q_tokens_per_req, num_heads, max_pos must be >= 1");
  if (static_cast<int64_t>(batch) * q_tokens_per_req * num_heads >= (1ll << 31))
    return fail(MLA_ERR_UNSUPPORTED, "mla_combine_inv_rope: too many query rows");
  if (rope0 < 0 || rope0 % 4 != 0 || rope0 + 64 > 512)
    return fail(MLA_ERR_INVALID_ARG, "mla_combine_inv_rope: rope0 = %d must be a multiple of 4 with rope0 + 64 <= 512",
                rope0);
  if ((part_out == nullptr) != (part_lse == nullptr))
    return fail(MLA_ERR_INVALID_ARG, "mla_combine_inv_rope: part_out and part_lse must be given together");
  if (!aligned16(out) || (part_out && !aligned16(part_out)) || (reinterpret_cast<uintptr_t>(freqs) & 3u))
    return fail(MLA_ERR_INVALID_ARG, "mla_combine_inv_rope: out and part_out must be 16-byte aligned");
  cudaError_t e = mla::launch_combine_inv_rope(part_out, part_lse, num_splits, batch, q_tokens_per_req, num_heads,
                                               sink, positions, freqs, max_pos, rope0, static_cast<uint16_t*>(out), lse,
                                               static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_combine_inv_rope: launch");
  return MLA_OK;
}

int mla_combine_v_up(const float* part_out, const float* part_lse, const int32_t* num_splits, int32_t batch,
                     int32_t q_tokens_per_req, int32_t num_heads, const float* sink, const void* w_uv, void* out,
                     float* lse, void* o_v, uint32_t* status, void* stream) {
  if (!num_splits || !w_uv || !out || !lse || !o_v)
    return fail(MLA_ERR_INVALID_ARG, "mla_combine_v_up: NULL pointer argument");
  if (batch < 1 || q_tokens_per_req < 1 || num_heads < 1)
    return fail(MLA_ERR_INVALID_ARG, "mla_combine_v_up: batch, q_tokens_per_req and num_heads must be >= 1");
  if (static_cast<int64_t>(batch) * q_tokens_per_req * num_heads >= (1ll << 31))
    return fail(MLA_ERR_UNSUPPORTED, "mla_combine_v_up: too many query rows");
  if ((part_out == nullptr) != (part_lse == nullptr))
    return fail(MLA_ERR_INVALID_ARG, "mla_combine_v_up: part_out and part_lse must be given together");
  if (!aligned16(w_uv) || !aligned16(out) || !aligned16(o_v) || (part_out && !aligned16(part_out)))
    return fail(MLA_ERR_INVALID_ARG, "mla_combine_v_up: w_uv, out, o_v and part_out must be 16-byte aligned");
  int enc_err = 0;
  EncodeTiledFn encode = get_encode_fn(&enc_err);
  if (enc_err) return fail(MLA_ERR_CUDA, "mla_combine_v_up: cuTensorMapEncodeTiled is unavailable");
  CUtensorMap w_map;
  std::memset(&w_map, 0, sizeof w_map);
  {
    const cuuint64_t dims[3] = {128, 512, static_cast<cuuint64_t>(num_heads)};
    const cuuint64_t strides[2] = {128 * 2, 512 * 128 * 2};
    const cuuint32_t box[3] = {64, 64, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    CUresult r = encode(&w_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w_uv), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MLA_ERR_CUDA, "mla_combine_v_up: encoding the W_UV tensor map failed (%d)", (int)r);
  }
  cudaError_t e = mla::launch_combine_v_up(part_out, part_lse, num_splits, batch, q_tokens_per_req, num_heads, sink,
                                           static_cast<uint16_t*>(out), lse, static_cast<uint16_t*>(o_v), status,
                                           w_map, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_combine_v_up: launch");
  return MLA_OK;
}

int mla_kv_write_norm_rope(const void* raw, const int32_t* slots, const int32_t* positions, const void* norm_weight,
                           float eps, const float* freqs, int32_t max_pos, int32_t n, void* kv_cache,
                           mla_kv_layout layout, int64_t num_pages, int32_t page_size, uint32_t* status,
                           void* stream) {
  if (n < 0) return fail(MLA_ERR_INVALID_ARG, "mla_kv_write_norm_rope: n < 0");
  if (n == 0) return MLA_OK;
  if (!raw || !slots || !positions || !norm_weight || !freqs || !kv_cache)
    return fail(MLA_ERR_INVALID_ARG, "mla_kv_write_norm_rope: NULL pointer");
  int64_t rb, pb;
  int dqk;
  if (layout_geometry(layout, page_size, &rb, &pb, &dqk) != 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_kv_write_norm_rope: unknown layout %d", static_cast<int>(layout));
  if (!pow2(page_size))
    return fail(MLA_ERR_INVALID_ARG, "mla_kv_write_norm_rope: page_size %d not a power of two", page_size);
  if (num_pages < 1) return fail(MLA_ERR_INVALID_ARG, "mla_kv_write_norm_rope: num_pages < 1");
  if (max_pos < 1) return fail(MLA_ERR_INVALID_ARG, "mla_kv_write_norm_rope: max_pos < 1");
  if (!(eps >= 0.f) || !(eps < 1e30f))
    return fail(MLA_ERR_INVALID_ARG, "mla_kv_write_norm_rope: eps must be a finite number >= 0");
  if (!aligned16(raw) || !aligned16(kv_cache) || !aligned16(norm_weight) ||
      (reinterpret_cast<uintptr_t>(freqs) & 3u) != 0)
    return fail(MLA_ERR_INVALID_ARG,
                "mla_kv_write_norm_rope: raw, norm_weight and kv_cache must be 16-byte aligned, freqs 4-byte aligned");
  cudaError_t e = mla::launch_kv_write_norm_rope(
      static_cast<const uint16_t*>(raw), slots, positions, static_cast<const uint16_t*>(norm_weight), eps, freqs,
      max_pos, n, static_cast<uint8_t*>(kv_cache), static_cast<int>(layout), num_pages, page_size, pb, status,
      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_kv_write_norm_rope: launch");
  return MLA_OK;
}

int mla_kv_gather(const void* kv_cache, mla_kv_layout layout, int64_t num_pages, int32_t page_size,
                  const int32_t* block_table_row, int32_t max_pages, int32_t length, float* out, void* stream) {
  if (length < 0) return fail(MLA_ERR_INVALID_ARG, "mla_kv_gather: length < 0");
  if (length == 0) return MLA_OK;
  if (!kv_cache || !block_table_row || !out) return fail(MLA_ERR_INVALID_ARG, "mla_kv_gather: NULL pointer");
  int64_t rb, pb;
  int dqk;
  if (layout_geometry(layout, page_size, &rb, &pb, &dqk) != 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_kv_gather: unknown layout %d", static_cast<int>(layout));
  if (!pow2(page_size) || max_pages < 1 || num_pages < 1)
    return fail(MLA_ERR_INVALID_ARG, "mla_kv_gather: bad page_size / max_pages / num_pages");
  cudaError_t e = mla::launch_kv_gather(static_cast<const uint8_t*>(kv_cache), static_cast<int>(layout), num_pages,
                                        page_size, pb, block_table_row, max_pages, length, out,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_kv_gather: launch");
  return MLA_OK;
}

int mla_workspace_init(void* workspace, void* stream) {
  if (!workspace) return fail(MLA_ERR_INVALID_ARG, "mla_workspace_init: NULL workspace");
  cudaError_t e = cudaMemsetAsync(workspace, 0, MLA_WORKSPACE_HEADER, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_workspace_init");
  return MLA_OK;
}

int mla_read_status(void* workspace, uint32_t* status, int32_t reset, void* stream) {
  if (!workspace || !status) return fail(MLA_ERR_INVALID_ARG, "mla_read_status: NULL argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "mla_read_status: stream synchronize");
  e = cudaMemcpy(status, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "mla_read_status: copy");
  if (reset) {
    e = cudaMemset(workspace, 0, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "mla_read_status: reset");
  }
  if (*status != 0)
    return fail(MLA_ERR_DEVICE_CHECK, "device status 0x%x:%s%s", *status,
                (*status & MLA_STATUS_WAIT_TIMEOUT) ? " pipeline wait timed out;" : "",
                (*status & MLA_STATUS_BAD_PAGE) ? " block_table entry out of range;" : "");
  return MLA_OK;
}

}  // extern "C"
