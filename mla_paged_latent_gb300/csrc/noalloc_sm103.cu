// mla_decode_static_workspace: mla_decode for callers that cannot allocate
// device memory.
//
// mla_decode needs a caller-provided workspace (a status word plus the split
// partials). Some callers cannot provide one: a host program that has handed
// the whole device memory budget to its own pool and forbids extensions from
// calling cudaMalloc, a latency-critical loop that must not pay for an
// allocation (cudaMalloc may synchronise the device), or a binding from a
// language runtime that has no way to allocate CUDA memory at all. For them
// this file keeps one workspace in a file-scope __device__ array that every GPU
// loading the library holds until the process exits.
//
// The array's name is only a host-side handle: passing it to a kernel from host
// code would hand the kernel a host address. Its device address is obtained
// once per device with cudaGetSymbolAddress, with that device current, on the
// first call made on that device; do that first call before any stream capture.
// All calls share the array, so calls that overlap on the GPU (two streams,
// two host threads) race on it.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "mla_decode.h"
#include "mla_kernels.h"

namespace mla {
int set_last_error(int code, const char* msg);
}

namespace {

constexpr size_t kStaticWorkspaceBytes = MLA_STATIC_WORKSPACE_BYTES;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_addr[kMaxDevices] = {};

// Device address of g_static_workspace on the current device (looked up once).
int static_workspace_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return mla::set_last_error(MLA_ERR_CUDA, "mla_decode_static_workspace: cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices)
    return mla::set_last_error(MLA_ERR_UNSUPPORTED, "mla_decode_static_workspace: device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess || p == nullptr) {
      char buf[256];
      snprintf(buf, sizeof buf, "mla_decode_static_workspace: cudaGetSymbolAddress failed: %s",
               cudaGetErrorString(e));
      return mla::set_last_error(MLA_ERR_CUDA, buf);
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" int mla_decode_static_workspace(const void* q, const void* kv_cache, mla_kv_layout layout,
                                           int64_t num_pages, int32_t page_size, const int32_t* block_table,
                                           int32_t max_pages, const int32_t* cache_seqlens, int32_t batch,
                                           int32_t q_tokens_per_req, int32_t num_heads, float sm_scale,
                                           const float* sink, const int32_t* indices, int32_t topk, int32_t causal,
                                           const int32_t* sched, const int32_t* num_splits, int32_t num_partitions,
                                           int32_t total_splits, void* out, float* lse, uint32_t* status_out,
                                           void* stream) {
  if (total_splits < 0 || q_tokens_per_req < 1 || num_heads < 1)
    return mla::set_last_error(MLA_ERR_INVALID_ARG, "mla_decode_static_workspace: bad sizes");
  // the size mla_decode checks its caller's workspace against
  const size_t need =
      mla::workspace_bytes_for(total_splits, static_cast<int64_t>(q_tokens_per_req) * static_cast<int64_t>(num_heads));
  if (need > kStaticWorkspaceBytes) {
    char buf[256];
    snprintf(buf, sizeof buf,
             "mla_decode_static_workspace: this plan needs %zu workspace bytes, more than the %zu-byte static "
             "workspace; use mla_decode with a caller-allocated workspace",
             need, kStaticWorkspaceBytes);
    return mla::set_last_error(MLA_ERR_WORKSPACE_TOO_SMALL, buf);
  }
  void* ws = nullptr;
  if (int rc = static_workspace_address(&ws)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the status word must start at zero; the partials are fully rewritten by each call
  cudaError_t e = cudaMemsetAsync(ws, 0, MLA_WORKSPACE_HEADER, s);
  if (e != cudaSuccess)
    return mla::set_last_error(MLA_ERR_CUDA, "mla_decode_static_workspace: clearing the status word failed");
  int rc = mla_decode(q, kv_cache, layout, num_pages, page_size, block_table, max_pages, cache_seqlens, batch,
                      q_tokens_per_req, num_heads, sm_scale, sink, indices, topk, causal, sched, num_splits,
                      num_partitions, total_splits, ws, kStaticWorkspaceBytes, out, lse, 0u, stream);
  if (rc != MLA_OK) return rc;
  if (status_out != nullptr) {
    e = cudaMemcpyAsync(status_out, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess)
      return mla::set_last_error(MLA_ERR_CUDA, "mla_decode_static_workspace: copying the status word failed");
  }
  return MLA_OK;
}
