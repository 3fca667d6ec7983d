// pkv_paged_attention_static_workspace: attention for callers that cannot
// allocate device memory (contract in include/pagedkv.h).
//
// The scratch that pkv_paged_attention takes from the caller (plan counters,
// per-request prefix sums, split-KV partials) lives here in one file-scope
// device array instead. Host code cannot use the array's name as a device
// address, so the first call on each device looks the address up with
// cudaGetSymbolAddress and keeps it; every call then runs the normal
// attention path on that memory. Nothing in this file allocates.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/pagedkv.h"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[PKV_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_static_workspace on the current device.
int32_t static_workspace_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess || !p) return PKV_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" int32_t pkv_paged_attention_static_workspace(
    void* out, const void* q, int64_t q_row_stride, const void* kv_cache,
    const int32_t* block_table, int32_t max_blocks_per_req, const int32_t* seq_lens,
    const int32_t* query_start_loc, const int32_t* num_computed_tokens, int32_t num_reqs,
    int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len, int32_t num_q_heads,
    float scale, pkv_cache_layout layout, const pkv_attention_options* options, void* stream) {
  const int64_t need = pkv_attention_workspace_size(num_reqs, num_q_heads, layout, options);
  if (need < 0) return static_cast<int32_t>(need);
  if (need > static_cast<int64_t>(PKV_STATIC_WORKSPACE_BYTES)) return PKV_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  const int32_t st = static_workspace_address(&ws);
  if (st != PKV_OK) return st;
  return pkv_paged_attention(out, q, q_row_stride, kv_cache, block_table, max_blocks_per_req,
                             seq_lens, query_start_loc, num_computed_tokens, num_reqs, num_tokens,
                             max_query_len, max_seq_len, num_q_heads, scale, layout, ws,
                             PKV_STATIC_WORKSPACE_BYTES, options, stream);
}
