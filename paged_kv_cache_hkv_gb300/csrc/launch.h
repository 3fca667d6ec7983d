// Internal launch interface between the C ABI shim and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace pkv {

// Header words at the start of the attention workspace (written by the plan
// kernel every call).
enum : int {
  kHdrDecodeBlocks = 0,  // sum of ceil(L/16) (16-key chunks) over decode requests
  kHdrPrefillReqs = 1,   // requests with query_len > 1
  kHdrPrefillItems = 2,  // prefill work items (tile x kv head)
  kHdrPrefillNext = 3,   // work counter of the persistent prefill kernel
  kHdrWords = 64,
};

// Device pointers into the attention workspace.
struct AttnWorkspace {
  uint32_t* hdr;         // [kHdrWords]
  int32_t* dec_prefix;   // [R + 1]: decode 16-key chunks before request r
  int32_t* pf_req;       // [R + 1]: request id of the k-th prefill request (-1: the
                         // shared-prefix items, listed after every prefill request)
  int32_t* pf_prefix;    // [R + 2]: prefill items before the k-th prefill request
  float2* part_ml;       // [slots][GW]: (running max in log2 units, sum)
  float* part_o;         // [slots][GW][D]: unnormalised partial outputs
  int* bound;            // [C]: request holding the first position of each decode CTA range
  // shared-prefix items (only when the call has a shared-prefix hint)
  int32_t* casc_use;     // [shared_num]: 1 if the request takes its prefix from the shared items
  float2* casc_ml;       // [pieces][shared_num][Hq]: (max in log2 units, sum) of each piece
  float* casc_o;         // [pieces][shared_num][Hq][D]: unnormalised output of each piece
};

struct AttnArgs {
  uint16_t* out;  // bf16 [T][Hq][D]
  const uint16_t* q;  // bf16 rows of q_stride elements
  long long q_stride;  // elements between token rows of q
  const void* kv_cache;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* seq_lens;
  const int32_t* qsl;
  const int32_t* num_computed;
  int num_reqs, num_tokens, max_query_len, max_seq_len;
  int num_q_heads, num_kv_heads, head_dim, num_blocks;
  int block_shift;  // log2 of the tokens per cache block (3, 4 or 5)
  float scale;
  // Shared-prefix hint: requests shared_first .. + shared_num - 1 share their
  // first shared_len tokens (0 = off). Their prefix is attended by shared
  // items of the prefill kernel: q tiles of their rows x kv heads x key
  // pieces of shared_tpp 128-key tiles (shared_pieces of them).
  int shared_len, shared_first, shared_num;
  int shared_pieces, shared_tpp;
  long long decode_splits;  // CTAs along the decode stream (C)
};

// Key pieces of the shared-prefix items: enough items to fill the device
// (q tiles x kv heads x pieces ~ num_sms), each piece at least two 128-key
// tiles so that both softmax warpgroups of a CTA take part.
// At most this many pieces: each adds one partial per row that the combine
// kernel reads, and pieces of a few tiles already fill the device.
constexpr int kMaxSharedPieces = 8;

inline void shared_split(int shared_num, int group, int num_kv_heads, int shared_len,
                         int num_sms, int* pieces, int* tpp) {
  const int qt = (shared_num + (128 / group) - 1) / (128 / group);
  const int tiles = (shared_len + 127) / 128;
  const int base = qt * num_kv_heads;
  int want = base > 0 ? num_sms / base : 1;
  if (want < 1) want = 1;
  int t = (tiles + want - 1) / want;
  if (t < 2) t = 2;
  if (t < (tiles + kMaxSharedPieces - 1) / kMaxSharedPieces)
    t = (tiles + kMaxSharedPieces - 1) / kMaxSharedPieces;
  if (t > tiles) t = tiles;
  *tpp = t;
  *pieces = (tiles + t - 1) / t;
}

// Raise a kernel's dynamic shared memory limit once per device: `done` is a
// per-kernel bit mask of devices already set up, so later launches (also
// those recorded into a CUDA graph) make no attribute call.
template <typename Kernel>
inline cudaError_t smem_attr_once(Kernel kern, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Launch with programmatic stream serialization: the kernel may begin while
// the previous kernel in the stream is still running; it calls pdl_wait()
// before reading that kernel's results.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
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

// Heads handled together by one decode warp, and head groups per kv head.
inline int decode_heads_per_warp(int group) { return group < 4 ? group : 4; }

// slots of split-KV partials the decode kernel may write: (request + CTA) *
// virtual heads + virtual head
inline long long decode_partial_slots(int num_reqs, int virt_heads, long long splits) {
  return (static_cast<long long>(num_reqs) + splits) * virt_heads;
}

// Virtual heads (consumer warps) and kv heads of one decode CTA for a shape.
void decode_slab(int num_kv_heads, int group, int* slab_vh, int* slab_kh);

cudaError_t launch_slot_mapping(int64_t* slots, const int32_t* block_table, int max_blocks,
                                const int32_t* qsl, const int32_t* num_computed, int num_reqs,
                                int num_tokens, int num_blocks, int block_size,
                                cudaStream_t stream);

struct WriteRowsArgs;
WriteRowsArgs write_rows_args(void* pool, const void* key, const void* value,
                              long long key_stride, long long value_stride, int64_t* slots,
                              const int32_t* block_table, int max_blocks, const int32_t* qsl,
                              const int32_t* num_computed, int num_reqs, int num_tokens,
                              int num_blocks, int block_size, int num_kv_heads, int head_dim);
cudaError_t launch_mapped_write(const WriteRowsArgs& w, cudaStream_t stream);
cudaError_t launch_kv_write(void* pool, const void* key, const void* value, long long key_stride,
                            long long value_stride, const int64_t* slots, int num_tokens,
                            int num_blocks, int block_size, int num_kv_heads, int head_dim,
                            int num_sms, cudaStream_t stream);

cudaError_t launch_copy_blocks(void* dst, int dst_num_blocks, const void* src, int src_num_blocks,
                               const int32_t* pairs, int num_pairs, int block_size,
                               int num_kv_heads, int head_dim, int num_sms, cudaStream_t stream);

// The plan kernel; with `write`, one launch that also maps the slots of the
// step's new tokens and writes their K and V rows (the write's CTAs next to
// the plan's).
cudaError_t launch_plan(const AttnArgs& a, const AttnWorkspace& ws, cudaStream_t stream,
                        const WriteRowsArgs* write = nullptr);

// Decode splits (CTAs along the decode stream) in one full wave of the device.
cudaError_t decode_full_wave_splits(int head_dim, int num_kv_heads, int group, int block_shift,
                                    int num_sms, long long* splits);

// trace: NULL or the caller's event array; event [3] is recorded between the
// decode and the combine kernel.
cudaError_t launch_decode(const AttnArgs& a, const AttnWorkspace& ws, const CUtensorMap& kv_map,
                          long long splits, int num_sms, cudaStream_t stream, void** trace);

cudaError_t launch_prefill(const AttnArgs& a, const AttnWorkspace& ws, const CUtensorMap& kv_map,
                           const CUtensorMap& q_map, int num_sms, cudaStream_t stream);

cudaError_t read_errors_kvwrite(uint32_t* out, bool clear);
cudaError_t read_errors_decode(uint32_t* out, bool clear);
cudaError_t read_errors_prefill(uint32_t* out, bool clear);
cudaError_t read_errors_plan(uint32_t* out, bool clear);

}  // namespace pkv
