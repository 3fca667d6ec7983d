// C ABI of libpagedkv.so: argument checks, launch planning, tensor maps.
// Declarations and the contract of every entry point: include/pagedkv.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>

#include "../../include/pagedkv.h"
#include "launch.h"
#include "write_rows.cuh"

namespace {

thread_local char g_cuda_error[256] = "";

int32_t cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(g_cuda_error, sizeof(g_cuda_error), "%s: %s", where, cudaGetErrorString(e));
  return PKV_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DeviceInfo {
  int num_sms = 0;
  bool ok = false;
  std::map<long long, long long> full_wave_splits;  // by (D, group, B, kv heads)
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_init[kMaxDevices] = {};

int32_t device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!g_dev_init[dev]) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    d.ok = (major == 10 && minor == 3);
    g_dev_init[dev] = true;
  }
  if (!d.ok) return PKV_ERR_DEVICE;
  *out = &d;
  return PKV_OK;
}

// cuTensorMapEncodeTiled, reached through the runtime so that the library
// does not link the driver library directly.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int32_t encode_fn(EncodeTiledFn* fn) {
  static EncodeTiledFn cached = nullptr;
  static std::once_flag once;
  static cudaError_t status = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                              cudaEnableDefault, &q);
    if (status == cudaSuccess && q == cudaDriverEntryPointSuccess)
      cached = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!cached) return cuda_fail(status == cudaSuccess ? cudaErrorSymbolNotFound : status,
                                "cuTensorMapEncodeTiled entry point");
  *fn = cached;
  return PKV_OK;
}

// bf16 map of `rank` dims (dims[0] contiguous); strides[i] is the byte
// stride of dims[i + 1].
int32_t make_map_n(CUtensorMap* map, const void* base, uint32_t rank, const cuuint64_t* dims,
                   const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn;
  int32_t st = encode_fn(&fn);
  if (st != PKV_OK) return st;
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_cuda_error, sizeof(g_cuda_error), "cuTensorMapEncodeTiled failed (%d)",
                  static_cast<int>(r));
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

// 3-D bf16 map: dims {d0, d1, d2} (d0 contiguous), byte strides of dims 1, 2.
int32_t make_map(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2,
                 CUtensorMapSwizzle swz) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1, stride2};
  const cuuint32_t box[3] = {b0, b1, b2};
  return make_map_n(map, base, 3, dims, strides, box, swz);
}

bool block_size_ok(int32_t b) { return b == 8 || b == 16 || b == 32; }

int block_shift_of(int32_t b) { return b == 8 ? 3 : (b == 16 ? 4 : 5); }

int32_t check_layout(const pkv_cache_layout& l) {
  if (l.num_blocks < 1 || l.num_kv_heads < 1 || l.head_dim < 1 || l.block_size < 1)
    return PKV_ERR_BAD_SHAPE;
  if (!block_size_ok(l.block_size)) return PKV_ERR_UNSUPPORTED;
  if (l.head_dim != 64 && l.head_dim != 128) return PKV_ERR_UNSUPPORTED;
  // pool rows (block * 2 + k|v) * B + offset are 32-bit TMA coordinates
  if (static_cast<long long>(l.num_blocks) * 2 * l.block_size >= (1ll << 31))
    return PKV_ERR_BAD_SHAPE;
  return PKV_OK;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// The shared-prefix hint of the options, checked (all zero = off).
struct SharedHint {
  int len = 0, first = 0, num = 0, pieces = 0, tpp = 0;
};

int32_t shared_hint(const pkv_attention_options* opt, const pkv_cache_layout& l, int group,
                    int num_reqs, int num_sms, SharedHint* h) {
  *h = SharedHint();
  if (!opt) return PKV_OK;
  const int len = opt->shared_prefix_len, first = opt->shared_first_req,
            num = opt->shared_num_reqs;
  if (len == 0 && first == 0 && num == 0) return PKV_OK;
  if (len <= 0 || first < 0 || num < 1) return PKV_ERR_BAD_SHAPE;
  if (len % 16 || len % l.block_size) return PKV_ERR_BAD_SHAPE;
  if (static_cast<long long>(first) + num > num_reqs) return PKV_ERR_BAD_SHAPE;
  h->len = len;
  h->first = first;
  h->num = num;
  pkv::shared_split(num, group, l.num_kv_heads, len, num_sms, &h->pieces, &h->tpp);
  return PKV_OK;
}

struct WsLayout {
  size_t hdr, dec_prefix, pf_req, pf_prefix, part_ml, part_o, bound, casc_use, casc_ml, casc_o,
      total;
};

WsLayout ws_layout(int num_reqs, int virt_heads, int gw, int head_dim, long long splits,
                   const SharedHint& sh, int num_q_heads) {
  WsLayout w;
  const long long slots = pkv::decode_partial_slots(num_reqs, virt_heads, splits);
  size_t off = 0;
  w.hdr = off;
  off += round256(pkv::kHdrWords * sizeof(uint32_t));
  w.dec_prefix = off;
  off += round256((num_reqs + 1) * sizeof(int32_t));
  w.pf_req = off;
  off += round256((num_reqs + 1) * sizeof(int32_t));
  w.pf_prefix = off;
  off += round256((num_reqs + 2) * sizeof(int32_t));
  w.part_ml = off;
  off += round256(static_cast<size_t>(slots) * gw * sizeof(float2));
  w.part_o = off;
  off += round256(static_cast<size_t>(slots) * gw * head_dim * sizeof(float));
  w.bound = off;
  off += round256(static_cast<size_t>(splits) * sizeof(int));
  const size_t shared_rows = static_cast<size_t>(sh.pieces) * sh.num * num_q_heads;
  w.casc_use = off;
  off += round256(static_cast<size_t>(sh.num) * sizeof(int32_t));
  w.casc_ml = off;
  off += round256(shared_rows * sizeof(float2));
  w.casc_o = off;
  off += round256(shared_rows * head_dim * sizeof(float));
  w.total = off;
  return w;
}

// Ranges (CTAs) the decode stream is split into: the caller's choice, else
// one full wave of the device for the shape (cached per device).
int32_t decode_splits_for(DeviceInfo* d, int head_dim, int num_kv_heads, int group,
                          int block_size, const pkv_attention_options* opt, long long* splits) {
  if (opt) {
    for (int i = 0; i < 4; ++i)
      if (opt->reserved[i] != 0) return PKV_ERR_BAD_SHAPE;
    if (opt->decode_splits < 0) return PKV_ERR_BAD_SHAPE;
    if (opt->decode_splits > 0) {
      *splits = opt->decode_splits;
      return PKV_OK;
    }
  }
  const int sh = block_shift_of(block_size);
  const long long key = ((static_cast<long long>(head_dim) * 16 + group) * 8 + sh) * 65536 +
                        num_kv_heads;
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = d->full_wave_splits.find(key);
  if (it == d->full_wave_splits.end()) {
    long long c = 0;
    cudaError_t e =
        pkv::decode_full_wave_splits(head_dim, num_kv_heads, group, sh, d->num_sms, &c);
    if (e != cudaSuccess) return cuda_fail(e, "decode occupancy");
    it = d->full_wave_splits.emplace(key, c).first;
  }
  *splits = it->second;
  return PKV_OK;
}

int32_t check_group(int num_q_heads, int num_kv_heads) {
  if (num_q_heads < 1 || num_q_heads % num_kv_heads) return PKV_ERR_BAD_SHAPE;
  const int g = num_q_heads / num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

}  // namespace

extern "C" {

int32_t pkv_abi_version(void) { return PKV_ABI_VERSION; }

const char* pkv_status_string(int32_t status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_NULL_POINTER: return "a required pointer is NULL";
    case PKV_ERR_BAD_SHAPE: return "a size or count is out of range";
    case PKV_ERR_UNSUPPORTED: return "unsupported block size, head_dim or head grouping";
    case PKV_ERR_MISALIGNED: return "pointer or row stride not 16-byte aligned";
    case PKV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case PKV_ERR_CUDA: return "CUDA call failed (see pkv_last_cuda_error)";
    case PKV_ERR_DEVICE: return "current device is not an sm_103 GPU";
    case PKV_ERR_SCRATCH_LIMIT:
      return "call needs more scratch than the built-in static workspace holds";
    default: return "unknown status";
  }
}

const char* pkv_last_cuda_error(void) { return g_cuda_error; }

int32_t pkv_slot_mapping(int64_t* slot_mapping, const int32_t* block_table,
                         int32_t max_blocks_per_req, const int32_t* query_start_loc,
                         const int32_t* num_computed_tokens, int32_t num_reqs,
                         int32_t num_tokens, int32_t num_blocks, int32_t block_size,
                         void* stream) {
  if (num_tokens < 0 || num_reqs < 0 || max_blocks_per_req < 0 || num_blocks < 1)
    return PKV_ERR_BAD_SHAPE;
  if (block_size < 1) return PKV_ERR_BAD_SHAPE;
  if (!block_size_ok(block_size)) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!slot_mapping || !query_start_loc) return PKV_ERR_NULL_POINTER;
  if (num_reqs > 0 && (!block_table || !num_computed_tokens)) return PKV_ERR_NULL_POINTER;
  DeviceInfo* d;
  int32_t st = device_info(&d);
  if (st != PKV_OK) return st;
  cudaError_t e = pkv::launch_slot_mapping(slot_mapping, block_table, max_blocks_per_req,
                                           query_start_loc, num_computed_tokens, num_reqs,
                                           num_tokens, num_blocks, block_size,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "slot_mapping launch");
}

int32_t pkv_paged_kv_write(void* kv_cache, const void* key, const void* value,
                           int64_t key_row_stride, int64_t value_row_stride,
                           const int64_t* slot_mapping, int32_t num_tokens,
                           pkv_cache_layout layout, void* stream) {
  int32_t st = check_layout(layout);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_BAD_SHAPE;
  const int64_t row = static_cast<int64_t>(layout.num_kv_heads) * layout.head_dim;
  if (key_row_stride == 0) key_row_stride = row;
  if (value_row_stride == 0) value_row_stride = row;
  if (key_row_stride < row || value_row_stride < row) return PKV_ERR_BAD_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!kv_cache || !key || !value || !slot_mapping) return PKV_ERR_NULL_POINTER;
  if (!aligned16(kv_cache) || !aligned16(key) || !aligned16(value) || (key_row_stride % 8) ||
      (value_row_stride % 8))
    return PKV_ERR_MISALIGNED;
  DeviceInfo* d;
  st = device_info(&d);
  if (st != PKV_OK) return st;
  cudaError_t e = pkv::launch_kv_write(kv_cache, key, value, key_row_stride, value_row_stride,
                                       slot_mapping, num_tokens, layout.num_blocks,
                                       layout.block_size, layout.num_kv_heads, layout.head_dim,
                                       d->num_sms,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "kv_write launch");
}

int32_t pkv_slot_mapping_and_write(void* kv_cache, const void* key, const void* value,
                                   int64_t key_row_stride, int64_t value_row_stride,
                                   int64_t* slot_mapping, const int32_t* block_table,
                                   int32_t max_blocks_per_req, const int32_t* query_start_loc,
                                   const int32_t* num_computed_tokens, int32_t num_reqs,
                                   int32_t num_tokens, pkv_cache_layout layout, void* stream) {
  int32_t st = check_layout(layout);
  if (st != PKV_OK) return st;
  if (num_tokens < 0 || num_reqs < 0 || max_blocks_per_req < 0) return PKV_ERR_BAD_SHAPE;
  const int64_t row = static_cast<int64_t>(layout.num_kv_heads) * layout.head_dim;
  if (key_row_stride == 0) key_row_stride = row;
  if (value_row_stride == 0) value_row_stride = row;
  if (key_row_stride < row || value_row_stride < row) return PKV_ERR_BAD_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!kv_cache || !key || !value || !query_start_loc) return PKV_ERR_NULL_POINTER;
  if (num_reqs > 0 && (!block_table || !num_computed_tokens)) return PKV_ERR_NULL_POINTER;
  if (!aligned16(kv_cache) || !aligned16(key) || !aligned16(value) || (key_row_stride % 8) ||
      (value_row_stride % 8))
    return PKV_ERR_MISALIGNED;
  DeviceInfo* d;
  st = device_info(&d);
  if (st != PKV_OK) return st;
  const pkv::WriteRowsArgs w = pkv::write_rows_args(
      kv_cache, key, value, key_row_stride, value_row_stride, slot_mapping, block_table,
      max_blocks_per_req, query_start_loc, num_computed_tokens, num_reqs, num_tokens,
      layout.num_blocks, layout.block_size, layout.num_kv_heads, layout.head_dim);
  cudaError_t e = pkv::launch_mapped_write(w, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "slot mapping and write launch");
}

int32_t pkv_copy_blocks(void* dst_pool, int32_t dst_num_blocks, const void* src_pool,
                        int32_t src_num_blocks, const int32_t* block_pairs, int32_t num_pairs,
                        pkv_cache_layout layout, void* stream) {
  pkv_cache_layout l = layout;
  l.num_blocks = dst_num_blocks > 0 ? dst_num_blocks : 1;
  int32_t st = check_layout(l);
  if (st != PKV_OK) return st;
  if (dst_num_blocks < 1 || src_num_blocks < 1 || num_pairs < 0) return PKV_ERR_BAD_SHAPE;
  if (static_cast<long long>(src_num_blocks) * 2 * layout.block_size >= (1ll << 31))
    return PKV_ERR_BAD_SHAPE;
  if (num_pairs == 0) return PKV_OK;
  if (!dst_pool || !src_pool || !block_pairs) return PKV_ERR_NULL_POINTER;
  if (!aligned16(dst_pool) || !aligned16(src_pool)) return PKV_ERR_MISALIGNED;
  DeviceInfo* d;
  st = device_info(&d);
  if (st != PKV_OK) return st;
  cudaError_t e = pkv::launch_copy_blocks(dst_pool, dst_num_blocks, src_pool, src_num_blocks,
                                          block_pairs, num_pairs, layout.block_size,
                                          layout.num_kv_heads, layout.head_dim, d->num_sms,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "copy_blocks launch");
}

int64_t pkv_attention_workspace_size(int32_t num_reqs, int32_t num_q_heads,
                                     pkv_cache_layout layout,
                                     const pkv_attention_options* options) {
  int32_t st = check_layout(layout);
  if (st != PKV_OK) return st;
  if (num_reqs < 0) return PKV_ERR_BAD_SHAPE;
  st = check_group(num_q_heads, layout.num_kv_heads);
  if (st != PKV_OK) return st;
  DeviceInfo* d;
  st = device_info(&d);
  if (st != PKV_OK) return st;
  const int group = num_q_heads / layout.num_kv_heads;
  long long splits = 0;
  st = decode_splits_for(d, layout.head_dim, layout.num_kv_heads, group, layout.block_size,
                         options, &splits);
  if (st != PKV_OK) return st;
  SharedHint sh;
  st = shared_hint(options, layout, group, num_reqs, d->num_sms, &sh);
  if (st != PKV_OK) return st;
  const int gw = pkv::decode_heads_per_warp(group);
  const int virt = layout.num_kv_heads * (group / gw);
  return static_cast<int64_t>(
      ws_layout(num_reqs, virt, gw, layout.head_dim, splits, sh, num_q_heads).total);
}

// pkv_paged_attention, and with `write` the step's slot mapping and cache
// write in the plan's launch (pkv_paged_attention_with_write).
static int32_t attention_impl(void* out, const void* q, int64_t q_row_stride, const void* kv_cache,
                       const int32_t* block_table, int32_t max_blocks_per_req,
                       const int32_t* seq_lens, const int32_t* query_start_loc,
                       const int32_t* num_computed_tokens, int32_t num_reqs, int32_t num_tokens,
                       int32_t max_query_len, int32_t max_seq_len, int32_t num_q_heads,
                       float scale, pkv_cache_layout layout, void* workspace,
                       size_t workspace_bytes, const pkv_attention_options* options, void* stream,
                       const pkv::WriteRowsArgs* write) {
  int32_t st = check_layout(layout);
  if (st != PKV_OK) return st;
  st = check_group(num_q_heads, layout.num_kv_heads);
  if (st != PKV_OK) return st;
  if (num_reqs < 0 || num_tokens < 0 || max_blocks_per_req < 0 || max_query_len < 0 ||
      max_seq_len < 0)
    return PKV_ERR_BAD_SHAPE;
  if (!(scale > 0.f) || scale > 3.0e38f) return PKV_ERR_BAD_SHAPE;  // positive and finite
  const int64_t row = static_cast<int64_t>(num_q_heads) * layout.head_dim;
  if (q_row_stride == 0) q_row_stride = row;
  if (q_row_stride < row) return PKV_ERR_BAD_SHAPE;
  if (num_reqs == 0 || num_tokens == 0 || max_query_len == 0) {
    // no attention to do; the write (padding rows: slots -1) still runs
    if (!write) return PKV_OK;
    cudaError_t e = pkv::launch_mapped_write(*write, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "slot mapping and write launch");
  }
  if (static_cast<long long>(max_seq_len) >
      static_cast<long long>(max_blocks_per_req) * layout.block_size)
    return PKV_ERR_BAD_SHAPE;
  if (!out || !q || !kv_cache || !block_table || !seq_lens || !query_start_loc ||
      !num_computed_tokens)
    return PKV_ERR_NULL_POINTER;
  if (!aligned16(out) || !aligned16(q) || !aligned16(kv_cache) || (q_row_stride % 8))
    return PKV_ERR_MISALIGNED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PKV_ERR_WORKSPACE;

  DeviceInfo* d;
  st = device_info(&d);
  if (st != PKV_OK) return st;
  const int group = num_q_heads / layout.num_kv_heads;
  long long splits = 0;
  st = decode_splits_for(d, layout.head_dim, layout.num_kv_heads, group, layout.block_size,
                         options, &splits);
  if (st != PKV_OK) return st;
  SharedHint sh;
  st = shared_hint(options, layout, group, num_reqs, d->num_sms, &sh);
  if (st != PKV_OK) return st;
  if (static_cast<long long>(sh.len) >
      static_cast<long long>(max_blocks_per_req) * layout.block_size)
    return PKV_ERR_BAD_SHAPE;
  const int gw = pkv::decode_heads_per_warp(group);
  const int virt = layout.num_kv_heads * (group / gw);
  const WsLayout wl = ws_layout(num_reqs, virt, gw, layout.head_dim, splits, sh, num_q_heads);
  if (workspace_bytes < wl.total) return PKV_ERR_WORKSPACE;
  // The decode stream holds at most num_reqs * ceil(max_seq_len / 16)
  // chunks: with the default split, never use more ranges than that (a small
  // batch then launches a few CTAs instead of a full wave). The workspace
  // sized for the full wave still fits.
  if (!(options && options->decode_splits > 0)) {
    const long long bound =
        static_cast<long long>(num_reqs) * ((static_cast<long long>(max_seq_len) + 15) / 16);
    if (bound < splits) splits = bound > 0 ? bound : 1;
  }

  char* wsb = static_cast<char*>(workspace);
  pkv::AttnWorkspace ws;
  ws.hdr = reinterpret_cast<uint32_t*>(wsb + wl.hdr);
  ws.dec_prefix = reinterpret_cast<int32_t*>(wsb + wl.dec_prefix);
  ws.pf_req = reinterpret_cast<int32_t*>(wsb + wl.pf_req);
  ws.pf_prefix = reinterpret_cast<int32_t*>(wsb + wl.pf_prefix);
  ws.part_ml = reinterpret_cast<float2*>(wsb + wl.part_ml);
  ws.part_o = reinterpret_cast<float*>(wsb + wl.part_o);
  ws.bound = reinterpret_cast<int*>(wsb + wl.bound);
  ws.casc_use = reinterpret_cast<int32_t*>(wsb + wl.casc_use);
  ws.casc_ml = reinterpret_cast<float2*>(wsb + wl.casc_ml);
  ws.casc_o = reinterpret_cast<float*>(wsb + wl.casc_o);

  pkv::AttnArgs a;
  a.out = static_cast<uint16_t*>(out);
  a.q = static_cast<const uint16_t*>(q);
  a.q_stride = q_row_stride;
  a.kv_cache = kv_cache;
  a.block_table = block_table;
  a.max_blocks = max_blocks_per_req;
  a.seq_lens = seq_lens;
  a.qsl = query_start_loc;
  a.num_computed = num_computed_tokens;
  a.num_reqs = num_reqs;
  a.num_tokens = num_tokens;
  a.max_query_len = max_query_len;
  a.max_seq_len = max_seq_len;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = layout.num_kv_heads;
  a.head_dim = layout.head_dim;
  a.num_blocks = layout.num_blocks;
  a.block_shift = block_shift_of(layout.block_size);
  a.scale = scale;
  a.shared_len = sh.len;
  a.shared_first = sh.first;
  a.shared_num = sh.num;
  a.shared_pieces = sh.pieces;
  a.shared_tpp = sh.tpp;

  const int D = layout.head_dim, Hkv = layout.num_kv_heads;
  const uint64_t row_bytes = static_cast<uint64_t>(Hkv) * D * 2;
  // pool as rows of one kv head: {d, kv head, (block*2 + k|v)*B + offset}.
  // A decode copy covers the kv heads of one CTA slab and a block's 32 K and
  // V rows (B = 16), 16 rows (half of the K or V rows of a 32-token block)
  // or the 16 K and V rows of an 8-token block.
  const int B = layout.block_size;
  const uint64_t pool_rows = static_cast<uint64_t>(layout.num_blocks) * 2 * B;
  const uint32_t dec_box = B == 16 ? 32u : 16u;
  int slab_vh = 0, slab_kh = 0;
  pkv::decode_slab(Hkv, group, &slab_vh, &slab_kh);
  CUtensorMap kv_map;
  st = make_map(&kv_map, kv_cache, D, Hkv, pool_rows, static_cast<uint64_t>(D) * 2, row_bytes, D,
                static_cast<uint32_t>(slab_kh), dec_box, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != PKV_OK) return st;

  a.decode_splits = splits;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void** ev = options ? options->trace_events : nullptr;
  auto mark = [&](int i) -> cudaError_t {
    return ev ? cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), s) : cudaSuccess;
  };
  cudaError_t e = mark(0);
  if (e == cudaSuccess) e = pkv::launch_plan(a, ws, s, write);
  if (e == cudaSuccess) e = mark(1);
  if (e != cudaSuccess) return cuda_fail(e, "plan launch");
  if (max_query_len > 1 || sh.num > 0) {
    // pool for the tensor-core path, as {64-element half row, row within an
    // 8-row group, d half, kv head, 8-row group}: one copy takes the K (or V)
    // rows of one block and one kv head, and lands as 128-byte swizzled
    // 8-row atoms ordered (group, d half, row)
    CUtensorMap kv_map_sw, q_map;
    {
      const cuuint64_t dims[5] = {64, 8, static_cast<cuuint64_t>(D / 64),
                                  static_cast<cuuint64_t>(Hkv), pool_rows / 8};
      const cuuint64_t strides[4] = {row_bytes, 128, static_cast<uint64_t>(D) * 2, row_bytes * 8};
      const cuuint32_t box[5] = {64, 8, static_cast<cuuint32_t>(D / 64), 1,
                                 static_cast<cuuint32_t>(B / 8)};
      st = make_map_n(&kv_map_sw, kv_cache, 5, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (st != PKV_OK) return st;
    st = make_map(&q_map, q, D, num_q_heads, num_tokens, static_cast<uint64_t>(D) * 2,
                  static_cast<uint64_t>(q_row_stride) * 2, 64, group, 128 / group,
                  CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != PKV_OK) return st;
    e = pkv::launch_prefill(a, ws, kv_map_sw, q_map, d->num_sms, s);
    if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  }
  e = mark(2);
  if (e == cudaSuccess) e = pkv::launch_decode(a, ws, kv_map, splits, d->num_sms, s, ev);
  if (e == cudaSuccess) e = mark(4);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return PKV_OK;
}

int32_t pkv_paged_attention(void* out, const void* q, int64_t q_row_stride, const void* kv_cache,
                            const int32_t* block_table, int32_t max_blocks_per_req,
                            const int32_t* seq_lens, const int32_t* query_start_loc,
                            const int32_t* num_computed_tokens, int32_t num_reqs,
                            int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
                            int32_t num_q_heads, float scale, pkv_cache_layout layout,
                            void* workspace, size_t workspace_bytes,
                            const pkv_attention_options* options, void* stream) {
  return attention_impl(out, q, q_row_stride, kv_cache, block_table, max_blocks_per_req,
                        seq_lens, query_start_loc, num_computed_tokens, num_reqs, num_tokens,
                        max_query_len, max_seq_len, num_q_heads, scale, layout, workspace,
                        workspace_bytes, options, stream, nullptr);
}

int32_t pkv_paged_attention_with_write(
    void* out, const void* q, int64_t q_row_stride, void* kv_cache, const void* key,
    const void* value, int64_t key_row_stride, int64_t value_row_stride, int64_t* slot_mapping,
    const int32_t* block_table, int32_t max_blocks_per_req, const int32_t* seq_lens,
    const int32_t* query_start_loc, const int32_t* num_computed_tokens, int32_t num_reqs,
    int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len, int32_t num_q_heads,
    float scale, pkv_cache_layout layout, void* workspace, size_t workspace_bytes,
    const pkv_attention_options* options, void* stream) {
  int32_t st = check_layout(layout);
  if (st != PKV_OK) return st;
  if (num_tokens < 0 || num_reqs < 0 || max_blocks_per_req < 0) return PKV_ERR_BAD_SHAPE;
  const int64_t row = static_cast<int64_t>(layout.num_kv_heads) * layout.head_dim;
  if (key_row_stride == 0) key_row_stride = row;
  if (value_row_stride == 0) value_row_stride = row;
  if (key_row_stride < row || value_row_stride < row) return PKV_ERR_BAD_SHAPE;
  if (num_tokens > 0) {
    if (!kv_cache || !key || !value || !query_start_loc) return PKV_ERR_NULL_POINTER;
    if (num_reqs > 0 && (!block_table || !num_computed_tokens)) return PKV_ERR_NULL_POINTER;
    if (!aligned16(kv_cache) || !aligned16(key) || !aligned16(value) || (key_row_stride % 8) ||
        (value_row_stride % 8))
      return PKV_ERR_MISALIGNED;
  }
  const pkv::WriteRowsArgs w = pkv::write_rows_args(
      kv_cache, key, value, key_row_stride, value_row_stride, slot_mapping, block_table,
      max_blocks_per_req, query_start_loc, num_computed_tokens, num_reqs, num_tokens,
      layout.num_blocks, layout.block_size, layout.num_kv_heads, layout.head_dim);
  return attention_impl(out, q, q_row_stride, kv_cache, block_table, max_blocks_per_req,
                        seq_lens, query_start_loc, num_computed_tokens, num_reqs, num_tokens,
                        max_query_len, max_seq_len, num_q_heads, scale, layout, workspace,
                        workspace_bytes, options, stream, num_tokens > 0 ? &w : nullptr);
}

int32_t pkv_get_device_errors(uint32_t* flags, int32_t clear, void* stream) {
  if (!flags) return PKV_ERR_NULL_POINTER;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t v = 0;
  e = pkv::read_errors_kvwrite(&v, clear != 0);
  if (e == cudaSuccess) e = pkv::read_errors_decode(&v, clear != 0);
  if (e == cudaSuccess) e = pkv::read_errors_prefill(&v, clear != 0);
  if (e == cudaSuccess) e = pkv::read_errors_plan(&v, clear != 0);
  if (e != cudaSuccess) return cuda_fail(e, "reading device error word");
  *flags = v;
  return PKV_OK;
}

}  // extern "C"
