// Slot mapping and the cache write (reshape_and_cache) for sm_103a.
//
// Slot of a new token ("vllm v1 源码精读（三）", §3.4), B tokens per block:
//   slot = block_table[r][pos / B] * B + pos % B,  pos = num_computed[r] + i.
// Write ("vLLM 架构源码解析（一）" §3.3.3; same page §3.4 of the v1 walk-through):
//   kv_cache[slot / B][0|1][slot % B][:][:] = key[t] | value[t].
// B is 8, 16 or 32 ("vLLM 架构源码解析（一）" §5.1 weighs the choice), passed
// as its log2 so that / and % are a shift and a mask.
//
// Both are memory moves. The write copies 16-byte vectors: a K or V row of
// one token is num_kv_heads * head_dim bf16 contiguous in the source and in
// the pool, so consecutive threads touch consecutive 16-byte words on both
// sides.
#include "common.cuh"
#include "launch.h"
#include "write_rows.cuh"

namespace pkv {

static __device__ uint32_t g_errors_kvwrite;

// One warp per request: its lanes cover the request's new tokens. Tokens at
// or past query_start_loc[num_reqs] (padding rows) are set to -1 by the
// threads of the trailing blocks of the grid.
__global__ void slot_mapping_kernel(int64_t* __restrict__ slots,
                                    const int32_t* __restrict__ block_table, int max_blocks,
                                    const int32_t* __restrict__ qsl,
                                    const int32_t* __restrict__ num_computed, int num_reqs,
                                    int num_tokens, int num_blocks, int shift, int req_blocks) {
  pdl_trigger();
  pdl_wait();
  if (static_cast<int>(blockIdx.x) >= req_blocks) {  // padding rows
    const int t = (blockIdx.x - req_blocks) * blockDim.x + threadIdx.x;
    if (t < num_tokens && t >= __ldg(qsl + num_reqs)) slots[t] = -1;
    return;
  }
  const int r = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, lane = threadIdx.x & 31;
  if (r >= num_reqs) return;
  const int q0 = __ldg(qsl + r), q1 = __ldg(qsl + r + 1);
  const int c = __ldg(num_computed + r);
  if (q0 < 0 || q1 < q0 || q1 > num_tokens || c < 0 || (r == 0 && q0 != 0)) {
    if (lane == 0) atomicOr(&g_errors_kvwrite, kErrLengths);
    // The request's rows (and, for request 0, every row before it) get -1:
    // a slot left over in the caller's buffer would otherwise send this
    // step's K/V into another sequence's block.
    const int t0 = r == 0 ? 0 : max(q0, 0);
    const int t1 = min(max(q1, q0), num_tokens);
    for (int t = t0 + lane; t < t1; t += 32) slots[t] = -1;
    return;
  }
  const long long row = static_cast<long long>(r) * max_blocks;
  for (int t = q0 + lane; t < q1; t += 32) {
    const long long pos = static_cast<long long>(c) + (t - q0);
    const long long lb = pos >> shift;
    int64_t slot = -1;
    if (lb >= max_blocks) {
      atomicOr(&g_errors_kvwrite, kErrLengths);
    } else {
      const int phys = __ldg(block_table + row + lb);
      if (phys < 0 || phys >= num_blocks)
        atomicOr(&g_errors_kvwrite, kErrBlockRange);
      else
        slot = (static_cast<int64_t>(phys) << shift) + (pos & ((1 << shift) - 1));
    }
    slots[t] = slot;
  }
}

// The write as one flat stream of 16-byte words: word w of the step is
// (token t, K|V, word e of the row) with w = (2 t + kv) * vec_per_row + e,
// so consecutive threads read consecutive words of a token's K row, then of
// its V row, and write them to consecutive words of the pool row. Every
// thread takes kWriteVecs words, a grid stride apart, and issues all their
// loads -- the slot and the data, which do not depend on each other --
// before any store, so each SM keeps tens of KB of reads in flight instead
// of one dependent slot-then-data chain per token. Index is int for steps
// of fewer than 2^31 words, else long long.
constexpr int kWriteVecs = 4;
constexpr int kWriteThreads = 512;

template <typename Index>
__global__ void __launch_bounds__(kWriteThreads)
    kv_write_kernel(uint4* __restrict__ pool, const uint4* __restrict__ key,
                    const uint4* __restrict__ value, long long key_stride_v,
                    long long value_stride_v, const int64_t* __restrict__ slots, Index total,
                    Index row_pair, int vec_per_row, int shift, long long num_slots) {
  pdl_trigger();
  pdl_wait();
  const Index stride = static_cast<Index>(gridDim.x) * blockDim.x;
  for (Index w0 = static_cast<Index>(blockIdx.x) * blockDim.x + threadIdx.x; w0 < total;
       w0 += stride * kWriteVecs) {
    uint4 val[kWriteVecs];
    long long slot[kWriteVecs];
    Index tok[kWriteVecs];
    int kv[kWriteVecs], e[kWriteVecs];
#pragma unroll
    for (int u = 0; u < kWriteVecs; ++u) {
      const Index w = w0 + u * stride;
      slot[u] = -1;
      if (w < total) {
        tok[u] = w / row_pair;
        const int rem = static_cast<int>(w - tok[u] * row_pair);
        kv[u] = rem >= vec_per_row;
        e[u] = rem - kv[u] * vec_per_row;
        slot[u] = __ldg(slots + tok[u]);
        const uint4* src = kv[u] ? value + static_cast<long long>(tok[u]) * value_stride_v
                                 : key + static_cast<long long>(tok[u]) * key_stride_v;
        val[u] = __ldg(src + e[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kWriteVecs; ++u) {
      const long long s = slot[u];
      if (s < 0) continue;  // padding row, or past the end
      if (s >= num_slots) {
        if (kv[u] == 0 && e[u] == 0) atomicOr(&g_errors_kvwrite, kErrSlotRange);
        continue;
      }
      const long long blk = s >> shift, off = s & ((1 << shift) - 1);
      pool[((((blk * 2 + kv[u]) << shift) + off) * vec_per_row) + e[u]] = val[u];
    }
  }
}

// The slot mapping fused into the write: one warp per new token (the body
// is write_token_rows).
constexpr int kMappedWarps = 8;  // warps (tokens) per CTA

__global__ void __launch_bounds__(kMappedWarps * 32) mapped_write_kernel(const WriteRowsArgs w) {
  pdl_trigger();
  pdl_wait();
  const long long t = static_cast<long long>(blockIdx.x) * kMappedWarps + (threadIdx.x >> 5);
  if (t < w.num_tokens) write_token_rows(w, t, &g_errors_kvwrite);
}

// Whole-block copies between two pools of one layout (copy-on-write of a
// shared block; swap-out / swap-in between the device pool and a pool in
// pinned host memory). One CTA per pair: 16-byte vectors, coalesced on both
// sides. vec_per_block = 2 * B * Hkv * D / 8.
__global__ void copy_blocks_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                   const int32_t* __restrict__ pairs, int num_pairs,
                                   int dst_num_blocks, int src_num_blocks, int vec_per_block) {
  pdl_trigger();
  pdl_wait();
  for (int i = blockIdx.x; i < num_pairs; i += gridDim.x) {
    const int s = __ldg(pairs + 2 * i), d = __ldg(pairs + 2 * i + 1);
    if (s < 0 || s >= src_num_blocks || d < 0 || d >= dst_num_blocks) {
      if (threadIdx.x == 0) atomicOr(&g_errors_kvwrite, kErrBlockRange);
      continue;
    }
    const uint4* from = src + static_cast<long long>(s) * vec_per_block;
    uint4* to = dst + static_cast<long long>(d) * vec_per_block;
    for (int e = threadIdx.x; e < vec_per_block; e += blockDim.x) to[e] = from[e];
  }
}

cudaError_t launch_copy_blocks(void* dst, int dst_num_blocks, const void* src, int src_num_blocks,
                               const int32_t* pairs, int num_pairs, int block_size,
                               int num_kv_heads, int head_dim, int num_sms, cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int vec_per_block = 2 * block_size * num_kv_heads * head_dim / 8;
  const long long cap = static_cast<long long>(num_sms) * 8;
  const int grid = static_cast<int>(num_pairs < cap ? num_pairs : cap);
  return launch_pdl(copy_blocks_kernel, dim3(grid), dim3(256), 0, stream, static_cast<uint4*>(dst),
                    static_cast<const uint4*>(src), pairs, num_pairs, dst_num_blocks,
                    src_num_blocks, vec_per_block);
}

cudaError_t launch_slot_mapping(int64_t* slots, const int32_t* block_table, int max_blocks,
                                const int32_t* qsl, const int32_t* num_computed, int num_reqs,
                                int num_tokens, int num_blocks, int block_size,
                                cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int threads = 256;
  const int req_blocks = (num_reqs + threads / 32 - 1) / (threads / 32);
  const int pad_blocks = (num_tokens + threads - 1) / threads;
  return launch_pdl(slot_mapping_kernel, dim3(req_blocks + pad_blocks), dim3(threads), 0, stream,
                    slots, block_table, max_blocks, qsl, num_computed, num_reqs, num_tokens,
                    num_blocks, static_cast<int>(__builtin_ctz(static_cast<unsigned>(block_size))),
                    req_blocks);
}

cudaError_t launch_kv_write(void* pool, const void* key, const void* value, long long key_stride,
                            long long value_stride, const int64_t* slots, int num_tokens,
                            int num_blocks, int block_size, int num_kv_heads, int head_dim,
                            int num_sms, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int vec_per_row = num_kv_heads * head_dim / 8;
  const long long total = static_cast<long long>(num_tokens) * 2 * vec_per_row;
  const long long per_cta = static_cast<long long>(kWriteThreads) * kWriteVecs;
  const long long cap = static_cast<long long>(num_sms) * 2;  // 2 x 512 threads per SM
  const long long need = (total + per_cta - 1) / per_cta;
  const int grid = static_cast<int>(need < cap ? need : cap);
  const int shift = static_cast<int>(__builtin_ctz(static_cast<unsigned>(block_size)));
  const long long num_slots = static_cast<long long>(num_blocks) * block_size;
  // int indexes while w0 + kWriteVecs * stride stays below 2^31
  if (total + static_cast<long long>(grid) * kWriteThreads * kWriteVecs < (1ll << 31))
    return launch_pdl(kv_write_kernel<int>, dim3(grid), dim3(kWriteThreads), 0, stream,
                      static_cast<uint4*>(pool), static_cast<const uint4*>(key),
                      static_cast<const uint4*>(value), key_stride / 8, value_stride / 8, slots,
                      static_cast<int>(total), 2 * vec_per_row, vec_per_row, shift, num_slots);
  return launch_pdl(kv_write_kernel<long long>, dim3(grid), dim3(kWriteThreads), 0, stream,
                    static_cast<uint4*>(pool), static_cast<const uint4*>(key),
                    static_cast<const uint4*>(value), key_stride / 8, value_stride / 8, slots,
                    total, static_cast<long long>(2 * vec_per_row), vec_per_row, shift,
                    num_slots);
}

WriteRowsArgs write_rows_args(void* pool, const void* key, const void* value,
                              long long key_stride, long long value_stride, int64_t* slots,
                              const int32_t* block_table, int max_blocks, const int32_t* qsl,
                              const int32_t* num_computed, int num_reqs, int num_tokens,
                              int num_blocks, int block_size, int num_kv_heads, int head_dim) {
  WriteRowsArgs w;
  w.pool = static_cast<uint4*>(pool);
  w.key = static_cast<const uint4*>(key);
  w.value = static_cast<const uint4*>(value);
  w.key_stride_v = key_stride / 8;
  w.value_stride_v = value_stride / 8;
  w.slots_out = slots;
  w.block_table = block_table;
  w.max_blocks = max_blocks;
  w.qsl = qsl;
  w.num_computed = num_computed;
  w.num_reqs = num_reqs;
  w.num_tokens = num_tokens;
  w.num_blocks = num_blocks;
  w.shift = static_cast<int>(__builtin_ctz(static_cast<unsigned>(block_size)));
  w.vec_per_row = num_kv_heads * head_dim / 8;
  return w;
}

cudaError_t launch_mapped_write(const WriteRowsArgs& w, cudaStream_t stream) {
  if (w.num_tokens == 0) return cudaSuccess;
  const int grid = (w.num_tokens + kMappedWarps - 1) / kMappedWarps;
  return launch_pdl(mapped_write_kernel, dim3(grid), dim3(kMappedWarps * 32), 0, stream, w);
}

cudaError_t read_errors_kvwrite(uint32_t* out, bool clear) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_errors_kvwrite, sizeof(v));
  if (e != cudaSuccess) return e;
  *out |= v;
  if (clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_errors_kvwrite, &z, sizeof(z));
  }
  return e;
}

}  // namespace pkv
