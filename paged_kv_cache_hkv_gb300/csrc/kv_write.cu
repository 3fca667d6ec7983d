// Slot mapping and the cache write (reshape_and_cache) for sm_103a.
//
// Slot of a new token ("vllm v1 源码精读（三）", §3.4):
//   slot = block_table[r][pos / 16] * 16 + pos % 16,  pos = num_computed[r] + i.
// Write ("vLLM 架构源码解析（一）" §3.3.3; same page §3.4 of the v1 walk-through):
//   kv_cache[slot / 16][0|1][slot % 16][:][:] = key[t] | value[t].
//
// Both are memory moves. The write copies 16-byte vectors: a K or V row of
// one token is num_kv_heads * head_dim bf16 contiguous in the source and in
// the pool, so consecutive threads touch consecutive 16-byte words on both
// sides.
#include "common.cuh"
#include "launch.h"

namespace pkv {

static __device__ uint32_t g_errors_kvwrite;

__global__ void slot_mapping_kernel(int64_t* __restrict__ slots,
                                    const int32_t* __restrict__ block_table, int max_blocks,
                                    const int32_t* __restrict__ qsl,
                                    const int32_t* __restrict__ num_computed, int num_reqs,
                                    int num_tokens, int num_blocks) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= num_tokens) return;
  const int total = __ldg(qsl + num_reqs);
  if (t >= total || num_reqs <= 0) {
    slots[t] = -1;
    return;
  }
  if (__ldg(qsl) > t) {  // query_start_loc[0] must be 0
    atomicOr(&g_errors_kvwrite, kErrLengths);
    slots[t] = -1;
    return;
  }
  const int r = upper_index(qsl, num_reqs, t);
  const long long pos = static_cast<long long>(__ldg(num_computed + r)) + (t - __ldg(qsl + r));
  const long long lb = pos / kBlockSize;
  if (pos < 0 || lb >= max_blocks) {
    atomicOr(&g_errors_kvwrite, kErrLengths);
    slots[t] = -1;
    return;
  }
  const int phys = __ldg(block_table + static_cast<long long>(r) * max_blocks + lb);
  if (phys < 0 || phys >= num_blocks) {
    atomicOr(&g_errors_kvwrite, kErrBlockRange);
    slots[t] = -1;
    return;
  }
  slots[t] = static_cast<int64_t>(phys) * kBlockSize + (pos % kBlockSize);
}

// One 16-byte vector per thread per iteration. vec_per_row = Hkv * D / 8.
__global__ void kv_write_kernel(uint4* __restrict__ pool, const uint4* __restrict__ key,
                                const uint4* __restrict__ value, long long key_stride_v,
                                long long value_stride_v, const int64_t* __restrict__ slots,
                                int num_tokens, int vec_per_row, long long num_slots) {
  const long long total = static_cast<long long>(num_tokens) * 2 * vec_per_row;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int t = static_cast<int>(i / (2 * vec_per_row));
    const int w = static_cast<int>(i - static_cast<long long>(t) * 2 * vec_per_row);
    const int kv = w >= vec_per_row;
    const int e = w - kv * vec_per_row;
    const long long s = __ldg(slots + t);
    if (s < 0) continue;
    if (s >= num_slots) {
      if (e == 0 && kv == 0) atomicOr(&g_errors_kvwrite, kErrSlotRange);
      continue;
    }
    const uint4 v = kv ? __ldg(value + t * value_stride_v + e) : __ldg(key + t * key_stride_v + e);
    const long long blk = s / kBlockSize, off = s % kBlockSize;
    pool[((blk * 2 + kv) * kBlockSize + off) * vec_per_row + e] = v;
  }
}

cudaError_t launch_slot_mapping(int64_t* slots, const int32_t* block_table, int max_blocks,
                                const int32_t* qsl, const int32_t* num_computed, int num_reqs,
                                int num_tokens, int num_blocks, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int threads = 256;
  const int grid = (num_tokens + threads - 1) / threads;
  slot_mapping_kernel<<<grid, threads, 0, stream>>>(slots, block_table, max_blocks, qsl,
                                                    num_computed, num_reqs, num_tokens,
                                                    num_blocks);
  return cudaGetLastError();
}

cudaError_t launch_kv_write(void* pool, const void* key, const void* value, long long key_stride,
                            long long value_stride, const int64_t* slots, int num_tokens,
                            int num_blocks, int num_kv_heads, int head_dim, int num_sms,
                            cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int vec_per_row = num_kv_heads * head_dim / 8;
  const long long total = static_cast<long long>(num_tokens) * 2 * vec_per_row;
  const int threads = 256;
  long long grid = (total + threads - 1) / threads;
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (grid > cap) grid = cap;
  kv_write_kernel<<<static_cast<int>(grid), threads, 0, stream>>>(
      static_cast<uint4*>(pool), static_cast<const uint4*>(key), static_cast<const uint4*>(value),
      key_stride / 8, value_stride / 8, slots, num_tokens, vec_per_row,
      static_cast<long long>(num_blocks) * kBlockSize);
  return cudaGetLastError();
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
