// The cache write of one new token with its slot computed on the device: the
// body shared by the fused slot-mapping-and-write kernel and the attention
// call's prologue kernel (sm_103a).
//
// Slot ("vllm v1 源码精读（三）" §3.4): request r's i-th new token, at position
// pos = num_computed[r] + i, goes to block_table[r][pos / B] * B + pos % B.
// Write ("vLLM 架构源码解析（一）" §3.3.3 step 2): kv_cache[slot / B][0|1]
// [slot % B][:][:] = key[t] | value[t].
#pragma once

#include "common.cuh"

namespace pkv {

struct WriteRowsArgs {
  uint4* pool;
  const uint4* key;
  const uint4* value;
  long long key_stride_v, value_stride_v;  // row strides in 16-byte words
  int64_t* slots_out;                      // may be null
  const int32_t* block_table;
  int max_blocks;
  const int32_t* qsl;
  const int32_t* num_computed;
  int num_reqs, num_tokens, num_blocks;
  int shift;        // log2 of the block size
  int vec_per_row;  // 16-byte words of one K (or V) row: Hkv * D / 8
};

constexpr int kWritePrefetch = 8;  // 16-byte words per lane loaded before the slot is known

// Token t by one whole warp. The warp issues the loads of the token's K and
// V rows first (the first kWritePrefetch words per lane of each), finds the
// token's request with a 32-way search of query_start_loc (non-decreasing),
// computes the slot and stores the rows. A token that the search puts in no
// request (before query_start_loc[0], at or past query_start_loc[num_reqs])
// or in a request with inconsistent lengths gets slot -1 and is not written;
// the error bits go to *err.
__device__ __forceinline__ void write_token_rows(const WriteRowsArgs& w, long long t,
                                                 uint32_t* err) {
  const int lane = threadIdx.x & 31;
  const uint4* ksrc = w.key + t * w.key_stride_v;
  const uint4* vsrc = w.value + t * w.value_stride_v;
  uint4 kw[kWritePrefetch], vw[kWritePrefetch];
#pragma unroll
  for (int i = 0; i < kWritePrefetch; ++i) {
    const int e = lane + 32 * i;
    if (e < w.vec_per_row) {
      kw[i] = __ldg(ksrc + e);
      vw[i] = __ldg(vsrc + e);
    }
  }
  const int tt = static_cast<int>(t);
  long long slot = -1;
  const int qend = __ldg(w.qsl + w.num_reqs), qfirst = __ldg(w.qsl);
  if (tt < qend && tt >= qfirst) {
    const int r = warp_upper_index(w.qsl, w.num_reqs, tt);
    const int q0 = __ldg(w.qsl + r), q1 = __ldg(w.qsl + r + 1);
    const int c = __ldg(w.num_computed + r);
    if (q0 < 0 || q1 < q0 || q1 > w.num_tokens || c < 0 || (r == 0 && q0 != 0)) {
      if (lane == 0) atomicOr(err, kErrLengths);
    } else {
      const long long pos = static_cast<long long>(c) + (tt - q0);
      const long long lb = pos >> w.shift;
      if (lb >= w.max_blocks) {
        if (lane == 0) atomicOr(err, kErrLengths);
      } else {
        const int phys = __ldg(w.block_table + static_cast<long long>(r) * w.max_blocks + lb);
        if (phys < 0 || phys >= w.num_blocks) {
          if (lane == 0) atomicOr(err, kErrBlockRange);
        } else {
          slot = (static_cast<long long>(phys) << w.shift) + (pos & ((1 << w.shift) - 1));
        }
      }
    }
  } else if (tt < qend || qfirst != 0) {  // rows before a non-zero query_start_loc[0]
    if (lane == 0) atomicOr(err, kErrLengths);
  }
  if (w.slots_out && lane == 0) w.slots_out[t] = slot;
  if (slot < 0) return;
  const long long blk = slot >> w.shift, off = slot & ((1 << w.shift) - 1);
  uint4* kdst = w.pool + (((blk * 2) << w.shift) + off) * w.vec_per_row;
  uint4* vdst = w.pool + (((blk * 2 + 1) << w.shift) + off) * w.vec_per_row;
#pragma unroll
  for (int i = 0; i < kWritePrefetch; ++i) {
    const int e = lane + 32 * i;
    if (e < w.vec_per_row) {
      kdst[e] = kw[i];
      vdst[e] = vw[i];
    }
  }
  for (int e = lane + 32 * kWritePrefetch; e < w.vec_per_row; e += 32) {  // rows over 4 KB
    kdst[e] = __ldg(ksrc + e);
    vdst[e] = __ldg(vsrc + e);
  }
}

}  // namespace pkv
