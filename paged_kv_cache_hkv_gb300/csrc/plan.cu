// The per-step plan (sm_103a): one CTA scans the requests' lengths and
// writes the decode stream's prefix sums, each decode CTA's first request,
// the prefill requests and work items, and checks the shared-prefix hint;
// the attention kernels read it. With the step's cache write fused in, the
// same launch also maps the new tokens' slots and writes their K and V rows
// (prologue_kernel).
#include "common.cuh"
#include "launch.h"
#include "write_rows.cuh"

namespace pkv {

static __device__ uint32_t g_errors_plan;

// ------------------------------------------------------------------ plan
// Block-wide exclusive scan of three counters (blockDim.x == 1024).
struct Int3 {
  int a, b, c;
};

__device__ __forceinline__ Int3 block_exclusive_scan(Int3 v, Int3* total) {
  __shared__ Int3 warp_tot[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  Int3 inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, inc.a, off);
    const int b = __shfl_up_sync(0xffffffffu, inc.b, off);
    const int c = __shfl_up_sync(0xffffffffu, inc.c, off);
    if (lane >= off) {
      inc.a += a;
      inc.b += b;
      inc.c += c;
    }
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    Int3 w = warp_tot[lane];
    Int3 wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, wi.a, off);
      const int b = __shfl_up_sync(0xffffffffu, wi.b, off);
      const int c = __shfl_up_sync(0xffffffffu, wi.c, off);
      if (lane >= off) {
        wi.a += a;
        wi.b += b;
        wi.c += c;
      }
    }
    warp_tot[lane] = Int3{wi.a - w.a, wi.b - w.b, wi.c - w.c};
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  const Int3 base = warp_tot[warp];
  __syncthreads();
  return Int3{base.a + inc.a - v.a, base.b + inc.b - v.b, base.c + inc.c - v.c};
}

// Counts of one request: decode 16-key chunks, is-prefill, prefill work items.
// A decode request that takes its shared prefix from the shared items
// streams only the chunks past the prefix.
__device__ __forceinline__ Int3 plan_counts(const AttnArgs& a, const AttnWorkspace& ws, int r,
                                            int tile_q, bool flag) {
  Int3 v{0, 0, 0};
  const int q0 = __ldg(a.qsl + r), q1 = __ldg(a.qsl + r + 1);
  const int n = q1 - q0, L = __ldg(a.seq_lens + r), c = __ldg(a.num_computed + r);
  bool bad = n < 0 || q0 < 0 || q1 > a.num_tokens || c < 0 || L != c + n || (r == 0 && q0 != 0);
  const long long nblk = (static_cast<long long>(L) + kChunkKeys - 1) / kChunkKeys;
  const long long nent = (static_cast<long long>(L) + (1 << a.block_shift) - 1) >> a.block_shift;
  if (!bad && n > 0 && nent > a.max_blocks) bad = true;
  if (bad) {
    if (flag) atomicOr(&g_errors_plan, kErrLengths);
  } else if (n == 1) {
    v.a = static_cast<int>(nblk);
    const int i = r - a.shared_first;
    if (a.shared_num > 0 && i >= 0 && i < a.shared_num && ws.casc_use[i])
      v.a -= a.shared_len / kChunkKeys;
  } else if (n > 1) {
    v.b = 1;
    v.c = ((n + tile_q - 1) / tile_q) * a.num_kv_heads;
  }
  return v;
}

// One CTA of 1024 threads, one pass: each thread takes a run of consecutive
// requests, counts decode blocks, prefill requests and prefill work items,
// and after one block scan writes the prefix sums and the compact list of
// prefill requests. Requests with inconsistent lengths are skipped and
// flagged.
// The shared-prefix hint, checked: every request of the run starts as a
// member; one whose table does not begin with the run's first request's
// entries, or whose context does not reach past the prefix, drops out (it is
// attended without the hint); one with other than a single new token turns
// the whole run off. Returns the number of shared-prefix work items.
__device__ int plan_shared(const AttnArgs& a, const AttnWorkspace& ws, int tile_q) {
  __shared__ int run_off, dropped;
  const int num = a.shared_num;
  if (threadIdx.x == 0) {
    run_off = 0;
    dropped = 0;
  }
  for (int i = threadIdx.x; i < num; i += blockDim.x) ws.casc_use[i] = 1;
  __syncthreads();
  for (int i = threadIdx.x; i < num; i += blockDim.x) {
    const int r = a.shared_first + i;
    if (__ldg(a.qsl + r + 1) - __ldg(a.qsl + r) != 1) run_off = 1;
    if (__ldg(a.seq_lens + r) <= a.shared_len) {
      ws.casc_use[i] = 0;
      dropped = 1;
    }
  }
  // table entries: request i's j-th against the first request's, four
  // (request, entry group) pairs per thread in flight; groups of 4 entries
  // (16-byte loads) when the rows allow it
  const int pb = a.shared_len >> a.block_shift;  // shared table entries
  const int32_t* row0 = a.block_table + static_cast<long long>(a.shared_first) * a.max_blocks;
  const bool vec = ((reinterpret_cast<uintptr_t>(row0) & 15u) == 0) && (a.max_blocks % 4 == 0) &&
                   (pb % 4 == 0);
  if (vec) {
    const int pb4 = pb / 4;
    const long long pairs = static_cast<long long>(num - 1) * pb4;
    const int4* r0 = reinterpret_cast<const int4*>(row0);
#pragma unroll 4
    for (long long x = threadIdx.x; x < pairs; x += blockDim.x) {
      const int i = 1 + static_cast<int>(x / pb4);
      const int j = static_cast<int>(x - static_cast<long long>(i - 1) * pb4);
      const int4 u = __ldg(r0 + static_cast<long long>(i) * (a.max_blocks / 4) + j);
      const int4 v = __ldg(r0 + j);
      if (u.x != v.x || u.y != v.y || u.z != v.z || u.w != v.w) {
        ws.casc_use[i] = 0;
        dropped = 1;
      }
    }
  } else {
    const long long pairs = static_cast<long long>(num - 1) * pb;
#pragma unroll 4
    for (long long x = threadIdx.x; x < pairs; x += blockDim.x) {
      const int i = 1 + static_cast<int>(x / pb);
      const int j = static_cast<int>(x - static_cast<long long>(i - 1) * pb);
      if (__ldg(row0 + static_cast<long long>(i) * a.max_blocks + j) != __ldg(row0 + j)) {
        ws.casc_use[i] = 0;
        dropped = 1;
      }
    }
  }
  __syncthreads();
  const bool off = run_off != 0;
  if (off)
    for (int i = threadIdx.x; i < num; i += blockDim.x) ws.casc_use[i] = 0;
  if (threadIdx.x == 0 && (off || dropped)) atomicOr(&g_errors_plan, kErrShared);
  __syncthreads();
  if (off) return 0;
  const int qtiles = (num + tile_q - 1) / tile_q;
  return qtiles * a.shared_pieces * a.num_kv_heads;
}

__device__ void plan_block(const AttnArgs& a, const AttnWorkspace& ws, int tile_q) {
  __shared__ Int3 total;
  const int shared_items = a.shared_num > 0 ? plan_shared(a, ws, tile_q) : 0;
  const int R = a.num_reqs;
  const int per = (R + 1023) / 1024;
  const int r0 = min(R, static_cast<int>(threadIdx.x) * per), r1 = min(R, r0 + per);
  Int3 sum{0, 0, 0};
  for (int r = r0; r < r1; ++r) {
    const Int3 v = plan_counts(a, ws, r, tile_q, true);
    sum.a += v.a;
    sum.b += v.b;
    sum.c += v.c;
  }
  Int3 run = block_exclusive_scan(sum, &total);
  // Request holding the first position floor(c * N / C) of each decode
  // CTA's range: request r (chunks [a, a + n) of the stream) holds the
  // starts of CTAs ceil(a C / N) .. ceil((a + n) C / N) - 1, so each CTA
  // reads its start instead of searching the prefix sums.
  const long long N = total.a, C = a.decode_splits;
  if (N == 0)
    for (long long c = threadIdx.x; c < C; c += blockDim.x) ws.bound[c] = -1;
  for (int r = r0; r < r1; ++r) {
    const Int3 v = plan_counts(a, ws, r, tile_q, false);
    if (v.a > 0) {
      const long long c_lo = (static_cast<long long>(run.a) * C + N - 1) / N;
      long long c_hi = ((static_cast<long long>(run.a) + v.a) * C + N - 1) / N;
      if (c_hi > C) c_hi = C;
      for (long long c = c_lo; c < c_hi; ++c) ws.bound[c] = r;
    }
    ws.dec_prefix[r] = run.a;
    if (v.b) {
      ws.pf_req[run.b] = r;
      ws.pf_prefix[run.b] = run.c;
    }
    run.a += v.a;
    run.b += v.b;
    run.c += v.c;
  }
  if (threadIdx.x == 0) {
    ws.dec_prefix[R] = total.a;
    int nreq = total.b, nitems = total.c;
    if (shared_items > 0) {  // the shared-prefix items come after every prefill request
      ws.pf_req[nreq] = -1;
      ws.pf_prefix[nreq] = nitems;
      nitems += shared_items;
      ++nreq;
    }
    ws.pf_prefix[nreq] = nitems;
    ws.hdr[kHdrDecodeBlocks] = static_cast<uint32_t>(total.a);
    ws.hdr[kHdrPrefillReqs] = static_cast<uint32_t>(nreq);
    ws.hdr[kHdrPrefillItems] = static_cast<uint32_t>(nitems);
    ws.hdr[kHdrPrefillNext] = 0u;
  }
}

__global__ void __launch_bounds__(1024) plan_kernel(AttnArgs a, AttnWorkspace ws, int tile_q) {
  pdl_trigger();
  pdl_wait();
  plan_block(a, ws, tile_q);
}

// The plan and the step's cache write in one launch: CTA 0 plans (it is
// dispatched first), CTAs 1 .. map the slots of kPrologueTokens new tokens
// each and write their rows (one warp per token; the CTA's other warps have
// nothing to do, so the tokens spread over twice as many SMs as full CTAs
// would). Neither part depends on the other; the attention kernels that
// follow wait for both.
constexpr int kPrologueTokens = 8;

__global__ void __launch_bounds__(1024)
    prologue_kernel(AttnArgs a, AttnWorkspace ws, int tile_q, WriteRowsArgs w) {
  pdl_trigger();
  pdl_wait();
  if (blockIdx.x == 0) {
    plan_block(a, ws, tile_q);
    return;
  }
  const int warp = threadIdx.x >> 5;
  if (warp >= kPrologueTokens) return;
  const long long t = static_cast<long long>(blockIdx.x - 1) * kPrologueTokens + warp;
  if (t < w.num_tokens) write_token_rows(w, t, &g_errors_plan);
}

cudaError_t launch_plan(const AttnArgs& a, const AttnWorkspace& ws, cudaStream_t stream,
                        const WriteRowsArgs* write) {
  const int group = a.num_q_heads / a.num_kv_heads;
  if (write && write->num_tokens > 0) {
    const int write_ctas = (write->num_tokens + kPrologueTokens - 1) / kPrologueTokens;
    return launch_pdl(prologue_kernel, dim3(1 + write_ctas), dim3(1024), 0, stream, a, ws,
                      128 / group, *write);
  }
  return launch_pdl(plan_kernel, dim3(1), dim3(1024), 0, stream, a, ws, 128 / group);
}

cudaError_t read_errors_plan(uint32_t* out, bool clear) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_errors_plan, sizeof(v));
  if (e != cudaSuccess) return e;
  *out |= v;
  if (clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_errors_plan, &z, sizeof(z));
  }
  return e;
}

}  // namespace pkv
