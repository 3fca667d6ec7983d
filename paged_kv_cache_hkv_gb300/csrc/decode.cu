// Split-KV paged decode attention and the split-KV combine (sm_103a).
//
// Decode ("vLLM 架构源码解析（一）" §3.3.3, §4.2; "vllm v1 源码精读（三）" §4.2):
// a request with one new token attends every one of its L cached keys, read
// block by block through its block table without gathering them into a
// contiguous buffer. GQA: the G = Hq/Hkv q heads of a kv head share every
// K/V row, so one warp handles up to 4 of them (a "virtual head") and each
// row is read from HBM once.
//
// Work split (split-KV, "PagedAttention v2" in §4.2 of the first page; the
// pages only name it): the decode KV stream of the whole step is the
// sequence of (request, 16-key chunk) in that order; CTA c of C takes the
// contiguous range [c*N/C, (c+1)*N/C) for a slab of up to 8 virtual heads
// (whole kv heads; the grid is C x slabs). Every CTA streams the same number
// of chunks whatever the length mix. A request cut by a range boundary
// leaves one partial (m, l, o) per CTA that touched it, which the combine
// kernel merges with the usual log-sum-exp rule; a request that falls
// inside one CTA's range is finished there and written straight to the
// output.
//
// The unit of the stream is a chunk of 16 keys, whatever the cache's block
// size B: a 16-token block, half of a 32-token block or two 8-token blocks.
// Inside a CTA one producer warp fills a ring of shared-memory stages, each
// holding one chunk's 16 K rows and 16 V rows of every kv head of the slab:
// one 3-D TMA copy for B = 16, where K and V of a block are 32 consecutive
// pool rows; two of 16 rows for B = 32 (half the K rows, half the V rows)
// and for B = 8 (the 8 K and 8 V rows of each block). On the first chunk of
// a request it also bulk-copies the slab's query rows. One consumer warp per
// virtual head reads its kv head's columns of each stage. Online softmax
// runs in base 2 with q pre-scaled by scale*log2(e).
#include <mutex>
#include <vector>

#include "common.cuh"
#include "launch.h"

namespace pkv {

static __device__ uint32_t g_errors_decode;

// ------------------------------------------------------------------ decode
// Work split: the decode stream of the step is the sequence of (request,
// 16-key chunk) positions; CTA c of C takes [c*N/C, (c+1)*N/C). A CTA holds
// one consumer warp per virtual head (GW q heads of one kv head) of its head
// slab -- up to 8 virtual heads, so 9 warps with the producer -- and each
// chunk's K and V rows of every kv head of the slab arrive in one TMA copy
// (one {D, KH, 32} box for 16-token blocks: 32 pool rows of KH*D*2
// contiguous bytes), which streams DRAM far better than one 256-byte row
// per kv head. A request cut by a range boundary leaves one partial per
// CTA that touched it, in slot (request + c) * V + virtual head; the
// combine kernel merges them.
struct DecodeParams {
  const uint16_t* q;
  long long q_stride;
  uint16_t* out;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* seq_lens;
  const int32_t* qsl;
  int num_reqs, num_q_heads, num_blocks;
  int head_groups;  // q-head groups of GW per kv head
  int virt_heads;   // V = num_kv_heads * head_groups
  int slab_vh;      // virtual heads per CTA slab (<= 8); slab s = virtual heads [s*slab_vh, ...)
  int slab_kh;      // kv heads per slab = slab_vh / head_groups
  long long splits; // C: CTAs along the stream (the grid is C x slabs)
  int stages;       // depth of the shared-memory ring of K/V chunks (>= 2)
  float scale_log2;
  const int32_t* dec_prefix;
  const uint32_t* hdr;
  float2* part_ml;
  float* part_o;
  const int* bound;  // [C]: request holding the first position of CTA c's range (-1: none)
  // Shared prefix: request shared_first + i with shared_use[i] streams only
  // its chunks from shared_chunks on and always leaves partials; the combine
  // kernel merges them with the shared items' partials of its row
  // (shared_pieces of them).
  int shared_first, shared_num, shared_chunks, shared_pieces;
  const int32_t* shared_use;
  const float2* shared_ml;
  const float* shared_o;
};

// CTA that owns position x of the decode stream: ranges start at floor(c * N / C).
__device__ __forceinline__ long long owner_cta(long long x, long long N, long long C) {
  return ((x + 1) * C + N - 1) / N - 1;
}

template <int D, int GW>
struct DecodeCfg {
  static constexpr int LPK = D / 8;     // lanes per key row (8 bf16 per lane)
  static constexpr int KPI = 32 / LPK;  // keys per warp instruction ("sub-groups")
  static constexpr int KPL = 16 / KPI;  // keys per lane per chunk
  static constexpr int NV = GW * KPL;   // partial scores per lane per chunk
  static constexpr int NPL = NV >= LPK ? NV / LPK : 1;  // full scores per lane
  static constexpr int DUP = NV >= LPK ? 1 : LPK / NV;  // lanes holding the same score
  static constexpr int LPH = LPK / GW;                  // lanes per head in a sub-group
  static_assert(KPL * KPI == 16, "chunk of 16 keys");
  static_assert(KPL % NPL == 0, "a lane's scores stay in one head");

  struct alignas(16) WarpScratch {
    float p[KPI][NV];
    float2 hs[GW];
  };
};

// Shared memory of a decode CTA (bytes from a 128-aligned base), the same on
// host and device: S stages of [32 rows][KH kv heads][D] K/V then the slab's
// q rows [VH * GW][D]; per-stage metadata; full / empty barriers; per-warp
// scratch.
template <int D, int GW>
struct DecodeLayout {
  uint32_t kv_bytes, row_bytes, stage_bytes, meta_off, bar_off, scratch_off, total;
  __host__ __device__ DecodeLayout(int kh, int vh, int S) {
    row_bytes = static_cast<uint32_t>(kh) * D * 2u;
    kv_bytes = 32u * row_bytes;
    const uint32_t q_bytes = static_cast<uint32_t>(vh) * GW * D * 2u;
    stage_bytes = (kv_bytes + q_bytes + 127u) & ~127u;
    meta_off = S * stage_bytes;
    bar_off = meta_off + S * 16u;
    scratch_off = (bar_off + 2u * S * 8u + 127u) & ~127u;
    total = scratch_off + static_cast<uint32_t>(vh) *
                              static_cast<uint32_t>(sizeof(typename DecodeCfg<D, GW>::WarpScratch));
  }
};

enum : int { kFirst = 1, kLast = 2, kInvalid = 4, kEnd = 8 };

// Stage rows of key j (0..15) of a chunk, SH = log2(B). 8-token blocks land
// as [K 0..7 | V 0..7 | K 8..15 | V 8..15], the others as [K 0..15 | V 0..15].
template <int SH>
__device__ __forceinline__ int k_row(int j) {
  return SH == 3 ? (j & 7) + ((j >> 3) << 4) : j;
}
template <int SH>
__device__ __forceinline__ int v_row(int j) {
  return SH == 3 ? (j & 7) + ((j >> 3) << 4) + 8 : 16 + j;
}

// Reduce-scatter across the LPK lanes of a sub-group. The caller stores at
// register position p the partial score of logical index p ^ (li * NV / LPK)
// (lane-dependent order of q heads and keys), so at every halving stage the
// lower half is the one this lane keeps and the upper half the one its
// partner keeps: no selects. On return v[0..NPL) hold full sums for logical
// indices (li * NV / LPK) + i.
template <int N, int OFF>
struct ReduceScatter {
  static __device__ __forceinline__ void run(float* v) {
    if constexpr (OFF >= 1) {
      if constexpr (N >= 2) {
        constexpr int H = N / 2;
#pragma unroll
        for (int i = 0; i < H; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i + H], OFF);
        ReduceScatter<H, OFF / 2>::run(v);
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], OFF);
        ReduceScatter<1, OFF / 2>::run(v);
      }
    }
  }
};

// The running max of a head is only moved (and o, l rescaled) when a chunk's
// max exceeds it by more than this many powers of two; in between, p may
// reach 2^8, far inside fp32 range. The result is the same softmax.
constexpr float kRescaleLog2 = 8.f;

constexpr int kDecodeMaxSlab = 8;                        // virtual heads per CTA at most
constexpr int kDecodeThreads = (kDecodeMaxSlab + 1) * 32;  // + the producer warp

template <int D, int GW, int SH>
__global__ void __launch_bounds__(kDecodeThreads)
    decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p) {
  using C = DecodeCfg<D, GW>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // dynamic shared memory is only guaranteed 16-byte aligned: round up
  unsigned char* base = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  const int VH = p.slab_vh, KH = p.slab_kh;
  const uint32_t S = static_cast<uint32_t>(p.stages);
  const DecodeLayout<D, GW> lay(KH, VH, p.stages);
  int4* meta = reinterpret_cast<int4*>(base + lay.meta_off);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + lay.bar_off);
  uint64_t* empty = full + S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the tensor map is a kernel parameter: its descriptor can be fetched
  // before the previous kernel is done
  if (warp == VH && lane == 0) prefetch_tensormap(&kv_map);
  // no early trigger here: a next kernel's CTAs, resident next to these for
  // the whole decode while they wait for it, slow the decode down
  pdl_wait();

  const long long Cn = p.splits, c = blockIdx.x;
  const int slab = blockIdx.y;
  // the stream's length and this CTA's start record are independent loads
  const long long N = p.hdr[kHdrDecodeBlocks];
  const int r_start = __ldg(p.bound + c);  // -1 when the step has no decode chunk
  const long long x0 = c * N / Cn, x1 = (c + 1) * N / Cn;

  // ---------------- locate position x0: (request r, chunk blk); the plan
  // recorded the request holding it (the combine kernel reads the same
  // records to find split requests)
  int r = -1, blk = 0, nblk = 0, pr = 0;
  if (x0 < N) {
    r = r_start;
    pr = __ldg(p.dec_prefix + r);  // stream position of the request's first chunk
    nblk = __ldg(p.dec_prefix + r + 1) - pr;
    blk = static_cast<int>(x0 - pr);
  }
  if (x0 >= x1) return;
  constexpr int sh = SH;
  // chunks of request rr before its first streamed one (its shared prefix)
  auto chunk_off = [&](int rr) -> int {
    const int i = rr - p.shared_first;
    return (p.shared_num > 0 && i >= 0 && i < p.shared_num && __ldg(p.shared_use + i))
               ? p.shared_chunks
               : 0;
  };
  // table entry of absolute chunk a
  auto entry_of = [&](int a) -> int { return (sh == 4) ? a : (sh == 5 ? a >> 1 : 2 * a); };
  // the producer's first loads go out before the barrier: the first
  // request's lengths and the 32 block-table entries from its first chunk on
  int L = 0, t = 0, nent = 0, skip = 0, win_r = -1, win_base = 0, win_val = -1;
  if (warp == VH) {
    L = __ldg(p.seq_lens + r);
    t = __ldg(p.qsl + r);
    skip = chunk_off(r);  // chunk = blk + skip
    nent = (L + (1 << sh) - 1) >> sh;  // table entries the request uses
    win_r = r;
    win_base = entry_of(blk + skip);
    const int j = win_base + lane;
    win_val = (j < nent) ? __ldg(p.block_table + static_cast<long long>(r) * p.max_blocks + j) : -1;
  }
  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], VH);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == VH) {
    // ================= producer warp: metadata, block-table lookups and the
    // copies of every chunk of the range, S stages ahead of the consumers
    // K/V rows are read once per step: evict them from L2 first, so that the
    // split-KV partials, q rows and tables stay (mixed step: 827 -> 819 us)
    const uint64_t l2_policy = l2_evict_first_policy();
    // The next request's lengths and the 32 entries of its block table row
    // from its first streamed chunk on, loaded one request ahead: a request
    // boundary then waits on no load.
    int nx_pn = -1, nx_L = 0, nx_t = 0, nx_win = -1, nx_off = 0;
    auto prefetch_next = [&]() {
      if (r + 1 < p.num_reqs) {
        nx_pn = __ldg(p.dec_prefix + r + 2);
        nx_L = __ldg(p.seq_lens + r + 1);
        nx_t = __ldg(p.qsl + r + 1);
        nx_off = chunk_off(r + 1);
        const int e = entry_of(nx_off) + lane;
        nx_win = e < p.max_blocks
                     ? __ldg(p.block_table + static_cast<long long>(r + 1) * p.max_blocks + e)
                     : -1;
      } else {
        nx_pn = -1;
      }
    };
    prefetch_next();
    int out_base = -1;
    bool new_piece = true;
    long long x = x0;
    uint32_t issued = 0;  // stages handed out so far
    uint32_t s = 0, eph = 0;  // ring slot of the next stage; parity of its empty barrier
    bool ok = true;
    for (;; ++issued) {
      if (issued >= S && !mbar_wait(&empty[s], eph)) {
        if (lane == 0) atomicOr(&g_errors_decode, kErrTimeout);
        ok = false;
        break;
      }
      if (x >= x1) {
        if (lane == 0) {
          meta[s] = make_int4(kEnd, 0, 0, 0);
          mbar_arrive(&full[s]);
        }
        ++issued;
        break;
      }
      if (new_piece) {
        // a request split over several CTAs, or one whose shared prefix is
        // attended elsewhere, leaves a partial for the combine kernel
        const long long a = pr;
        const long long cf = owner_cta(a, N, Cn), cl = owner_cta(a + nblk - 1, N, Cn);
        out_base = (cf == cl && skip == 0) ? -1 : static_cast<int>((r + c) * p.virt_heads);
      }
      // table entries of chunk blk: e0, and e0 + 1 for 8-token blocks
      const int ab = blk + skip;  // the chunk's place in the request
      const int e0 = entry_of(ab);
      const int e_hi = (sh == 3) ? e0 + 1 : e0;
      if (r != win_r || e0 < win_base || e_hi >= win_base + 32) {
        win_r = r;
        win_base = e0;
        const int j = e0 + lane;
        win_val = (j < nent) ? __ldg(p.block_table + static_cast<long long>(r) * p.max_blocks + j) : -1;
      }
      const int phys = __shfl_sync(0xffffffffu, win_val, e0 - win_base);
      const int nvalid = min(kChunkKeys, L - ab * kChunkKeys);
      bool valid = phys >= 0 && phys < p.num_blocks;
      bool second = false;  // 8-token blocks: the chunk's keys 8..15 exist
      int phys1 = -1;
      if constexpr (sh == 3) {
        phys1 = __shfl_sync(0xffffffffu, win_val, e_hi - win_base);
        second = nvalid > 8;
        if (second) valid = valid && phys1 >= 0 && phys1 < p.num_blocks;
      }
      const int flags = (new_piece ? kFirst : 0) | ((blk == nblk - 1 || x == x1 - 1) ? kLast : 0) |
                        (valid ? 0 : kInvalid);
      if (lane == 0) {
        meta[s] = make_int4(flags, nvalid, t, out_base);
        unsigned char* stage = base + s * lay.stage_bytes;
        const uint32_t kv_tx = (sh == 3 && !second) ? lay.kv_bytes / 2 : lay.kv_bytes;
        const uint32_t q_tx = static_cast<uint32_t>(VH) * GW * D * 2u;
        const uint32_t tx = (valid ? kv_tx : 0u) + (new_piece ? q_tx : 0u);
        if (!valid) atomicOr(&g_errors_decode, kErrBlockRange);
        if (tx) {
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(&full[s], tx);
          if (valid) {
            // pool rows of the slab's kv heads: (block * 2 + k|v) * B + offset
            const int hk0 = slab * KH;
            if constexpr (sh == 4) {  // K and V of the block: 32 consecutive rows
              tma_load_3d_hint(stage, &kv_map, 0, hk0, phys * 32, &full[s], l2_policy);
            } else if constexpr (sh == 5) {  // half (blk & 1) of the K rows and of the V rows
              const int row = phys * 64 + (blk & 1) * 16;
              tma_load_3d_hint(stage, &kv_map, 0, hk0, row, &full[s], l2_policy);
              tma_load_3d_hint(stage + 16 * lay.row_bytes, &kv_map, 0, hk0, row + 32, &full[s],
                               l2_policy);
            } else {  // two blocks of 8, each its 16 consecutive K and V rows
              tma_load_3d_hint(stage, &kv_map, 0, hk0, phys * 16, &full[s], l2_policy);
              if (second)
                tma_load_3d_hint(stage + 16 * lay.row_bytes, &kv_map, 0, hk0, phys1 * 16, &full[s],
                                 l2_policy);
            }
          }
          if (new_piece)  // the slab's q rows of the request (contiguous in the token row)
            bulk_load(stage + lay.kv_bytes,
                      p.q + static_cast<long long>(t) * p.q_stride + slab * VH * GW * D, q_tx,
                      &full[s]);
        } else {
          mbar_arrive(&full[s]);
        }
      }
      if (++s == S) {  // ring wraps; from the second wrap on, the empty parity flips
        s = 0;
        if (issued + 1 > S) eph ^= 1u;
      }
      // advance (request, chunk)
      ++x;
      ++blk;
      new_piece = false;
      if (blk == nblk) {
        blk = 0;
        new_piece = true;
        if (x < x1) {
          pr += nblk;  // empty requests in between add no chunks
          if (nx_pn - pr > 0) {  // the next request has chunks: its data is here
            ++r;
            nblk = nx_pn - pr;
            L = nx_L;
            t = nx_t;
            skip = nx_off;
            nent = (L + (1 << sh) - 1) >> sh;
            win_r = r;
            win_base = entry_of(skip);
            win_val = win_base + lane < nent ? nx_win : -1;
          } else {
            do {
              ++r;
              nblk = __ldg(p.dec_prefix + r + 1) - __ldg(p.dec_prefix + r);
            } while (nblk == 0);
            L = __ldg(p.seq_lens + r);
            t = __ldg(p.qsl + r);
            skip = chunk_off(r);
            nent = (L + (1 << sh) - 1) >> sh;
          }
          prefetch_next();
        }
      }
    }
    if (!ok && lane == 0) {
      // let every copy in flight land before the shared memory goes away
      for (uint32_t k = (issued > S ? issued - S : 0); k < issued; ++k)
        mbar_wait(&full[k % S], (k / S) & 1u, kDrainLimitNs);
    }
    return;
  }

  // ================= consumer warp: virtual head vg = slab * VH + warp
  const int vg = slab * VH + warp;
  const int hk_local = warp / p.head_groups;  // kv head within the slab
  auto& scr = reinterpret_cast<typename C::WarpScratch*>(base + lay.scratch_off)[warp];
  const int sub = lane / C::LPK, li = lane % C::LPK;
  // Position p of the per-chunk score registers holds logical index
  // p ^ perm: q head (p / KPL) ^ perm_h, key slot (p % KPL) ^ perm_k.
  const int perm = (li * C::NV) / C::LPK;
  const int perm_h = perm / C::KPL, perm_k = perm % C::KPL;
  const int hm = perm_h;  // head of this lane's full scores after the reduction
  float2 q2[GW][4];  // q * scale * log2(e), position order (head hp ^ perm_h)
  float2 o2[GW][4];  // unnormalised output, logical heads, dims li*8 .. li*8+7
  float m_run = -INFINITY, l_run = 0.f;  // for head hm of this lane
  const uint32_t RS = lay.row_bytes;    // bytes between stage rows

  for (uint32_t s = 0, fph = 0;;) {  // ring slot, parity of its full barrier
    if (!mbar_wait(&full[s], fph)) {
      atomicOr(&g_errors_decode, kErrTimeout);
      break;
    }
    const int4 m = meta[s];
    if (m.x & kEnd) break;
    const int flags = m.x, nvalid = m.y, row = m.z, out_base = m.w;
    const unsigned char* stage = base + s * lay.stage_bytes;
    const uint32_t kv_base = smem_u32(stage) + hk_local * D * 2 + li * 16;

    if (flags & kFirst) {
      const uint32_t qa = smem_u32(stage + lay.kv_bytes) + warp * GW * D * 2 + li * 16;
#pragma unroll
      for (int hp = 0; hp < GW; ++hp) {
        const uint4 qv = ld_shared_v4(qa + (hp ^ perm_h) * D * 2);
        const uint32_t wd[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          q2[hp][e] = make_float2(bf16_lo(wd[e]) * p.scale_log2, bf16_hi(wd[e]) * p.scale_log2);
          o2[hp][e] = make_float2(0.f, 0.f);
        }
      }
      m_run = -INFINITY;
      l_run = 0.f;
    }
    const bool bvalid = !(flags & kInvalid);

    // ---- scores, partial over this lane's 8 dims
    float acc[C::NV];
#pragma unroll
    for (int jp = 0; jp < C::KPL; ++jp) {
      const int key = (jp ^ perm_k) * C::KPI + sub;
      const uint4 kv4 = ld_shared_v4(kv_base + k_row<SH>(key) * RS);
      const uint32_t wd[4] = {kv4.x, kv4.y, kv4.z, kv4.w};
      float2 k2[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) k2[e] = make_float2(bf16_lo(wd[e]), bf16_hi(wd[e]));
#pragma unroll
      for (int hp = 0; hp < GW; ++hp) {
        float2 a2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 4; ++e) a2 = ffma2(q2[hp][e], k2[e], a2);
        acc[hp * C::KPL + jp] = a2.x + a2.y;
      }
    }
    ReduceScatter<C::NV, C::LPK / 2>::run(acc);

    // ---- online softmax for head hm
    float sc[C::NPL];
    float lmax = -INFINITY;
#pragma unroll
    for (int q = 0; q < C::NPL; ++q) {
      const int key = ((perm + q) % C::KPL) * C::KPI + sub;
      sc[q] = (bvalid && key < nvalid) ? acc[q] : -INFINITY;
      lmax = fmaxf(lmax, sc[q]);
    }
#pragma unroll
    for (int off = 1; off < C::LPH; off <<= 1)
      lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, off));
#pragma unroll
    for (int off = C::LPK; off < 32; off <<= 1)
      lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, off));
    if (__any_sync(0xffffffffu, lmax > m_run + kRescaleLog2)) {
      const float m_new = fmaxf(m_run, lmax);
      const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
      l_run *= alpha;
      m_run = m_new;
      if (sub == 0 && (li % C::LPH) == 0) scr.hs[hm].x = alpha;
      __syncwarp();
#pragma unroll
      for (int h = 0; h < GW; ++h) {
        const float a = scr.hs[h].x;
#pragma unroll
        for (int e = 0; e < 4; ++e) o2[h][e] = make_float2(o2[h][e].x * a, o2[h][e].y * a);
      }
    }
    float psum = 0.f;
#pragma unroll
    for (int q = 0; q < C::NPL; ++q) {
      const float pv = (sc[q] == -INFINITY || m_run == -INFINITY) ? 0.f : exp2f(sc[q] - m_run);
      scr.p[sub][perm + q] = pv;
      psum += pv;
    }
    l_run += psum;
    __syncwarp();

    // ---- o += sum_j p_j v_j
    {
      float pj[C::NV];
#pragma unroll
      for (int q = 0; q < C::NV; q += 4) {
        const float4 f = ld_shared_f4(smem_u32(&scr.p[sub][q]));
        pj[q] = f.x;
        pj[q + 1] = f.y;
        pj[q + 2] = f.z;
        pj[q + 3] = f.w;
      }
      auto pv_key = [&](int j) {
        const int key = j * C::KPI + sub;
        const uint4 vv = ld_shared_v4(kv_base + v_row<SH>(key) * RS);
        const uint32_t wd[4] = {vv.x, vv.y, vv.z, vv.w};
        float2 v2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v2[e] = make_float2(bf16_lo(wd[e]), bf16_hi(wd[e]));
#pragma unroll
        for (int h = 0; h < GW; ++h) {
          const float pp = pj[h * C::KPL + j];
          const float2 p2 = make_float2(pp, pp);
#pragma unroll
          for (int e = 0; e < 4; ++e) o2[h][e] = ffma2(p2, v2[e], o2[h][e]);
        }
      };
      if (bvalid && nvalid == kChunkKeys) {
#pragma unroll
        for (int j = 0; j < C::KPL; ++j) pv_key(j);
      } else {
#pragma unroll
        for (int j = 0; j < C::KPL; ++j)
          if (bvalid && j * C::KPI + sub < nvalid) pv_key(j);
      }
    }
    __syncwarp();

    // ---- end of this CTA's piece of the request
    if (flags & kLast) {
#pragma unroll
      for (int off = C::LPK; off < 32; off <<= 1)
#pragma unroll
        for (int h = 0; h < GW; ++h)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            o2[h][e].x += __shfl_xor_sync(0xffffffffu, o2[h][e].x, off);
            o2[h][e].y += __shfl_xor_sync(0xffffffffu, o2[h][e].y, off);
          }
      float lo = (C::DUP == 1 || (li % C::DUP) == 0) ? l_run : 0.f;
#pragma unroll
      for (int off = 1; off < C::LPH; off <<= 1) lo += __shfl_xor_sync(0xffffffffu, lo, off);
#pragma unroll
      for (int off = C::LPK; off < 32; off <<= 1) lo += __shfl_xor_sync(0xffffffffu, lo, off);
      if (sub == 0 && (li % C::LPH) == 0) scr.hs[hm] = make_float2(m_run, lo);
      __syncwarp();
      const long long slot = out_base < 0 ? -1 : static_cast<long long>(out_base) + vg;
      if (sub == 0) {
#pragma unroll
        for (int h = 0; h < GW; ++h) {
          const float2 ml = scr.hs[h];
          if (slot < 0) {
            const float inv = 1.f / ml.y;
            uint4 ov;
            ov.x = pack_bf16x2(o2[h][0].x * inv, o2[h][0].y * inv);
            ov.y = pack_bf16x2(o2[h][1].x * inv, o2[h][1].y * inv);
            ov.z = pack_bf16x2(o2[h][2].x * inv, o2[h][2].y * inv);
            ov.w = pack_bf16x2(o2[h][3].x * inv, o2[h][3].y * inv);
            const long long off =
                (static_cast<long long>(row) * p.num_q_heads + vg * GW + h) * D + li * 8;
            *reinterpret_cast<uint4*>(p.out + off) = ov;
          } else {
            float4* dst = reinterpret_cast<float4*>(p.part_o + (slot * GW + h) * D + li * 8);
            dst[0] = make_float4(o2[h][0].x, o2[h][0].y, o2[h][1].x, o2[h][1].y);
            dst[1] = make_float4(o2[h][2].x, o2[h][2].y, o2[h][3].x, o2[h][3].y);
            if (li == 0) p.part_ml[slot * GW + h] = ml;
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // the stage may be refilled
    if (++s == S) {
      s = 0;
      fph ^= 1u;
    }
  }
}

// ------------------------------------------------------------------ combine
// One CTA per (range boundary c of the split, virtual head vg), one warp per
// q head. A request is split when a boundary falls strictly inside its
// chunks; the first such boundary is the one right after the CTA that owns
// the request's first chunk, and that boundary's CTAs merge the request's
// partials (one per non-empty range that touched it):
//   M = max_p m_p,  o = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p.
// CTAs c >= C (one per request of a shared-prefix run) merge such a
// request's decode partials with the shared-prefix items' partials of its
// row; the boundary CTAs leave those requests to them.
// Lanes first read the (m, l) of up to 32 pieces at once, then every lane
// sums its dims over the pieces with independent loads.
template <int D, int GW>
__global__ void __launch_bounds__(GW * 32) combine_kernel(const DecodeParams p) {
  const long long c = blockIdx.x;
  const int vg = blockIdx.y;
  const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long Cn = p.splits;
  pdl_trigger();
  pdl_wait();
  auto in_shared_run = [&](int rr) -> bool {
    const int i = rr - p.shared_first;
    return p.shared_num > 0 && i >= 0 && i < p.shared_num && __ldg(p.shared_use + i);
  };
  int r, si = -1;  // si: the request's place in the shared-prefix run, if it has one
  if (c >= Cn) {
    si = static_cast<int>(c - Cn);
    if (si >= p.shared_num || !__ldg(p.shared_use + si)) return;
    r = p.shared_first + si;
  } else {
    if (c < 1) return;
    r = p.bound[c];
    if (r < 0) return;
  }
  const int pr = __ldg(p.dec_prefix + r);
  const int nblk = __ldg(p.dec_prefix + r + 1) - pr;
  const long long N = p.hdr[kHdrDecodeBlocks];
  const long long cf = owner_cta(pr, N, Cn);
  if (si < 0 && (cf != c - 1 || in_shared_run(r))) return;
  // pieces j < nd: the decode partial of CTA cf + j, in slot (r + cf + j) * V
  // + vg; pieces nd .. nd + ns - 1: the shared-prefix items' partials
  const int nd = static_cast<int>(owner_cta(pr + nblk - 1, N, Cn) - cf + 1);
  const int ns = si >= 0 ? p.shared_pieces : 0;
  const int npieces = nd + ns;
  const long long srow = static_cast<long long>(si) * p.num_q_heads + vg * GW + h;
  const long long sstride = static_cast<long long>(p.shared_num) * p.num_q_heads;

  // (m, l) of piece j; empty ranges wrote nothing and weigh zero
  auto piece_ml = [&](int j) -> float2 {
    if (j >= npieces) return make_float2(-INFINITY, 0.f);
    if (j >= nd) return p.shared_ml[srow + (j - nd) * sstride];
    const long long cc = cf + j;
    if (cc * N / Cn == (cc + 1) * N / Cn) return make_float2(-INFINITY, 0.f);
    return p.part_ml[((r + cc) * p.virt_heads + vg) * GW + h];
  };
  auto piece_o = [&](int j) -> const float* {
    if (j >= nd) return p.shared_o + (srow + (j - nd) * sstride) * D;
    return p.part_o + (((r + cf + j) * p.virt_heads + vg) * GW + h) * D;
  };
  float M = -INFINITY;
  for (int j0 = 0; j0 < npieces; j0 += 32) M = fmaxf(M, piece_ml(j0 + lane).x);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  constexpr int E = D / 32;  // dims per lane
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float Ls = 0.f;
  for (int j0 = 0; j0 < npieces; j0 += 32) {
    const float2 ml = piece_ml(j0 + lane);
    const float wgt = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
    Ls += wgt * ml.y;
    const int cnt = min(32, npieces - j0);
    // 8 pieces' loads in flight per lane; a piece of weight 0 (an empty
    // range, which wrote no partial) reads piece 0's slot and adds nothing
#pragma unroll 8
    for (int j = 0; j < cnt; ++j) {
      const float wj = __shfl_sync(0xffffffffu, wgt, j);
      const float* src = piece_o(wj == 0.f ? 0 : j0 + j) + lane * E;
      if constexpr (E == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] += wj * v.x;
        acc[1] += wj * v.y;
        acc[2] += wj * v.z;
        acc[3] += wj * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] += wj * v.x;
        acc[1] += wj * v.y;
      }
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
  const float inv = 1.f / Ls;
  const int row = __ldg(p.qsl + r);
  uint16_t* dst =
      p.out + (static_cast<long long>(row) * p.num_q_heads + vg * GW + h) * D + lane * E;
  if constexpr (E == 4) {
    uint2 ov;
    ov.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    ov.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = ov;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
}

// ------------------------------------------------------------------ host
#ifndef PKV_DECODE_MAX_STAGES
#define PKV_DECODE_MAX_STAGES 6
#endif
// Ring depth: as many stages as the CTA's share of the SM's shared memory
// holds, within these bounds (one stage per 16-key chunk of the slab's kv
// heads; more stages keep more bytes in flight per SM: 2 -> 3 stages of
// 64 KB took the mixed-step decode from 830 to 788 us)
constexpr int kDecodeMinStages = 2;
constexpr int kDecodeMaxStages = PKV_DECODE_MAX_STAGES;

// Consumer warps per SM the default split aims at (CTAs per SM = this / slab
// size, at least one): about the count that streamed fastest.
constexpr int kDecodeWarpsPerSm = 8;

// Decode slab of a shape: virtual heads per CTA and kv heads per CTA.
void decode_slab(int num_kv_heads, int group, int* vh, int* kh) {
  const int gw = decode_heads_per_warp(group);
  const int hg = group / gw;
  const int V = num_kv_heads * hg;
  int s = V <= kDecodeMaxSlab ? V : kDecodeMaxSlab;
  while (V % s || s % hg) --s;  // whole kv heads per slab, equal slabs
  *vh = s;
  *kh = s / hg;
}

template <int D, int GW>
static size_t decode_smem_bytes(int kh, int vh, int stages, int ctas_per_sm) {
  // More than 1 / (ctas_per_sm + 1) of an SM's shared memory (228 KB), so
  // that no SM ever holds more CTAs than the split assumes -- also when the
  // grid is launched early (programmatic dependent launch) and its first
  // CTAs land on the few SMs the previous kernel has already left.
  const size_t used = DecodeLayout<D, GW>(kh, vh, stages).total + 128;
  const size_t share = 228u * 1024u / (ctas_per_sm + 1) + 1024u;
  return used > share ? used : share;
}

template <int D, int GW, int SH>
static std::atomic<unsigned long long> g_decode_attr_done{0};

// Launch shape of one decode instantiation on one device for a slab shape,
// worked out once (the occupancy query costs microseconds of host time per
// call, which short steps would pay on every launch).
struct DecodePrep {
  int dev, kh, vh, num_sms, stages;
  long long splits;
  size_t smem;
};

template <int D, int GW, int SH>
static std::vector<DecodePrep> g_decode_prep;
static std::mutex g_decode_prep_mu;

template <int D, int GW, int SH>
static cudaError_t decode_prepare(int kh, int vh, int num_sms, long long* splits, int* stages,
                                  size_t* smem) {
  auto kern = decode_kernel<D, GW, SH>;
  cudaError_t e = smem_attr_once(kern, 227 * 1024, g_decode_attr_done<D, GW, SH>);
  if (e != cudaSuccess) return e;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lock(g_decode_prep_mu);
    for (const DecodePrep& d : g_decode_prep<D, GW, SH>)
      if (d.dev == dev && d.kh == kh && d.vh == vh && d.num_sms == num_sms) {
        *stages = d.stages;
        *smem = d.smem;
        if (splits) *splits = d.splits;
        return cudaSuccess;
      }
  }
  int want = kDecodeWarpsPerSm / vh;
  if (want < 1) want = 1;
  const size_t least = DecodeLayout<D, GW>(kh, vh, kDecodeMinStages).total + 128;
  int fit = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, kern, (vh + 1) * 32, least);
  if (e != cudaSuccess) return e;
  const int ctas = fit < want ? (fit < 1 ? 1 : fit) : want;
  // deepest ring within the CTA's share (the SM's 228 KB less 1 KB reserved per CTA)
  const size_t budget = 228u * 1024u / ctas - 1024u;
  int S = kDecodeMinStages;
  while (S < kDecodeMaxStages && DecodeLayout<D, GW>(kh, vh, S + 1).total + 128 <= budget) ++S;
  *stages = S;
  *smem = decode_smem_bytes<D, GW>(kh, vh, S, ctas);
  const long long full = static_cast<long long>(num_sms) * ctas;
  if (splits) *splits = full;
  std::lock_guard<std::mutex> lock(g_decode_prep_mu);
  g_decode_prep<D, GW, SH>.push_back(DecodePrep{dev, kh, vh, num_sms, S, full, *smem});
  return cudaSuccess;
}

template <int D, int GW, int SH>
static cudaError_t launch_decode_t(const DecodeParams& p, const CUtensorMap& kv_map,
                                   int num_sms, cudaStream_t stream, void** trace) {
  size_t smem = 0;
  DecodeParams q = p;
  cudaError_t e = decode_prepare<D, GW, SH>(p.slab_kh, p.slab_vh, num_sms, nullptr, &q.stages, &smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(p.splits), static_cast<unsigned>(p.virt_heads / p.slab_vh));
  e = launch_pdl(decode_kernel<D, GW, SH>, grid, dim3((p.slab_vh + 1) * 32), smem, stream, kv_map, q);
  if (e == cudaSuccess && trace) e = cudaEventRecord(static_cast<cudaEvent_t>(trace[3]), stream);
  if (e != cudaSuccess) return e;
  return launch_pdl(combine_kernel<D, GW>,
                    dim3(static_cast<unsigned>(p.splits + p.shared_num),
                         static_cast<unsigned>(p.virt_heads)),
                    dim3(GW * 32), 0, stream, p);
}

// Calls F<D, GW, SH>::run(args...) for the instantiated shapes: head_dim 64 or
// 128, 1, 2 or 4 heads per warp, blocks of 8, 16 or 32 tokens.
template <template <int, int, int> class F, typename... A>
static cudaError_t decode_dispatch(int head_dim, int gw, int sh, A&&... args) {
#define PKV_DECODE_CASE(D_, GW_, SH_) \
  if (head_dim == D_ && gw == GW_ && sh == SH_) return F<D_, GW_, SH_>::run(args...);
#define PKV_DECODE_SH(D_, GW_) \
  PKV_DECODE_CASE(D_, GW_, 3) PKV_DECODE_CASE(D_, GW_, 4) PKV_DECODE_CASE(D_, GW_, 5)
  PKV_DECODE_SH(128, 4) PKV_DECODE_SH(128, 2) PKV_DECODE_SH(128, 1)
  PKV_DECODE_SH(64, 4) PKV_DECODE_SH(64, 2) PKV_DECODE_SH(64, 1)
#undef PKV_DECODE_SH
#undef PKV_DECODE_CASE
  return cudaErrorInvalidValue;
}

template <int D, int GW, int SH>
struct PrepareOp {
  static cudaError_t run(int kh, int vh, int sms, long long* splits) {
    size_t smem = 0;
    int stages = 0;
    return decode_prepare<D, GW, SH>(kh, vh, sms, splits, &stages, &smem);
  }
};

template <int D, int GW, int SH>
struct LaunchOp {
  static cudaError_t run(const DecodeParams& p, const CUtensorMap& m, int sms, cudaStream_t s,
                         void** t) {
    return launch_decode_t<D, GW, SH>(p, m, sms, s, t);
  }
};

cudaError_t decode_full_wave_splits(int head_dim, int num_kv_heads, int group, int block_shift,
                                    int num_sms, long long* splits) {
  int vh = 0, kh = 0;
  decode_slab(num_kv_heads, group, &vh, &kh);
  return decode_dispatch<PrepareOp>(head_dim, decode_heads_per_warp(group), block_shift, kh, vh,
                                    num_sms, splits);
}


cudaError_t launch_decode(const AttnArgs& a, const AttnWorkspace& ws, const CUtensorMap& kv_map,
                          long long splits, int num_sms, cudaStream_t stream, void** trace) {
  const int group = a.num_q_heads / a.num_kv_heads;
  const int gw = decode_heads_per_warp(group);
  DecodeParams p;
  p.q = a.q;
  p.q_stride = a.q_stride;
  p.out = a.out;
  p.block_table = a.block_table;
  p.max_blocks = a.max_blocks;
  p.seq_lens = a.seq_lens;
  p.qsl = a.qsl;
  p.num_reqs = a.num_reqs;
  p.num_q_heads = a.num_q_heads;
  p.num_blocks = a.num_blocks;
  p.head_groups = group / gw;
  p.virt_heads = a.num_kv_heads * p.head_groups;
  decode_slab(a.num_kv_heads, group, &p.slab_vh, &p.slab_kh);
  p.splits = splits;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.dec_prefix = ws.dec_prefix;
  p.hdr = ws.hdr;
  p.part_ml = ws.part_ml;
  p.part_o = ws.part_o;
  p.bound = ws.bound;
  p.shared_first = a.shared_first;
  p.shared_num = a.shared_num;
  p.shared_chunks = a.shared_len / kChunkKeys;
  p.shared_pieces = a.shared_pieces;
  p.shared_use = ws.casc_use;
  p.shared_ml = ws.casc_ml;
  p.shared_o = ws.casc_o;
  return decode_dispatch<LaunchOp>(a.head_dim, gw, a.block_shift, p, kv_map, num_sms, stream,
                                   trace);
}

cudaError_t read_errors_decode(uint32_t* out, bool clear) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_errors_decode, sizeof(v));
  if (e != cudaSuccess) return e;
  *out |= v;
  if (clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_errors_decode, &z, sizeof(z));
  }
  return e;
}

}  // namespace pkv
