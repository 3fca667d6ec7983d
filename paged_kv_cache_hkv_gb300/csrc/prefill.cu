// Causal chunked-prefill attention over the paged cache on the 5th-generation
// tensor cores (tcgen05, TMEM accumulators, TMA operands), sm_103a.
//
// What it computes ("vllm v1 源码精读（三）" §4.2; "Inside vLLM" §3.4-3.5):
// request r has c = num_computed tokens already cached and n > 1 new tokens
// (a prompt chunk). Its i-th new token, at absolute position c + i, attends
// keys 0 .. c + i of its own sequence -- the cached prefix and the chunk up to
// itself -- all read through the block table (the chunk's own K/V was written
// into the pool first).
//
// Work item = (request, tile of 128 query rows, kv head). The 128 rows of a
// tile are the G = Hq/Hkv q heads of one kv head for 128/G consecutive
// queries, so every K/V tile feeds all G heads (GQA). For each tile of 128
// keys (8 pool blocks):
//   S = Q K^T        tcgen05.mma M=128 N=128, A = Q (smem), B = K (smem)
//   softmax          each thread owns one row: tcgen05.ld of S, causal
//                    mask, running max/sum in base 2, P rounded to bf16 into
//                    smem, O rescaled in TMEM when the max moves
//   O += P V         tcgen05.mma M=128 N=D, A = P (smem), B = V (smem)
// Q, K and V arrive by TMA with 128-byte swizzle (one 16-token block of one
// kv head per copy), the layout the tensor core reads. Accumulators: S in
// TMEM columns [0, 128), O in [128, 128 + D).
//
// Every wait is bounded; on a timeout the kernel records
// PKV_DEVERR_TIMEOUT, drains its copies, frees TMEM and returns.
#include "common.cuh"
#include "launch.h"

namespace pkv {

static __device__ uint32_t g_errors_prefill;

namespace tc {

// Shared-memory matrix descriptor (tcgen05), 128-byte swizzle.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) |  // version
         (2ull << 61);                                                         // SWIZZLE_128B
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator,
// A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

}  // namespace tc

constexpr int kTileM = 128;  // query rows (query x head) per tile
constexpr int kTileN = 128;  // keys per tile (8 blocks)
constexpr uint32_t kTmemCols = 256;

template <int D>
struct PrefillLayout {
  static constexpr int DH = D / 64;  // 64-element (128-byte) column chunks
  static constexpr uint32_t kChunk = kTileM * 128;  // one 128-row x 128-byte chunk: 16 KB
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + DH * kChunk;  // 2 stages
  static constexpr uint32_t kV = kK + 2 * DH * kChunk;
  static constexpr uint32_t kP = kV + 2 * DH * kChunk;  // 2 chunks (128 keys)
  static constexpr uint32_t kBar = kP + 2 * kChunk;
  static constexpr uint32_t kBytes = kBar + 128;
  static constexpr uint32_t kAlloc = kBytes + 1024;  // room to align the base
};

struct PrefillParams {
  uint16_t* out;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* seq_lens;
  const int32_t* qsl;
  const int32_t* num_computed;
  int num_q_heads, num_kv_heads, group, num_blocks;
  float scale_log2;
  uint32_t* hdr;
  const int32_t* pf_req;
  const int32_t* pf_prefix;
};

struct PrefillShared {
  uint64_t q_full;
  uint64_t kv_full[2];
  uint64_t s_full;
  uint64_t o_full;
  uint32_t tmem;
  int item;
  int abort;
  uint32_t mask[2];
};

template <int D>
__global__ void __launch_bounds__(128, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
                   const PrefillParams p) {
  using Lay = PrefillLayout<D>;
  constexpr int DH = Lay::DH;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  PrefillShared& sh = *reinterpret_cast<PrefillShared*>(gbase + Lay::kBar);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int G = p.group, QT = kTileM / G;

  if (tid == 0) {
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.kv_full[0], 1);
    mbar_init(&sh.kv_full[1], 1);
    mbar_init(&sh.s_full, 1);
    mbar_init(&sh.o_full, 1);
    sh.abort = 0;
    fence_barrier_init();
    prefetch_tensormap(&kv_map);
    prefetch_tensormap(&q_map);
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sh.tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh.tmem;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t t_s = tmem + lane_base;         // S: columns [0, 128)
  const uint32_t t_o = tmem + lane_base + 128u;  // O: columns [128, 128 + D)

  constexpr uint32_t idesc_qk = tc::idesc_bf16(kTileM, kTileN, 0);
  constexpr uint32_t idesc_pv = tc::idesc_bf16(kTileM, D, 1);
  const uint32_t n_items = p.hdr[kHdrPrefillItems];
  const int n_req = static_cast<int>(p.hdr[kHdrPrefillReqs]);

  uint32_t n_q = 0, n_s = 0, n_o = 0, tiles = 0;  // completed phases per barrier
  bool failed = false;

  while (true) {
    if (tid == 0) sh.item = static_cast<int>(atomicAdd(&p.hdr[kHdrPrefillNext], 1u));
    __syncthreads();
    const int item = sh.item;
    if (item >= static_cast<int>(n_items)) break;

    // ---- which (request, tile, kv head)
    const int k = upper_index(p.pf_prefix, n_req, item);
    const int r = __ldg(p.pf_req + k);
    const int local = item - __ldg(p.pf_prefix + k);
    const int g = local % p.num_kv_heads;
    const int c = __ldg(p.num_computed + r);
    const int q0 = __ldg(p.qsl + r);
    const int n = __ldg(p.qsl + r + 1) - q0;
    const int ntile = (n + QT - 1) / QT;
    const int mt = ntile - 1 - local / p.num_kv_heads;  // longest tiles first
    const int i0 = mt * QT;
    const int i_last = min(i0 + QT, n) - 1;
    const int kv_len = c + i_last + 1;
    const int nkv = (kv_len + kTileN - 1) / kTileN;
    const long long bt_row = static_cast<long long>(r) * p.max_blocks;

    auto issue_tile = [&](int kt, int st) {  // thread 0 only
      const int left = kv_len - kt * kTileN;
      const int nb = min(8, (left + kBlockSize - 1) / kBlockSize);
      uint32_t mask = 0, bytes = 0;
      int phys[8];
      for (int b = 0; b < nb; ++b) {
        phys[b] = __ldg(p.block_table + bt_row + kt * 8 + b);
        if (phys[b] >= 0 && phys[b] < p.num_blocks) {
          mask |= 1u << b;
          bytes += 2u * DH * 2048u;
        } else {
          atomicOr(&g_errors_prefill, kErrBlockRange);
        }
      }
      sh.mask[st] = mask;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&sh.kv_full[st], bytes);
      for (int b = 0; b < nb; ++b) {
        if (!(mask >> b & 1u)) continue;
#pragma unroll
        for (int dh = 0; dh < DH; ++dh) {
          tma_load_3d(gbase + Lay::kK + (st * DH + dh) * Lay::kChunk + b * 2048, &kv_map, dh * 64,
                      g, phys[b] * 32, &sh.kv_full[st]);
          tma_load_3d(gbase + Lay::kV + (st * DH + dh) * Lay::kChunk + b * 2048, &kv_map, dh * 64,
                      g, phys[b] * 32 + 16, &sh.kv_full[st]);
        }
      }
    };

    if (tid == 0) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&sh.q_full, DH * Lay::kChunk);
#pragma unroll
      for (int dh = 0; dh < DH; ++dh)
        tma_load_3d(gbase + Lay::kQ + dh * Lay::kChunk, &q_map, dh * 64, g * G, q0 + i0,
                    &sh.q_full);
      issue_tile(0, tiles & 1);
      if (nkv > 1) issue_tile(1, (tiles + 1) & 1);
    }

    // this thread's row: query i0 + tid / G, head g * G + tid % G
    const int qi = i0 + tid / G;
    const int lim = min(c + qi, kv_len - 1);  // last key this row may see
    float m_run = -INFINITY, l_run = 0.f;

    for (int kt = 0; kt < nkv; ++kt) {
      const uint32_t tg = tiles + kt;
      const int st = tg & 1;
      bool ok = mbar_wait(&sh.kv_full[st], (tg >> 1) & 1u);
      if (kt == 0) ok = mbar_wait(&sh.q_full, n_q & 1u) && ok;
      const uint32_t mask = sh.mask[st];
      {  // zero the V rows of keys that are past kv_len or were not loaded
        const int j = kt * kTileN + tid;
        if (j >= kv_len || !(mask >> (tid >> 4) & 1u)) {
#pragma unroll
          for (int dh = 0; dh < DH; ++dh) {
            uint4* row = reinterpret_cast<uint4*>(gbase + Lay::kV + (st * DH + dh) * Lay::kChunk +
                                                  tid * 128);
#pragma unroll
            for (int x = 0; x < 8; ++x) row[x] = make_uint4(0, 0, 0, 0);
          }
        }
      }
      fence_proxy_async_smem();
      if (!ok) sh.abort = 1;
      __syncthreads();
      if (sh.abort) {
        failed = true;
        break;
      }
      if (tid == 0) {  // S = Q K^T
        tc::fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * Lay::kChunk + (kk & 3) * 32;
          const uint64_t a = tc::sw128_desc(base + Lay::kQ + off, 16, 1024);
          const uint64_t b = tc::sw128_desc(base + Lay::kK + st * DH * Lay::kChunk + off, 16, 1024);
          tc::mma_bf16(tmem, a, b, idesc_qk, kk > 0);
        }
        tc::commit(&sh.s_full);
      }
      ok = mbar_wait(&sh.s_full, n_s & 1u);
      ++n_s;
      tc::fence_after_sync();

      // ---- softmax over this row's 128 scores
      float s[kTileN];
#pragma unroll
      for (int q = 0; q < 4; ++q) tc::ld32(t_s + q * 32, s + q * 32);
      tc::wait_ld();
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < kTileN; ++j) {
        const int key = kt * kTileN + j;
        const bool vis = key <= lim && (mask >> (j >> 4) & 1u);
        s[j] = vis ? s[j] * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, s[j]);
      }
      const float m_new = fmaxf(m_run, mx);
      const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
      const float msub = (m_new == -INFINITY) ? 0.f : m_new;

      if (kt > 0) {  // PV of the previous tile must be done: O and P are reused
        ok = mbar_wait(&sh.o_full, n_o & 1u) && ok;
        ++n_o;
        tc::fence_after_sync();
        if (tid == 0 && kt + 1 < nkv) issue_tile(kt + 1, (tg + 1) & 1);
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            float o[32];
            tc::ld32(t_o + q * 32, o);
            tc::wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] *= alpha;
            tc::st32(t_o + q * 32, o);
          }
        }
      }
      float psum = 0.f;
      unsigned char* prow = gbase + Lay::kP + tid * 128;
#pragma unroll
      for (int c8 = 0; c8 < kTileN / 8; ++c8) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a0 = exp2f(s[c8 * 8 + 2 * e] - msub);
          const float a1 = exp2f(s[c8 * 8 + 2 * e + 1] - msub);
          w[e] = pack_bf16x2(a0, a1);
          psum += bf16_lo(w[e]) + bf16_hi(w[e]);
        }
        const int chunk = c8 & 7, half = c8 >> 3;
        *reinterpret_cast<uint4*>(prow + half * Lay::kChunk + ((chunk ^ (tid & 7)) << 4)) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
      l_run = l_run * alpha + psum;
      m_run = m_new;
      fence_proxy_async_smem();
      tc::wait_st();
      tc::fence_before_sync();
      if (!ok) sh.abort = 1;
      __syncthreads();
      if (sh.abort) {
        failed = true;
        break;
      }
      if (tid == 0) {  // O += P V
        tc::fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          const uint64_t a = tc::sw128_desc(base + Lay::kP + (kk >> 2) * Lay::kChunk + (kk & 3) * 32,
                                            16, 1024);
          const uint64_t b = tc::sw128_desc(base + Lay::kV + st * DH * Lay::kChunk + kk * 2048,
                                            Lay::kChunk, 1024);
          tc::mma_bf16(tmem + 128u, a, b, idesc_pv, (kt > 0 || kk > 0) ? 1u : 0u);
        }
        tc::commit(&sh.o_full);
      }
    }
    if (failed) break;

    // ---- epilogue: O / l -> bf16 rows of the output
    bool ok = mbar_wait(&sh.o_full, n_o & 1u);
    ++n_o;
    tc::fence_after_sync();
    if (!ok) sh.abort = 1;
    const float inv = 1.f / l_run;
    const bool store = qi < n;
    uint16_t* dst = p.out + (static_cast<long long>(q0 + qi) * p.num_q_heads + g * G + tid % G) * D;
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
      float o[32];
      tc::ld32(t_o + q * 32, o);
      tc::wait_ld();
      if (store) {
        uint4* d4 = reinterpret_cast<uint4*>(dst + q * 32);
#pragma unroll
        for (int x = 0; x < 4; ++x)
          d4[x] = make_uint4(pack_bf16x2(o[8 * x] * inv, o[8 * x + 1] * inv),
                             pack_bf16x2(o[8 * x + 2] * inv, o[8 * x + 3] * inv),
                             pack_bf16x2(o[8 * x + 4] * inv, o[8 * x + 5] * inv),
                             pack_bf16x2(o[8 * x + 6] * inv, o[8 * x + 7] * inv));
      }
    }
    tc::fence_before_sync();
    __syncthreads();
    tiles += nkv;
    ++n_q;
    if (sh.abort) {
      failed = true;
      break;
    }
  }

  if (failed) {
    if (tid == 0) {
      atomicOr(&g_errors_prefill, kErrTimeout);
      // let copies still in flight land before the shared memory goes away
      mbar_wait(&sh.kv_full[0], 0, kDrainLimitNs);
      mbar_wait(&sh.kv_full[1], 0, kDrainLimitNs);
      mbar_wait(&sh.q_full, n_q & 1u, kDrainLimitNs);
    }
    __syncthreads();
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

template <int D>
static cudaError_t launch_prefill_t(const PrefillParams& p, const CUtensorMap& kv_map,
                                    const CUtensorMap& q_map, int grid, cudaStream_t stream) {
  auto kern = prefill_kernel<D>;
  const int smem = static_cast<int>(PrefillLayout<D>::kAlloc);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, 128, smem, stream>>>(kv_map, q_map, p);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const AttnArgs& a, const AttnWorkspace& ws, const CUtensorMap& kv_map,
                           const CUtensorMap& q_map, int num_sms, cudaStream_t stream) {
  PrefillParams p;
  p.out = a.out;
  p.block_table = a.block_table;
  p.max_blocks = a.max_blocks;
  p.seq_lens = a.seq_lens;
  p.qsl = a.qsl;
  p.num_computed = a.num_computed;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.num_blocks = a.num_blocks;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.hdr = ws.hdr;
  p.pf_req = ws.pf_req;
  p.pf_prefix = ws.pf_prefix;
  // upper bound of work items from the host hints: every row can be in a tile
  const long long tile_q = kTileM / p.group;
  const long long max_items =
      ((static_cast<long long>(a.num_tokens) + tile_q - 1) / tile_q + a.num_reqs) * a.num_kv_heads;
  const int grid = static_cast<int>(max_items < num_sms ? max_items : num_sms);
  if (grid <= 0) return cudaSuccess;
  if (a.head_dim == 128) return launch_prefill_t<128>(p, kv_map, q_map, grid, stream);
  if (a.head_dim == 64) return launch_prefill_t<64>(p, kv_map, q_map, grid, stream);
  return cudaErrorInvalidValue;
}

cudaError_t read_errors_prefill(uint32_t* out, bool clear) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_errors_prefill, sizeof(v));
  if (e != cudaSuccess) return e;
  *out |= v;
  if (clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_errors_prefill, &z, sizeof(z));
  }
  return e;
}

}  // namespace pkv
