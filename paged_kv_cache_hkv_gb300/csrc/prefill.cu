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
// queries, so every K/V tile feeds all G heads (GQA). The item's key tiles
// (128 keys = 8 chunks of 16 keys: 8 blocks of 16 tokens, 4 of 32 or 16 of
// 8) are split between two softmax warpgroups:
// warpgroup w takes tiles w, w+2, ... with its own accumulators
// (TMEM columns [256w, 256w+128) for S, [256w+128, 256w+128+D) for O).
// Two copy warps stream K and V tiles through a 2-stage ring by TMA (128-byte
// swizzle, one 16-key chunk of one kv head per copy, two copies of 8 rows
// for 8-token blocks) and one MMA thread issues
//   S_w = Q K^T      tcgen05.mma M=128 N=128, A = Q (smem), B = K (smem)
//   O_w += P_w V     tcgen05.mma M=128 N=D, A = P_w (smem), B = V (smem)
// while the warpgroups run the softmax: each thread owns one row, reads S
// with tcgen05.ld, applies the causal mask, keeps a base-2 running max
// (rescaling O in TMEM only when it grows by more than 2^8) and sum, and
// writes P as bf16 into its warpgroup's smem buffer. One warpgroup's softmax
// runs while the tensor core works on the other's tiles; each warpgroup's
// next K/V tile streams in by TMA while the other one computes. At the end the two
// partial (max, sum, O) are merged and each warpgroup writes half of the
// output columns.
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
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }



// 16 consecutive 32-bit columns of this thread's TMEM lane (asynchronous:
// the registers hold the data only after wait16 on them).
__device__ __forceinline__ void ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// 32 consecutive 32-bit columns (asynchronous, like ld16).
__device__ __forceinline__ void ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// tcgen05.wait::ld pinning 32 loaded registers (see wait16).
__device__ __forceinline__ void wait32(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// tcgen05.wait::ld with the loaded registers as operands, so that no use of
// them can be scheduled before the wait.
__device__ __forceinline__ void wait16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

__device__ __forceinline__ void st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

}  // namespace tc

constexpr int kTileM = 128;  // query rows (query x head) per tile
constexpr int kTileN = 128;  // keys per tile (8 blocks)
constexpr int kStages = 2;   // K and V tile rings: tile kt uses slot (tiles + kt) % 2
constexpr uint32_t kTmemCols = 512;
constexpr int kThreads = 352;  // 2 softmax warpgroups + MMA warp + K-copy warp + V-copy warp
constexpr int kIssuer = 256;   // thread that issues the MMAs (warp 8, lane 0)
constexpr float kRescaleLog2 = 8.f;  // lazy rescale threshold (powers of two)

template <int D>
struct PrefillLayout {
  static constexpr int DH = D / 64;                 // 64-element (128-byte) column chunks
  static constexpr uint32_t kChunk = kTileM * 128;  // 128 rows x 128 bytes = 16 KB
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kTileKV = DH * kChunk;     // K (or V) of one 128-key tile
  static constexpr uint32_t kK = kQ + DH * kChunk;     // K ring, kStages tiles
  static constexpr uint32_t kV = kK + kStages * kTileKV;  // V ring, kStages tiles
  static constexpr uint32_t kP = kV + kStages * kTileKV;  // P of warpgroup w: 2 chunks each
  static constexpr uint32_t kBar = kP + 2 * 2 * kChunk;
  static constexpr uint32_t kBytes = kBar + 256;
  static constexpr uint32_t kAlloc = kBytes + 1024;  // room to align the base
  static_assert(kAlloc <= 232448, "shared memory");
};

struct PrefillParams {
  uint16_t* out;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* seq_lens;
  const int32_t* qsl;
  const int32_t* num_computed;
  int num_q_heads, num_kv_heads, group, num_blocks;
  int block_shift;  // log2 of the tokens per cache block (3, 4 or 5)
  float scale_log2;
  uint32_t* hdr;
  const int32_t* pf_req;
  const int32_t* pf_prefix;
};

struct PrefillShared {
  uint64_t q_full;
  uint64_t k_full[kStages];
  uint64_t v_full[kStages];
  uint64_t s_full[2];   // S of warpgroup w computed
  uint64_t p_ready[2];  // P of warpgroup w in smem, V rows cleaned (128 arrivals)
  uint64_t pv_done[2];  // O of warpgroup w updated
  uint64_t drain;
  uint32_t tmem;
  int item;
  int abort;
};

// Bounded wait that also gives up once another thread has flagged an abort.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort) return false;
      if (global_ns() - t0 > kWaitLimitNs) {
        *abort = 1;
        atomicOr(&g_errors_prefill, kErrTimeout);
        return false;
      }
    }
  }
}

// Work item: (request, 128-row query tile, kv head). Two softmax warpgroups
// split the item's key tiles (warpgroup w takes tiles w, w+2, ...), each with
// its own S and O accumulators in TMEM and its own running max and sum; one
// thread streams K/V tiles through a 3-stage ring by TMA and issues every
// MMA: S_w = Q K^T into TMEM, then O_w += P_w V with P_w (bf16) read from
// TMEM where the softmax wrote it over S_w. At the end the two partial
// results are merged (log-sum-exp) and each warpgroup writes half of the
// output columns.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
                   const PrefillParams p) {
  using Lay = PrefillLayout<D>;
  constexpr int DH = Lay::DH;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  PrefillShared& sh = *reinterpret_cast<PrefillShared*>(gbase + Lay::kBar);
  volatile int* abort_flag = &sh.abort;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int wg = tid >> 7;          // 0, 1 softmax warpgroups; 2 = issuer warp
  const int row = tid & 127;        // query row of this softmax thread (TMEM lane)
  const int G = p.group, QT = kTileM / G;

  if (tid == kIssuer) {
    mbar_init(&sh.q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sh.k_full[i], 1);
      mbar_init(&sh.v_full[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.p_ready[i], 128);
      mbar_init(&sh.pv_done[i], 1);
    }
    mbar_init(&sh.drain, 1);
    sh.abort = 0;
    fence_barrier_init();
    prefetch_tensormap(&kv_map);
    prefetch_tensormap(&q_map);
  }
  if (warp == 8) {
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
  constexpr uint32_t idesc_qk = tc::idesc_bf16(kTileM, kTileN, 0);
  constexpr uint32_t idesc_pv = tc::idesc_bf16(kTileM, D, 1);
  const uint32_t n_items = p.hdr[kHdrPrefillItems];
  const int n_req = static_cast<int>(p.hdr[kHdrPrefillReqs]);

  // phase counters, identical in every thread
  uint32_t n_q = 0, tiles = 0, cnt[2] = {0, 0};
  uint32_t drains = 0;

  while (true) {
    if (tid == kIssuer) sh.item = static_cast<int>(atomicAdd(&p.hdr[kHdrPrefillNext], 1u));
    __syncthreads();
    const int item = sh.item;
    if (item >= static_cast<int>(n_items) || sh.abort) break;

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
    auto stage_of = [&](int kt) { return static_cast<int>((tiles + kt) % kStages); };
    auto stage_par = [&](int kt) { return ((tiles + kt) / kStages) & 1u; };
    // block table entry e of the request if it holds keys < kv_len and its id
    // is in the pool, else -1
    const int bsh = p.block_shift;
    auto entry_id = [&](int e) -> int {
      if ((e << bsh) >= kv_len) return -1;
      const int id = __ldg(p.block_table + bt_row + e);
      return (id >= 0 && id < p.num_blocks) ? id : -1;
    };
    // chunk b (keys 16b .. 16b+15) of tile kt holds keys < kv_len, all of
    // them in blocks of the pool
    auto chunk_ok = [&](int kt, int b) -> bool {
      const int k0 = kt * kTileN + b * kChunkKeys;
      if (k0 >= kv_len) return false;
      if (bsh == 4) return entry_id(k0 >> 4) >= 0;
      if (bsh == 5) return entry_id(k0 >> 5) >= 0;
      return entry_id(k0 >> 3) >= 0 && (k0 + 8 >= kv_len || entry_id((k0 >> 3) + 1) >= 0);
    };

    if (warp >= 8) {
      // ================= producer warps, each with in-order blocking waits:
      //   warp 9:  K(kt) TMA copies, once S(kt - 2) is done (its K slot is free)
      //   warp 10: V(kt) TMA copies, once PV(kt - 2) is done (its V slot is free)
      //   warp 8:  MMAs: S(kt) once K(kt) landed and softmax(kt - 2) read S_w;
      //            PV(kt) once softmax(kt) wrote P_w and V(kt) landed
      // Lane (chunk b, d half dh), lanes 0 .. 8*DH-1, issues the copies of
      // that chunk (one of 16 rows, or two of 8 rows for 8-token blocks); the
      // block ids of a 32-entry window of the block table sit in the lanes'
      // registers.
      const int ln = tid & 31;
      auto phase = [&](int kt) { return (cnt[kt & 1] + (kt >> 1)) & 1u; };
      bool ok = true;
      if (warp == 9 || warp == 10) {
        const int is_v = warp == 10;
        if (!is_v && ln == 0) {
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(&sh.q_full, DH * Lay::kChunk);
#pragma unroll
          for (int dh = 0; dh < DH; ++dh)
            tma_load_3d(gbase + Lay::kQ + dh * Lay::kChunk, &q_map, dh * 64, g * G, q0 + i0,
                        &sh.q_full);
        }
        int win_base = -1000000, win_val = -1;
        for (int kt = 0; ok && kt < nkv; ++kt) {
          if (kt >= kStages) {  // the slot's previous tile (kt - 2) must be done with it
            ok = wait_or_abort(is_v ? &sh.pv_done[kt & 1] : &sh.s_full[kt & 1], phase(kt - 2),
                               abort_flag);
            if (!ok) break;
          }
          const int st = stage_of(kt);
          const int E = kTileN >> bsh;  // table entries per tile
          if (kt * E + E > win_base + 32) {
            win_base = kt * E;
            const int e = win_base + ln;
            win_val = entry_id(e);
            if (!is_v && (e << bsh) < kv_len && win_val < 0)
              atomicOr(&g_errors_prefill, kErrBlockRange);
          }
          const int b = (ln / DH) & 7, dh = ln % DH;
          // pool rows of one kv head: (block * 2 + k|v) * B + offset
          int id0, id1 = -1, row0, row1 = 0;
          if (bsh == 4) {
            id0 = __shfl_sync(0xffffffffu, win_val, kt * 8 + b - win_base);
            row0 = id0 * 32 + (is_v ? 16 : 0);
          } else if (bsh == 5) {
            id0 = __shfl_sync(0xffffffffu, win_val, kt * 4 + (b >> 1) - win_base);
            row0 = id0 * 64 + (b & 1) * 16 + (is_v ? 32 : 0);
          } else {
            id0 = __shfl_sync(0xffffffffu, win_val, kt * 16 + 2 * b - win_base);
            id1 = __shfl_sync(0xffffffffu, win_val, kt * 16 + 2 * b + 1 - win_base);
            row0 = id0 * 16 + (is_v ? 8 : 0);
            row1 = id1 * 16 + (is_v ? 8 : 0);
          }
          const bool mine0 = ln < 8 * DH && id0 >= 0;
          const bool mine1 = ln < 8 * DH && id1 >= 0;
          const uint32_t bytes = bsh == 3 ? (mine0 ? 1024u : 0u) + (mine1 ? 1024u : 0u)
                                         : (mine0 ? 2048u : 0u);
          const uint32_t tx = __reduce_add_sync(0xffffffffu, bytes);
          uint64_t* bar = is_v ? &sh.v_full[st] : &sh.k_full[st];
          if (ln == 0) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar, tx);
          }
          __syncwarp();
          unsigned char* dst = gbase + (is_v ? Lay::kV : Lay::kK) + st * Lay::kTileKV +
                               dh * Lay::kChunk + b * 2048;
          if (mine0) tma_load_3d(dst, &kv_map, dh * 64, g, row0, bar);
          if (mine1) tma_load_3d(dst + 1024, &kv_map, dh * 64, g, row1, bar);
        }
      } else if (warp == 8 && ln == 0) {
        auto issue_s = [&](int kt) {  // S_w = Q K^T for tile kt
          const int w = kt & 1, st = stage_of(kt);
          tc::fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * Lay::kChunk + (kk & 3) * 32;
            const uint64_t a = tc::sw128_desc(base + Lay::kQ + off, 16, 1024);
            const uint64_t b = tc::sw128_desc(base + Lay::kK + st * Lay::kTileKV + off, 16, 1024);
            tc::mma_bf16(tmem + w * 256u, a, b, idesc_qk, kk > 0);
          }
          tc::commit(&sh.s_full[w]);
        };
        auto issue_pv = [&](int kt) {  // O_w += P_w V for tile kt, P_w from smem
          const int w = kt & 1, st = stage_of(kt);
          tc::fence_after_sync();
          const uint32_t vbase = base + Lay::kV + st * Lay::kTileKV;
          const uint32_t pbase = base + Lay::kP + w * 2 * Lay::kChunk;
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk) {
            const uint64_t a =
                tc::sw128_desc(pbase + (kk >> 2) * Lay::kChunk + (kk & 3) * 32, 16, 1024);
            const uint64_t b = tc::sw128_desc(vbase + kk * 2048, Lay::kChunk, 1024);
            tc::mma_bf16(tmem + w * 256u + 128u, a, b, idesc_pv, (kt >= 2 || kk > 0) ? 1u : 0u);
          }
          tc::commit(&sh.pv_done[w]);
        };
        ok = wait_or_abort(&sh.q_full, n_q & 1u, abort_flag);
        for (int kt = 0; ok && kt < 2 && kt < nkv; ++kt) {
          ok = wait_or_abort(&sh.k_full[stage_of(kt)], stage_par(kt), abort_flag);
          if (ok) issue_s(kt);
        }
        // after softmax(kt): S(kt + 2) first (the warpgroup's next softmax
        // waits on it), then PV(kt) (needed only before its next P write)
        for (int kt = 0; ok && kt < nkv; ++kt) {
          ok = wait_or_abort(&sh.p_ready[kt & 1], phase(kt), abort_flag);
          if (ok && kt + 2 < nkv) {
            ok = wait_or_abort(&sh.k_full[stage_of(kt + 2)], stage_par(kt + 2), abort_flag);
            if (ok) issue_s(kt + 2);
          }
          if (ok) ok = wait_or_abort(&sh.v_full[stage_of(kt)], stage_par(kt), abort_flag);
          if (!ok) break;
          issue_pv(kt);
        }
        if (!ok) {  // let issued MMAs finish before anything is torn down
          tc::commit(&sh.drain);
          mbar_wait(&sh.drain, drains & 1u, kDrainLimitNs);
        }
      }
      if (warp == 8) drains += __shfl_sync(0xffffffffu, ok ? 0u : 1u, 0);
    } else if (wg < 2) {
      // ================= softmax warpgroup wg: tiles wg, wg + 2, ...
      const int qi = i0 + row / G;              // query of this row
      const int lim = min(c + qi, kv_len - 1);  // last key this row may see
      const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const uint32_t t_s = tmem + lane_base + wg * 256u;
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      int nmine = 0;
      const int lane = tid & 31;
      // block ids of this warpgroup's next tile, loaded one tile ahead by lanes 0..7
      auto load_ids = [&](int kt) -> int {
        return (lane < 8 && kt < nkv && chunk_ok(kt, lane)) ? 1 : -1;
      };
      int next_id = load_ids(wg);
      for (int kt = wg; ok && kt < nkv; kt += 2, ++nmine) {
        const uint32_t ph = cnt[wg] + (kt >> 1);
        const uint32_t mask = __ballot_sync(0xffffffffu, next_id >= 0) & 0xFFu;
        next_id = load_ids(kt + 2);
        ok = wait_or_abort(&sh.s_full[wg], ph & 1u, abort_flag);
        if (!ok) break;
        tc::fence_after_sync();
        // a tile every row sees in full needs no mask; otherwise column j is
        // visible iff j <= jlim and its 16-key chunk was loaded (chunk c =
        // columns 16c .. 16c+15)
        const bool full = kt * kTileN + kTileN - 1 <= c + i0 && mask == 0xFFu;
        const int jlim = lim - kt * kTileN;
        // the whole S row in one TMEM round trip: 4 x 32 columns, one wait
        uint32_t sr[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tc::ld32(t_s + q * 32, sr[q]);
#pragma unroll
        for (int q = 0; q < 4; ++q) tc::wait32(sr[q]);
        // invisible columns become -inf
        if (!full) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int j = q * 32 + i;
              if (!(((mask >> (j >> 4)) & 1u) && j <= jlim)) sr[q][i] = __float_as_uint(-INFINITY);
            }
        }
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int i = 0; i < 32; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], __uint_as_float(sr[q][i]));
        const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * p.scale_log2;
        // (scale > 0 keeps the argmax)
        // PV(kt - 2) must be done before O_wg is rescaled and P_wg rewritten
        if (kt >= 2) {
          ok = wait_or_abort(&sh.pv_done[wg], (ph - 1) & 1u, abort_flag);
          if (!ok) break;
          tc::fence_after_sync();
        }
        if (__any_sync(0xffffffffu, mx > m_run + kRescaleLog2)) {
          const float m_new = fmaxf(m_run, mx);
          const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
          l_run *= alpha;
          m_run = m_new;
          if (kt >= 2) {
#pragma unroll 1
            for (int q = 0; q < D / 16; ++q) {
              uint32_t o[16];
              tc::ld16(t_s + 128u + q * 16, o);
              tc::wait16(o);
#pragma unroll
              for (int x = 0; x < 16; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
              tc::st16(t_s + 128u + q * 16, o);
            }
          }
        }
        // P = 2^(s * scale - m) as bf16 (-inf -> 0), row `row` of P_wg in smem
        // (K-major, 128-byte swizzle: 16-byte chunk c of a row sits at c ^ (row % 8))
        float ps4[4] = {0.f, 0.f, 0.f, 0.f};
        const float msub = (m_run == -INFINITY) ? 0.f : m_run;
        unsigned char* prow = gbase + Lay::kP + wg * 2 * Lay::kChunk + row * 128;
#pragma unroll
        for (int c8 = 0; c8 < 16; ++c8) {  // 8 keys = one 16-byte chunk
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = c8 * 8 + 2 * e;
            const float p0 = exp2f(__uint_as_float(sr[j >> 5][j & 31]) * p.scale_log2 - msub);
            const float p1 = exp2f(__uint_as_float(sr[(j + 1) >> 5][(j + 1) & 31]) * p.scale_log2 - msub);
            w[e] = pack_bf16x2(p0, p1);
            ps4[e] += p0 + p1;
          }
          *reinterpret_cast<uint4*>(prow + (c8 >> 3) * Lay::kChunk + (((c8 & 7) ^ (row & 7)) << 4)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
        l_run += (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
        // V rows of keys past kv_len or of chunks not loaded must be zero
        // (0 * NaN): for such a tile wait for its V copy first
        if (kt * kTileN + kTileN > kv_len || mask != 0xFFu) {
          ok = wait_or_abort(&sh.v_full[stage_of(kt)], stage_par(kt), abort_flag);
          if (!ok) break;
          const int key = kt * kTileN + row;
          if (key >= kv_len || !(mask >> (row >> 4) & 1u)) {
            unsigned char* vrow = gbase + Lay::kV + stage_of(kt) * Lay::kTileKV;
#pragma unroll
            for (int dh = 0; dh < DH; ++dh) {
              uint4* v4 = reinterpret_cast<uint4*>(vrow + dh * Lay::kChunk + row * 128);
#pragma unroll
              for (int x = 0; x < 8; ++x) v4[x] = make_uint4(0, 0, 0, 0);
            }
          }
        }
        fence_proxy_async_smem();
        tc::wait_st();
        tc::fence_before_sync();
        mbar_arrive(&sh.p_ready[wg]);
      }
      if (ok && nmine > 0)  // this warpgroup's last PV
        ok = wait_or_abort(&sh.pv_done[wg], (cnt[wg] + nmine - 1) & 1u, abort_flag);
      tc::fence_after_sync();
      // ---- merge the two partial results. Each warpgroup posts its (max,
      // sum) in its own P buffer, which no MMA reads any more (its last PV is
      // done, or it had no tiles); Q may still be in use by the other's MMAs.
      float2* ml_own = reinterpret_cast<float2*>(gbase + Lay::kP + wg * 2 * Lay::kChunk);
      ml_own[row] = make_float2(m_run, l_run);
      tc::fence_before_sync();
      asm volatile("bar.sync 1, 256;" ::: "memory");
      tc::fence_after_sync();
      const float2 ml0 = reinterpret_cast<const float2*>(gbase + Lay::kP)[row];
      const float2 ml1 = reinterpret_cast<const float2*>(gbase + Lay::kP + 2 * Lay::kChunk)[row];
      const float M = fmaxf(ml0.x, ml1.x);
      const float a0 = (ml0.x == -INFINITY) ? 0.f : exp2f(ml0.x - M);
      const float a1 = (ml1.x == -INFINITY) ? 0.f : exp2f(ml1.x - M);
      const float inv = 1.f / (ml0.y * a0 + ml1.y * a1);
      const bool has1 = nkv > 1;
      const bool store = ok && qi < n;
      uint16_t* dst = p.out + (static_cast<long long>(q0 + qi) * p.num_q_heads + g * G + row % G) * D;
      const uint32_t t_o0 = tmem + lane_base + 128u, t_o1 = tmem + lane_base + 256u + 128u;
#pragma unroll 1
      for (int q = 0; q < D / 32; ++q) {  // this warpgroup's D/2 columns, 16 at a time
        const int col = wg * (D / 2) + q * 16;
        uint32_t o0[16], o1[16];
        tc::ld16(t_o0 + col, o0);
        if (has1) tc::ld16(t_o1 + col, o1);
        tc::wait16(o0);
        if (has1) tc::wait16(o1);
        if (store) {
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float v[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int x = 2 * e + h;
              v[h] = (__uint_as_float(o0[x]) * a0 + (has1 ? __uint_as_float(o1[x]) * a1 : 0.f)) * inv;
            }
            w[e] = pack_bf16x2(v[0], v[1]);
          }
          uint4* d4 = reinterpret_cast<uint4*>(dst + col);
          d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
          d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    }
    tc::fence_before_sync();
    __syncthreads();  // O read, merge space reusable, next item may overwrite TMEM
    tc::fence_after_sync();
    tiles += nkv;
    cnt[0] += (nkv + 1) / 2;
    cnt[1] += nkv / 2;
    ++n_q;
  }

  if (sh.abort && tid == kIssuer) {
    // let copies in flight land before the shared memory goes away
    for (int st = 0; st < kStages; ++st) {
      mbar_wait(&sh.k_full[st], 0, kDrainLimitNs);
      mbar_wait(&sh.v_full[st], 0, kDrainLimitNs);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 8) {
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
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = smem_attr_once(kern, smem, attr_done);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, stream>>>(kv_map, q_map, p);
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
  p.block_shift = a.block_shift;
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
