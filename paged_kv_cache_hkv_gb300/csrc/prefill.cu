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
// queries, so every K/V tile feeds all G heads (GQA). Per key tile (128 keys
// = 8 chunks of 16 keys: 8 blocks of 16 tokens, 4 of 32 or 16 of 8):
//   S = Q K^T      tcgen05.mma M=128 N=128, A = Q (smem), B = K (smem)
//   O += P V       tcgen05.mma M=128 N=D, A = P (TMEM), B = V (smem)
// with S in one of three TMEM buffers (tile T of the CTA's stream uses
// buffer T % 3) and one O accumulator. Eight softmax warps share every
// tile: each holds 16 query rows, and each row is split between two threads
// (keys 0..63 and 64..127). A thread reads its half row of S with
// tcgen05.ld, applies the causal mask, keeps a base-2 running max (rescaling
// its half of O in TMEM only when the max grows by more than 2^8) and sum,
// and writes P as bf16 pairs over the S buffer's columns with tcgen05.st.
// A K-copy warp (3-slot ring) and a V-copy warp (2-slot ring) stream the
// tiles by TMA (128-byte swizzle, one copy per cache block and kv head: the
// fewer and larger the copies, the faster one SM's copy engine goes); one
// thread issues every S and another every PV. The
// CTAs are persistent and take items from a counter; the roles meet only at
// mbarriers, so consecutive items overlap.
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

// Same, with the A operand (M rows x 16 K elements) in tensor memory: lane i
// holds row i, 32-bit column c holds K elements 2c (low half) and 2c + 1.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
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

// tcgen05.wait::ld with the 32 loaded registers as operands, so that no use
// of them can be scheduled before the wait.
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

// The 16-lane x 2 access shape: 16 TMEM lanes from the address's lane,
// threads 0-15 at columns col .. col+31 of lanes 0-15, threads 16-31 at
// columns col+OFF .. col+OFF+31 of the same lanes (asynchronous: the
// registers hold the data only after wait32 on them).
template <int OFF>
__device__ __forceinline__ void ld_half32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32], %33;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr), "n"(OFF));
}

template <int OFF>
__device__ __forceinline__ void st_half16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], %1, {%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17};" ::"r"(taddr),
      "n"(OFF), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
      "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),
      "r"(v[14]), "r"(v[15])
      : "memory");
}

template <int OFF>
__device__ __forceinline__ void st_half32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x32.b32 [%0], %1, {%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33};" ::"r"(
          taddr),
      "n"(OFF), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
      "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),
      "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]),
      "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

}  // namespace tc


constexpr int kTileM = 128;    // query rows (query x head) per tile
constexpr int kTileN = 128;    // keys per tile (8 chunks of 16)
constexpr int kKStages = 3;    // K ring: global tile T uses slot T % 3
constexpr int kVStages = 2;    // V ring: global tile T uses slot T % 2
constexpr int kSBufs = 3;      // S (then P) buffers in TMEM: global tile T uses buffer T % 3
static_assert(kKStages == kSBufs, "K slot T % 3 is freed by the commit of S buffer T % 3");
constexpr uint32_t kTmemS = 128;  // TMEM columns: O at [0, D), S buffer b at [128 + 128b, +128)
constexpr uint32_t kTmemCols = 512;
constexpr int kItemQ = 4;      // claimed work items in flight between the roles
constexpr int kMetaReqs = 128;  // prefill requests whose metadata a CTA keeps in shared memory
constexpr int kThreads = 384;  // 8 softmax warps, S-MMA warp, K-copy warp, V-copy warp, PV-MMA warp
constexpr float kRescaleLog2 = 8.f;  // lazy rescale threshold (powers of two)

template <int D>
struct PrefillLayout {
  static constexpr int DH = D / 64;                 // 64-element (128-byte) column chunks
  static constexpr uint32_t kChunk = kTileM * 128;  // 128 rows x 128 bytes = 16 KB
  static constexpr uint32_t kQ = 0;
  // K (or V) of one 128-key tile: 16 groups of 8 keys, each DH 128-byte
  // swizzled 8-row atoms (one per 64-element half of d), group-major
  static constexpr uint32_t kGroupBytes = DH * 1024;
  static constexpr uint32_t kTileKV = 16 * kGroupBytes;
  static constexpr uint32_t kK = kQ + DH * kChunk;         // K ring
  static constexpr uint32_t kV = kK + kKStages * kTileKV;  // V ring
  // request metadata: int4 (request, cached, first row, new tokens) [kMetaReqs],
  // then the item prefix int [kMetaReqs + 1]
  static constexpr uint32_t kMeta = kV + kVStages * kTileKV;
  static constexpr uint32_t kBar = kMeta + kMetaReqs * 16 + (kMetaReqs + 1) * 4 + 124;
  static constexpr uint32_t kBytes = kBar + 512;
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
  // shared-prefix items (see AttnArgs): their partial results go to
  // shared_ml / shared_o instead of the output
  int shared_len, shared_first, shared_num, shared_pieces, shared_tpp;
  float2* shared_ml;
  float* shared_o;
};

// mbarriers. "commit" ones are arrived on by a tcgen05.commit of an MMA thread
// (S: s_full, q_free, drain[0]; PV: pv_done, o_full, drain[1]).
struct PrefillShared {
  uint64_t q_full;               // Q tile of the item landed (TMA)
  uint64_t q_free;               // commit: the item's last S read Q
  uint64_t k_full[kKStages];     // K tile landed (TMA)
  uint64_t v_full[kVStages];     // V tile landed (TMA)
  uint64_t s_full[kSBufs];       // commit: S of the buffer's tile in TMEM (and the
                                 // K slot of the same index free: both rings have 3)
  uint64_t pv_done[kSBufs];      // commit: PV of the buffer's tile done (its P read,
                                 // its V slot free, O updated)
  uint64_t p_ready[kSBufs];      // 256 arrivals: P of the buffer's tile in TMEM, O
                                 // rescaled, V cleaned (and, for an item's first tile,
                                 // the previous item's O read)
  uint64_t o_full;               // commit: the item's last PV done
  uint64_t drain[2];             // commit: every MMA of the S / PV thread done (teardown)
  uint64_t iq_full[kItemQ];      // item id j published in item_q[j % kItemQ]
  uint64_t iq_free[kItemQ];      // 11 arrivals: every role has read it
  int item_q[kItemQ];
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(PrefillShared) <= 512, "barrier area");



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

// Consumers of the item queue (the MMA thread, the V-copy warp, each softmax
// warp): item id number j of this CTA, or -1 after an abort. The calling
// warp's lane 0 releases the slot once every lane has read it.
__device__ __forceinline__ int take_item(PrefillShared& sh, int j, volatile int* abort,
                                         bool whole_warp) {
  const int slot = j % kItemQ;
  if (!wait_or_abort(&sh.iq_full[slot], (j / kItemQ) & 1u, abort)) return -1;
  const int item = *reinterpret_cast<volatile int*>(&sh.item_q[slot]);
  if (whole_warp) __syncwarp();
  if (!whole_warp || (threadIdx.x & 31) == 0) mbar_arrive(&sh.iq_free[slot]);
  return item;
}

// One work item: (request, 128-row query tile, kv head).
struct PrefillItem {
  int g;       // kv head
  int c;       // cached tokens of the request
  int q0;      // batch row of the request's first query
  int n;       // new tokens of the request
  int i0;      // first query of the tile (within the request)
  int kv_len;  // keys the tile's last query sees (shared items: end of the piece)
  int nkv;     // key tiles
  int kt0;     // first key tile (0, or a shared item's piece start)
  int piece;   // shared items: key piece, else -1
  long long bt_row;  // offset of the request's block table row
};

// Items of the k-th prefill request are numbered tile-major, longest tile
// first: local index l -> kv head l % Hkv, tile ntile - 1 - l / Hkv. The
// request's metadata comes from the CTA's shared-memory copy when it holds
// every prefill request (meta != nullptr), else from global memory.
__device__ __forceinline__ PrefillItem prefill_item(const PrefillParams& p, int n_req, int item,
                                                    int QT, const int4* meta,
                                                    const int* meta_prefix) {
  PrefillItem m;
  int r, local;
  if (meta) {
    int lo = 0, hi = n_req;  // meta_prefix[lo] <= item < meta_prefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (meta_prefix[mid] <= item) lo = mid; else hi = mid;
    }
    const int4 v = meta[lo];
    r = v.x;
    m.c = v.y;
    m.q0 = v.z;
    m.n = v.w;
    local = item - meta_prefix[lo];
  } else {
    const int k = upper_index(p.pf_prefix, n_req, item);
    r = __ldg(p.pf_req + k);
    local = item - __ldg(p.pf_prefix + k);
    if (r >= 0) {
      m.c = __ldg(p.num_computed + r);
      m.q0 = __ldg(p.qsl + r);
      m.n = __ldg(p.qsl + r + 1) - m.q0;
    } else {
      m.c = p.shared_len;
      m.q0 = __ldg(p.qsl + p.shared_first);
      m.n = p.shared_num;
    }
  }
  m.g = local % p.num_kv_heads;
  if (r < 0) {
    // shared-prefix item: rows = the run's decode rows (one per request) x
    // the kv head's q heads, keys = one piece of the shared prefix, all of
    // them visible to every row
    const int rest = local / p.num_kv_heads;
    m.piece = rest % p.shared_pieces;
    m.i0 = (rest / p.shared_pieces) * QT;
    const int tiles = (p.shared_len + kTileN - 1) / kTileN;
    m.kt0 = m.piece * p.shared_tpp;
    m.nkv = min(p.shared_tpp, tiles - m.kt0);
    m.kv_len = min((m.kt0 + m.nkv) * kTileN, p.shared_len);
    m.bt_row = static_cast<long long>(p.shared_first) * p.max_blocks;
    return m;
  }
  m.piece = -1;
  m.kt0 = 0;
  const int ntile = (m.n + QT - 1) / QT;
  const int mt = ntile - 1 - local / p.num_kv_heads;
  m.i0 = mt * QT;
  const int i_last = min(m.i0 + QT, m.n) - 1;
  m.kv_len = m.c + i_last + 1;
  m.nkv = (m.kv_len + kTileN - 1) / kTileN;
  m.bt_row = static_cast<long long>(r) * p.max_blocks;
  return m;
}

// Block table entry e of the item's request if it holds keys < kv_len and its
// id is in the pool, else -1.
__device__ __forceinline__ int entry_id(const PrefillParams& p, const PrefillItem& m, int e) {
  if ((e << p.block_shift) >= m.kv_len) return -1;
  const int id = __ldg(p.block_table + m.bt_row + e);
  return (id >= 0 && id < p.num_blocks) ? id : -1;
}

// Chunk b (keys 16b .. 16b+15) of tile kt holds keys < kv_len, all of them in
// blocks of the pool.
__device__ __forceinline__ bool chunk_ok(const PrefillParams& p, const PrefillItem& m, int kt, int b) {
  const int k0 = kt * kTileN + b * kChunkKeys;
  if (k0 >= m.kv_len) return false;
  const int bsh = p.block_shift;
  if (bsh == 4) return entry_id(p, m, k0 >> 4) >= 0;
  if (bsh == 5) return entry_id(p, m, k0 >> 5) >= 0;
  return entry_id(p, m, k0 >> 3) >= 0 && (k0 + 8 >= m.kv_len || entry_id(p, m, (k0 >> 3) + 1) >= 0);
}

// Persistent CTAs; CTA b takes items b, b + gridDim.x, ... (items come
// longest first within a request). Every role walks that list on its own and
// the roles meet only at mbarriers, so the next item's Q/K/V copies and first
// S MMAs overlap the current item's last tiles and epilogue.
//   warp 9:  Q copy (once the previous item's last S is done) and K tiles
//            into a 3-slot ring (a slot is refilled once its S is done);
//   warp 10: V tiles into a 2-slot ring (refilled once its PV is done);
//   warp 8, lane 0: every MMA, per item in the order S(0), S(1), S(2),
//            PV(0), S(3), PV(1), S(4), ...: S(kt) = Q K^T into S buffer
//            (T+kt) % 3, and O += P V with P read from TMEM, where the
//            softmax warps wrote it over the tile's S (bf16 pairs, one pair
//            per 32-bit column). MMAs run in issue order, so S(kt+3)
//            overwrites P(kt) only after PV(kt) read it.
//   warps 0..7: the softmax of every tile, 16 query rows per warp and half
//            of each row per thread, and the item's epilogue (each thread
//            normalises and writes half of its row's output columns).
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
  const int G = p.group, QT = kTileM / G;

  if (tid == 0) {
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.q_free, 1);
    for (int i = 0; i < kKStages; ++i) mbar_init(&sh.k_full[i], 1);
    for (int i = 0; i < kVStages; ++i) mbar_init(&sh.v_full[i], 1);
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.pv_done[i], 1);
      mbar_init(&sh.p_ready[i], 256);
    }
    mbar_init(&sh.o_full, 1);
    mbar_init(&sh.drain[0], 1);
    mbar_init(&sh.drain[1], 1);
    for (int i = 0; i < kItemQ; ++i) {
      mbar_init(&sh.iq_full[i], 1);
      mbar_init(&sh.iq_free[i], 11);
    }
    sh.abort = 0;
    fence_barrier_init();
  }
  if (tid == 32 * 9) {
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
  pdl_trigger();
  // barriers, tensor maps and TMEM above do not depend on the plan; its output does
  pdl_wait();
  const int n_items = static_cast<int>(p.hdr[kHdrPrefillItems]);
  const int n_req = static_cast<int>(p.hdr[kHdrPrefillReqs]);
  int4* meta_s = reinterpret_cast<int4*>(gbase + Lay::kMeta);
  int* meta_prefix_s = reinterpret_cast<int*>(gbase + Lay::kMeta + kMetaReqs * 16);
  if (n_req <= kMetaReqs) {
    for (int i = tid; i <= n_req; i += kThreads) {
      meta_prefix_s[i] = __ldg(p.pf_prefix + i);
      if (i < n_req) {
        const int r = __ldg(p.pf_req + i);
        if (r >= 0) {
          const int q0 = __ldg(p.qsl + r);
          meta_s[i] = make_int4(r, __ldg(p.num_computed + r), q0, __ldg(p.qsl + r + 1) - q0);
        } else {  // the shared-prefix items
          meta_s[i] = make_int4(-1, p.shared_len, __ldg(p.qsl + p.shared_first), p.shared_num);
        }
      }
    }
  }
  // the first work item is claimed while the CTA sets up
  int first_claim = 0;
  if (tid == 32 * 9) first_claim = static_cast<int>(atomicAdd(&p.hdr[kHdrPrefillNext], 1u));
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh.tmem;
  const int4* meta = n_req <= kMetaReqs ? meta_s : nullptr;
  const int* meta_prefix = meta_prefix_s;
  auto valid = [&](int item) { return item >= 0 && item < n_items; };

  if (warp == 9 || warp == 10) {
    // ================= copy warps. Lane (chunk b, d half dh), lanes
    // 0 .. 8*DH-1, issues the copies of that chunk (one of 16 rows, or two of
    // 8 rows for 8-token blocks); the block ids of a 32-entry window of the
    // block table sit in the lanes' registers.
    const int ln = tid & 31;
    const bool is_v = warp == 10;
    const int S = is_v ? kVStages : kKStages;
    uint64_t* full = is_v ? sh.v_full : sh.k_full;
    const uint32_t ring = is_v ? Lay::kV : Lay::kK;
    const int bsh = p.block_shift;
    const int E = kTileN >> bsh;  // table entries per tile
    uint32_t T = 0;               // tiles issued so far (all items)
    bool ok = true;
    int q_loads = 0;
    for (int it = 0; ok; ++it) {
      int item;
      if (!is_v) {
        // the Q buffer is free once the previous item's last S is done; only
        // then is the next item claimed (work counter), so that items go to
        // the CTAs that are about to be idle
        if (it > 0) ok = wait_or_abort(&sh.q_free, (it - 1) & 1u, abort_flag);
        if (!ok) break;
        item = n_items;
        if (ln == 0) {
          const int slot = it % kItemQ;
          if (it >= kItemQ) ok = wait_or_abort(&sh.iq_free[slot], ((it - kItemQ) / kItemQ) & 1u, abort_flag);
          if (ok) item = it == 0 ? first_claim : static_cast<int>(atomicAdd(&p.hdr[kHdrPrefillNext], 1u));
          sh.item_q[slot] = item;
          mbar_arrive(&sh.iq_full[slot]);
        }
        item = __shfl_sync(0xffffffffu, item, 0);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      } else {
        item = take_item(sh, it, abort_flag, true);
        if (item < 0) ok = false;
      }
      if (!ok || !valid(item)) break;
      const PrefillItem m = prefill_item(p, n_req, item, QT, meta, meta_prefix);
      if (!is_v) {
        if (ln == 0) {
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(&sh.q_full, DH * Lay::kChunk);
#pragma unroll
          for (int dh = 0; dh < DH; ++dh)
            tma_load_3d(gbase + Lay::kQ + dh * Lay::kChunk, &q_map, dh * 64, m.g * G, m.q0 + m.i0,
                        &sh.q_full);
        }
        ++q_loads;
      }
      int win_base = -1000000, win_val = -1;
      for (int kt = 0; kt < m.nkv; ++kt) {
        const int slot = static_cast<int>(T % S);
        if (T >= static_cast<uint32_t>(S)) {
          // K slot T % 3 is free once S(T-3) is done; V slot T % 2 once
          // PV(T-2) is done
          const uint32_t Tp = T - S;
          ok = is_v ? wait_or_abort(&sh.pv_done[Tp % kSBufs], (Tp / kSBufs) & 1u, abort_flag)
                    : wait_or_abort(&sh.s_full[Tp % kSBufs], (Tp / kSBufs) & 1u, abort_flag);
          if (!ok) break;
        }
        const int ka = m.kt0 + kt;  // key tile (keys ka*128 ..)
        if (ka * E + E > win_base + 32) {
          win_base = ka * E;
          const int e = win_base + ln;
          win_val = entry_id(p, m, e);
          if (!is_v && (e << bsh) < m.kv_len && win_val < 0)
            atomicOr(&g_errors_prefill, kErrBlockRange);
        }
        // lane j < E copies the K (or V) rows of table entry ka*E + j, kv
        // head g: one box of B rows x D, 8-row groups of pool row
        // (block * 2 + k|v) * B
        const int id = __shfl_sync(0xffffffffu, win_val, (ka * E + (ln & (E - 1)) - win_base) & 31);
        const bool mine = ln < E && id >= 0;
        const uint32_t box = static_cast<uint32_t>(Lay::kGroupBytes) << (bsh - 3);
        const uint32_t tx = __reduce_add_sync(0xffffffffu, mine ? box : 0u);
        if (ln == 0) {
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(&full[slot], tx);
        }
        __syncwarp();
        if (mine)
          tma_load_5d(gbase + ring + slot * Lay::kTileKV + ln * box, &kv_map, 0, 0, 0, m.g,
                      ((id * 2 + (is_v ? 1 : 0)) << bsh) >> 3, &full[slot]);
        ++T;
      }
    }
    if (!ok) {  // let the copies in flight land before the shared memory goes away
      for (int s = 0; s < S; ++s)
        if (T > static_cast<uint32_t>(s)) {
          const uint32_t last = s + S * ((T - 1 - s) / S);
          mbar_wait(&full[s], (last / S) & 1u, kDrainLimitNs);
        }
      if (!is_v && q_loads > 0) mbar_wait(&sh.q_full, (q_loads - 1) & 1u, kDrainLimitNs);
    }
  } else if (warp == 8 || warp == 11) {
    // ================= MMA threads: warp 8 issues every S, warp 11 every PV
    if ((tid & 31) == 0) {
      const bool is_s = warp == 8;
      constexpr uint32_t idesc_qk = tc::idesc_bf16(kTileM, kTileN, 0);
      constexpr uint32_t idesc_pv = tc::idesc_bf16(kTileM, D, 1);
      uint32_t T = 0;  // tiles of earlier items
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int item = take_item(sh, it, abort_flag, false);
        if (item < 0) ok = false;
        if (!ok || !valid(item)) break;
        const PrefillItem m = prefill_item(p, n_req, item, QT, meta, meta_prefix);
        const int nkv = m.nkv;
        if (is_s) {
          ok = wait_or_abort(&sh.q_full, it & 1u, abort_flag);
          for (int kt = 0; ok && kt < nkv; ++kt) {
            // S(Tk) = Q K^T into buffer Tk % 3, once PV(Tk-3) has read the
            // P that the buffer holds and K(Tk) has landed
            const uint32_t Tk = T + kt;
            const uint32_t b = Tk % kSBufs;
            if (Tk >= static_cast<uint32_t>(kSBufs))
              ok = wait_or_abort(&sh.pv_done[b], ((Tk - kSBufs) / kSBufs) & 1u, abort_flag);
            if (ok) ok = wait_or_abort(&sh.k_full[b], (Tk / kKStages) & 1u, abort_flag);
            if (!ok) break;
            tc::fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t sub = (kk & 3) * 32;  // 16 elements within the 64-element half
              const uint64_t a = tc::sw128_desc(base + Lay::kQ + (kk >> 2) * Lay::kChunk + sub, 16, 1024);
              const uint64_t bd = tc::sw128_desc(
                  base + Lay::kK + b * Lay::kTileKV + (kk >> 2) * 1024 + sub, 16, Lay::kGroupBytes);
              tc::mma_bf16(tmem + kTmemS + kTileN * b, a, bd, idesc_qk, kk > 0);
            }
            tc::commit(&sh.s_full[b]);  // S in TMEM, and the K slot free
            if (kt == nkv - 1) tc::commit(&sh.q_free);
          }
        } else {
          for (int kt = 0; ok && kt < nkv; ++kt) {
            // O += P V for tile Tg, P read from its S buffer. The first PV of
            // an item overwrites O: the softmax warps publish P of an item's
            // first tile only after their epilogue of the previous item has
            // read O.
            const uint32_t Tg = T + kt;
            const uint32_t b = Tg % kSBufs;
            const int slot = static_cast<int>(Tg % kVStages);
            ok = wait_or_abort(&sh.p_ready[b], (Tg / kSBufs) & 1u, abort_flag);
            if (ok) ok = wait_or_abort(&sh.v_full[slot], (Tg / kVStages) & 1u, abort_flag);
            if (!ok) break;
            tc::fence_after_sync();
            const uint32_t vbase = base + Lay::kV + slot * Lay::kTileKV;
#pragma unroll
            for (int kk = 0; kk < kTileN / 16; ++kk) {
              // keys 16kk .. 16kk+15: two 8-key groups (SBO), d halves 1 KB apart (LBO)
              const uint64_t bd = tc::sw128_desc(vbase + kk * 2 * Lay::kGroupBytes, 1024, Lay::kGroupBytes);
              tc::mma_bf16_ts(tmem, tmem + kTmemS + kTileN * b + kk * 8u, bd, idesc_pv,
                              (kt > 0 || kk > 0) ? 1u : 0u);
            }
            tc::commit(&sh.pv_done[b]);  // P's buffer and the V slot free
            if (kt == nkv - 1) tc::commit(&sh.o_full);  // the item's O is complete
          }
        }
        T += nkv;
      }
      // every MMA of this thread (and the arrivals of its commits) done
      // before teardown
      tc::commit(&sh.drain[is_s ? 0 : 1]);
      mbar_wait(&sh.drain[is_s ? 0 : 1], 0, ok ? kWaitLimitNs : kDrainLimitNs);
    }
    __syncwarp();
  } else {
    // ================= softmax warps 0..7: every tile of every item. Warp w
    // owns TMEM lanes (query rows) lane0 .. lane0+15 with lane0 = 32*(w%4) +
    // 16*(w/4) (warp w reaches lanes 32*(w%4) .. +31 only). Of each row,
    // thread t < 16 takes keys 0..63 of every tile and thread t + 16 keys
    // 64..127 (the 16x32bx2 TMEM access shape), so a row's max needs one
    // shuffle and no warp waits for another.
    constexpr int HC = D / 2;  // O columns per thread
    const int lane = tid & 31;
    const int ch = lane >> 4;  // key half of this thread
    const int lane0 = 32 * (warp & 3) + 16 * (warp >> 2);
    const int row = lane0 + (lane & 15);  // query row of this thread (TMEM lane)
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(lane0) << 16);
    uint32_t T = 0;
    bool ok = true;
    // chunk validity of tile kt of item m (lanes 0..7), read one tile ahead
    auto load_ids = [&](const PrefillItem& mm, int kt) -> int {
      return (lane < 8 && kt < mm.nkv && chunk_ok(p, mm, mm.kt0 + kt, lane)) ? 1 : -1;
    };
    int item = take_item(sh, 0, abort_flag, true);
    PrefillItem m{};
    int next_id = -1;
    if (valid(item)) {
      m = prefill_item(p, n_req, item, QT, meta, meta_prefix);
      next_id = load_ids(m, 0);
    }
    for (int it = 0; ok && valid(item); ++it) {
      const int nkv = m.nkv;
      const int qi = m.i0 + row / G;                // query of this row
      const int lim = min(m.c + qi, m.kv_len - 1);  // last key this row may see
      float m_run = -INFINITY, l_run = 0.f;
      for (int kt = 0; kt < nkv; ++kt) {
        const uint32_t Tg = T + kt;
        const uint32_t b = Tg % kSBufs;
        const uint32_t t_s = t_lane + kTmemS + kTileN * b;
        const uint32_t mask = __ballot_sync(0xffffffffu, next_id >= 0) & 0xFFu;
        ok = wait_or_abort(&sh.s_full[b], (Tg / kSBufs) & 1u, abort_flag);
        if (!ok) break;
        tc::fence_after_sync();
        // a tile every row sees in full needs no mask; otherwise key j of the
        // tile is visible iff j <= lim - 128 ka and its 16-key chunk was
        // loaded (chunk c = keys 16c .. 16c+15)
        const int ka = m.kt0 + kt;  // key tile (keys ka*128 ..)
        const bool full = ka * kTileN + kTileN - 1 <= m.c + m.i0 && mask == 0xFFu;
        // this thread's keys 64ch .. 64ch+63 of the tile: sr[0] the first 32
        uint32_t sr[2][32];
        tc::ld_half32<64>(t_s, sr[0]);
        tc::ld_half32<64>(t_s + 32, sr[1]);
        tc::wait32(sr[0]);
        tc::wait32(sr[1]);
        if (!full) {  // invisible keys become -inf
          const int jlim = lim - ka * kTileN - 64 * ch;
          const uint32_t cm = mask >> (4 * ch);
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int j = q * 32 + i;
              if (!(((cm >> (j >> 4)) & 1u) && j <= jlim)) sr[q][i] = __float_as_uint(-INFINITY);
            }
        }
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            mx4[(i >> 1) & 3] =
                max3f(mx4[(i >> 1) & 3], __uint_as_float(sr[q][i]), __uint_as_float(sr[q][i + 1]));
        float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        // (scale > 0 keeps the argmax; both threads of the row get the same bits)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16)) * p.scale_log2;
        if (__any_sync(0xffffffffu, mx > m_run + kRescaleLog2)) {
          const float m_new = fmaxf(m_run, mx);
          const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
          l_run *= alpha;
          m_run = m_new;
          if (kt > 0) {
            // O holds PV of the item's earlier tiles; the last of them is PV(Tg-1)
            const uint32_t Tp = Tg - 1;
            ok = wait_or_abort(&sh.pv_done[Tp % kSBufs], (Tp / kSBufs) & 1u, abort_flag);
            if (!ok) break;
            tc::fence_after_sync();
#pragma unroll 1
            for (int q = 0; q < HC / 32; ++q) {  // this thread's O columns HC*ch + 32q ..
              uint32_t o[32];
              tc::ld_half32<HC>(t_lane + 32 * q, o);
              tc::wait32(o);
#pragma unroll
              for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
              tc::st_half32<HC>(t_lane + 32 * q, o);
            }
          }
        }
        // P = 2^(s * scale - m) as bf16 (-inf -> 0) over the S buffer: column
        // c holds keys 2c (low half) and 2c+1, so this thread's keys land in
        // columns 32ch .. 32ch+31 (pairs of keys in the packed fp32x2 FMA / add)
        float2 ps4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        const float msub = (m_run == -INFINITY) ? 0.f : m_run;
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(-msub, -msub);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 e = ffma2(
                make_float2(__uint_as_float(sr[q][2 * j]), __uint_as_float(sr[q][2 * j + 1])), sc2, nm2);
            const float2 pp = make_float2(exp2f(e.x), exp2f(e.y));
            pk[j] = pack_bf16x2(pp.x, pp.y);
            ps4[j & 3] = fadd2(ps4[j & 3], pp);
          }
          tc::st_half16<32>(t_s + 16 * q, pk);
        }
        l_run += ((ps4[0].x + ps4[1].x) + (ps4[2].x + ps4[3].x)) +
                 ((ps4[0].y + ps4[1].y) + (ps4[2].y + ps4[3].y));
        // V rows of keys past kv_len or of chunks not loaded must be zero
        // (0 * NaN): for such a tile wait for its V copy first; thread (row,
        // ch) clears 64-element chunk ch of V row `row`
        if (ka * kTileN + kTileN > m.kv_len || mask != 0xFFu) {
          const int slot = static_cast<int>(Tg % kVStages);
          // S(Tg) done only implies PV(Tg-3) done, so the slot's copy
          // barrier may be anywhere from V(Tg-2) pending to V(Tg) landed;
          // once PV(Tg-2) is done (slot released) it is V(Tg) pending or landed
          if (Tg >= static_cast<uint32_t>(kVStages)) {
            const uint32_t Tp = Tg - kVStages;
            ok = wait_or_abort(&sh.pv_done[Tp % kSBufs], (Tp / kSBufs) & 1u, abort_flag);
          }
          if (ok) ok = wait_or_abort(&sh.v_full[slot], (Tg / kVStages) & 1u, abort_flag);
          if (!ok) break;
          if (ch < DH && (ka * kTileN + row >= m.kv_len || !(mask >> (row >> 4) & 1u))) {
            uint4* v4 = reinterpret_cast<uint4*>(gbase + Lay::kV + slot * Lay::kTileKV +
                                                 (row >> 3) * Lay::kGroupBytes + ch * 1024 +
                                                 (row & 7) * 128);
#pragma unroll
            for (int x = 0; x < 8; ++x) v4[x] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tc::wait_st();
        tc::fence_before_sync();
        mbar_arrive(&sh.p_ready[b]);
        next_id = load_ids(m, kt + 1);  // its latency hides under the next S wait
      }
      if (!ok) break;
      // ---- the next item's id and metadata, while the last PV runs
      const int item_n = take_item(sh, it + 1, abort_flag, true);
      if (item_n < 0) {  // aborted
        ok = false;
        break;
      }
      PrefillItem m_next{};
      if (valid(item_n)) {
        m_next = prefill_item(p, n_req, item_n, QT, meta, meta_prefix);
        next_id = load_ids(m_next, 0);
      }
      // ---- epilogue: this thread's O columns HC*ch .. HC*ch + HC - 1 of its row
      ok = wait_or_abort(&sh.o_full, it & 1u, abort_flag);
      if (!ok) break;
      tc::fence_after_sync();
      const float l_tot = l_run + __shfl_xor_sync(0xffffffffu, l_run, 16);
      const float inv = 1.f / l_tot;
      const bool store = qi < m.n;
      const int head = m.g * G + row % G;
      // shared-prefix items keep the row's partial (max, sum, unnormalised O)
      // for the decode of request shared_first + qi: slot of (piece, qi, head)
      const bool partial = m.piece >= 0;
      const long long pslot = (static_cast<long long>(m.piece) * p.shared_num + qi) * p.num_q_heads + head;
      if (partial && store && ch == 0) p.shared_ml[pslot] = make_float2(m_run, l_tot);
      uint16_t* dst = p.out + (static_cast<long long>(m.q0 + qi) * p.num_q_heads + head) * D + HC * ch;
#pragma unroll 1
      for (int q = 0; q < HC / 32; ++q) {
        uint32_t o[32];
        tc::ld_half32<HC>(t_lane + 32 * q, o);
        tc::wait32(o);
        if (!store) continue;
        if (partial) {
          float4* d4 = reinterpret_cast<float4*>(p.shared_o + pslot * D + HC * ch + 32 * q);
#pragma unroll
          for (int x = 0; x < 8; ++x)
            d4[x] = make_float4(__uint_as_float(o[4 * x]), __uint_as_float(o[4 * x + 1]),
                                __uint_as_float(o[4 * x + 2]), __uint_as_float(o[4 * x + 3]));
        } else {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * q);
#pragma unroll
          for (int x = 0; x < 4; ++x) d4[x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
        }
      }
      T += nkv;
      m = m_next;
      item = item_n;
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
  return launch_pdl(kern, dim3(grid), dim3(kThreads), static_cast<size_t>(smem), stream, kv_map,
                    q_map, p);
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
  p.shared_len = a.shared_len;
  p.shared_first = a.shared_first;
  p.shared_num = a.shared_num;
  p.shared_pieces = a.shared_pieces;
  p.shared_tpp = a.shared_tpp;
  p.shared_ml = ws.casc_ml;
  p.shared_o = ws.casc_o;
  // upper bound of work items from the host hints: every row can be in a
  // tile (only rows of requests with more than one new token are, when the
  // call has no shared prefix), plus the shared-prefix items
  const long long tile_q = kTileM / p.group;
  long long max_items = a.max_query_len > 1
      ? ((static_cast<long long>(a.num_tokens) + tile_q - 1) / tile_q + a.num_reqs) *
            a.num_kv_heads
      : 0;
  if (a.shared_num > 0)
    max_items += (a.shared_num + tile_q - 1) / tile_q * a.shared_pieces * a.num_kv_heads;
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
