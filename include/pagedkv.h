/*
 * pagedkv.h -- C ABI of libpagedkv.so, the GB300 (sm_103a) hot path of a
 * paged KV cache: slot mapping, the cache write, and paged attention over a
 * block-table-indexed pool for one mixed continuous-batching step.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers named as device buffers are CUDA device pointers on the current
 *   device, owned by the caller. The library never allocates, frees or keeps
 *   them past the call, and never synchronises the stream inside a compute
 *   call: work is only enqueued on `stream` (a cudaStream_t passed as void*;
 *   NULL = the legacy default stream).
 * - bf16 tensors are IEEE bfloat16 bit patterns. Row strides are counted in
 *   elements and must keep every row 16-byte aligned.
 * - Every call returns PKV_OK (0) or a negative PKV_ERR_* status. Argument
 *   checks run on the host before anything is enqueued; a failed check
 *   enqueues nothing. A CUDA launch error returns PKV_ERR_CUDA and
 *   pkv_last_cuda_error() gives its text.
 * - Bad *contents* of device arrays (a slot or block id outside the pool,
 *   inconsistent lengths) cannot be seen by the host without a sync. Kernels
 *   skip such entries instead of touching memory out of range and set bits in
 *   a sticky per-device error word, read by pkv_get_device_errors().
 *
 * Pool layout (the pages' physical KV cache, "vllm v1 源码精读（三）", §3.3):
 *   kv_cache[num_blocks][2][block_size][num_kv_heads][head_dim], bf16,
 *   contiguous; index 0 of the second dimension holds K, 1 holds V.
 *   block_size (B) is 8, 16 or 32 tokens: 16 is the pages' default and 8
 *   and 32 the two other points of "vLLM 架构源码解析（一）" §5.1 (less
 *   last-block waste vs fewer block-table entries); other sizes return
 *   PKV_ERR_UNSUPPORTED. num_blocks * 2 * B must stay below 2^31.
 *   head_dim must be 64 or 128.
 *
 * Launches: every kernel is launched with programmatic stream serialization.
 * A kernel may start (set up barriers, allocate tensor memory, fetch the
 * descriptors passed as its own parameters) while the previous kernel in the
 * stream is still running, and it waits for that kernel to complete -- and
 * its writes to be visible -- before reading any buffer. Work the caller
 * queued earlier on the stream is therefore seen as with plain stream order.
 * The write calls (pkv_slot_mapping, pkv_paged_kv_write,
 * pkv_slot_mapping_and_write) and the attention calls that take the caller's
 * workspace (pkv_paged_attention, pkv_paged_attention_with_write) can be
 * recorded into a CUDA graph.
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_ABI_VERSION 2

/* status codes */
#define PKV_OK 0
#define PKV_ERR_NULL_POINTER (-1) /* a required pointer is NULL             */
#define PKV_ERR_BAD_SHAPE (-2)    /* a size or count is out of range         */
#define PKV_ERR_UNSUPPORTED (-3)  /* valid but not built (block size, d, G)  */
#define PKV_ERR_MISALIGNED (-4)   /* pointer or stride not 16-byte aligned   */
#define PKV_ERR_WORKSPACE (-5)    /* workspace missing or too small          */
#define PKV_ERR_CUDA (-6)         /* a CUDA runtime / driver call failed     */
#define PKV_ERR_DEVICE (-7)       /* the current device is not sm_103        */
#define PKV_ERR_SCRATCH_LIMIT (-8) /* the call needs more scratch than the
                                      library's built-in array holds (see
                                      pkv_paged_attention_static_workspace)    */

/* bits of the sticky device error word */
#define PKV_DEVERR_SLOT_RANGE 0x1u  /* slot >= num_blocks * block_size: row skipped */
#define PKV_DEVERR_BLOCK_RANGE 0x2u /* table entry outside [0, num_blocks) in the
                                       used range: its keys are masked out       */
#define PKV_DEVERR_LENGTHS 0x4u     /* query_start_loc / seq_lens /
                                       num_computed_tokens inconsistent, or a
                                       sequence needs more than
                                       max_blocks_per_req blocks                 */
#define PKV_DEVERR_TIMEOUT 0x8u     /* an on-chip wait (TMA / tensor core) gave
                                       up after its time limit                    */
#define PKV_DEVERR_SHARED 0x10u     /* the shared-prefix hint of
                                       pkv_attention_options did not hold for
                                       some request; it was attended without
                                       the hint (results unaffected)            */

/* Shape of the physical pool. */
typedef struct pkv_cache_layout {
  int32_t num_blocks;   /* physical blocks in the pool, >= 1                  */
  int32_t block_size;   /* tokens per block: 8, 16 or 32                       */
  int32_t num_kv_heads; /* kv heads per token                                 */
  int32_t head_dim;     /* 64 or 128                                          */
} pkv_cache_layout;

/* Optional tuning and tracing of pkv_paged_attention; pass NULL for the
 * defaults. */
typedef struct pkv_attention_options {
  /* Ranges the step's decode KV stream of (request, 16-key chunk) positions
   * is cut into, one CTA each (split-KV). 0 = one full wave of the device,
   * or fewer when the hints bound the stream below that (num_reqs *
   * ceil(max_seq_len / 16)). A single range means no split at all; tests use
   * other values to vary the partitioning. */
  int32_t decode_splits;
  /* Shared prefix of a run of decode requests (prefix caching: "vLLM
   * 架构源码解析（一）" §4.3.1, blocks with ref_cnt > 1 at the head of
   * several block tables). shared_num_reqs > 0 declares that the requests
   * shared_first_req .. shared_first_req + shared_num_reqs - 1 are decodes
   * (one new token each) whose first shared_prefix_len tokens live in the
   * same physical blocks: block_table[r][j] == block_table[shared_first_req][j]
   * for j < shared_prefix_len / B. The call then attends those requests'
   * query rows over the shared prefix once, as one dense tensor-core
   * contraction (rows = requests x q heads, the prefix's keys read once
   * per kv head), and each request's decode covers only its own keys past
   * the prefix, starting from that partial result. The output is the same
   * attention (shared blocks behave as private copies); only the traffic
   * changes.
   *   - shared_prefix_len: tokens, a multiple of 16 and of B, >= 16; 0 =
   *     off (then the other two fields must be 0).
   *   - The hint is checked on the device: a request of the run whose
   *     table does not start with the shared entries, or whose seq_len is
   *     not above shared_prefix_len, is attended without it; if a request of
   *     the run has a query_len other than 1 the whole run is. Either sets
   *     PKV_DEVERR_SHARED. The results stay correct in every case.
   *   - The workspace grows with shared_num_reqs
   *     (pkv_attention_workspace_size takes the same options). */
  int32_t shared_prefix_len;
  int32_t shared_first_req;
  int32_t shared_num_reqs;
  int32_t reserved[4]; /* must be zero */
  /* Tracing: NULL, or PKV_TRACE_EVENTS cudaEvent_t handles (as void*) owned
   * by the caller. The call records them on `stream` around its kernels:
   * [0] before the plan kernel, [1] before the prefill kernel, [2] before
   * the decode kernel, [3] before the combine kernel, [4] after it.
   * Consecutive pairs bracket one kernel each (an empty bracket when a
   * kernel is not needed). The events keep the kernels from overlapping
   * (see "Launches" above), so a traced call can be a little slower. */
  void** trace_events;
} pkv_attention_options;

#define PKV_TRACE_EVENTS 5

/* Library version (PKV_ABI_VERSION). */
int32_t pkv_abi_version(void);

/* Text for a status code; never NULL. */
const char* pkv_status_string(int32_t status);

/* Text of the last CUDA error this thread saw inside the library. */
const char* pkv_last_cuda_error(void);

/*
 * pkv_slot_mapping -- physical slot of every new token of the varlen batch.
 *
 * "vllm v1 源码精读（三）" §3.4: request r's i-th new token sits at position
 * pos = num_computed_tokens[r] + i and goes to
 *   slot = block_table[r][pos / block_size] * block_size + pos % block_size
 * (the page's worked examples: request 0 pos 17 -> 193, request 2 pos 32 ->
 * 144 with tables [[5,12,-1],[3,-1,-1],[7,21,9]]).
 *
 * slot_mapping        out, device int64 [num_tokens]. Token t belongs to the
 *                     request r with query_start_loc[r] <= t <
 *                     query_start_loc[r+1]; tokens at or past
 *                     query_start_loc[num_reqs] get -1 (padding). A token
 *                     whose table entry is missing or outside the pool gets
 *                     -1 and sets PKV_DEVERR_BLOCK_RANGE / _LENGTHS. Every
 *                     row of a request with inconsistent lengths
 *                     (query_start_loc[r] < 0, query_start_loc[r+1] <
 *                     query_start_loc[r] or > num_tokens,
 *                     num_computed_tokens[r] < 0, or query_start_loc[0] !=
 *                     0) gets -1 and sets PKV_DEVERR_LENGTHS; so does every
 *                     row before query_start_loc[0] when that is not 0. No
 *                     row keeps what the buffer held before the call.
 * block_table         device int32 [num_reqs][max_blocks_per_req], -1 = unused.
 * query_start_loc     device int32 [num_reqs + 1], non-decreasing, [0] = 0.
 * num_computed_tokens device int32 [num_reqs].
 * num_blocks          pool size, for the range check.
 * block_size          tokens per block: 8, 16 or 32 (else PKV_ERR_UNSUPPORTED).
 */
int32_t pkv_slot_mapping(int64_t* slot_mapping, const int32_t* block_table,
                         int32_t max_blocks_per_req,
                         const int32_t* query_start_loc,
                         const int32_t* num_computed_tokens, int32_t num_reqs,
                         int32_t num_tokens, int32_t num_blocks,
                         int32_t block_size, void* stream);

/*
 * pkv_paged_kv_write -- reshape_and_cache: store each new token's K and V rows
 * into the pool at its slot ("vLLM 架构源码解析（一）" §3.3.3 step 2;
 * "vllm v1 源码精读（三）" §3.4, reshape_and_cache_flash). A bit copy:
 *   kv_cache[s / B][0][s % B][:][:] = key[t],  [..][1][..] = value[t]
 * for every t with s = slot_mapping[t] >= 0 (B = layout.block_size).
 * Negative slots are skipped; slots >= num_blocks * B are skipped and set
 * PKV_DEVERR_SLOT_RANGE. Two
 * tokens with the same slot race (undefined which wins).
 *
 * kv_cache      in/out, device bf16 pool (layout above).
 * key, value    device bf16 [num_tokens][num_kv_heads][head_dim]; row t starts
 *               at key + t * key_row_stride (0 = num_kv_heads * head_dim).
 * slot_mapping  device int64 [num_tokens].
 */
int32_t pkv_paged_kv_write(void* kv_cache, const void* key, const void* value,
                           int64_t key_row_stride, int64_t value_row_stride,
                           const int64_t* slot_mapping, int32_t num_tokens,
                           pkv_cache_layout layout, void* stream);

/*
 * pkv_slot_mapping_and_write -- pkv_slot_mapping and pkv_paged_kv_write fused
 * into one kernel (the pages compute the slot mapping on the device and then
 * store the rows: "vllm v1 源码精读（三）" §3.4; "vLLM 架构源码解析（一）"
 * §3.3.3 step 2). Each new token's slot is computed as pkv_slot_mapping
 * defines it, and its K and V rows are stored there as pkv_paged_kv_write
 * does, with one launch instead of two.
 *
 * slot_mapping  out, device int64 [num_tokens], or NULL (not stored). For a
 *               non-decreasing query_start_loc it receives exactly what
 *               pkv_slot_mapping writes; a token with slot -1 is not written.
 *               Tokens are assigned to requests by searching
 *               query_start_loc, so where it decreases (inconsistent
 *               lengths, PKV_DEVERR_LENGTHS) the rows that get -1 may differ
 *               from pkv_slot_mapping's.
 * kv_cache, key, value, key_row_stride, value_row_stride, layout
 *               as pkv_paged_kv_write (layout.num_blocks is the range check).
 * block_table, max_blocks_per_req, query_start_loc, num_computed_tokens,
 * num_reqs, num_tokens   as pkv_slot_mapping.
 */
int32_t pkv_slot_mapping_and_write(void* kv_cache, const void* key, const void* value,
                                   int64_t key_row_stride, int64_t value_row_stride,
                                   int64_t* slot_mapping, const int32_t* block_table,
                                   int32_t max_blocks_per_req, const int32_t* query_start_loc,
                                   const int32_t* num_computed_tokens, int32_t num_reqs,
                                   int32_t num_tokens, pkv_cache_layout layout, void* stream);

/*
 * pkv_copy_blocks -- copy whole blocks (K and V of every kv head) between two
 * pools of the same block shape:
 *   - copy-on-write: before a new token is written into a block that other
 *     sequences also reference, the writer gets its own copy of the block
 *     ("vLLM 架构源码解析（一）" §4.3.2, parallel sampling), src_pool ==
 *     dst_pool;
 *   - swap-out / swap-in of a preempted request ("vLLM 架构源码解析（一）"
 *     §1.1, v0 preemption by swapping the KV cache to CPU memory), one pool
 *     on the device and the other in pinned host memory.
 *   dst_pool[d][...] = src_pool[s][...] for every pair (s, d): a bit copy of
 *   2 * B * num_kv_heads * head_dim bf16.
 *
 * dst_pool, src_pool  pools [num_blocks][2][B][num_kv_heads][head_dim] bf16:
 *                     device memory, or pinned host memory the device can
 *                     address with the same pointer (unified addressing).
 * dst_num_blocks, src_num_blocks  pool sizes, for the range checks.
 * block_pairs         device int32 [num_pairs][2] = (source block, destination
 *                     block). A pair out of range is skipped and sets
 *                     PKV_DEVERR_BLOCK_RANGE. Pairs with the same destination,
 *                     or a destination that is another pair's source within one
 *                     call, race (undefined contents).
 * layout              block shape; its num_blocks field is ignored.
 */
int32_t pkv_copy_blocks(void* dst_pool, int32_t dst_num_blocks, const void* src_pool,
                        int32_t src_num_blocks, const int32_t* block_pairs,
                        int32_t num_pairs, pkv_cache_layout layout, void* stream);

/*
 * pkv_attention_workspace_size -- bytes of device workspace that
 * pkv_paged_attention needs for `num_reqs` requests on the current device
 * with the given options (NULL = defaults). Returns a negative status on bad
 * arguments. The size does not depend on sequence lengths.
 */
int64_t pkv_attention_workspace_size(int32_t num_reqs, int32_t num_q_heads,
                                     pkv_cache_layout layout,
                                     const pkv_attention_options* options);

/*
 * pkv_paged_attention -- attention of one mixed step over the paged cache.
 *
 * Run it after pkv_paged_kv_write of the same step: the step's new tokens are
 * read back from the pool ("vLLM 架构源码解析（一）" §3.3.3: write, then
 * attend through the block tables; "vllm v1 源码精读（三）" §4.2: one varlen
 * call holds prefill chunks and decodes; "Inside vLLM" §3.4: each sequence
 * attends only its own tokens).
 *
 * For request r with c = num_computed_tokens[r], n = query_start_loc[r+1] -
 * query_start_loc[r] and L = seq_lens[r] = c + n: its i-th query row
 * (batch row query_start_loc[r] + i, absolute position c + i) and q head h
 * attend keys j = 0 .. c + i of kv head h / (num_q_heads / num_kv_heads):
 *   out = sum_j softmax_j(scale * q . k_j) v_j,
 * key j read from block block_table[r][j / B], offset j % B.
 * Rows with n == 1 run on the split-KV decode kernels (+ combine); rows of
 * requests with n > 1 run on the tensor-core prefill kernel.
 *
 * out            device bf16 [num_tokens][num_q_heads][head_dim], contiguous.
 *                Rows past query_start_loc[num_reqs] are not written.
 * q              device bf16 [num_tokens][num_q_heads][head_dim]; row t at
 *                q + t * q_row_stride (0 = num_q_heads * head_dim).
 * kv_cache       device bf16 pool (layout above), read only.
 * block_table    device int32 [num_reqs][max_blocks_per_req], -1 = unused;
 *                entries from ceil(L / B) on are never read;
 *                max_seq_len <= max_blocks_per_req * B.
 * seq_lens, query_start_loc, num_computed_tokens: device int32 as above.
 * num_tokens     rows of q / out (>= query_start_loc[num_reqs]).
 * max_query_len  host hint: >= every n (like max_seqlen_q).
 * max_seq_len    host hint: >= every L (like max_seqlen_k).
 * num_q_heads    multiple of num_kv_heads; num_q_heads / num_kv_heads must be
 *                1, 2, 4 or 8.
 * scale          softmax scale, positive and finite (1/sqrt(head_dim) on the
 *                pages' models); anything else is PKV_ERR_BAD_SHAPE.
 * workspace      device buffer of at least pkv_attention_workspace_size()
 *                bytes, 256-byte aligned, private to this call while it runs
 *                (no zeroing needed).
 */
int32_t pkv_paged_attention(void* out, const void* q, int64_t q_row_stride,
                            const void* kv_cache, const int32_t* block_table,
                            int32_t max_blocks_per_req, const int32_t* seq_lens,
                            const int32_t* query_start_loc,
                            const int32_t* num_computed_tokens, int32_t num_reqs,
                            int32_t num_tokens, int32_t max_query_len,
                            int32_t max_seq_len, int32_t num_q_heads, float scale,
                            pkv_cache_layout layout, void* workspace,
                            size_t workspace_bytes,
                            const pkv_attention_options* options, void* stream);

/*
 * pkv_paged_attention_with_write -- the whole step of one layer in one call:
 * the slot mapping and cache write of every new token
 * (pkv_slot_mapping_and_write) and then pkv_paged_attention over the pool
 * that now holds them, as the pages' engine does per layer ("vLLM 架构源码解析
 * （一）" §3.3.3: write the step's K/V, then attend; "Inside vLLM" §3.4-3.5:
 * one attention call over the mixed batch). The write runs in the same
 * launch as the attention's plan (its own CTAs next to the plan's), so the
 * step takes one launch fewer than the two calls.
 *
 * Arguments: those of pkv_paged_attention, plus key, value,
 * key_row_stride, value_row_stride and slot_mapping (out, may be NULL) as in
 * pkv_slot_mapping_and_write; kv_cache is written. Results, error bits and
 * the workspace are those of the two calls. A call with no attention to do
 * (num_reqs, num_tokens or max_query_len 0) still maps and writes (padding
 * rows get slot -1). With trace_events, bracket [0, 1) covers the write and
 * the plan.
 */
int32_t pkv_paged_attention_with_write(
    void* out, const void* q, int64_t q_row_stride, void* kv_cache, const void* key,
    const void* value, int64_t key_row_stride, int64_t value_row_stride, int64_t* slot_mapping,
    const int32_t* block_table, int32_t max_blocks_per_req, const int32_t* seq_lens,
    const int32_t* query_start_loc, const int32_t* num_computed_tokens, int32_t num_reqs,
    int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len, int32_t num_q_heads,
    float scale, pkv_cache_layout layout, void* workspace, size_t workspace_bytes,
    const pkv_attention_options* options, void* stream);

/*
 * pkv_paged_attention_static_workspace -- pkv_paged_attention for callers
 * that cannot allocate device memory. The pages have no counterpart to this
 * entry point; it exists for how the library is called, not for what it
 * computes.
 *
 * Some callers have no way to hand the library a workspace: a server that
 * gave all device memory to its own caching allocator and KV pool at start-up
 * and may not call cudaMalloc afterwards, a plugin inside a host framework
 * that forbids raw device allocations, or a plain C caller with no allocator
 * at all. This call takes the same arguments as pkv_paged_attention except the
 * workspace, and uses instead one scratch array compiled into the library:
 * PKV_STATIC_WORKSPACE_BYTES of device memory that every GPU which loads the
 * library holds until the process exits. It never calls cudaMalloc, cudaFree
 * or any allocating routine.
 *
 * - Size limit: if the call would need more scratch than the array holds
 *   (pkv_attention_workspace_size() > PKV_STATIC_WORKSPACE_BYTES) it returns
 *   PKV_ERR_SCRATCH_LIMIT and enqueues nothing. With the default options the
 *   Llama-3-8B layer shape (32 q / 8 kv heads, d = 128) fits about 1860
 *   requests per call on a 152-SM GB300.
 * - First call per device: it looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current. The address is kept
 *   for the life of the process: do not call this entry point again on a device after
 *   cudaDeviceReset (or after its primary context was released and made
 *   anew), since the library's device memory may then sit elsewhere.
 * - Shared state: every call on a device uses the same array and leaves its
 *   contents behind. Nothing needs to start at zero (each call re-plans the
 *   whole scratch area first). Calls whose kernels overlap on the GPU (on
 *   different streams, or from different threads) race on the array and give
 *   wrong results: keep them ordered, e.g. on one stream.
 */
#define PKV_STATIC_WORKSPACE_BYTES (32u * 1024u * 1024u)

int32_t pkv_paged_attention_static_workspace(
    void* out, const void* q, int64_t q_row_stride, const void* kv_cache,
    const int32_t* block_table, int32_t max_blocks_per_req, const int32_t* seq_lens,
    const int32_t* query_start_loc, const int32_t* num_computed_tokens, int32_t num_reqs,
    int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len, int32_t num_q_heads,
    float scale, pkv_cache_layout layout, const pkv_attention_options* options,
    void* stream);

/*
 * pkv_get_device_errors -- checked path: synchronise `stream`, then return
 * in *flags the PKV_DEVERR_* bits that kernels on the current device have set
 * since the last clear; clear them when `clear` is nonzero.
 */
int32_t pkv_get_device_errors(uint32_t* flags, int32_t clear, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */
