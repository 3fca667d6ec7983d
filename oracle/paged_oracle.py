"""Plain fp64 CPU statement of the paged KV cache hot path (test infrastructure).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
legs may use this module. It shares nothing with the CUDA library.

Sources (pages by title, with the section each step follows):

* [P1] "vLLM 架构源码解析（一）：从 API 请求到 Token 生成" -- §3.3.2 (positions
  start..end of each request), §3.3.3 (write the new K/V into the cache, then
  attend through the block table), §4.2 (block table maps logical to physical
  blocks; 1/sqrt(d_k) scaling).
* [P2] "Inside vLLM: Anatomy of a High-Throughput LLM Inference System" --
  §3.3 (ceil(tokens/16) blocks, 17 -> 2), §3.4 (all sequences flattened into one
  super-sequence; positions and the mask keep each sequence to its own
  tokens), §3.5 (a chunk continues where the previous one stopped).
* [P3] nano-vllm / cleanvllm walk-through -- ``Sequence.num_blocks`` and
  ``last_block_num_tokens``.
* [P4] "vllm v1 源码精读（三）：KV Cache 管理、Chunked Prefill 与异步架构" --
  §3.3 (pool layout [num_blocks, 2, block_size, num_kv_heads, head_dim],
  index 0 = K, 1 = V), §3.4 (block table with -1 padding; slot of a token;
  worked examples 193 and 144; write by slot_mapping, read by block_table),
  §4.2 (mixed varlen batch: each request's queries attend only that request's
  cached plus new keys).

Readings where the pages are silent or garbled:

* The slot formula is lost in the text of [P4] §3.4; its two worked examples
  fix it as ``block_table[pos // B] * B + pos % B``.
* GQA head map (not stated): q head h reads kv head ``h // (Hq / Hkv)``.
* A query at absolute position p = num_computed + i sees keys 0..p
  (bottom-right causal); a decode row is the case query_len = 1.
* ``seq_len = num_computed + query_len``; the new tokens are written first and
  read back from the cache.
* Softmax is the standard one with max subtraction; ``scale`` is applied to
  q.k before it.
* A negative slot in ``slot_mapping`` means "skip this token" (padding).

All floating point is fp64 on the exact bf16 input values.
"""

from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as fp64: a bf16 is the top
    half of an fp32."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def blocks_for_tokens(n_tokens, block_size: int = 16):
    """Blocks a sequence of ``n_tokens`` needs: ceil(n / B) ([P2] §3.3:
    17 new tokens need 2 blocks; [P3] ``Sequence.num_blocks``)."""
    n = np.asarray(n_tokens, dtype=np.int64)
    return (n + block_size - 1) // block_size


def last_block_fill(n_tokens, block_size: int = 16):
    """Tokens held by the last block ([P3] ``last_block_num_tokens``)."""
    n = np.asarray(n_tokens, dtype=np.int64)
    return n - (blocks_for_tokens(n, block_size) - 1) * block_size


def kv_bytes_per_token(num_kv_heads: int, head_dim: int, dtype_bytes: int = 2) -> int:
    """Cache bytes one token takes in one layer: K and V, each
    num_kv_heads x head_dim elements ([P2] §3.1 block-size formula divided by
    block_size; [P4] §3.1: 2 x 8 x 128 x 2 = 4096 for LLaMA-3-8B)."""
    return 2 * num_kv_heads * head_dim * dtype_bytes


def slot_of(table_row: np.ndarray, pos: int, block_size: int = 16) -> int:
    """Physical slot of the token at absolute position ``pos`` ([P4] §3.4):
    logical block pos // B is looked up in the table, the offset inside the
    block is pos % B."""
    return int(table_row[pos // block_size]) * block_size + pos % block_size


def slot_mapping(block_table: np.ndarray, query_start_loc: np.ndarray,
                 num_computed: np.ndarray, block_size: int = 16) -> np.ndarray:
    """One slot per new token of the varlen batch ([P4] §3.4, [P1] §3.3.2).

    Request r owns batch rows query_start_loc[r] .. query_start_loc[r+1]-1; its
    i-th new token sits at position num_computed[r] + i."""
    T = int(query_start_loc[-1])
    out = np.full(T, -1, dtype=np.int64)
    for r in range(len(num_computed)):
        t0, t1 = int(query_start_loc[r]), int(query_start_loc[r + 1])
        for t in range(t0, t1):
            pos = int(num_computed[r]) + (t - t0)
            out[t] = slot_of(block_table[r], pos, block_size)
    return out


def kv_write(kv_cache: np.ndarray, k: np.ndarray, v: np.ndarray,
             slots: np.ndarray) -> np.ndarray:
    """Return a copy of the pool with each new token's K and V rows stored at
    its slot ([P1] §3.3.3 step 2; [P4] §3.4 ``reshape_and_cache_flash``).

    kv_cache: uint16 [NB, 2, B, Hkv, D]; k, v: uint16 [N, Hkv, D];
    slots: int [N], negative = skip. A pure bit copy."""
    out = kv_cache.copy()
    B = kv_cache.shape[2]
    for t in range(len(slots)):
        s = int(slots[t])
        if s < 0:
            continue
        out[s // B, 0, s % B] = k[t]
        out[s // B, 1, s % B] = v[t]
    return out


def copy_blocks(dst_pool: np.ndarray, src_pool: np.ndarray, pairs) -> np.ndarray:
    """Return a copy of dst_pool with block d replaced by src_pool's block s
    for every pair (s, d), in order: copy-on-write of a shared block before a
    write ([P1] §4.3.2) and swap-out / swap-in of a preempted request's blocks
    between device and host memory ([P1] §1.1)."""
    out = dst_pool.copy()
    for s, d in np.asarray(pairs, dtype=np.int64).reshape(-1, 2):
        out[d] = src_pool[s]
    return out


def gather_request_kv(kv_cache: np.ndarray, table_row: np.ndarray,
                      seq_len: int) -> np.ndarray:
    """Logical-order copy of one request's cached K/V: uint16 [L, 2, Hkv, D].

    Key j lives in block table_row[j // B] at offset j % B ([P4] §3.3-3.4).
    Entries from ceil(L / B) on are never read; a -1 inside the used range is
    an error."""
    B = kv_cache.shape[2]
    j = np.arange(seq_len)
    blk = np.asarray(table_row, dtype=np.int64)[j // B]
    if seq_len and blk.min() < 0:
        raise ValueError("block table has -1 inside the used range")
    return kv_cache[blk, :, j % B]


def attend_rows(q_bits: np.ndarray, kv_bits: np.ndarray, positions: np.ndarray,
                scale: float) -> np.ndarray:
    """Causal softmax attention of one request's query rows over its keys.

    q_bits: uint16 [n, Hq, D]; kv_bits: uint16 [L, 2, Hkv, D] (logical order);
    positions: [n] absolute positions. Row i, head h attends keys
    0..positions[i] of kv head h // (Hq / Hkv):
    s_j = scale * q.k_j, w = exp(s - max s) / sum exp(s - max s), o = sum w_j v_j.
    Returns fp64 [n, Hq, D]."""
    n, Hq, D = q_bits.shape
    L, _, Hkv, _ = kv_bits.shape
    G = Hq // Hkv
    out = np.empty((n, Hq, D), dtype=np.float64)
    visible = np.arange(L)[None, :] <= np.asarray(positions)[:, None]
    for g in range(Hkv):
        K = bf16_bits_to_f64(kv_bits[:, 0, g, :])
        V = bf16_bits_to_f64(kv_bits[:, 1, g, :])
        for h in range(g * G, (g + 1) * G):
            Q = bf16_bits_to_f64(q_bits[:, h, :])
            s = scale * (Q @ K.T)
            s = np.where(visible, s, -np.inf)
            w = np.exp(s - s.max(axis=1, keepdims=True))
            out[:, h, :] = (w @ V) / w.sum(axis=1, keepdims=True)
    return out


def paged_attention(q: np.ndarray, kv_cache: np.ndarray, block_table: np.ndarray,
                    seq_lens: np.ndarray, query_start_loc: np.ndarray,
                    num_computed: np.ndarray, scale: float,
                    rows=None) -> np.ndarray:
    """Attention output of one mixed step, fp64 [T, Hq, D] ([P4] §4.2, [P1]
    §3.3.3, [P2] §3.4).

    The cache must already hold the step's new tokens (write first). For
    request r: its rows are query_start_loc[r]..[r+1]-1, the i-th one at
    position num_computed[r] + i, seeing keys 0..position of that request.
    ``rows`` (optional iterable of batch row indices) limits the work to those
    rows; other rows are NaN."""
    T = int(query_start_loc[-1])
    Hq, D = q.shape[1], q.shape[2]
    out = np.full((T, Hq, D), np.nan)
    want = None if rows is None else np.zeros(T, dtype=bool)
    if want is not None:
        want[np.asarray(list(rows), dtype=np.int64)] = True
    for r in range(len(seq_lens)):
        t0, t1 = int(query_start_loc[r]), int(query_start_loc[r + 1])
        if t1 == t0:
            continue
        idx = np.arange(t0, t1)
        if want is not None:
            idx = idx[want[t0:t1]]
            if len(idx) == 0:
                continue
        L, c = int(seq_lens[r]), int(num_computed[r])
        if L != c + (t1 - t0):
            raise ValueError("seq_len must equal num_computed + query_len")
        kv = gather_request_kv(kv_cache, block_table[r], L)
        out[idx] = attend_rows(q[idx], kv, c + (idx - t0), scale)
    return out


def partial_attention(q_row: np.ndarray, kv_bits: np.ndarray, j0: int, j1: int,
                      scale: float):
    """Split-KV partial of one query row over keys j0..j1-1.

    Returns (m [Hq], l [Hq], o [Hq, D]) with m = max s, l = sum exp(s - m),
    o = sum exp(s - m) v / l. The pages only name split-KV ("PagedAttention
    v2", online softmax, [P1] §4.2 and §6.4); this is the plain reading."""
    Hq, D = q_row.shape
    Hkv = kv_bits.shape[2]
    G = Hq // Hkv
    m = np.empty(Hq)
    lsum = np.empty(Hq)
    o = np.empty((Hq, D))
    for h in range(Hq):
        g = h // G
        K = bf16_bits_to_f64(kv_bits[j0:j1, 0, g, :])
        V = bf16_bits_to_f64(kv_bits[j0:j1, 1, g, :])
        s = scale * (K @ bf16_bits_to_f64(q_row[h]))
        m[h] = s.max()
        w = np.exp(s - m[h])
        lsum[h] = w.sum()
        o[h] = (w @ V) / lsum[h]
    return m, lsum, o


def combine_partials(ms, ls, os_):
    """Merge split-KV partials: M = max m_p, weight_p = exp(m_p - M) l_p,
    o = sum_p weight_p o_p / sum_p weight_p."""
    ms = np.asarray(ms, dtype=np.float64)
    ls = np.asarray(ls, dtype=np.float64)
    os_ = np.asarray(os_, dtype=np.float64)
    M = ms.max(axis=0)
    wgt = np.exp(ms - M) * ls
    return (wgt[..., None] * os_).sum(axis=0) / wgt.sum(axis=0)[..., None]
