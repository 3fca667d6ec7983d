"""Seeded synthetic inputs for one paged-attention step.

This module builds the inputs that both the CUDA path and the CPU oracle
consume: the physical KV block pool, per-request block tables, the varlen
batch metadata and the bf16 Q/K/V values. It holds none of the attention
arithmetic and it never computes a slot id; it only plays the role of the
block allocator and of the model layer that produces Q/K/V.

What it mirrors on the pages:

* "vllm v1 源码精读（三）" §3.2-3.3: the pool is one tensor
  ``kv_cache[num_blocks, 2, block_size, num_kv_heads, head_dim]`` (index 0 = K,
  1 = V), allocated once; free blocks sit in a queue and allocation pops from
  its head (``popleft``).
* same page §3.4: the block table is int32 ``[num_reqs, max_blocks]`` with
  ``-1`` in unused entries.
* "Inside vLLM" §3.3: a request needs ceil(tokens / 16) blocks (17 tokens -> 2).
* "vLLM 架构源码解析（一）" §4.3.1 and "Inside vLLM" §3.6: prefix sharing puts
  the same physical block ids at the head of several tables (ref_cnt > 1).
* "vllm v1 源码精读（三）" §4.2 and "Inside vLLM" §3.4: all requests' new
  tokens are concatenated into one varlen batch; ``query_start_loc`` marks the
  boundaries, ``seq_lens`` counts cached plus new tokens.

Allocation is simulated block by block (a new block is taken when the current
one is full, as nano-vllm's ``may_append`` does), and every history token is
placed at the (block, offset) the walk hands out. Slots that hold no token are
filled with a bf16 NaN so that any read of them shows up in the output.

Values are N(0, 1) drawn in fp32 and rounded to bf16 (round to nearest even).
bf16 tensors are carried as ``uint16`` bit patterns.
"""

from __future__ import annotations

import math
from collections import deque
from dataclasses import dataclass, field

import numpy as np

BF16_NAN = np.uint16(0x7FC0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits.

    Only finite inputs are expected (normal draws)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


@dataclass(frozen=True)
class RequestSpec:
    """One request in the step.

    num_computed: tokens already in the cache when the step starts.
    query_len:    new tokens scheduled this step (1 = decode).
    shares_prefix: the request's first ``prefix_tokens`` tokens live in the
                   shared prefix blocks (they must be whole blocks).
    """

    num_computed: int
    query_len: int
    shares_prefix: bool = False

    @property
    def seq_len(self) -> int:
        return self.num_computed + self.query_len


@dataclass
class PagedStep:
    """Every input of one mixed step, host side.

    kv_cache, q, k, v are uint16 bf16 bit patterns.
    """

    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    specs: list
    num_computed: np.ndarray  # int32 [R]
    query_len: np.ndarray  # int32 [R]
    seq_lens: np.ndarray  # int32 [R]
    query_start_loc: np.ndarray  # int32 [R+1]
    block_table: np.ndarray  # int32 [R, max_blocks], -1 padded
    ref_cnt: np.ndarray  # int32 [num_blocks]
    kv_cache: np.ndarray | None  # uint16 [NB, 2, B, Hkv, D]
    q: np.ndarray | None  # uint16 [T, Hq, D]
    k: np.ndarray | None  # uint16 [T, Hkv, D]
    v: np.ndarray | None  # uint16 [T, Hkv, D]
    scale: float
    prefix_tokens: int = 0
    # per new token: the (physical block, offset) the allocator handed out;
    # used only by generator self-checks, never passed to a kernel.
    new_token_place: np.ndarray | None = None  # int64 [T, 2]
    meta: dict = field(default_factory=dict)

    @property
    def num_reqs(self) -> int:
        return len(self.specs)

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def max_blocks_per_req(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_query_len(self) -> int:
        return int(self.query_len.max()) if len(self.query_len) else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if len(self.seq_lens) else 0


class _FreeQueue:
    """Free-block queue: allocation pops from the head (popleft)."""

    def __init__(self, order: np.ndarray):
        self._q = deque(int(b) for b in order)

    def popleft(self) -> int:
        if not self._q:
            raise RuntimeError("block pool exhausted")
        return self._q.popleft()

    def __len__(self) -> int:
        return len(self._q)


def _walk(blocks_out: list, free: _FreeQueue, n_tokens: int, B: int,
          first_fill: int = 0):
    """Hand out (block, offset) for ``n_tokens`` appended tokens.

    ``blocks_out`` is the request's block list; when it is empty or its last
    block is full (``first_fill == B``) a new block is popped from the free
    queue. Returns (block ids, offsets) per token and the fill of the last
    block."""
    blk_ids = []
    offs = []
    fill = first_fill if blocks_out else B
    left = n_tokens
    while left > 0:
        if fill == B:
            blocks_out.append(free.popleft())
            fill = 0
        take = min(B - fill, left)
        blk_ids.append(np.full(take, blocks_out[-1], dtype=np.int64))
        offs.append(np.arange(fill, fill + take, dtype=np.int64))
        fill += take
        left -= take
    if blk_ids:
        return np.concatenate(blk_ids), np.concatenate(offs), fill
    return np.zeros(0, np.int64), np.zeros(0, np.int64), fill


def make_step(specs, *, num_q_heads: int, num_kv_heads: int, head_dim: int,
              block_size: int = 16, num_blocks: int | None = None,
              pool_slack: float = 1.1, seed: int = 0, shuffle_pool: bool = True,
              prefix_tokens: int = 0, table_width: int | None = None,
              materialize: bool = True, scale: float | None = None,
              chunk_tokens: int = 32768, key_drift: float = 0.0,
              spike: float = 0.0) -> PagedStep:
    """Build one step's inputs.

    specs: list of RequestSpec, in batch order.
    num_blocks: pool size; default ceil(needed * pool_slack).
    shuffle_pool: the free queue starts as a seeded permutation of the pool
        (physically scattered tables); False gives the identity order.
    prefix_tokens: length of the shared prefix (whole blocks) used by specs
        with ``shares_prefix``.
    materialize: also draw the pool contents and Q/K/V (False gives only the
        metadata, for cheap host-side checks).
    key_drift: value profile with scores that move along the sequence. Every
        K row (cached and new) at absolute position p gets ``key_drift * p``
        added to its first head_dim/2 components, and those components of q
        head h are shifted by +1, 0 or -1 for h % 3 = 0, 1, 2. So the scores
        of one head in three climb steadily with the key position (the
        running max of an online softmax keeps moving), one in three stay
        level and one in three fall.
    spike: value profile with one key that outweighs all others. For each
        decode request (one new token) with cached tokens of its own, one
        cached key near the end of its context (within its last 48 cached
        positions, outside any shared prefix) is replaced, in every kv head,
        by ``spike`` times the sum of that kv head's q rows of the request, so
        its score dwarfs every other score of the request. 0 = off.
    """
    B = block_size
    Hq, Hkv, D = num_q_heads, num_kv_heads, head_dim
    specs = list(specs)
    R = len(specs)
    if Hq % Hkv:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    if prefix_tokens % B:
        raise ValueError("the shared prefix must be whole blocks")
    for s in specs:
        if s.query_len < 0 or s.num_computed < 0:
            raise ValueError("negative length")
        if s.shares_prefix and s.num_computed < prefix_tokens:
            raise ValueError("a sharing request must have the whole prefix cached")

    any_shared = any(s.shares_prefix for s in specs)
    shared_blocks = prefix_tokens // B if any_shared else 0
    needed = shared_blocks
    for s in specs:
        own = s.seq_len - (prefix_tokens if s.shares_prefix else 0)
        needed += -(-own // B)
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(needed * pool_slack)))
    if needed > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {needed}")

    ss = np.random.SeedSequence(seed)
    s_pool, s_prefix, s_hist, s_new, s_spike = ss.spawn(5)
    rng_pool = np.random.Generator(np.random.PCG64(s_pool))
    order = rng_pool.permutation(num_blocks) if shuffle_pool else np.arange(num_blocks)
    free = _FreeQueue(order)
    ref_cnt = np.zeros(num_blocks, np.int32)

    # shared prefix blocks: allocated once, referenced by every sharing request
    shared_list: list = []
    shared_blk = shared_off = np.zeros(0, np.int64)
    if shared_blocks:
        shared_blk, shared_off, _ = _walk(shared_list, free, prefix_tokens, B)

    tables = []
    hist_blk, hist_off, hist_pos = [], [], []
    new_blk, new_off = [], []
    for s in specs:
        blocks: list = []
        start = 0
        fill = B
        if s.shares_prefix:
            blocks.extend(shared_list)
            start = prefix_tokens
            fill = B  # prefix is whole blocks: the next token opens a new block
        hb, ho, fill = _walk(blocks, free, s.num_computed - start, B, fill)
        nb, no, fill = _walk(blocks, free, s.query_len, B, fill)
        hist_blk.append(hb)
        hist_off.append(ho)
        hist_pos.append(np.arange(start, s.num_computed, dtype=np.int64))
        new_blk.append(nb)
        new_off.append(no)
        tables.append(blocks)
        for b in blocks:
            ref_cnt[b] += 1

    width = max([len(t) for t in tables] + [1])
    if table_width is not None:
        if table_width < width:
            raise ValueError("table_width too small")
        width = table_width
    block_table = np.full((R, width), -1, np.int32)
    for i, t in enumerate(tables):
        block_table[i, : len(t)] = t

    num_computed = np.array([s.num_computed for s in specs], np.int32)
    query_len = np.array([s.query_len for s in specs], np.int32)
    seq_lens = (num_computed + query_len).astype(np.int32)
    qsl = np.zeros(R + 1, np.int32)
    qsl[1:] = np.cumsum(query_len)
    T = int(qsl[-1])

    new_place = np.stack([np.concatenate(new_blk) if new_blk else np.zeros(0, np.int64),
                          np.concatenate(new_off) if new_off else np.zeros(0, np.int64)],
                         axis=1)
    # no new token may land in a block that another request also references
    # (copy-on-write: shared blocks are read-only for the step)
    if T and np.any(ref_cnt[new_place[:, 0]] > 1):
        raise AssertionError("a new token would be written into a shared block")
    if T and len(np.unique(new_place[:, 0] * B + new_place[:, 1])) != T:
        raise AssertionError("two new tokens were given the same place")

    step = PagedStep(
        num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=B,
        num_blocks=num_blocks, specs=specs, num_computed=num_computed,
        query_len=query_len, seq_lens=seq_lens, query_start_loc=qsl,
        block_table=block_table, ref_cnt=ref_cnt, kv_cache=None, q=None, k=None,
        v=None, scale=float(scale if scale is not None else 1.0 / math.sqrt(D)),
        prefix_tokens=prefix_tokens if any_shared else 0, new_token_place=new_place,
        meta={"seed": seed, "needed_blocks": needed},
    )
    if not materialize:
        return step

    pool = np.full((num_blocks, 2, B, Hkv, D), BF16_NAN, np.uint16)

    def fill_rows(rng, blk, off):
        n = len(blk)
        for c0 in range(0, n, chunk_tokens):
            c1 = min(n, c0 + chunk_tokens)
            vals = f32_to_bf16_bits(
                rng.standard_normal((c1 - c0, 2, Hkv, D), dtype=np.float32))
            pool[blk[c0:c1], 0, off[c0:c1]] = vals[:, 0]
            pool[blk[c0:c1], 1, off[c0:c1]] = vals[:, 1]

    if shared_blocks:
        fill_rows(np.random.Generator(np.random.PCG64(s_prefix)), shared_blk, shared_off)
    rng_hist = np.random.Generator(np.random.PCG64(s_hist))
    if hist_blk:
        fill_rows(rng_hist, np.concatenate(hist_blk), np.concatenate(hist_off))

    rng_new = np.random.Generator(np.random.PCG64(s_new))
    step.q = f32_to_bf16_bits(rng_new.standard_normal((T, Hq, D), dtype=np.float32))
    step.k = f32_to_bf16_bits(rng_new.standard_normal((T, Hkv, D), dtype=np.float32))
    step.v = f32_to_bf16_bits(rng_new.standard_normal((T, Hkv, D), dtype=np.float32))
    step.kv_cache = pool
    if key_drift:
        _apply_key_drift(step, key_drift, shared_blk, shared_off, hist_blk, hist_off, hist_pos)
    if spike:
        _apply_spike(step, spike, hist_blk, hist_off, hist_pos,
                     np.random.Generator(np.random.PCG64(s_spike)))
    return step


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact fp32 value of bf16 bit patterns (a bf16 is the top half of an
    fp32)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _apply_key_drift(step, drift, shared_blk, shared_off, hist_blk, hist_off, hist_pos):
    """The ``key_drift`` value profile (see make_step)."""
    D, Hq = step.head_dim, step.num_q_heads
    half = D // 2
    pool = step.kv_cache

    def drift_rows(rows_bits, pos):
        vals = bf16_bits_to_f32(rows_bits[..., :half]) + np.float32(drift) * pos.astype(
            np.float32).reshape((-1,) + (1,) * (rows_bits.ndim - 1))
        out = rows_bits.copy()
        out[..., :half] = f32_to_bf16_bits(vals)
        return out

    if len(shared_blk):
        pos = np.arange(len(shared_blk), dtype=np.int64)
        pool[shared_blk, 0, shared_off] = drift_rows(pool[shared_blk, 0, shared_off], pos)
    for blk, off, pos in zip(hist_blk, hist_off, hist_pos):
        if len(blk):
            pool[blk, 0, off] = drift_rows(pool[blk, 0, off], pos)
    new_pos = np.concatenate([np.arange(c, c + n, dtype=np.int64) for c, n in
                              zip(step.num_computed, step.query_len)] + [np.zeros(0, np.int64)])
    if len(new_pos):
        step.k = drift_rows(step.k, new_pos)
    shift = np.array([1.0, 0.0, -1.0], np.float32)[np.arange(Hq) % 3]
    qv = bf16_bits_to_f32(step.q[..., :half]) + shift[None, :, None]
    step.q = step.q.copy()
    step.q[..., :half] = f32_to_bf16_bits(qv)
    step.meta["key_drift"] = float(drift)


def _apply_spike(step, spike, hist_blk, hist_off, hist_pos, rng):
    """The ``spike`` value profile (see make_step)."""
    G = step.num_q_heads // step.num_kv_heads
    placed = {}
    for r in range(step.num_reqs):
        if step.query_len[r] != 1 or len(hist_pos[r]) == 0:
            continue
        j = len(hist_pos[r]) - 1 - int(rng.integers(0, min(len(hist_pos[r]), 48)))
        t = int(step.query_start_loc[r])
        qf = bf16_bits_to_f32(step.q[t]).reshape(step.num_kv_heads, G, step.head_dim)
        krow = f32_to_bf16_bits(np.float32(spike) * qf.sum(axis=1))
        step.kv_cache[hist_blk[r][j], 0, hist_off[r][j]] = krow
        placed[r] = int(hist_pos[r][j])
    step.meta["spike"] = float(spike)
    step.meta["spike_pos"] = placed


# ---------------------------------------------------------------------------
# The five workloads (Llama-3-8B layer shapes: 32 q heads, 8 kv heads, d=128)
# ---------------------------------------------------------------------------

LLAMA = dict(num_q_heads=32, num_kv_heads=8, head_dim=128)


def _decodes(lengths):
    return [RequestSpec(int(L) - 1, 1) for L in lengths]


def tiny_decode(seed: int = 1, **kw) -> PagedStep:
    """4 decodes, contexts {5,16,17,40}, 4 q / 2 kv heads, d=64, pool of 32
    blocks handed out in a seeded random order."""
    return make_step(_decodes([5, 16, 17, 40]), num_q_heads=4, num_kv_heads=2,
                     head_dim=64, num_blocks=32, seed=seed, **kw)


def llama_decode(seed: int = 2, **kw) -> PagedStep:
    """64 decodes, contexts uniform in [512, 4096], pool of 20000 blocks."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(512, 4096, size=64, endpoint=True)
    return make_step(_decodes(lengths), num_blocks=20000, seed=seed, **LLAMA, **kw)


def mixed_step_specs(seed: int = 3, num_decodes: int = 1280):
    rng = np.random.default_rng(seed)
    specs = [RequestSpec(1536, 512)]
    specs += [RequestSpec(0, 64) for _ in range(8)]
    lengths = rng.integers(128, 2048, size=num_decodes, endpoint=True)
    specs += _decodes(lengths)
    return specs


def mixed_step(seed: int = 3, num_decodes: int = 1280, **kw) -> PagedStep:
    """One chunked-prefill step: a 512-token chunk over 1536 cached tokens,
    8 fresh 64-token prefills and ``num_decodes`` decodes with contexts
    uniform in [128, 2048]."""
    return make_step(mixed_step_specs(seed, num_decodes), seed=seed, **LLAMA, **kw)


def mixed_step_2048(seed: int = 3, **kw) -> PagedStep:
    """The mixed step under its 2048-token-budget reading: the same chunk and
    prefills with 1024 decodes instead of 1280."""
    return mixed_step(seed, num_decodes=1024, **kw)


def prefill_rows(seed: int = 3, **kw) -> PagedStep:
    """The mixed step's prefill requests alone: the 512-token chunk over 1536
    cached tokens and the 8 fresh 64-token prefills."""
    return make_step(mixed_step_specs(seed, num_decodes=0), seed=seed, **LLAMA, **kw)


def prefix_sharing(seed: int = 4, **kw) -> PagedStep:
    """128 decodes sharing a 1024-token (64-block) prefix, private suffixes of
    16..256 tokens."""
    rng = np.random.default_rng(seed)
    suffix = rng.integers(16, 256, size=128, endpoint=True)
    specs = [RequestSpec(1024 + int(s) - 1, 1, shares_prefix=True) for s in suffix]
    return make_step(specs, prefix_tokens=1024, seed=seed, **LLAMA, **kw)


def long_context(seed: int = 5, **kw) -> PagedStep:
    """8 decodes with contexts uniform in [32768, 131072]."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(32768, 131072, size=8, endpoint=True)
    return make_step(_decodes(lengths), seed=seed, **LLAMA, **kw)


def long_prefill(seed: int = 6, **kw) -> PagedStep:
    """Prefill at scale: 4 prompt chunks of 2048 new tokens over 6144 cached
    tokens each (keys up to 8192 per query), no decodes."""
    return make_step([RequestSpec(6144, 2048) for _ in range(4)], seed=seed, **LLAMA, **kw)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "llama_decode": llama_decode,
    "mixed_step": mixed_step,
    "mixed_step_2048": mixed_step_2048,
    "prefill_rows": prefill_rows,
    "prefix_sharing": prefix_sharing,
    "long_context": long_context,
    "long_prefill": long_prefill,
}
