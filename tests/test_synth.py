"""Generator invariants (host only)."""

import numpy as np
import pytest

from paged_kv_cache_hkv_gb300 import synth
from paged_kv_cache_hkv_gb300.synth import BF16_NAN, RequestSpec, make_step


def _check_tables(step):
    B = step.block_size
    used = []
    for r, s in enumerate(step.specs):
        row = step.block_table[r]
        n = -(-s.seq_len // B)
        assert (row[:n] >= 0).all() and (row[:n] < step.num_blocks).all()
        assert (row[n:] == -1).all()
        used.append(row[:n])
    ids, counts = np.unique(np.concatenate(used), return_counts=True)
    assert np.array_equal(step.ref_cnt[ids], counts)
    assert step.ref_cnt.sum() == counts.sum()


def test_tiny_decode_shape_and_poison():
    st = synth.tiny_decode()
    assert st.num_blocks == 32
    assert list(st.seq_lens) == [5, 16, 17, 40]
    assert list(st.query_len) == [1, 1, 1, 1]
    # 5, 16, 17, 40 tokens need 1, 1, 2, 3 blocks (17 -> 2)
    assert [(row >= 0).sum() for row in st.block_table] == [1, 1, 2, 3]
    _check_tables(st)
    # unreferenced blocks are all poison
    free = np.setdiff1d(np.arange(32), st.block_table[st.block_table >= 0])
    assert (st.kv_cache[free] == BF16_NAN).all()
    # new tokens' places are poison until the write
    for blk, off in st.new_token_place:
        assert (st.kv_cache[blk, :, off] == BF16_NAN).all()
    assert st.q.shape == (4, 4, 64) and st.k.shape == (4, 2, 64)


def test_tiny_decode_tables_are_scattered_and_seeded():
    a, b = synth.tiny_decode(seed=1), synth.tiny_decode(seed=1)
    assert np.array_equal(a.block_table, b.block_table)
    assert np.array_equal(a.kv_cache, b.kv_cache)
    c = synth.tiny_decode(seed=9)
    assert not np.array_equal(a.block_table, c.block_table)


def test_history_slots_filled_and_tail_poisoned():
    st = make_step([RequestSpec(20, 3), RequestSpec(0, 5), RequestSpec(33, 1)],
                   num_q_heads=4, num_kv_heads=2, head_dim=8, seed=3)
    B = 16
    for r, s in enumerate(st.specs):
        row = st.block_table[r]
        # walk the table: token p is the p-th slot of the walk
        k = 0
        for blk in row[row >= 0]:
            for off in range(B):
                cell = st.kv_cache[blk, :, off]
                if k < s.num_computed:
                    assert not (cell == BF16_NAN).any()
                else:
                    assert (cell == BF16_NAN).all()
                k += 1


def test_identity_pool_order():
    st = make_step([RequestSpec(40, 1), RequestSpec(10, 2)], num_q_heads=2,
                   num_kv_heads=1, head_dim=8, shuffle_pool=False, seed=1)
    assert list(st.block_table[0][:3]) == [0, 1, 2]
    assert st.block_table[1][0] == 3


def test_prefix_sharing_metadata():
    st = synth.prefix_sharing(materialize=False)
    assert st.num_reqs == 128
    shared = st.block_table[:, :64]
    assert (shared == shared[0]).all()
    assert (st.ref_cnt[shared[0]] == 128).all()
    _check_tables(st)
    # every new token lands in a private block
    assert (st.ref_cnt[st.new_token_place[:, 0]] == 1).all()
    assert ((st.seq_lens >= 1024 + 16) & (st.seq_lens <= 1024 + 256)).all()


def test_mixed_step_metadata():
    st = synth.mixed_step(materialize=False)
    assert st.num_reqs == 1 + 8 + 1280
    assert st.num_tokens == 512 + 8 * 64 + 1280
    assert st.specs[0] == RequestSpec(1536, 512)
    assert all(s == RequestSpec(0, 64) for s in st.specs[1:9])
    dec = st.seq_lens[9:]
    assert ((dec >= 128) & (dec <= 2048)).all()
    assert st.max_query_len == 512 and st.max_seq_len == 2048
    _check_tables(st)
    assert st.num_blocks >= st.meta["needed_blocks"]


def test_llama_and_long_metadata():
    st = synth.llama_decode(materialize=False)
    assert st.num_blocks == 20000 and st.num_reqs == 64
    assert ((st.seq_lens >= 512) & (st.seq_lens <= 4096)).all()
    _check_tables(st)
    lc = synth.long_context(materialize=False)
    assert ((lc.seq_lens >= 32768) & (lc.seq_lens <= 131072)).all()
    _check_tables(lc)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.140625], np.float32)
    bits = synth.f32_to_bf16_bits(x)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa wins (1.0)
    assert list(bits) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x4049]
