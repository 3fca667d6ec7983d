"""CPU restatement of the per-token slot rule of the fused write
(write_token_rows: one warp per new token, used by
pkv_slot_mapping_and_write and by the attention call's prologue).

The warp finds its token's request with a 32-way search of query_start_loc:
each round the 32 lanes test 32 evenly spaced candidates of the current
interval, and the interval shrinks to the gap between the last candidate
that is <= t and the next one. These tests replay that search lane by lane
and check it against a plain bisection, then check the whole per-token rule
(padding rows, rows before a non-zero query_start_loc[0], requests with
inconsistent lengths, missing table entries) against the oracle's slot
mapping and the separate slot-mapping kernel's rules.
"""

import numpy as np
import pytest

import oracle


def warp_upper_index(a, n, x):
    """Largest i in [0, n) with a[i] <= x (a non-decreasing, a[0] <= x), as
    32 lanes find it."""
    lo, hi = 0, n
    while hi - lo > 1:
        idx = [lo + (lane * (hi - lo)) // 32 for lane in range(32)]
        le = [a[i] <= x for i in idx]
        k = max(lane for lane in range(32) if le[lane])  # lane 0 (idx lo) always is
        idx_next = idx[k + 1] if k < 31 else hi
        lo, hi = idx[k], idx_next if k < 31 else hi
    return lo


def token_slot(t, qsl, num_computed, block_table, num_tokens, B, num_blocks):
    """The fused write's slot of token t, -1 when it writes nothing."""
    R = len(num_computed)
    qend, qfirst = int(qsl[R]), int(qsl[0])
    if not (qfirst <= t < qend):
        return -1
    r = warp_upper_index(qsl, R, t)
    q0, q1, c = int(qsl[r]), int(qsl[r + 1]), int(num_computed[r])
    if q0 < 0 or q1 < q0 or q1 > num_tokens or c < 0 or (r == 0 and q0 != 0):
        return -1
    pos = c + (t - q0)
    lb = pos // B
    if lb >= block_table.shape[1]:
        return -1
    phys = int(block_table[r, lb])
    if phys < 0 or phys >= num_blocks:
        return -1
    return phys * B + pos % B


def test_search_matches_bisection():
    rng = np.random.default_rng(0)
    for _ in range(3000):
        n = int(rng.integers(1, 3000))
        steps = rng.integers(0, 4, size=n)
        a = np.concatenate([[0], np.cumsum(steps)]).astype(np.int64)
        x = int(rng.integers(0, a[-1] + 2))
        got = warp_upper_index(a, n, x)
        ref = int(np.searchsorted(a[:n], x, side="right")) - 1
        assert got == ref, (n, x)


def random_batch(rng, R, B, num_blocks):
    qlen = rng.choice([0, 1, 1, 1, 2, 7, 33], size=R)
    qlen[0] = max(1, qlen[0])
    computed = rng.integers(0, 300, size=R)
    qsl = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    width = int(np.max((computed + qlen + B - 1) // B)) + 1
    table = np.full((R, width), -1, dtype=np.int32)
    perm = rng.permutation(num_blocks)
    k = 0
    for r in range(R):
        for j in range((int(computed[r] + qlen[r]) + B - 1) // B):
            table[r, j] = perm[k % num_blocks]
            k += 1
    return qsl, computed.astype(np.int32), table


@pytest.mark.parametrize("B", [8, 16, 32])
def test_rule_matches_the_oracle_on_valid_batches(B):
    rng = np.random.default_rng(B)
    for _ in range(60):
        R = int(rng.integers(1, 60))
        qsl, nc, table = random_batch(rng, R, B, num_blocks=4096)
        T = int(qsl[-1])
        ref = oracle.slot_mapping(table, qsl, nc, B)
        pad = int(rng.integers(0, 4))
        got = [token_slot(t, qsl, nc, table, T + pad, B, 4096) for t in range(T + pad)]
        assert got[:T] == ref.tolist()
        assert all(s == -1 for s in got[T:])  # padding rows


def test_bad_lengths_and_missing_entries_give_minus_one():
    rng = np.random.default_rng(7)
    B = 16
    qsl, nc, table = random_batch(rng, 12, B, num_blocks=512)
    T = int(qsl[-1])
    ref = oracle.slot_mapping(table, qsl, nc, B)
    # a request with a negative cached count: all its rows -1, the rest exact
    bad = int(np.flatnonzero(np.diff(qsl) > 0)[1])
    nc2 = nc.copy()
    nc2[bad] = -1
    got = [token_slot(t, qsl, nc2, table, T, B, 512) for t in range(T)]
    rows = range(int(qsl[bad]), int(qsl[bad + 1]))
    for t in range(T):
        assert got[t] == (-1 if t in rows else ref[t])
    # a missing table entry or one outside the pool: that token only
    t = int(qsl[bad])
    r, pos = bad, int(nc[bad])
    for value in (-1, 512, 10 ** 6):
        tb = table.copy()
        tb[r, pos // B] = value
        got = [token_slot(x, qsl, nc, tb, T, B, 512) for x in range(T)]
        # the tokens of request r whose position falls in that table entry
        hit = [x for x in range(int(qsl[r]), int(qsl[r + 1]))
               if (int(nc[r]) + x - int(qsl[r])) // B == pos // B]
        for x in range(T):
            assert got[x] == (-1 if x in hit else ref[x])


def test_rows_before_a_non_zero_first_offset():
    # query_start_loc = [1, 2, 6]: request 0 is inconsistent (it must start at
    # 0) and row 0 belongs to no request; request 1 is fine
    qsl = np.array([1, 2, 6], dtype=np.int32)
    nc = np.array([5, 30], dtype=np.int32)
    table = np.arange(2 * 4, dtype=np.int32).reshape(2, 4)
    got = [token_slot(t, qsl, nc, table, 6, 16, 64) for t in range(6)]
    assert got[:2] == [-1, -1]
    assert got[2:] == [table[1, (30 + i) // 16] * 16 + (30 + i) % 16 for i in range(4)]
