"""CPU restatement of the decode kernel's integer work split and lane maps.

The split-KV decode kernel cuts the step's stream of (request, 16-key chunk)
positions into C equal ranges, one per CTA (every head of a request's chunk
is handled by the same CTA); a request that straddles ranges leaves one
partial per CTA that touched it, in slot (request + CTA) * V + virtual head,
and the combine kernel merges them. These tests walk that rule in Python for
many random shapes and check that every chunk is visited exactly once, that
the partial slots never collide, and that the combine finds exactly the CTAs
that wrote. A second test replays the warp reduce-scatter of partial dot
products lane by lane for every (head_dim, heads-per-warp) variant.
"""

import numpy as np
import pytest


def owner(x, N, C):
    """CTA whose range [floor(c*N/C), floor((c+1)*N/C)) holds position x."""
    return ((x + 1) * C + N - 1) // N - 1


def walk_split(nblk, V, C):
    """Replay every CTA's range: (request, chunk) visits and partial slots."""
    R = len(nblk)
    prefix = np.concatenate([[0], np.cumsum(nblk)]).astype(np.int64)
    N = int(prefix[-1])
    seen, slots = {}, {}
    for c in range(C):
        x0, x1 = c * N // C, (c + 1) * N // C
        if x0 >= x1:
            continue
        r = max(i for i in range(R) if prefix[i] <= x0)
        nb = int(prefix[r + 1] - prefix[r])
        assert nb > 0
        blk = x0 - int(prefix[r])
        x, new_piece = x0, True
        while x < x1:
            if new_piece:
                a = int(prefix[r])
                cf, cl = owner(a, N, C), owner(a + nb - 1, N, C)
                assert cf <= c <= cl
                if cf != cl:
                    for vg in range(V):
                        slot = (r + c) * V + vg
                        assert 0 <= slot < (R + C) * V
                        assert slot not in slots
                        slots[slot] = (r, vg)
            key = (r, blk)
            assert key not in seen
            seen[key] = c
            x += 1
            blk += 1
            new_piece = False
            if blk == nb:
                blk, new_piece = 0, True
                if x < x1:
                    r += 1
                    nb = int(prefix[r + 1] - prefix[r])
                    while nb == 0:
                        r += 1
                        nb = int(prefix[r + 1] - prefix[r])
    return prefix, N, seen, slots


@pytest.mark.parametrize("trial", range(60))
def test_stream_k_split_covers_every_chunk_once(trial):
    rng = np.random.default_rng(trial)
    R = int(rng.integers(1, 12))
    nblk = rng.integers(0, 30, size=R)
    if nblk.sum() == 0:
        nblk[0] = 3
    V = int(rng.choice([1, 2, 4, 8, 16]))
    C = int(rng.integers(1, 300))
    prefix, N, seen, slots = walk_split(nblk, V, C)
    assert len(seen) == N
    for r in range(R):
        nb = int(prefix[r + 1] - prefix[r])
        if nb == 0:
            continue
        a = int(prefix[r])
        cf, cl = owner(a, N, C), owner(a + nb - 1, N, C)
        writers = {seen[(r, b)] for b in range(nb)}
        if cf == cl:
            assert writers == {cf}
        else:
            # the combine skips CTAs whose range is empty
            used = {c for c in range(cf, cl + 1) if c * N // C != (c + 1) * N // C}
            assert writers == used
            for vg in range(V):
                assert all(slots[(r + c) * V + vg] == (r, vg) for c in used)


@pytest.mark.parametrize("D,GW", [(64, 1), (64, 2), (64, 4), (128, 1), (128, 2), (128, 4)])
def test_reduce_scatter_lane_map(D, GW):
    LPK = D // 8
    KPI = 32 // LPK
    KPL = 16 // KPI
    NV = GW * KPL
    NPL = NV // LPK if NV >= LPK else 1
    LPH = LPK // GW
    rng = np.random.default_rng(D + GW)
    vals = rng.standard_normal((32, NV))
    v = vals.copy()
    n, off = NV, LPK // 2
    while off >= 1:
        new = v.copy()
        if n >= 2:
            H = n // 2
            for lane in range(32):
                upper = (lane % LPK) & off
                peer = lane ^ off
                for i in range(H):
                    keep = v[lane, i + H] if upper else v[lane, i]
                    send = v[peer, i] if ((peer % LPK) & off) else v[peer, i + H]
                    new[lane, i] = keep + send
            n = H
        else:
            for lane in range(32):
                new[lane, 0] = v[lane, 0] + v[lane ^ off, 0]
        v = new
        off //= 2
    for lane in range(32):
        sub, li = lane // LPK, lane % LPK
        base = (li * NV) // LPK
        group = [sub * LPK + k for k in range(LPK)]
        for i in range(NPL):
            assert abs(v[lane, i] - vals[group, base + i].sum()) < 1e-9
            assert (base + i) // KPL == li // LPH  # a lane's scores stay in one head


@pytest.mark.parametrize("D,GW", [(64, 1), (64, 2), (64, 4), (128, 1), (128, 2), (128, 4)])
def test_select_free_reduce_scatter_with_permuted_lanes(D, GW):
    """The kernel stores, at register position p, the score of logical index
    p ^ M(lane) with M = (li * NV) // LPK (q heads and keys visited in a
    lane-dependent order). Then every halving stage is v[i] += shfl_xor(v[i+H])
    with no select, and lane li ends with logical indices M + i."""
    LPK = D // 8
    KPI = 32 // LPK
    KPL = 16 // KPI
    NV = GW * KPL
    NPL = NV // LPK if NV >= LPK else 1
    rng = np.random.default_rng(7 * D + GW)
    logical = rng.standard_normal((32, NV))  # lane's partial for logical index
    v = np.empty_like(logical)
    for lane in range(32):
        li = lane % LPK
        M = (li * NV) // LPK
        for p in range(NV):
            h, j = (p // KPL) ^ (M // KPL), (p % KPL) ^ (M % KPL)
            assert h < GW and j < KPL
            v[lane, p] = logical[lane, h * KPL + j]
    n, off = NV, LPK // 2
    while off >= 1:
        new = v.copy()
        if n >= 2:
            H = n // 2
            for lane in range(32):
                for i in range(H):
                    new[lane, i] = v[lane, i] + v[lane ^ off, i + H]
            n = H
        else:
            for lane in range(32):
                new[lane, 0] = v[lane, 0] + v[lane ^ off, 0]
        v = new
        off //= 2
    for lane in range(32):
        sub, li = lane // LPK, lane % LPK
        M = (li * NV) // LPK
        group = [sub * LPK + k for k in range(LPK)]
        for i in range(NPL):
            assert abs(v[lane, i] - logical[group, M + i].sum()) < 1e-9


def request_at(x, prefix):
    """Request holding stream position x."""
    return max(i for i in range(len(prefix) - 1) if prefix[i] <= x and prefix[i + 1] > x)


@pytest.mark.parametrize("trial", range(60))
def test_each_split_request_is_combined_by_exactly_one_boundary(trial):
    """Boundary CTA c (1 <= c < C) reads the request holding start(c) (empty
    ranges included) and combines it iff the request's first chunk belongs
    to CTA c - 1."""
    rng = np.random.default_rng(1000 + trial)
    R = int(rng.integers(1, 10))
    nblk = rng.integers(0, 25, size=R)
    if nblk.sum() == 0:
        nblk[-1] = 2
    C = int(rng.integers(1, 400))
    prefix = np.concatenate([[0], np.cumsum(nblk)]).astype(np.int64)
    N = int(prefix[-1])
    claimed = {}
    for c in range(1, C):
        x = c * N // C
        if x >= N:
            continue
        r = request_at(x, prefix)
        if owner(int(prefix[r]), N, C) == c - 1:
            assert r not in claimed
            claimed[r] = c
    for r in range(R):
        nb = int(prefix[r + 1] - prefix[r])
        if nb == 0:
            continue
        split = owner(int(prefix[r]), N, C) != owner(int(prefix[r]) + nb - 1, N, C)
        assert (r in claimed) == split


def warp_upper_index(a, n, x):
    """Host restatement of the decode kernel's warp search: 32 lanes test 32
    evenly spaced candidates per round; a ballot picks the interval."""
    lo, hi, rounds = 0, n, 0
    while hi - lo > 1:
        idx = [lo + (lane * (hi - lo) >> 5) for lane in range(32)]
        le = [a[i] <= x for i in idx]
        k = max(lane for lane in range(32) if le[lane])
        assert all(le[:k + 1]) and not any(le[k + 1:])  # the true lanes form a prefix
        hi = idx[k + 1] if k < 31 else hi
        lo = idx[k]
        rounds += 1
    return lo, rounds


@pytest.mark.parametrize("seed", range(20))
def test_warp_search_equals_bisection(seed):
    import bisect
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 5000))
    # chunk counts per request, many zero (requests with no decode chunks)
    counts = rng.integers(0, 5, size=n) * (rng.random(n) < 0.7)
    counts[rng.integers(0, n)] += 1  # at least one chunk
    a = np.concatenate([[0], np.cumsum(counts)]).tolist()
    N = a[n]
    for x in sorted(set([0, N - 1] + rng.integers(0, N, size=50).tolist())):
        got, rounds = warp_upper_index(a, n, x)
        want = bisect.bisect_right(a, x, 0, n) - 1  # largest r < n with a[r] <= x
        assert got == want
        assert a[got] <= x < a[got + 1]  # the request holding position x has chunks
        assert rounds <= int(np.ceil(np.log(max(n, 2)) / np.log(32))) + 2


def producer_walk(prefix, n_reqs, x0, x1):
    """Host restatement of the decode producer's walk over its range
    [x0, x1): the request at x0 from the warp search, then request by
    request with the next request's prefix loaded one request ahead; a next
    request with no chunks falls back to a scan."""
    r, _ = warp_upper_index(prefix, n_reqs, x0)
    pr = prefix[r]
    nblk = prefix[r + 1] - pr
    blk = x0 - pr
    nx_pn = prefix[r + 2] if r + 1 < n_reqs else -1
    out = []
    x = x0
    while x < x1:
        out.append((r, blk))
        x += 1
        blk += 1
        if blk == nblk:
            blk = 0
            if x < x1:
                pr += nblk
                if nx_pn - pr > 0:  # the lookahead's request has chunks
                    r += 1
                    nblk = nx_pn - pr
                else:
                    while True:
                        r += 1
                        nblk = prefix[r + 1] - prefix[r]
                        if nblk:
                            break
                    assert prefix[r] == pr  # empty requests add no chunks
                nx_pn = prefix[r + 2] if r + 1 < n_reqs else -1
    return out


@pytest.mark.parametrize("seed", range(20))
def test_producer_walk_with_lookahead_visits_its_range_in_order(seed):
    rng = np.random.default_rng(500 + seed)
    n = int(rng.integers(1, 300))
    counts = rng.integers(0, 6, size=n) * (rng.random(n) < 0.6)  # many empty requests
    counts[rng.integers(0, n)] += 1
    prefix = [0] + np.cumsum(counts).tolist()
    N = prefix[n]
    want = [(r, b) for r in range(n) for b in range(counts[r])]
    for C in sorted({1, 2, 3, 7, 152, int(rng.integers(1, 2 * N + 2))}):
        got = []
        for c in range(C):
            x0, x1 = c * N // C, (c + 1) * N // C
            if x0 < x1:
                got += producer_walk(prefix, n, x0, x1)
        assert got == want


def plan_bounds(nblk, C):
    """The plan kernel's rule for the request holding the first position of
    every decode CTA's range: request r (chunks [a, a + n) of the stream)
    holds the starts of CTAs ceil(a * C / N) .. ceil((a + n) * C / N) - 1."""
    N = int(sum(nblk))
    bound = [-1] * C
    if N == 0:
        return bound
    a = 0
    for r, n in enumerate(nblk):
        if n:
            c_lo = -(-(a * C) // N)
            c_hi = min(C, -(-((a + n) * C) // N))
            for c in range(c_lo, c_hi):
                bound[c] = r
        a += n
    return bound


@pytest.mark.parametrize("trial", range(200))
def test_plan_bounds_equal_the_search_of_each_range_start(trial):
    rng = np.random.default_rng(500 + trial)
    R = int(rng.integers(1, 40))
    nblk = rng.integers(0, 50, size=R) * (rng.random(R) < 0.8)
    C = int(rng.integers(1, 400))
    bound = plan_bounds(nblk, C)
    prefix = np.concatenate([[0], np.cumsum(nblk)])
    N = int(prefix[-1])
    for c in range(C):
        x0 = c * N // C
        if N == 0:
            assert bound[c] == -1
            continue
        # brute force: the request whose chunks hold position x0
        r = int(np.searchsorted(prefix, x0, side="right")) - 1
        while nblk[r] == 0:  # an empty request holds no position
            r += 1
        assert bound[c] == r, (c, x0, r, bound[c])
