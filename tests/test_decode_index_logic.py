"""CPU restatement of the decode kernel's integer work split and lane maps.

The split-KV decode kernel cuts the step's stream of (request, kv head,
block) positions into W equal ranges, one per warp; a (request, kv head)
that straddles ranges is merged by the combine kernel from one partial slot
per warp that touched it. These tests walk that rule in Python for many
random shapes and check that every block is visited exactly once, that the
partial slots never collide, and that the combine finds exactly the warps
that wrote. A second test replays the warp reduce-scatter of partial dot
products lane by lane for every (head_dim, heads-per-warp) variant.
"""

import numpy as np
import pytest


def owner(x, N, W):
    """Warp whose range [floor(w*N/W), floor((w+1)*N/W)) holds position x."""
    return ((x + 1) * W + N - 1) // N - 1


def walk_split(nblk, Hv, W):
    R = len(nblk)
    prefix = np.concatenate([[0], np.cumsum(nblk)]).astype(np.int64)
    N = Hv * int(prefix[-1])
    seen, slots = {}, {}
    for w in range(W):
        x0, x1 = w * N // W, (w + 1) * N // W
        if x0 >= x1:
            continue
        u = x0 // Hv
        r = max(i for i in range(R) if prefix[i] <= u)
        nb = int(prefix[r + 1] - prefix[r])
        assert nb > 0
        rem = x0 - Hv * int(prefix[r])
        vg, blk = rem // nb, rem % nb
        x, new_piece = x0, True
        while x < x1:
            if new_piece:
                a = Hv * int(prefix[r]) + vg * nb
                wf, wl = owner(a, N, W), owner(a + nb - 1, N, W)
                assert wf <= w <= wl
                if wf != wl:
                    slot = r * Hv + vg + w
                    assert 0 <= slot < R * Hv + W
                    assert slot not in slots
                    slots[slot] = (r, vg)
            key = (r, vg, blk)
            assert key not in seen
            seen[key] = w
            x += 1
            blk += 1
            new_piece = False
            if blk == nb:
                blk, new_piece = 0, True
                vg += 1
                if vg == Hv:
                    vg = 0
                    if x < x1:
                        r += 1
                        nb = int(prefix[r + 1] - prefix[r])
                        while nb == 0:
                            r += 1
                            nb = int(prefix[r + 1] - prefix[r])
    return prefix, N, seen, slots


@pytest.mark.parametrize("trial", range(60))
def test_stream_k_split_covers_every_block_once(trial):
    rng = np.random.default_rng(trial)
    R = int(rng.integers(1, 12))
    nblk = rng.integers(0, 30, size=R)
    if nblk.sum() == 0:
        nblk[0] = 3
    Hv = int(rng.choice([1, 2, 4, 8]))
    W = int(rng.integers(1, 300))
    prefix, N, seen, slots = walk_split(nblk, Hv, W)
    assert len(seen) == N
    for r in range(R):
        nb = int(prefix[r + 1] - prefix[r])
        for vg in range(Hv if nb else 0):
            a = Hv * int(prefix[r]) + vg * nb
            wf, wl = owner(a, N, W), owner(a + nb - 1, N, W)
            writers = {seen[(r, vg, b)] for b in range(nb)}
            if wf == wl:
                assert writers == {wf}
            else:
                # the combine skips warps whose range is empty
                used = {w for w in range(wf, wl + 1) if w * N // W != (w + 1) * N // W}
                assert writers == used
                assert all(slots[r * Hv + vg + w] == (r, vg) for w in used)


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


def pair_at(x, prefix, Hv):
    """(request, virtual head) holding stream position x."""
    u = x // Hv
    r = max(i for i in range(len(prefix) - 1) if prefix[i] <= u)
    nb = int(prefix[r + 1] - prefix[r])
    return r, (x - Hv * int(prefix[r])) // nb


@pytest.mark.parametrize("trial", range(60))
def test_each_split_pair_is_combined_by_exactly_one_boundary(trial):
    """Boundary warp w (1 <= w < W) reads the pair holding start(w) (empty
    ranges included) and combines it iff the pair's first block belongs to
    warp w - 1."""
    rng = np.random.default_rng(1000 + trial)
    R = int(rng.integers(1, 10))
    nblk = rng.integers(0, 25, size=R)
    if nblk.sum() == 0:
        nblk[-1] = 2
    Hv = int(rng.choice([1, 2, 4, 8]))
    W = int(rng.integers(1, 400))
    prefix = np.concatenate([[0], np.cumsum(nblk)]).astype(np.int64)
    N = Hv * int(prefix[-1])
    claimed = {}
    for w in range(1, W):
        x = w * N // W
        if x >= N:
            continue
        r, vg = pair_at(x, prefix, Hv)
        nb = int(prefix[r + 1] - prefix[r])
        a = Hv * int(prefix[r]) + vg * nb
        if owner(a, N, W) == w - 1:
            assert (r, vg) not in claimed
            claimed[(r, vg)] = w
    for r in range(R):
        nb = int(prefix[r + 1] - prefix[r])
        for vg in range(Hv if nb else 0):
            a = Hv * int(prefix[r]) + vg * nb
            split = owner(a, N, W) != owner(a + nb - 1, N, W)
            assert ((r, vg) in claimed) == split
