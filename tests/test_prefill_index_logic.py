"""CPU restatement of the prefill kernel's work items and tile rules.

A prefill request (c cached tokens, n > 1 new ones) is cut into work items
(q tile mt, kv head g). A tile holds QT = 128 / G consecutive queries times
the G q heads of kv head g: row r of the tile is query i0 + r // G and q
head g * G + r % G. Items of a request are numbered longest first: local
index l -> kv head l % Hkv, tile ntile - 1 - l // Hkv. The item's last
query sees keys 0 .. kv_len - 1, which take nkv = ceil(kv_len / 128) key
tiles. A key tile every row of the item sees whole needs no mask.

These tests restate those rules and check them against brute force.
"""

import numpy as np
import pytest


def items_of(c, n, Hkv, G):
    QT = 128 // G
    ntile = -(-n // QT)
    out = []
    for l in range(ntile * Hkv):
        g = l % Hkv
        mt = ntile - 1 - l // Hkv
        i0 = mt * QT
        i_last = min(i0 + QT, n) - 1
        kv_len = c + i_last + 1
        out.append({"g": g, "i0": i0, "kv_len": kv_len, "nkv": -(-kv_len // 128)})
    return out


def full_tile(kt, c, i0):
    """The kernel's test for a key tile that every row of the item sees whole
    (every chunk loaded)."""
    return kt * 128 + 127 <= c + i0


SHAPES = [(32, 8), (16, 8), (8, 8), (4, 4), (16, 2), (8, 1), (12, 3)]


@pytest.mark.parametrize("Hq,Hkv", SHAPES)
def test_items_cover_every_query_and_head_once(Hq, Hkv):
    G = Hq // Hkv
    QT = 128 // G
    rng = np.random.default_rng(Hq * 31 + Hkv)
    for _ in range(30):
        c, n = int(rng.integers(0, 3000)), int(rng.integers(2, 700))
        seen = np.zeros((n, Hq), dtype=np.int32)
        for it in items_of(c, n, Hkv, G):
            for r in range(128):
                qi = it["i0"] + r // G
                if qi < n:  # rows past the request's queries are not stored
                    seen[qi, it["g"] * G + r % G] += 1
        assert (seen == 1).all()


@pytest.mark.parametrize("Hq,Hkv", SHAPES)
def test_items_come_longest_first_and_key_tiles_are_tight(Hq, Hkv):
    G = Hq // Hkv
    QT = 128 // G
    rng = np.random.default_rng(Hq * 7 + Hkv)
    for _ in range(30):
        c, n = int(rng.integers(0, 3000)), int(rng.integers(2, 700))
        its = items_of(c, n, Hkv, G)
        nkv = [it["nkv"] for it in its]
        assert nkv == sorted(nkv, reverse=True)
        for it in its:
            # the last query of the tile sees key kv_len - 1 and no later one
            last_q = min(it["i0"] + QT, n) - 1
            assert it["kv_len"] == c + last_q + 1
            assert (it["nkv"] - 1) * 128 < it["kv_len"] <= it["nkv"] * 128


def test_full_tile_rule_is_exact():
    """A tile passes the no-mask test iff every key of it is visible to every
    query of the item (query i sees keys 0 .. c + i)."""
    rng = np.random.default_rng(5)
    for _ in range(400):
        c, n, G = int(rng.integers(0, 2000)), int(rng.integers(2, 500)), int(rng.choice([1, 2, 4, 8]))
        QT = 128 // G
        for it in items_of(c, n, 1, G):
            i0 = it["i0"]
            for kt in range(it["nkv"]):
                brute = all(kt * 128 + 127 <= c + i for i in range(i0, min(i0 + QT, n)))
                assert full_tile(kt, c, i0) == brute
