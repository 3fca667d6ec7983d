"""Pins for the CPU oracle: values the pages print, closed forms, brute force.

Each test checks the oracle against something other than itself. The helpers
here place tokens by walking the block table entry by entry (no slot
arithmetic), and the brute-force attention is written with scalar loops over
contiguous per-request arrays (no paging at all).
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import paged_oracle as po
from paged_kv_cache_hkv_gb300.synth import BF16_NAN, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# helpers independent of the oracle
# ---------------------------------------------------------------------------

def walk_places(table_row, n_tokens, B=16):
    """(block, offset) of tokens 0..n-1, by walking the table entries in
    order and filling each block's offsets one after another."""
    places = []
    for blk in table_row:
        for off in range(B):
            if len(places) == n_tokens:
                return places
            places.append((int(blk), off))
    assert len(places) == n_tokens
    return places


def scatter(pool, table_row, kv_seq):
    """Store a contiguous [L, 2, Hkv, D] sequence into the pool along the
    table walk."""
    for j, (blk, off) in enumerate(walk_places(table_row, len(kv_seq), pool.shape[2])):
        pool[blk, :, off] = kv_seq[j]


def to_f(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def textbook_attention(q_rows, kv_seq, positions, scale):
    """Scalar-loop softmax attention on contiguous data.

    q_rows [n, Hq, D] bits, kv_seq [L, 2, Hkv, D] bits. Consecutive q heads
    share a kv head (head map h // (Hq / Hkv))."""
    qf, kf, vf = to_f(q_rows), to_f(kv_seq[:, 0]), to_f(kv_seq[:, 1])
    n, Hq, D = qf.shape
    Hkv = kf.shape[1]
    G = Hq // Hkv
    out = np.zeros((n, Hq, D))
    for i in range(n):
        for h in range(Hq):
            g = h // G
            scores = []
            for j in range(int(positions[i]) + 1):
                acc = 0.0
                for d in range(D):
                    acc += qf[i, h, d] * kf[j, g, d]
                scores.append(scale * acc)
            mx = max(scores)
            ws = [math.exp(s - mx) for s in scores]
            tot = sum(ws)
            for d in range(D):
                acc = 0.0
                for j, w in enumerate(ws):
                    acc += w * vf[j, g, d]
                out[i, h, d] = acc / tot
    return out


def rand_bits(rng, shape):
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def build_case(rng, lens_q, lens_c, Hq, Hkv, D, NB=64, B=16, shuffle=True):
    """Random small batch built without any slot arithmetic.

    Returns dict with pool (post-write contents), tables, metadata, q and the
    contiguous per-request sequences."""
    R = len(lens_q)
    order = rng.permutation(NB) if shuffle else np.arange(NB)
    nxt = 0
    seqs, tables = [], []
    for r in range(R):
        L = lens_c[r] + lens_q[r]
        nblk = 0
        row = []
        while nblk * B < L:
            row.append(int(order[nxt]))
            nxt += 1
            nblk += 1
        tables.append(row)
        seqs.append(rand_bits(rng, (L, 2, Hkv, D)))
    width = max(len(t) for t in tables)
    bt = np.full((R, width + 1), -1, np.int32)
    for r, t in enumerate(tables):
        bt[r, : len(t)] = t
    pool = np.full((NB, 2, B, Hkv, D), BF16_NAN, np.uint16)
    for r in range(R):
        scatter(pool, bt[r], seqs[r])
    qsl = np.zeros(R + 1, np.int32)
    qsl[1:] = np.cumsum(lens_q)
    q = rand_bits(rng, (int(qsl[-1]), Hq, D))
    return dict(pool=pool, bt=bt, seqs=seqs, qsl=qsl, q=q,
                nc=np.array(lens_c, np.int32),
                sl=np.array([c + n for c, n in zip(lens_c, lens_q)], np.int32))


# ---------------------------------------------------------------------------
# the oracle's input decoder
# ---------------------------------------------------------------------------

# bfloat16 is the top half of an IEEE-754 binary32: sign, 8 exponent bits, 7
# fraction bits. Each pattern below is decoded by hand from that definition.
BF16_LITERALS = [
    (0x3F80, 1.0),             # exponent 127, fraction 0
    (0xC020, -2.5),            # sign, exponent 128, fraction 0b0100000 -> -(1 + 1/4) * 2
    (0x4049, 3.140625),        # exponent 128, fraction 0b1001001 -> (1 + 73/128) * 2
    (0x0000, 0.0),
    (0x8000, -0.0),
    (0x0080, 2.0 ** -126),     # smallest normal
    (0x0001, 2.0 ** -133),     # smallest subnormal: 2^-126 * 2^-7
    (0x7F7F, (2 - 2.0 ** -7) * 2.0 ** 127),  # largest finite
    (0x7F80, math.inf),
    (0xFF80, -math.inf),
]


def test_bf16_decoder_literal_values():
    bits = np.array([b for b, _ in BF16_LITERALS], np.uint16)
    got = oracle.bf16_bits_to_f64(bits)
    for (b, want), g in zip(BF16_LITERALS, got):
        assert g == want and math.copysign(1.0, g) == math.copysign(1.0, want), hex(b)
    nan = oracle.bf16_bits_to_f64(np.array([0x7FC0, 0xFFC1], np.uint16))
    assert np.isnan(nan).all()


# ---------------------------------------------------------------------------
# slot and block arithmetic
# ---------------------------------------------------------------------------

def test_worked_slot_examples():
    g = _load("slot_mapping_worked_example.json")
    bt = np.array(g["block_table"], np.int32)
    for ex in g["slots"]:
        assert oracle.slot_of(bt[ex["request"]], ex["pos"], g["block_size"]) == ex["slot"]
    assert list(oracle.blocks_for_tokens(g["prompt_tokens"], g["block_size"])) == g["blocks_needed"]
    # the table's used width is exactly the blocks each prompt needs
    used = [(row >= 0).sum() for row in bt]
    assert used == g["blocks_needed"]


def test_block_arithmetic_values():
    g = _load("block_arithmetic.json")
    bn = g["blocks_needed"]
    assert int(oracle.blocks_for_tokens(bn["tokens"], bn["block_size"])) == bn["blocks"]
    a, b = g["kv_bytes_per_token_layer"]
    assert oracle.kv_bytes_per_token(a["num_kv_heads"], a["head_dim"], a["dtype_bytes"]) == a["bytes"]
    assert a["bytes"] * a["layers"] == a["bytes_all_layers"]
    per_block = (oracle.kv_bytes_per_token(b["num_kv_heads"], b["head_dim"], b["dtype_bytes"])
                 * b["block_size"] * b["layers"])
    assert per_block == b["bytes_per_block_all_layers"]


# block sizes the pages weigh against each other (vLLM 架构源码解析（一）, §5.1)
BLOCK_SIZES = [8, 16, 32]


@pytest.mark.parametrize("B", BLOCK_SIZES)
def test_last_block_fill_matches_walk(B):
    for n in range(1, 200):
        places = walk_places(list(range(100)), n, B)
        nblocks = len({p[0] for p in places})
        assert int(oracle.blocks_for_tokens(n, B)) == nblocks
        assert int(oracle.last_block_fill(n, B)) == sum(1 for p in places if p[0] == places[-1][0])


@pytest.mark.parametrize("B", BLOCK_SIZES)
def test_slot_of_equals_table_walk(B):
    rng = np.random.default_rng(11)
    for _ in range(20):
        row = rng.permutation(500)[:40]
        n = int(rng.integers(1, 40 * B))
        for pos, (blk, off) in enumerate(walk_places(row, n, B)):
            assert oracle.slot_of(row, pos, B) == blk * B + off


@pytest.mark.parametrize("B", BLOCK_SIZES)
def test_slot_mapping_varlen_batch(B):
    rng = np.random.default_rng(12)
    case = build_case(rng, [1, 7, 33, 1], [40, 0, 17, 15], 4, 2, 8, B=B)
    sm = oracle.slot_mapping(case["bt"], case["qsl"], case["nc"], B)
    for r in range(len(case["nc"])):
        places = walk_places(case["bt"][r], int(case["sl"][r]), B)
        for i, t in enumerate(range(case["qsl"][r], case["qsl"][r + 1])):
            blk, off = places[int(case["nc"][r]) + i]
            assert sm[t] == blk * B + off


# ---------------------------------------------------------------------------
# the write
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B", BLOCK_SIZES)
def test_kv_write_roundtrip_and_untouched(B):
    rng = np.random.default_rng(13)
    NB, Hkv, D = 12, 2, 8
    pool = rand_bits(rng, (NB, 2, B, Hkv, D))
    N = 30
    slots = rng.permutation(NB * B)[:N].astype(np.int64)
    slots[[3, 17]] = -1  # padding rows are skipped
    k, v = rand_bits(rng, (N, Hkv, D)), rand_bits(rng, (N, Hkv, D))
    out = oracle.kv_write(pool, k, v, slots)
    flat_in = pool.transpose(0, 2, 1, 3, 4).reshape(NB * B, 2, Hkv, D)
    flat_out = out.transpose(0, 2, 1, 3, 4).reshape(NB * B, 2, Hkv, D)
    written = set()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        written.add(int(s))
        assert np.array_equal(flat_out[s, 0], k[t])
        assert np.array_equal(flat_out[s, 1], v[t])
    for s in range(NB * B):
        if s not in written:
            assert np.array_equal(flat_out[s], flat_in[s])


def test_kv_write_bytes_per_token_llama():
    rng = np.random.default_rng(14)
    NB, B, Hkv, D = 3, 16, 8, 128
    pool = np.zeros((NB, 2, B, Hkv, D), np.uint16)
    k = np.full((2, Hkv, D), 0x3F80, np.uint16)
    v = np.full((2, Hkv, D), 0x4000, np.uint16)
    out = oracle.kv_write(pool, k, v, np.array([5, 40]))
    changed_bytes = int((out != pool).sum()) * 2
    assert changed_bytes == 2 * oracle.kv_bytes_per_token(Hkv, D) == 2 * 4096


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def _oracle_out(case, scale, pool=None, bt=None):
    return oracle.paged_attention(case["q"], case["pool"] if pool is None else pool,
                                  case["bt"] if bt is None else bt, case["sl"],
                                  case["qsl"], case["nc"], scale)


@pytest.mark.parametrize("Hq,Hkv,D,B", [(4, 2, 8, 16), (4, 4, 4, 16), (8, 2, 6, 16),
                                        (4, 2, 8, 8), (8, 2, 6, 32)])
def test_attention_equals_textbook_on_contiguous(Hq, Hkv, D, B):
    rng = np.random.default_rng(100 + Hq + D)
    lens_q, lens_c = [1, 5, 1, 3], [19, 0, 4, 30]
    case = build_case(rng, lens_q, lens_c, Hq, Hkv, D, B=B)
    scale = 1.0 / math.sqrt(D)
    got = _oracle_out(case, scale)
    for r in range(len(lens_q)):
        t0, t1 = case["qsl"][r], case["qsl"][r + 1]
        pos = lens_c[r] + np.arange(lens_q[r])
        ref = textbook_attention(case["q"][t0:t1], case["seqs"][r], pos, scale)
        np.testing.assert_allclose(got[t0:t1], ref, rtol=0, atol=1e-12)


def test_paging_independence_identity_vs_permuted():
    rng = np.random.default_rng(21)
    lens_q, lens_c = [1, 9, 1], [70, 20, 33]
    case = build_case(rng, lens_q, lens_c, 4, 2, 16, shuffle=False)
    scale = 0.25
    ident = _oracle_out(case, scale)
    # move every request's blocks to other physical ids, same logical content
    NB = case["pool"].shape[0]
    perm = rng.permutation(NB)
    pool2 = np.full_like(case["pool"], BF16_NAN)
    bt2 = case["bt"].copy()
    for r in range(len(lens_q)):
        for j, b in enumerate(case["bt"][r]):
            if b >= 0:
                bt2[r, j] = perm[b]
                pool2[perm[b]] = case["pool"][b]
    assert not np.array_equal(bt2, case["bt"])
    moved = _oracle_out(case, scale, pool=pool2, bt=bt2)
    assert np.array_equal(ident, moved)  # bit for bit


def test_block_size_does_not_change_the_result():
    """The block size decides only where a token's K/V sits, never what is
    computed: one logical batch stored with 8-, 16- and 32-token blocks gives
    the same output bit for bit."""
    lens_q, lens_c = [1, 12, 1], [45, 9, 80]
    outs = []
    for B in BLOCK_SIZES:
        case = build_case(np.random.default_rng(31), lens_q, lens_c, 4, 2, 8, NB=40, B=B)
        outs.append(_oracle_out(case, 0.3))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_shared_prefix_equals_private_copies():
    rng = np.random.default_rng(22)
    B, Hkv, D, Hq = 16, 2, 8, 4
    NB = 40
    prefix = rand_bits(rng, (48, 2, Hkv, D))  # 3 full blocks
    suffixes = [rand_bits(rng, (n, 2, Hkv, D)) for n in (5, 16, 21)]
    pool_s = np.full((NB, 2, B, Hkv, D), BF16_NAN, np.uint16)
    pool_p = pool_s.copy()
    shared_ids = [7, 2, 30]
    scatter(pool_s, shared_ids, prefix)
    bt_s = np.full((3, 8), -1, np.int32)
    bt_p = np.full((3, 8), -1, np.int32)
    nxt = iter([1, 3, 4, 5, 6, 8, 9, 10, 11, 12, 13, 14, 15, 16, 17, 18, 19, 20, 21])
    for r, suf in enumerate(suffixes):
        own = [next(nxt) for _ in range(-(-len(suf) // B))]
        bt_s[r, :3] = shared_ids
        bt_s[r, 3:3 + len(own)] = own
        scatter(pool_s, own, suf)
        priv = [next(nxt) for _ in range(3)]
        bt_p[r, :3] = priv
        bt_p[r, 3:3 + len(own)] = own
        scatter(pool_p, priv, prefix)
        scatter(pool_p, own, suf)
    sl = np.array([48 + len(s) for s in suffixes], np.int32)
    nc = sl - 1
    qsl = np.arange(4, dtype=np.int32)
    q = rand_bits(rng, (3, Hq, D))
    a = oracle.paged_attention(q, pool_s, bt_s, sl, qsl, nc, 0.3)
    b = oracle.paged_attention(q, pool_p, bt_p, sl, qsl, nc, 0.3)
    assert np.array_equal(a, b)


def test_constant_keys_give_mean_of_v():
    rng = np.random.default_rng(23)
    case = build_case(rng, [1, 6], [37, 10], 4, 2, 8)
    for r, seq in enumerate(case["seqs"]):
        seq[:, 0] = seq[0, 0]  # every key equal
        scatter(case["pool"], case["bt"][r], seq)
    out = _oracle_out(case, 0.5)
    for r, seq in enumerate(case["seqs"]):
        V = to_f(seq[:, 1])
        for i, t in enumerate(range(case["qsl"][r], case["qsl"][r + 1])):
            p = case["nc"][r] + i
            for h in range(4):
                np.testing.assert_allclose(out[t, h], V[: p + 1, h // 2].mean(axis=0),
                                           rtol=0, atol=1e-12)


def test_single_key_gives_v0():
    rng = np.random.default_rng(24)
    case = build_case(rng, [1], [0], 4, 2, 8)
    out = _oracle_out(case, 1.0)
    v0 = to_f(case["seqs"][0][0, 1])
    for h in range(4):
        assert np.array_equal(out[0, h], v0[h // 2])


def test_chunked_prefill_equals_one_shot_and_decode_equals_last_row():
    rng = np.random.default_rng(25)
    L = 45
    one = build_case(rng, [L], [0], 4, 2, 8)
    full = _oracle_out(one, 0.35)
    # the same request split into chunks (0,20) (20,17) (37,7) and a decode (44,1)
    pieces = [(0, 20), (20, 17), (37, 7), (44, 1)]
    for c, n in pieces:
        sl = np.array([c + n], np.int32)
        got = oracle.paged_attention(one["q"][c:c + n], one["pool"], one["bt"], sl,
                                     np.array([0, n], np.int32), np.array([c], np.int32), 0.35)
        np.testing.assert_allclose(got, full[c:c + n], rtol=0, atol=1e-12)


def test_request_independence_in_mixed_batch():
    rng = np.random.default_rng(26)
    lens_q, lens_c = [1, 12, 1, 1, 7], [50, 3, 1, 16, 0]
    case = build_case(rng, lens_q, lens_c, 4, 2, 8)
    mixed = _oracle_out(case, 0.4)
    for r in range(len(lens_q)):
        t0, t1 = case["qsl"][r], case["qsl"][r + 1]
        alone = oracle.paged_attention(case["q"][t0:t1], case["pool"], case["bt"][r:r + 1],
                                       case["sl"][r:r + 1], np.array([0, t1 - t0], np.int32),
                                       case["nc"][r:r + 1], 0.4)
        np.testing.assert_allclose(alone, mixed[t0:t1], rtol=0, atol=1e-12)


@pytest.mark.parametrize("part", [1, 16, 512, 700])
def test_split_kv_combine_equals_unsplit(part):
    rng = np.random.default_rng(27)
    L = 700
    case = build_case(rng, [1], [L - 1], 8, 2, 16, NB=60)
    full = _oracle_out(case, 0.25)[0]
    kv = oracle.gather_request_kv(case["pool"], case["bt"][0], L)
    ms, ls, os_ = [], [], []
    for j0 in range(0, L, part):
        m, l, o = oracle.partial_attention(case["q"][0], kv, j0, min(L, j0 + part), 0.25)
        ms.append(m)
        ls.append(l)
        os_.append(o)
    np.testing.assert_allclose(oracle.combine_partials(ms, ls, os_), full, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# planted mistakes: each plausible slip in the oracle must fail a pin above
# ---------------------------------------------------------------------------

def _bad_attend_head_map(q_bits, kv_bits, positions, scale):
    n, Hq, D = q_bits.shape
    Hkv = kv_bits.shape[2]
    out = np.empty((n, Hq, D))
    vis = np.arange(kv_bits.shape[0])[None, :] <= np.asarray(positions)[:, None]
    for h in range(Hq):
        g = h % Hkv  # interleaved instead of consecutive grouping
        K, V, Q = to_f(kv_bits[:, 0, g]), to_f(kv_bits[:, 1, g]), to_f(q_bits[:, h])
        s = np.where(vis, scale * Q @ K.T, -np.inf)
        w = np.exp(s - s.max(1, keepdims=True))
        out[:, h] = w @ V / w.sum(1, keepdims=True)
    return out


def _bad_attend_causal(q_bits, kv_bits, positions, scale):
    # off by one: a query also sees the next key
    return po.__dict__["_orig_attend"](q_bits, kv_bits, np.asarray(positions) + 1, scale)


def _bad_attend_no_scale(q_bits, kv_bits, positions, scale):
    return po.__dict__["_orig_attend"](q_bits, kv_bits, positions, 1.0)


@pytest.mark.parametrize("bad", [_bad_attend_head_map, _bad_attend_causal, _bad_attend_no_scale])
def test_planted_attention_mistakes_are_caught(monkeypatch, bad):
    monkeypatch.setitem(po.__dict__, "_orig_attend", po.attend_rows)
    monkeypatch.setattr(po, "attend_rows", bad)
    rng = np.random.default_rng(31)
    lens_q, lens_c = [1, 4], [9, 2]
    case = build_case(rng, lens_q, lens_c, 4, 2, 4)
    got = _oracle_out(case, 0.5)
    worst = 0.0
    for r in range(2):
        t0, t1 = case["qsl"][r], case["qsl"][r + 1]
        pos = lens_c[r] + np.arange(lens_q[r])
        ref = textbook_attention(case["q"][t0:t1], case["seqs"][r], pos, 0.5)
        worst = max(worst, float(np.nan_to_num(np.abs(got[t0:t1] - ref), nan=1e9).max()))
    assert worst > 1e-6


def test_planted_slot_mistake_is_caught(monkeypatch):
    def bad_slot(row, pos, B=16):
        return int(row[pos // B]) * B + (pos + 1) % B

    monkeypatch.setattr(po, "slot_of", bad_slot)
    g = _load("slot_mapping_worked_example.json")
    bt = np.array(g["block_table"], np.int32)
    assert any(po.slot_of(bt[e["request"]], e["pos"]) != e["slot"] for e in g["slots"])


# ---------------------------------------------------------------------------
# block copies (copy-on-write, swap)
# ---------------------------------------------------------------------------

def test_copy_blocks_moves_whole_blocks_only():
    rng = np.random.default_rng(41)
    src = rand_bits(rng, (9, 2, 16, 2, 8))
    dst = rand_bits(rng, (7, 2, 16, 2, 8))
    pairs = [(3, 0), (8, 6), (3, 2)]
    out = oracle.copy_blocks(dst, src, pairs)
    for s_, d in pairs:
        assert np.array_equal(out[d], src[s_])
    for d in (1, 3, 4, 5):
        assert np.array_equal(out[d], dst[d])


def test_copy_on_write_keeps_the_sharer_intact():
    """Two sequences share a partly filled block; the one that writes first
    gets its own copy ([P1] §4.3.2). Afterwards the other one still sees the
    original block and the writer sees its copy plus its new token, exactly
    as if it had owned private blocks from the start."""
    rng = np.random.default_rng(42)
    B, Hkv, D, Hq = 16, 2, 8, 4
    prefix = rand_bits(rng, (24, 2, Hkv, D))  # 1.5 blocks: the second block is shared and partial
    pool = np.full((10, 2, B, Hkv, D), BF16_NAN, np.uint16)
    scatter(pool, [4, 7], prefix)
    new_kv = rand_bits(rng, (1, 2, Hkv, D))
    pool_cow = oracle.copy_blocks(pool, pool, [(7, 9)])  # the writer's copy of block 7
    slot = oracle.slot_of(np.array([4, 9]), 24)
    pool_cow = oracle.kv_write(pool_cow, new_kv[:, 0], new_kv[:, 1], np.array([slot]))
    assert np.array_equal(pool_cow[7], pool[7])  # the sharer's block is untouched
    q = rand_bits(rng, (2, Hq, D))
    bt = np.array([[4, 7, -1], [4, 9, -1]], np.int32)
    out = oracle.paged_attention(q, pool_cow, bt, np.array([24, 25], np.int32),
                                 np.array([0, 1, 2], np.int32), np.array([23, 24], np.int32), 0.3)
    # reference: the sharer alone, and the writer with private blocks from the start
    ref_pool = np.full_like(pool, BF16_NAN)
    scatter(ref_pool, [1, 2], np.concatenate([prefix, new_kv]))
    scatter(ref_pool, [5, 6], prefix)
    ref = oracle.paged_attention(q, ref_pool, np.array([[5, 6, -1], [1, 2, -1]], np.int32),
                                 np.array([24, 25], np.int32), np.array([0, 1, 2], np.int32),
                                 np.array([23, 24], np.int32), 0.3)
    assert np.array_equal(out, ref)
