"""CPU restatement of the kernels' online-softmax update and combine.

The decode and prefill kernels keep a running max in base 2 and move it
lazily: only when a new chunk (decode: 16 keys) or tile (prefill: 128 keys)
beats it by more than 2^8 -- decided once per warp, for every head or row the
warp holds -- are the running sum and the unnormalised output rescaled by
alpha = 2^(m_old - m_new). In the prefill each query row is split between
two threads of one warp (keys 0..63 and 64..127 of every tile, and the two
halves of O's columns): the row max is taken over both halves, each half
keeps its own running sum and both rescale with the same alpha; the row's
sum is the two halves' sums added at the end. A warp holds 16 rows. A
decode request cut by split-KV ranges leaves one partial per range, merged
by the combine kernel with weights 2^(m_p - M).

These tests restate those rules in numpy fp32 (the kernels' precision; the
prefill's P rounded to bf16 before P.V as on the tensor cores) on the
rescale-path inputs of ``rescale_cases`` -- the same inputs the GPU parity
tests run -- and require the oracle's result within the attention tolerance.
They also check that the inputs really drive each branch (rescales that keep
weight on earlier keys, alphas and combine weights that underflow to zero),
and that each plausible slip in the update (a wrong alpha, a missing rescale
of the sum or of (half of) the output, a half-row sum left out, a wrong
combine weight) fails against the oracle.
"""

import numpy as np
import pytest

import oracle
from parity import ABS_TOL, REL_TOL
from rescale_cases import DECODE_CASES, PREFILL_CASES, case

F32 = np.float32
LOG2E = F32(1.4426950408889634)
THRESH = F32(8.0)  # lazy rescale threshold, powers of two
CHUNK, TILE = 16, 128

# planted slips overflow on purpose
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def to_f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_round(x):
    """fp32 -> nearest bf16 (ties to even) -> fp32, as the P store does."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    r = ((u + ((u >> 16) & 1) + 0x7FFF) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def request_kv(step, r):
    """K and V of request r in key order, [L, Hkv, D] fp32 each, read by
    walking its block table."""
    B, L = step.block_size, int(step.seq_lens[r])
    pos = np.arange(L)
    blk = step.block_table[r, pos // B]
    return to_f32(step_pool(step)[blk, 0, pos % B]), to_f32(step_pool(step)[blk, 1, pos % B])


_POOLS = {}


def step_pool(step):
    """The pool after the step's cache write (new tokens at their places)."""
    key = id(step)
    if key not in _POOLS:
        pool = step.kv_cache.copy()
        for t, (b, o) in enumerate(step.new_token_place):
            pool[b, 0, o] = step.k[t]
            pool[b, 1, o] = step.v[t]
        _POOLS[key] = pool
    return _POOLS[key]


class Stats:
    def __init__(self):
        self.rescales_with_weight = 0  # mid-stream rescales keeping > 5% of the weight
        self.zero_alphas = 0           # mid-stream rescales whose alpha underflowed
        self.zero_weights = 0          # merge / combine weights that underflowed


# ---------------------------------------------------------------- decode
def decode_piece(qs, K, V, j0, j1, gw, bug=None, st=None):
    """One CTA's piece of a decode request: keys j0..j1-1 (whole 16-key
    chunks of the request, the last one maybe partial) for every q head.

    qs: [Hq, D] fp32 already multiplied by scale * log2(e); K, V: [L, Hq, D]
    (each q head's kv head already selected). Heads are grouped gw to a warp:
    the warp rescales when any of its heads needs it."""
    Hq, D = qs.shape
    m = np.full(Hq, -np.inf, F32)
    lsum = np.zeros(Hq, F32)
    o = np.zeros((Hq, D), F32)
    for c0 in range(j0, j1, CHUNK):
        c1 = min(c0 + CHUNK, j1)
        s = np.einsum("hd,jhd->hj", qs, K[c0:c1]).astype(F32)
        lmax = s.max(axis=1)
        need = (lmax > m + THRESH).reshape(-1, gw).any(axis=1).repeat(gw)
        if need.any():
            m_new = np.where(need, np.maximum(m, lmax), m)
            with np.errstate(invalid="ignore", over="ignore"):
                if bug == "alpha_inverted":
                    alpha = np.exp2(m_new - m)
                else:
                    alpha = np.exp2(m - m_new)
            alpha = np.where(m_new == -np.inf, F32(1), alpha).astype(F32)
            if st is not None:
                mid = need & np.isfinite(m)
                old = alpha * lsum
                new = np.exp2(s - m_new[:, None]).sum(axis=1)
                st.rescales_with_weight += int((mid & (old > 0.05 * (old + new))).sum())
                st.zero_alphas += int((mid & (alpha == 0)).sum())
            if bug != "l_not_rescaled":
                lsum = lsum * alpha
            if bug != "o_not_rescaled":
                o = o * alpha[:, None]
            m = m_new.astype(F32)
        with np.errstate(over="ignore", invalid="ignore"):
            p = np.where(np.isfinite(m)[:, None], np.exp2(s - m[:, None]), F32(0)).astype(F32)
        lsum = lsum + p.sum(axis=1, dtype=F32)
        o = o + np.einsum("hj,jhd->hd", p, V[c0:c1]).astype(F32)
    return m, lsum, o


def combine(parts, bug=None, st=None):
    """Merge the (m, l, o) partials of one request's pieces."""
    ms = np.stack([p[0] for p in parts])
    M = ms.max(axis=0)
    with np.errstate(over="ignore", invalid="ignore"):
        w = np.exp2(M - ms) if bug == "combine_weight_inverted" else np.exp2(ms - M)
    w = np.where(ms == -np.inf, F32(0), w).astype(F32)
    if st is not None:
        st.zero_weights += int(((w == 0) & np.stack([p[1] > 0 for p in parts])).sum())
    ls = np.stack([p[1] for p in parts])
    acc = sum(w[i][:, None] * parts[i][2] for i in range(len(parts)))
    den = w.sum(axis=0) if bug == "combine_forgets_l" else (w * ls).sum(axis=0)
    return acc / den[:, None]


def decode_restated(step, r, rng, bug=None, st=None):
    """Output of decode request r, its chunks cut into random pieces."""
    Hq, Hkv = step.num_q_heads, step.num_kv_heads
    G = Hq // Hkv
    gw = min(G, 4)
    L = int(step.seq_lens[r])
    K, V = request_kv(step, r)
    head_kv = np.arange(Hq) // G
    K, V = K[:, head_kv], V[:, head_kv]
    scale_log2 = F32(step.scale) * LOG2E
    qs = (to_f32(step.q[int(step.query_start_loc[r])]) * scale_log2).astype(F32)
    nchunk = -(-L // CHUNK)
    ncut = int(rng.integers(0, min(nchunk, 6)))
    cuts = sorted(set(rng.choice(np.arange(1, nchunk), size=ncut, replace=False).tolist())
                  if nchunk > 1 and ncut else [])
    bounds = [0] + [c * CHUNK for c in cuts] + [L]
    parts = [decode_piece(qs, K, V, a, b, gw, bug, st) for a, b in zip(bounds[:-1], bounds[1:])]
    if len(parts) == 1:
        m, lsum, o = parts[0]
        return o / lsum[:, None]
    return combine(parts, bug, st)


# ---------------------------------------------------------------- prefill
def prefill_rows(S_tiles, keep, scale_log2, bug=None, st=None):
    """The softmax warps over an item's tiles, in order. S_tiles: list of
    ([rows, 128] unscaled scores, masked keys at -inf; [128, D] V); keep:
    [rows] rows that take part in the warp vote. Each row's keys 0..63 and
    64..127 (and O's first and second halves of columns) belong to two
    threads; rows are grouped 16 to a warp. Returns the normalised output,
    with P rounded to bf16 before P.V."""
    rows = S_tiles[0][0].shape[0]
    D = S_tiles[0][1].shape[1]
    m = np.full(rows, -np.inf, F32)
    lh = np.zeros((2, rows), F32)  # the two halves' running sums
    O = np.zeros((rows, D), F32)
    for kt, (S, Vt) in enumerate(S_tiles):
        # each half's max, then the pair's (both threads get the same value)
        mh = np.stack([S[:, :64].max(axis=1), S[:, 64:].max(axis=1)])
        mx = (mh.max(axis=0) * scale_log2).astype(F32)
        vote = (mx > m + THRESH) & keep
        need = vote.reshape(-1, 16).any(axis=1).repeat(16)
        if need.any():
            m_new = np.where(need, np.maximum(m, mx), m)
            with np.errstate(invalid="ignore", over="ignore"):
                alpha = np.exp2(m_new - m) if bug == "alpha_inverted" else np.exp2(m - m_new)
            alpha = np.where(m_new == -np.inf, F32(1), alpha).astype(F32)
            if st is not None:
                mid = need & np.isfinite(m) & keep
                st.zero_alphas += int((mid & (alpha == 0)).sum())
                old = alpha * (lh[0] + lh[1])
                with np.errstate(over="ignore", invalid="ignore"):
                    new = np.exp2(S * scale_log2 - m_new[:, None]).sum(axis=1)
                st.rescales_with_weight += int((mid & (old > 0.05 * (old + new))).sum())
            lh = lh * alpha[None, :]
            if kt > 0 and bug != "o_not_rescaled":
                O[:, : D // 2] *= alpha[:, None]
                if bug != "o_half_not_rescaled":
                    O[:, D // 2:] *= alpha[:, None]
            m = m_new.astype(F32)
        msub = np.where(np.isfinite(m), m, F32(0))
        with np.errstate(over="ignore", invalid="ignore"):
            p = np.exp2((S * scale_log2).astype(F32) - msub[:, None]).astype(F32)
        lh[0] += p[:, :64].sum(axis=1, dtype=F32)
        lh[1] += p[:, 64:].sum(axis=1, dtype=F32)
        O = O + (bf16_round(p) @ Vt).astype(F32)
    l_row = lh[0] if bug == "l_half_missing" else lh[0] + lh[1]
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        return O / l_row[:, None]


def prefill_restated(step, r, g, bug=None, st=None):
    """Rows of prefill request r for kv head g: [n, G, D]."""
    Hq, Hkv, D = step.num_q_heads, step.num_kv_heads, step.head_dim
    G = Hq // Hkv
    QT = TILE // G
    c, n = int(step.num_computed[r]), int(step.query_len[r])
    q0 = int(step.query_start_loc[r])
    K, V = request_kv(step, r)
    K, V = K[:, g], V[:, g]
    Q = to_f32(step.q[q0:q0 + n, g * G:(g + 1) * G])  # [n, G, D]
    scale_log2 = F32(step.scale) * LOG2E
    out = np.zeros((n, G, D), F32)
    for i0 in range(0, n, QT):
        qi = i0 + np.arange(QT)
        valid = qi < n
        rows_q = np.repeat(np.minimum(qi, n - 1), G)  # row = query offset * G + head
        rows_h = np.tile(np.arange(G), QT)
        keep = np.repeat(valid, G)
        Qr = Q[rows_q, rows_h]  # [128, D]
        kv_len = c + int(qi[valid].max()) + 1
        lim = np.minimum(c + rows_q, kv_len - 1)
        nkv = -(-kv_len // TILE)
        tiles = []
        for kt in range(nkv):
            k0, k1 = kt * TILE, min(kt * TILE + TILE, kv_len)
            S = np.full((TILE, TILE), -np.inf, F32)
            S[:, : k1 - k0] = Qr @ K[k0:k1].T
            j = k0 + np.arange(TILE)
            S[j[None, :] > lim[:, None]] = -np.inf
            Vt = np.zeros((TILE, D), F32)
            Vt[: k1 - k0] = V[k0:k1]
            tiles.append((S, Vt))
        res = prefill_rows(tiles, keep, scale_log2, bug, st)
        res = res.reshape(QT, G, D)
        out[qi[valid]] = res[valid]
    return out


# ---------------------------------------------------------------- checks
def within_tolerance(got, ref):
    err = np.abs(got.astype(np.float64) - ref)
    return bool((err <= np.maximum(ABS_TOL, REL_TOL * np.abs(ref))).all())


_STEPS = {}


def get_case(name, D):
    key = (name, D)
    if key not in _STEPS:
        Hq, Hkv = (32, 8) if D == 128 else (16, 4)
        step = case(name, Hq=Hq, Hkv=Hkv, D=D, seed=D)
        slots = oracle.slot_mapping(step.block_table, step.query_start_loc, step.num_computed,
                                    step.block_size)
        pool = oracle.kv_write(step.kv_cache, step.k, step.v, slots)
        ref = oracle.paged_attention(step.q, pool, step.block_table, step.seq_lens,
                                     step.query_start_loc, step.num_computed, step.scale)
        _STEPS[key] = (step, ref)
    return _STEPS[key]


def run_decode(name, D, bug=None, st=None, reqs=6):
    step, ref = get_case(name, D)
    rng = np.random.default_rng(5)
    ok = True
    dec = [r for r in range(step.num_reqs) if step.query_len[r] == 1][:reqs]
    for r in dec:
        got = decode_restated(step, r, rng, bug, st)
        ok &= within_tolerance(got, ref[int(step.query_start_loc[r])])
    return ok


def run_prefill(name, D, bug=None, st=None):
    step, ref = get_case(name, D)
    G = step.num_q_heads // step.num_kv_heads
    ok = True
    for r in range(step.num_reqs):
        if step.query_len[r] < 2:
            continue
        q0, n = int(step.query_start_loc[r]), int(step.query_len[r])
        for g in (0, step.num_kv_heads - 1):
            got = prefill_restated(step, r, g, bug, st)
            ok &= within_tolerance(got, ref[q0:q0 + n, g * G:(g + 1) * G])
    return ok


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("name", DECODE_CASES)
def test_decode_update_and_combine_match_the_oracle(name, D):
    assert run_decode(name, D)


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("name", PREFILL_CASES)
def test_prefill_update_matches_the_oracle(name, D):
    assert run_prefill(name, D)


def test_the_inputs_drive_every_branch():
    """The drift cases rescale partials that still hold weight; the steep
    and spike cases make alphas and combine weights underflow to exactly
    zero."""
    st = {n: Stats() for n in DECODE_CASES + PREFILL_CASES}
    for n in DECODE_CASES:
        run_decode(n, 128, st=st[n])
    for n in PREFILL_CASES:
        run_prefill(n, 128, st=st[n])
    assert st["decode_drift"].rescales_with_weight > 100
    assert st["decode_scale"].rescales_with_weight > 0
    assert st["decode_steep"].zero_weights > 0 and st["decode_spike"].zero_weights > 0
    assert st["decode_spike"].zero_alphas > 0 or st["decode_steep"].zero_alphas > 0
    assert st["prefill_drift"].rescales_with_weight > 100
    assert st["prefill_steep"].zero_alphas > 0


@pytest.mark.parametrize("bug,cases", [
    ("alpha_inverted", ["decode_drift", "decode_scale"]),
    ("l_not_rescaled", ["decode_drift", "decode_scale"]),
    ("o_not_rescaled", ["decode_drift", "decode_scale"]),
    ("combine_weight_inverted", ["decode_spike", "decode_steep"]),
    ("combine_forgets_l", ["decode_drift", "decode_spike"]),
])
def test_planted_decode_slips_fail(bug, cases):
    assert not all(run_decode(n, 128, bug=bug) for n in cases)


@pytest.mark.parametrize("bug", ["alpha_inverted", "o_not_rescaled", "o_half_not_rescaled",
                                 "l_half_missing"])
def test_planted_prefill_slips_fail(bug):
    assert not all(run_prefill(n, 128, bug=bug) for n in ("prefill_drift", "prefill_steep"))
