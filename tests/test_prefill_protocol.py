"""Model check of the prefill kernel's barrier protocol, on the CPU.

Every role of a prefill CTA is restated as the sequence of mbarrier waits
and arrivals it performs:
- the K-copy warp claims items and copies Q and K tiles;
- the V-copy warp copies V tiles;
- the MMA thread issues S and PV;
- the two softmax warpgroups take tile T of the CTA's stream on warpgroup
  T & 1, finish one-tile items alone and merge longer ones.

Copies and MMA completions are asynchronous events. Copies complete in any
order; MMA commits complete in issue order. Random item lists run under
many random interleavings.

Each wait names the barrier phase it means (from the role's own counters),
and a parity wait is only correct if the barrier is then at that phase or
one past it. The model checks that, that no barrier receives more arrivals
than a phase takes, and that the CTA never deadlocks.
"""

import random

import pytest

K_STAGES, V_STAGES, ITEM_Q = 3, 2, 4
# arrivals per phase: item queue slots are released by the MMA thread, the
# V-copy warp and the 8 softmax warps (4 per warpgroup)
IQ_FREE_ARRIVALS = 10


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.phases = name, count, 0, 0

    def arrive(self, n=1):
        self.pending += n
        assert self.pending <= self.count, f"{self.name}: more arrivals than a phase takes"
        if self.pending == self.count:
            self.pending = 0
            self.phases += 1


class Cta:
    def __init__(self, items):
        self.items = items  # key tiles of each item, in claim order
        b = {}

        def mk(name, count):
            b[name] = Barrier(name, count)

        mk("q_full", 1)
        mk("q_free", 1)
        for i in range(K_STAGES):
            mk(f"k_full{i}", 1)
            mk(f"k_free{i}", 1)
        for i in range(V_STAGES):
            mk(f"v_full{i}", 1)
            mk(f"v_free{i}", 1)
        for w in range(2):
            mk(f"s_full{w}", 1)
            mk(f"p_ready{w}", 1)  # the warpgroup's 128 arrivals, as one
            mk(f"o_full{w}", 1)
            mk(f"o_free{w}", 2)   # two warpgroups' worth of readers
            mk(f"ml_full{w}", 2)  # one per warpgroup
        for i in range(ITEM_Q):
            mk(f"iq_full{i}", 1)
            mk(f"iq_free{i}", IQ_FREE_ARRIVALS)
        self.b = b
        self.item_q = [None] * ITEM_Q
        self.next_claim = 0
        self.tma = []  # copies in flight: (barrier) -- complete in any order
        self.mma = []  # MMA commits in flight -- complete in issue order

    def claim(self):
        j = self.next_claim
        self.next_claim += 1
        return j if j < len(self.items) else None


# Operations a role yields: ("wait", barrier, phase index), ("arrive", barrier, n),
# ("tma", barrier), ("commit", barrier), ("do", callable).

def k_warp(cta):
    T = 0
    it = 0
    while True:
        if it > 0:
            yield ("wait", "q_free", it - 1)
        slot = it % ITEM_Q
        if it >= ITEM_Q:
            yield ("wait", f"iq_free{slot}", (it - ITEM_Q) // ITEM_Q)
        item = cta.claim()
        cta.item_q[slot] = item
        yield ("arrive", f"iq_full{slot}", 1)
        if item is None:
            return
        yield ("tma", "q_full")
        for _ in range(cta.items[item]):
            s = T % K_STAGES
            if T >= K_STAGES:
                yield ("wait", f"k_free{s}", (T - K_STAGES) // K_STAGES)
            yield ("tma", f"k_full{s}")
            T += 1
        it += 1


def take(cta, j, arrivals):
    slot = j % ITEM_Q
    yield ("wait", f"iq_full{slot}", j // ITEM_Q)
    item = cta.item_q[slot]
    yield ("arrive", f"iq_free{slot}", arrivals)
    return item


def v_warp(cta):
    T = 0
    it = 0
    while True:
        item = yield from take(cta, it, 1)
        if item is None:
            return
        for _ in range(cta.items[item]):
            s = T % V_STAGES
            if T >= V_STAGES:
                yield ("wait", f"v_free{s}", (T - V_STAGES) // V_STAGES)
            yield ("tma", f"v_full{s}")
            T += 1
        it += 1


def mma_thread(cta):
    T = 0
    np_ = [0, 0]
    uses = [0, 0]
    it = 0
    while True:
        item = yield from take(cta, it, 1)
        if item is None:
            return
        nkv = cta.items[item]
        rot = T & 1

        def issue_s(kt):
            w = (kt + rot) & 1
            s = (T + kt) % K_STAGES
            yield ("wait", f"k_full{s}", (T + kt) // K_STAGES)
            yield ("commit", f"s_full{w}")
            yield ("commit", f"k_free{s}")
            if kt == nkv - 1:
                yield ("commit", "q_free")

        yield ("wait", "q_full", it)
        yield from issue_s(0)
        if nkv > 1:
            yield from issue_s(1)
        for kt in range(nkv):
            w = (kt + rot) & 1
            yield ("wait", f"p_ready{w}", np_[w])
            np_[w] += 1
            if kt < 2:
                if uses[w] > 0:
                    yield ("wait", f"o_free{w}", uses[w] - 1)
                uses[w] += 1
            s = (T + kt) % V_STAGES
            yield ("wait", f"v_full{s}", (T + kt) // V_STAGES)
            yield ("commit", f"v_free{s}")
            if kt >= nkv - 2:
                yield ("commit", f"o_full{w}")
            if kt + 2 < nkv:
                yield from issue_s(kt + 2)
        T += nkv
        it += 1


def softmax_wg(cta, wg):
    T = 0
    ns = 0
    uses = [0, 0]
    mi = 0
    it = 0
    item = yield from take(cta, 0, 4)
    while item is not None:
        nkv = cta.items[item]
        rot = T & 1
        for kt in range((wg - rot) & 1, nkv, 2):
            yield ("wait", f"s_full{wg}", ns)
            ns += 1
            # a tile with keys past the end or chunks not loaded waits for its
            # V copy before cleaning it; the model lets every tile do so (a
            # superset of the kernel's waits, which change no phase)
            s = (T + kt) % V_STAGES
            yield ("wait", f"v_full{s}", (T + kt) // V_STAGES)
            yield ("arrive", f"p_ready{wg}", 1)
        item_n = yield from take(cta, it + 1, 4)
        if nkv > 1:
            yield ("wait", "o_full0", uses[0])
            yield ("wait", "o_full1", uses[1])
            yield ("arrive", f"ml_full{mi & 1}", 1)
            yield ("wait", f"ml_full{mi & 1}", mi >> 1)
            yield ("arrive", "o_free0", 1)
            yield ("arrive", "o_free1", 1)
            uses[0] += 1
            uses[1] += 1
            mi += 1
        else:
            if wg == rot:
                yield ("wait", f"o_full{wg}", uses[wg])
                yield ("arrive", f"o_free{wg}", 2)  # the only reader: both shares
            uses[rot] += 1
        T += nkv
        item = item_n
        it += 1


def run(items, seed, mma=None, wg=None):
    rng = random.Random(seed)
    cta = Cta(items)
    wg_role = wg or softmax_wg
    roles = {"k": k_warp(cta), "v": v_warp(cta), "mma": (mma or mma_thread)(cta),
             "wg0": wg_role(cta, 0), "wg1": wg_role(cta, 1)}
    pending = {name: next(g) for name, g in roles.items()}
    done = set()
    steps = 0
    while len(done) < len(roles) or cta.tma or cta.mma:
        steps += 1
        assert steps < 200000, "model did not finish"
        runnable = []
        for name, op in pending.items():
            if name in done:
                continue
            if op[0] == "wait":
                bar = cta.b[op[1]]
                k = op[2]
                # a parity wait is only correct within one phase of its target
                assert bar.phases in (k, k + 1), (
                    f"{name} waits for phase {k} of {op[1]}, which has completed {bar.phases}")
                if bar.phases == k:
                    continue  # blocked
            runnable.append(name)
        events = (["copy done"] if cta.tma else []) + (["mma done"] if cta.mma else [])
        choices = runnable + events
        assert choices, f"deadlock: {pending}"
        c = rng.choice(choices)
        if c == "copy done":
            cta.b[cta.tma.pop(rng.randrange(len(cta.tma)))].arrive()
            continue
        if c == "mma done":
            cta.b[cta.mma.pop(0)].arrive()
            continue
        op = pending[c]
        if op[0] == "arrive":
            cta.b[op[1]].arrive(op[2])
        elif op[0] == "tma":
            cta.tma.append(op[1])
        elif op[0] == "commit":
            cta.mma.append(op[1])
        try:
            pending[c] = roles[c].send(None)
        except StopIteration:
            done.add(c)
    # every item was claimed, and every barrier ended between phases
    assert cta.next_claim == len(items) + 1
    for bar in cta.b.values():
        assert bar.pending == 0, f"{bar.name} left with {bar.pending} arrivals"


@pytest.mark.parametrize("case", range(60))
def test_prefill_protocol_random_items_and_interleavings(case):
    rng = random.Random(1000 + case)
    n = rng.randint(1, 14)
    # one-tile items (short prefills) mixed with items of several tiles
    items = [rng.choice([1, 1, 1, 2, 3, rng.randint(1, 9)]) for _ in range(n)]
    for s in range(40):
        run(items, seed=case * 1000 + s)


def test_prefill_protocol_all_one_tile_and_all_long():
    for items in ([1] * 20, [7] * 6, [2, 1, 1, 1, 2, 1, 3, 1, 1], [1, 2] * 8):
        for s in range(100):
            run(items, seed=s)


def _late_o_free_wait(cta):
    """The MMA thread with one planted mistake: it waits for the O buffer's
    free phase one use too late."""
    g = mma_thread(cta)
    op = next(g)
    while True:
        if op[0] == "wait" and op[1].startswith("o_free"):
            op = ("wait", op[1], op[2] + 1)
        yield op
        try:
            op = next(g)
        except StopIteration:
            return


def _single_arrival_owner(cta, wg):
    """A softmax warpgroup with one planted mistake: finishing a one-tile item
    alone, it arrives once on the O free barrier instead of for both shares."""
    g = softmax_wg(cta, wg)
    op = next(g)
    while True:
        if op[0] == "arrive" and op[1].startswith("o_free") and op[2] == 2:
            op = ("arrive", op[1], 1)
        yield op
        try:
            op = next(g)
        except StopIteration:
            return


@pytest.mark.parametrize("mistake", ["late_o_free_wait", "single_arrival_owner"])
def test_model_catches_planted_protocol_mistakes(mistake):
    """The model is not vacuous: each planted mistake is caught (a wait at the
    wrong phase, or a deadlock)."""
    overrides = ({"mma": _late_o_free_wait} if mistake == "late_o_free_wait"
                 else {"wg": _single_arrival_owner})
    with pytest.raises(AssertionError):
        for s in range(50):
            run([1, 1, 2, 1, 1, 3, 1], seed=s, **overrides)
