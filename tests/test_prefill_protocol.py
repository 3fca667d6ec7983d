"""Model check of the prefill kernel's barrier protocol, on the CPU.

Every role of a prefill CTA is restated as the sequence of mbarrier waits
and arrivals it performs:
- the K-copy warp claims items and copies Q and K tiles (K slot T % 3 is
  refilled once S(T-3) is done);
- the V-copy warp copies V tiles (V slot T % 2 is refilled once PV(T-2) is
  done);
- the S thread issues S(T) into TMEM buffer T % 3 once PV(T-3) is done and
  K(T) landed;
- the PV thread issues PV(T) once P(T) is published and V(T) landed, into
  one O accumulator;
- the softmax warps (modelled as N_SOFTMAX independent agents, each owning
  some query rows) take every tile of every item, sometimes rescale O
  (after PV of the previous tile is done), sometimes clean V rows (after the
  V copy landed), publish P, and write the item's output once its last PV
  is done.

Copies and MMA completions are asynchronous events. Copies complete in any
order; each MMA thread's commits complete in its issue order. Random item
lists run under many random interleavings, and the optional waits are taken
at random.

Each wait names the barrier phase it means (from the role's own counters),
and a parity wait is only correct if the barrier is then at that phase or
one past it. The model checks that, that no barrier receives more arrivals
than a phase takes, that the CTA never deadlocks, and the TMEM hazards:
S(T) overwrites buffer T % 3 only after every agent read S(T-3) and PV(T-3)
read P(T-3); the first PV of an item overwrites O only after every agent
read the previous item's O; a rescale finds PV(T-1) done and PV(T) not yet
issued.
"""

import random

import pytest

K_STAGES, V_STAGES, S_BUFS, ITEM_Q = 3, 2, 3, 4
N_SOFTMAX = 4
# arrivals per phase: item queue slots are released by the two MMA threads,
# the V-copy warp and every softmax agent
IQ_FREE_ARRIVALS = 3 + N_SOFTMAX


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
    def __init__(self, items, rng):
        self.items = items  # key tiles of each item, in claim order
        self.rng = rng
        b = {}

        def mk(name, count):
            b[name] = Barrier(name, count)

        mk("q_full", 1)
        mk("q_free", 1)
        for i in range(K_STAGES):
            mk(f"k_full{i}", 1)
        for i in range(V_STAGES):
            mk(f"v_full{i}", 1)
        for i in range(S_BUFS):
            mk(f"s_full{i}", 1)
            mk(f"pv_done{i}", 1)
            mk(f"p_ready{i}", N_SOFTMAX)
        mk("o_full", 1)
        for i in range(ITEM_Q):
            mk(f"iq_full{i}", 1)
            mk(f"iq_free{i}", IQ_FREE_ARRIVALS)
        self.b = b
        self.item_q = [None] * ITEM_Q
        self.next_claim = 0
        self.tma = []  # copies in flight: (barrier) -- complete in any order
        self.mma = {"s": [], "pv": []}  # each MMA thread's commits, in issue order
        # TMEM bookkeeping for the hazard checks
        self.s_read = {}     # tile -> agents that read its S (and wrote P)
        self.pv_issued = set()
        self.pv_done = set()
        self.o_read = {}     # item -> agents whose epilogue read O

    def claim(self):
        j = self.next_claim
        self.next_claim += 1
        return j if j < len(self.items) else None


# Operations a role yields: ("wait", barrier, phase index), ("arrive", barrier, n),
# ("tma", barrier), ("commit", barrier), ("pv", tile) -- a PV whose completion
# is recorded in issue order with that thread's commits.

def k_warp(cta, phase_slip=0):
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
                Tp = T - K_STAGES
                yield ("wait", f"s_full{Tp % S_BUFS}", Tp // S_BUFS + phase_slip)
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
                Tp = T - V_STAGES
                yield ("wait", f"pv_done{Tp % S_BUFS}", Tp // S_BUFS)
            yield ("tma", f"v_full{s}")
            T += 1
        it += 1


def s_thread(cta, skip_pv_wait=False):
    T = 0
    it = 0
    while True:
        item = yield from take(cta, it, 1)
        if item is None:
            return
        nkv = cta.items[item]
        yield ("wait", "q_full", it)
        for kt in range(nkv):
            Tk = T + kt
            if Tk >= S_BUFS and not skip_pv_wait:
                Tp = Tk - S_BUFS
                yield ("wait", f"pv_done{Tp % S_BUFS}", Tp // S_BUFS)
            yield ("wait", f"k_full{Tk % K_STAGES}", Tk // K_STAGES)
            # S(Tk) overwrites buffer Tk % 3: S(Tk-3) read by every agent and
            # P(Tk-3) read by its PV
            if Tk >= S_BUFS:
                assert cta.s_read.get(Tk - S_BUFS, 0) == N_SOFTMAX, f"S({Tk}) over unread S"
                assert (Tk - S_BUFS) in cta.pv_done, f"S({Tk}) before PV({Tk - S_BUFS}) done"
            yield ("commit", "s", f"s_full{Tk % S_BUFS}")
            if kt == nkv - 1:
                yield ("commit", "s", "q_free")
        T += nkv
        it += 1


def pv_thread(cta):
    T = 0
    it = 0
    while True:
        item = yield from take(cta, it, 1)
        if item is None:
            return
        nkv = cta.items[item]
        for kt in range(nkv):
            Tg = T + kt
            yield ("wait", f"p_ready{Tg % S_BUFS}", Tg // S_BUFS)
            yield ("wait", f"v_full{Tg % V_STAGES}", Tg // V_STAGES)
            if kt == 0 and it > 0:  # O is overwritten: the last item's O read by all
                assert cta.o_read.get(it - 1, 0) == N_SOFTMAX, f"item {it} PV(0) over unread O"
            cta.pv_issued.add(Tg)
            yield ("pv", Tg)
            yield ("commit", "pv", f"pv_done{Tg % S_BUFS}")
            if kt == nkv - 1:
                yield ("commit", "pv", "o_full")
        T += nkv
        it += 1


def softmax_agent(cta, a, v_clean_one_wait=False):
    rng = random.Random(cta.rng.random())
    T = 0
    it = 0
    item = yield from take(cta, 0, 1)
    while item is not None:
        nkv = cta.items[item]
        for kt in range(nkv):
            Tg = T + kt
            yield ("wait", f"s_full{Tg % S_BUFS}", Tg // S_BUFS)
            cta.s_read[Tg] = cta.s_read.get(Tg, 0) + 1
            if kt > 0 and rng.random() < 0.3:  # the max grew: rescale O
                Tp = Tg - 1
                yield ("wait", f"pv_done{Tp % S_BUFS}", Tp // S_BUFS)
                assert Tp in cta.pv_done, f"rescale at {Tg} before PV({Tp}) done"
                assert Tg not in cta.pv_issued, f"rescale at {Tg} after PV({Tg}) issued"
            if rng.random() < 0.3:  # a ragged tile: clean V rows after the copy
                # PV(Tg-2) first: S(Tg) only implies PV(Tg-3) done, so the V
                # slot's barrier may be anywhere from V(Tg-2) pending to V(Tg)
                # landed; once PV(Tg-2) is done it is at V(Tg) pending or landed
                if Tg >= V_STAGES and not v_clean_one_wait:
                    Tp = Tg - V_STAGES
                    yield ("wait", f"pv_done{Tp % S_BUFS}", Tp // S_BUFS)
                yield ("wait", f"v_full{Tg % V_STAGES}", Tg // V_STAGES)
            yield ("arrive", f"p_ready{Tg % S_BUFS}", 1)
        item_n = yield from take(cta, it + 1, 1)
        yield ("wait", "o_full", it)
        assert (T + nkv - 1) in cta.pv_done
        cta.o_read[it] = cta.o_read.get(it, 0) + 1
        T += nkv
        item = item_n
        it += 1


def softmax_agent_epilogue_late(cta, a):
    """A softmax agent with one planted mistake: it publishes P of an item's
    first tile before its epilogue of the previous item has read O."""
    T = 0
    it = 0
    pending_epilogue = None
    item = yield from take(cta, 0, 1)
    while item is not None:
        nkv = cta.items[item]
        for kt in range(nkv):
            Tg = T + kt
            yield ("wait", f"s_full{Tg % S_BUFS}", Tg // S_BUFS)
            cta.s_read[Tg] = cta.s_read.get(Tg, 0) + 1
            yield ("arrive", f"p_ready{Tg % S_BUFS}", 1)
            if kt == 0 and pending_epilogue is not None:
                yield ("wait", "o_full", pending_epilogue)
                cta.o_read[pending_epilogue] = cta.o_read.get(pending_epilogue, 0) + 1
                pending_epilogue = None
        item_n = yield from take(cta, it + 1, 1)
        pending_epilogue = it
        T += nkv
        item = item_n
        it += 1
    if pending_epilogue is not None:
        yield ("wait", "o_full", pending_epilogue)
        cta.o_read[pending_epilogue] = cta.o_read.get(pending_epilogue, 0) + 1


def run(items, seed, roles_override=None):
    rng = random.Random(seed)
    cta = Cta(items, rng)
    ro = roles_override or {}
    roles = {"k": ro.get("k", k_warp)(cta), "v": v_warp(cta), "s": ro.get("s", s_thread)(cta),
             "pv": pv_thread(cta)}
    agent = ro.get("agent", softmax_agent)
    for a in range(N_SOFTMAX):
        roles[f"sm{a}"] = agent(cta, a)
    pending = {name: next(g) for name, g in roles.items()}
    done = set()
    steps = 0
    while len(done) < len(roles) or cta.tma or cta.mma["s"] or cta.mma["pv"]:
        steps += 1
        assert steps < 400000, "model did not finish"
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
        events = (["copy done"] if cta.tma else []) + [f"mma {q}" for q in ("s", "pv") if cta.mma[q]]
        choices = runnable + events
        assert choices, f"deadlock: {pending}"
        c = rng.choice(choices)
        if c == "copy done":
            cta.b[cta.tma.pop(rng.randrange(len(cta.tma)))].arrive()
            continue
        if c.startswith("mma "):
            ev = cta.mma[c[4:]].pop(0)
            if isinstance(ev, tuple):
                cta.pv_done.add(ev[1])
            else:
                cta.b[ev].arrive()
            continue
        op = pending[c]
        if op[0] == "arrive":
            cta.b[op[1]].arrive(op[2])
        elif op[0] == "tma":
            cta.tma.append(op[1])
        elif op[0] == "commit":
            cta.mma[op[1]].append(op[2])
        elif op[0] == "pv":
            cta.mma["pv"].append(("pv", op[1]))
        try:
            pending[c] = roles[c].send(None)
        except StopIteration:
            done.add(c)
    # every item was claimed, and every barrier ended between phases
    assert cta.next_claim == len(items) + 1
    for bar in cta.b.values():
        assert bar.pending == 0, f"{bar.name} left with {bar.pending} arrivals"
    assert all(cta.o_read.get(i, 0) == N_SOFTMAX for i in range(len(items)))


@pytest.mark.parametrize("case", range(60))
def test_prefill_protocol_random_items_and_interleavings(case):
    rng = random.Random(1000 + case)
    n = rng.randint(1, 14)
    # one-tile items (short prefills) mixed with items of several tiles
    items = [rng.choice([1, 1, 1, 2, 3, 4, rng.randint(1, 9)]) for _ in range(n)]
    for s in range(30):
        run(items, seed=case * 1000 + s)


def test_prefill_protocol_all_one_tile_and_all_long():
    for items in ([1] * 20, [7] * 6, [2, 1, 1, 1, 2, 1, 3, 1, 1], [1, 2] * 8, [3, 4, 5, 1]):
        for s in range(60):
            run(items, seed=s)


PLANTED = {
    # S issued as soon as K landed, without waiting for PV(T-3)
    "s_without_pv_wait": {"s": lambda cta: s_thread(cta, skip_pv_wait=True)},
    # P of an item's first tile published before the epilogue read O
    "epilogue_late": {"agent": softmax_agent_epilogue_late},
    # V rows cleaned after a wait for the tile's own copy alone
    "v_clean_one_wait": {"agent": lambda cta, a: softmax_agent(cta, a, v_clean_one_wait=True)},
    # the K-copy warp waits for the phase after the one it means
    "k_slot_phase_late": {"k": lambda cta: k_warp(cta, phase_slip=1)},
}


@pytest.mark.parametrize("mistake", sorted(PLANTED))
def test_model_catches_planted_protocol_mistakes(mistake):
    """The model is not vacuous: each planted mistake is caught (a wait at the
    wrong phase, a TMEM hazard, or a deadlock)."""
    with pytest.raises(AssertionError):
        for s in range(200):
            run([1, 5, 2, 1, 6, 3, 1, 4], seed=s, roles_override=PLANTED[mistake])
