"""Model check of the decode kernel's shared-memory ring, on the CPU.

One producer warp fills a ring of S stages (S chosen at launch, 2 to 6):
for the i-th stage it hands out it waits, from the second round on, for
the slot's empty barrier (one arrival per consumer warp) and then fills the
slot (a copy completing the full barrier), ending with an end-marker stage.
Each of the VH consumer warps waits for the full barrier of every stage and
arrives on its empty barrier.

The kernel tracks the ring slot and the parities incrementally: the
consumers' full parity flips on every wrap; the producer's empty parity
from the second wrap on. This model restates those updates and runs them
under random interleavings, with copies completing in any order. Every wait
must find its barrier at the phase it means or one past it (no parity
aliasing), no phase may be over-arrived, and nothing may deadlock.
"""

import random

import pytest


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.phases = count, 0, 0

    def arrive(self):
        self.pending += 1
        assert self.pending <= self.count
        if self.pending == self.count:
            self.pending, self.phases = 0, self.phases + 1


def producer(S, n_chunks):
    s, eph = 0, 0
    issued = 0
    while True:
        if issued >= S:
            # the phase this wait means: round (issued // S) - 1 of the slot
            yield ("wait", ("empty", s), issued // S - 1, eph)
        if issued == n_chunks:  # the end marker
            yield ("fill", s)
            return
        yield ("fill", s)
        if s + 1 == S:  # the kernel's update: ring wraps; from the second wrap on, flip
            s = 0
            if issued + 1 > S:
                eph ^= 1
        else:
            s += 1
        issued += 1


def consumer(S, n_chunks):
    s, fph = 0, 0
    i = 0
    while True:
        yield ("wait", ("full", s), i // S, fph)
        if i == n_chunks:  # read the end marker
            return
        yield ("arrive", ("empty", s))
        s += 1
        if s == S:
            s, fph = 0, fph ^ 1
        i += 1


def run(S, VH, n_chunks, seed):
    rng = random.Random(seed)
    bars = {}
    for s in range(S):
        bars[("full", s)] = Barrier(1)
        bars[("empty", s)] = Barrier(VH)
    roles = {"p": producer(S, n_chunks)}
    for w in range(VH):
        roles[f"c{w}"] = consumer(S, n_chunks)
    pending = {k: next(g) for k, g in roles.items()}
    copies = []
    done = set()
    while len(done) < len(roles) or copies:
        runnable = []
        for name, op in pending.items():
            if name in done:
                continue
            if op[0] == "wait":
                bar, k, parity = bars[op[1]], op[2], op[3]
                assert parity == k & 1, f"{name}: tracked parity {parity} for phase {k}"
                assert bar.phases in (k, k + 1), f"{name}: phase {k} of {op[1]}, at {bar.phases}"
                if bar.phases == k:
                    continue
            runnable.append(name)
        choices = runnable + (["copy done"] if copies else [])
        assert choices, "deadlock"
        c = rng.choice(choices)
        if c == "copy done":
            bars[copies.pop(rng.randrange(len(copies)))].arrive()
            continue
        op = pending[c]
        if op[0] == "fill":
            copies.append(("full", op[1]))
        elif op[0] == "arrive":
            bars[op[1]].arrive()
        try:
            pending[c] = next(roles[c])
        except StopIteration:
            done.add(c)


@pytest.mark.parametrize("S", [2, 3, 4, 5, 6])
@pytest.mark.parametrize("VH", [1, 2, 8])
def test_decode_ring_parities_and_progress(S, VH):
    for n in (0, 1, S - 1, S, S + 1, 2 * S, 2 * S + 1, 5 * S + 3, 40):
        for seed in range(15):
            run(S, VH, n, seed * 100 + n)


def test_model_catches_a_parity_flip_on_the_first_wrap():
    """The model is not vacuous: flipping the producer's empty parity on the
    first wrap too (the natural slip) is caught."""
    global producer
    saved = producer

    def flips_early(S, n_chunks):
        s, eph, issued = 0, 0, 0
        while True:
            if issued >= S:
                yield ("wait", ("empty", s), issued // S - 1, eph)
            if issued == n_chunks:
                yield ("fill", s)
                return
            yield ("fill", s)
            s += 1
            if s == S:
                s, eph = 0, eph ^ 1
            issued += 1

    producer = flips_early
    try:
        with pytest.raises(AssertionError):
            run(3, 2, 10, 0)
    finally:
        producer = saved
