"""The work queue of the persistent backward passes (csrc/fa_queue.cuh), checked on a randomised
model (no GPU).

Several CTAs share one work counter.  In each CTA a fetching thread (the TMA producer) publishes
round r's id into ring slot r % 4 once the slot's empty barrier shows that every consumer warp
has read round r - 4, one round ahead of its own use (it publishes round r+1 before it works on
round r); the consumers (the MMA warp, and elementwise warps that look one round ahead) wait on
the slot's full barrier by parity and free the slot with one arrive per warp.  Barriers follow
mbarrier semantics: a parity wait cannot tell phase k from phase k + 2.  Random interleavings
are checked for:
  - deadlock;
  - a consumer reading a slot before its round was published, or after it was overwritten by a
    later round (parity aliasing);
  - every id 0 .. total-1 handed to exactly one CTA, and every role of a CTA seeing the same ids
    in the same order, ending with the -1 that stops it.
Planted mistakes (no empty wait, a consumer that does not free its slot, fetching on the spot
instead of one round ahead while a consumer looks ahead) must be caught.
"""
import random

import pytest

SLOTS = 4


class Hazard(Exception):
    pass


class Bar:
    def __init__(self, count):
        self.count, self.phase, self.pending = count, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.phase += 1

    def done(self, parity):  # mbarrier.try_wait.parity
        return (self.phase & 1) != parity


def run(n_cta, total, consumers, seed, lag=0, mistake=None, lookahead=True, max_steps=200000):
    """`lag`: how many rounds the fetcher's loads may run ahead of the slowest consumer (None:
    unbounded, deep enough buffers)."""
    rnd = random.Random(seed)
    counter = [0]
    seen = {}  # cta -> {role: [ids]}
    prog = {}  # cta -> {consumer: the round it works on}
    agents = []
    for c in range(n_cta):
        full = [Bar(1) for _ in range(SLOTS)]
        empty = [Bar(consumers) for _ in range(SLOTS)]
        slot = [("none", None)] * SLOTS  # (round, id)
        seen[c] = {}

        def fetcher(c=c, full=full, empty=empty, slot=slot):
            got = []
            seen[c]["fetch"] = got

            def push(r, exhausted):
                s = r % SLOTS
                if r >= SLOTS and mistake != "no_empty_wait":
                    while not empty[s].done(((r // SLOTS) - 1) & 1):
                        yield
                idv = -1
                if not exhausted:
                    idv = counter[0]
                    counter[0] += 1
                    if idv >= total:
                        idv = -1
                slot[s] = (r, idv)
                full[s].arrive()
                return idv

            if mistake == "fetch_on_the_spot":
                r = 0
                while True:
                    idv = yield from push(r, False)
                    if idv < 0:
                        break
                    got.append(idv)
                    while lag is not None and min(prog[c].values()) < r - lag:
                        yield
                    for _ in range(rnd.randint(0, 3)):  # the round's work
                        yield
                    r += 1
                return
            nxt = yield from push(0, False)
            r = 0
            while True:
                idv = nxt
                if idv < 0:
                    break
                nxt = yield from push(r + 1, False)
                got.append(idv)
                # the round's loads reuse buffers that the consumers free only once they reach
                # this round (one key/value slot, one dO/LSE slot)
                while lag is not None and min(prog[c].values()) < r - lag:
                    yield
                for _ in range(rnd.randint(0, 3)):
                    yield
                r += 1

        def consumer(name, ahead, c=c, full=full, empty=empty, slot=slot):
            got = []
            seen[c][name] = got

            def pop(r):
                s = r % SLOTS
                while not full[s].done((r // SLOTS) & 1):
                    yield
                rr, idv = slot[s]
                if rr != r:
                    raise Hazard(f"CTA {c} {name}: round {r} read slot {s} holding round {rr}")
                if not (mistake == "no_free" and name == "mma"):
                    empty[s].arrive()
                return idv

            if ahead:  # the elementwise warps: round r+1 read while round r runs
                cur = yield from pop(0)
                r = 0
                while cur >= 0:
                    nxt = yield from pop(r + 1)
                    got.append(cur)
                    prog[c][name] = r
                    for _ in range(rnd.randint(0, 3)):
                        yield
                    cur = nxt
                    r += 1
                prog[c][name] = 1 << 30
            else:
                r = 0
                while True:
                    idv = yield from pop(r)
                    if idv < 0:
                        break
                    got.append(idv)
                    prog[c][name] = r
                    for _ in range(rnd.randint(0, 3)):
                        yield
                    r += 1
                prog[c][name] = 1 << 30

        names = ["mma"] + [f"ew{i}" for i in range(consumers - 1)]
        prog[c] = {n: -1 for n in names}
        for i, n in enumerate(names):
            agents.append(consumer(n, lookahead and i > 0))
        agents.append(fetcher())

    live = list(agents)
    steps = 0
    while live:
        a = rnd.choice(live)
        try:
            next(a)
        except StopIteration:
            live.remove(a)
        steps += 1
        if steps > max_steps:
            raise Hazard("deadlock")
    ids = sorted(i for c in seen for i in seen[c]["fetch"])
    if ids != list(range(total)):
        raise Hazard(f"ids handed out: {ids[:10]}... of {total}")
    for c in seen:
        ref = seen[c]["fetch"]
        for role, got in seen[c].items():
            if got != ref:
                raise Hazard(f"CTA {c}: {role} saw {got}, the fetcher published {ref}")
    return steps


@pytest.mark.parametrize("seed", range(40))
def test_queue_protocol_holds(seed):
    rnd = random.Random(seed)
    run(n_cta=rnd.randint(1, 5), total=rnd.randint(0, 40), consumers=rnd.randint(2, 5),
        seed=seed, lag=rnd.choice([0, 1, 2, None]))


# The slot reuse only goes wrong when the fetcher can run more than kQueueSlots rounds ahead,
# so that mistake is planted with deep buffers; fetching on the spot deadlocks only when the
# loads wait for the consumers.
@pytest.mark.parametrize("mistake,lag", [("no_empty_wait", None), ("no_free", 0),
                                         ("no_free", None), ("fetch_on_the_spot", 0)])
def test_queue_mistakes_caught(mistake, lag):
    caught = 0
    for seed in range(60):
        try:
            run(n_cta=3, total=30, consumers=3, seed=seed, lag=lag, mistake=mistake,
                max_steps=20000)
        except Hazard:
            caught += 1
    assert caught >= 50, (mistake, caught)
