"""The barrier protocol of the persistent dQ kernel (fa_bwd_dq_kernel_persistent), checked on a
randomised model (no GPU).

The model runs the kernel's roles as coroutines: the TMA producer, the MMA issuer, one or more
elementwise warp groups, an in-order tensor core (MMAs and commits execute in issue order) and
out-of-order TMA completions.  Every barrier wait, arrival and commit is the kernel's, in the
kernel's order, over a CTA's sequence of query tiles (each with its own number of key tiles);
phases count key-tile iterations (or tiles) over the CTA's lifetime as in the kernel.  Random
interleavings are checked for:
  - deadlock;
  - mbarrier parity aliasing: a barrier must never complete a second phase while a waiter for
    an earlier one is pending (a parity wait would then miss it);
  - data hazards: every read of Q, a K/V ring slot, S, dP, dS, dO or the dQ accumulator sees
    the version it needs, and nothing is overwritten while an MMA that reads it is pending.
Planted mistakes (a dropped wait, a misplaced commit, dO staged too early) must be caught.
"""
import random

import pytest


class Hazard(Exception):
    pass


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.phase, self.pending, self.waiters = name, count, 0, 0, []

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.phase += 1
            for k in self.waiters:
                if self.phase > k + 1:
                    raise Hazard(f"{self.name} completed phase {self.phase - 1} while a waiter "
                                 f"for phase {k} was pending")


def simulate(tiles, stages, groups, seed, skip=frozenset()):
    """One CTA's run over query tiles with `tiles[t]` key tiles each.  `skip` names planted
    mistakes.  Raises Hazard on any violation."""
    rnd = random.Random(seed)
    bar = {n: Bar(n, c) for n, c in [("sf", 1), ("df", 1), ("sr", groups), ("dpr", groups),
                                      ("pd", groups), ("dqd", 1), ("q", 1), ("qe", 1),
                                      ("qt", groups), ("done", 1), ("dqr", groups), ("fin", 1)]}
    kvf = [Bar(f"kvf{i}", 1) for i in range(stages)]
    kve = [Bar(f"kve{i}", 1) for i in range(stages)]
    first = [0]
    for n in tiles:
        first.append(first[-1] + n)
    st = {"Q": None, "slot": [None] * stages, "S": None, "DP": None, "DO": None, "DQ": None,
          "DQn": 0, "dp_done": -1, "dq_done": -1}
    reads = {}        # buffer -> MMAs issued but not executed that read it
    count = {}        # (what, index) -> arrivals of all groups
    queue, tma = [], []

    def bump(key):
        count[key] = count.get(key, 0) + 1

    def need(key):
        return count.get(key, 0) == groups

    def wait(b, k):
        if b.phase not in (k, k + 1):
            raise Hazard(f"wait on {b.name} for phase {k} at phase {b.phase}")
        b.waiters.append(k)
        while b.phase < k + 1:
            yield
        b.waiters.remove(k)

    def issue(fn, bufs, commit=None):
        for x in bufs:
            reads[x] = reads.get(x, 0) + 1
        queue.append(("mma", fn, bufs))
        if commit is not None:
            queue.append(("commit", commit, None))

    def s_mma(g, t):
        def run():
            if st["Q"] != t or st["slot"][g % stages] != g:
                raise Hazard(f"S({g}) read Q {st['Q']} / K {st['slot'][g % stages]}")
            if g > 0 and not need(("Sread", g - 1)):
                raise Hazard(f"S({g}) overwrote S({g - 1}) before it was read")
            st["S"] = g
        return run

    def dp_mma(g, t):
        def run():
            if st["DO"] != t or not need(("DO", t)) or st["slot"][g % stages] != g:
                raise Hazard(f"dP({g}) read dO of tile {st['DO']} / V {st['slot'][g % stages]}")
            if g > 0 and not need(("DPread", g - 1)):
                raise Hazard(f"dP({g}) overwrote dP({g - 1}) before it was read")
            st["DP"] = g
            st["dp_done"] = g
        return run

    def dq_mma(g, t, j):
        def run():
            if not need(("DS", g)) or st["slot"][g % stages] != g:
                raise Hazard(f"dQ({g}) read an incomplete dS or K {st['slot'][g % stages]}")
            if j == 0:
                if t > 0 and not need(("DQread", t - 1)):
                    raise Hazard(f"tile {t} overwrote dQ of tile {t - 1} before its read-out")
                st["DQ"], st["DQn"] = t, 1
            else:
                st["DQn"] += 1
            st["dq_done"] = g
        return run

    def producer():
        gk = 0
        for t, n in enumerate(tiles):
            if t > 0 and "qe_wait" not in skip:
                yield from wait(bar["qe"], t - 1)
            if reads.get("Q", 0):
                raise Hazard(f"Q of tile {t} loaded while an S still reads the previous Q")
            tma.append((bar["q"], lambda t=t: st.__setitem__("Q", t)))
            for _ in range(n):
                s = gk % stages
                if gk >= stages and "kve_wait" not in skip:
                    yield from wait(kve[s], gk // stages - 1)
                if reads.get(("slot", s), 0):
                    raise Hazard(f"ring slot {s} refilled while an MMA reads it")

                def land(s=s, g=gk):
                    st["slot"][s] = g
                tma.append((kvf[s], land))
                gk += 1
            yield

    def mma():
        g = 0
        for t, n in enumerate(tiles):
            yield from wait(bar["q"], t)
            yield from wait(bar["qt"], t)
            if g > 0:
                yield from wait(bar["sr"], g - 1)
                yield from wait(bar["dpr"], g - 1)
            yield from wait(kvf[g % stages], g // stages)
            issue(s_mma(g, t), ["Q", ("slot", g % stages)], bar["sf"])
            if n == 1:
                queue.append(("commit", bar["qe"], None))
            issue(dp_mma(g, t), ["DO", ("slot", g % stages)], bar["df"])
            for j in range(n):
                gg = g + j
                if j + 1 < n:
                    yield from wait(kvf[(gg + 1) % stages], (gg + 1) // stages)
                    yield from wait(bar["sr"], gg)
                    issue(s_mma(gg + 1, t), ["Q", ("slot", (gg + 1) % stages)], bar["sf"])
                    if j + 2 == n + (1 if "qe_commit_late" in skip else 0):
                        queue.append(("commit", bar["qe"], None))
                    yield from wait(bar["dpr"], gg)
                    issue(dp_mma(gg + 1, t), ["DO", ("slot", (gg + 1) % stages)], bar["df"])
                yield from wait(bar["pd"], gg)
                if j == 0 and t > 0:
                    yield from wait(bar["dqr"], t - 1)
                issue(dq_mma(gg, t, j), ["DS", ("slot", gg % stages)])
                queue.append(("commit", kve[gg % stages], None))
                queue.append(("commit", bar["dqd"], None))
            queue.append(("commit", bar["done"], None))
            g += n
        queue.append(("commit", bar["fin"], None))
        yield from wait(bar["fin"], 0)

    def stage(t):
        if reads.get("DO", 0) or (t > 0 and st["dp_done"] < first[t] - 1):
            raise Hazard(f"dO of tile {t} staged while a dP of tile {t - 1} still reads dO")
        st["DO"] = t
        bump(("DO", t))
        bar["qt"].arrive()

    def elementwise():
        stage(0)
        g = 0
        for t, n in enumerate(tiles):
            for j in range(n):
                gg = g + j
                if j == n - 1 and t + 1 < len(tiles) and "stage_early" in skip:
                    stage(t + 1)
                    yield
                yield from wait(bar["sf"], gg)
                if st["S"] != gg:
                    raise Hazard(f"read S({st['S']}) for iteration {gg}")
                bump(("Sread", gg))
                bar["sr"].arrive()
                yield
                yield from wait(bar["df"], gg)
                if st["DP"] != gg:
                    raise Hazard(f"read dP({st['DP']}) for iteration {gg}")
                bump(("DPread", gg))
                bar["dpr"].arrive()
                yield
                if gg > 0 and "dqd_wait" not in skip:
                    yield from wait(bar["dqd"], gg - 1)
                if gg > 0 and st["dq_done"] < gg - 1:
                    raise Hazard(f"dS({gg}) written before dQ({gg - 1}) read dS({gg - 1})")
                bump(("DS", gg))
                bar["pd"].arrive()
                yield
                if j == n - 1 and t + 1 < len(tiles) and "stage_early" not in skip:
                    stage(t + 1)
                    yield
            yield from wait(bar["done"], t)
            if st["DQ"] != t or st["DQn"] != n:
                raise Hazard(f"read out dQ of tile {st['DQ']} after {st['DQn']} of {n} updates")
            bump(("DQread", t))
            bar["dqr"].arrive()
            yield
            g += n

    actors = {"producer": producer(), "mma": mma()}
    for e in range(groups):
        actors[f"ew{e}"] = elementwise()
    finished = set()
    for _ in range(200000):
        choices = [a for a in actors if a not in finished]
        choices += ["tensor"] * bool(queue) + ["tma"] * bool(tma)
        if not choices:
            return
        a = rnd.choice(choices)
        if a == "tensor":
            kind, x, bufs = queue.pop(0)
            if kind == "mma":
                x()
                for b in bufs:
                    reads[b] -= 1
            else:
                x.arrive()
        elif a == "tma":
            b, land = tma.pop(rnd.randrange(len(tma)))
            land()
            b.arrive()
        else:
            try:
                next(actors[a])
            except StopIteration:
                finished.add(a)
    raise Hazard("deadlock: " + ", ".join(a for a in actors if a not in finished))


def cases(n):
    for seed in range(n):
        rnd = random.Random(seed)
        n_tiles = rnd.randint(1, 6)
        causal = rnd.random() < 0.5
        tiles = ([rnd.randint(1, 5) for _ in range(n_tiles)] if causal
                 else [rnd.randint(1, 4)] * n_tiles)
        yield tiles, rnd.choice([2, 3, 4, 6]), rnd.choice([1, 2, 3]), seed


def test_protocol_holds_under_random_interleavings():
    for tiles, stages, groups, seed in cases(2000):
        simulate(tiles, stages, groups, seed)


@pytest.mark.parametrize("mistake", ["qe_wait", "kve_wait", "dqd_wait", "qe_commit_late",
                                     "stage_early"])
def test_planted_mistakes_are_caught(mistake):
    with pytest.raises(Hazard):
        for tiles, stages, groups, seed in cases(400):
            simulate(tiles, stages, groups, seed, skip=frozenset({mistake}))
