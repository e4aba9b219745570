"""Event model of the barrier protocol of attn_wide_kernel (csrc/attn_wide.cu), the
d_k = 128 forward: a TMA loader, one MMA issuer per slot passing a turn token, and one
softmax warpgroup per slot, synchronised through mbarriers with phase parities.

The roles below follow the kernel's loops step for step (key-tile ranges per slot,
fill indices and stage parities of the K and V rings, the token, the commits), in
both instantiations: two query tiles of one head per CTA, and two heads of a single
query and key tile each.  Every asynchronous operation completes at a random later
time: TMA copies in any order, each issuer's MMAs and commits in issue order (one
thread's tcgen05 operations execute in order), the two issuers' streams interleaved
at random.  The model checks that no role waits forever, that every MMA reads the
K or V tile it should from its stage (a refill clears the stage while it is in
flight), that each P V reads the P of its own tile and each S overwrites P only
after that P V, that O holds exactly the finished tiles when the softmax sees the
next S (so it may rescale) and when the epilogue reads it, and that no S MMA is
left to read the slot's Q buffer when the epilogue stages its output tile there.
A mutant with stage-release barriers that expect one commit instead of two must be
caught.
"""
import random

import pytest

KB = 128  # rows per query tile, keys per key tile


def slot_range(m, n, length, causal, window, q0):
    """Key tiles [lo, hi) that query rows q0 .. min(m, q0 + 128) - 1 can see."""
    if q0 >= m:
        return 0, 0
    kv_end = min(length, q0 + KB) if causal else length
    first = 0
    if window >= 0:
        first = max(0, q0 - window) // KB
        kv_end = min(kv_end, min(m, q0 + KB) + window)
    if kv_end <= first * KB:
        return 0, 0
    return first, (kv_end + KB - 1) // KB


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.phase = count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, parity):
        """Phase of this parity has completed (the mbarrier parity test)."""
        return (self.phase & 1) != parity


class Deadlock(Exception):
    pass


def simulate(ranges, head_pairs, rng, release_count=2):
    """ranges: [(lo, hi)] per slot.  Raises AssertionError on a protocol violation and
    Deadlock when no role can make progress."""
    lo = [r[0] for r in ranges]
    hi = [r[1] for r in ranges]
    busy = [s for s in range(2) if hi[s] > lo[s]]
    if not busy:
        return
    t_lo, t_hi = min(lo[s] for s in busy), max(hi[s] for s in busy)
    n_fill = t_hi - t_lo
    bar = {}
    for s in range(2):
        bar[f"q{s}"], bar[f"s{s}"], bar[f"p{s}"], bar[f"o{s}"] = Barrier(1), Barrier(1), Barrier(KB), Barrier(1)
        bar[f"turn{s}"] = Barrier(1)
        bar[f"kf{s}"], bar[f"vf{s}"] = Barrier(1), Barrier(1)
        bar[f"ke{s}"], bar[f"ve{s}"] = Barrier(release_count), Barrier(release_count)
    stage = {"K": [None, None], "V": [None, None]}
    tmem = {"S": [None, None], "O": [[], []]}
    copies = []           # TMA completions, any order
    pipes = [[], []]      # each issuer's MMAs and commits, in issue order

    def load(kind, st, tile, full):
        stage[kind][st] = None  # being overwritten

        def land():
            stage[kind][st] = tile
            bar[full].arrive()
        copies.append(land)

    def loader():
        for s in range(2):
            if hi[s] == lo[s]:
                continue
            copies.append(lambda s=s: bar[f"q{s}"].arrive())
            if head_pairs:
                load("K", s, (s, 0), f"kf{s}")
                load("V", s, (s, 0), f"vf{s}")
        if head_pairs:
            return
        for f in range(n_fill):
            st, par = f % 2, ((f // 2) & 1) ^ 1
            while not bar[f"ke{st}"].done(par):
                yield
            load("K", st, (None, t_lo + f), f"kf{st}")
            while not bar[f"ve{st}"].done(par):
                yield
            load("V", st, (None, t_lo + f), f"vf{st}")

    def issuer(s):
        q_in = False
        for t in range(t_lo, t_hi + 1):
            f = t - t_lo
            st = s if head_pairs else f % 2
            pst = s if head_pairs else (f + 1) % 2
            k_par = 0 if head_pairs else (f // 2) & 1
            v_par = 0 if head_pairs else ((f - 1) // 2) & 1
            do_pv, do_s = lo[s] <= t - 1 < hi[s], lo[s] <= t < hi[s]
            if t > t_lo and (not head_pairs or do_pv):
                while not bar[f"vf{pst}"].done(v_par):
                    yield
            if do_pv:
                while not bar[f"p{s}"].done((t - 1 - lo[s]) & 1):
                    yield
            if t < t_hi and (not head_pairs or do_s):
                while not bar[f"kf{st}"].done(k_par):
                    yield
            if do_s and not q_in:
                while not bar[f"q{s}"].done(0):
                    yield
                q_in = True
            if s == 1 or t > t_lo:
                while not bar[f"turn{s}"].done((f if s == 1 else f - 1) & 1):
                    yield
            tile = (s, 0) if head_pairs else (None, t)
            prev = (s, 0) if head_pairs else (None, t - 1)
            if do_pv:
                pipes[s].append(("pv", s, pst, prev, t - 1))
                if t == hi[s]:
                    pipes[s].append(("commit", f"o{s}"))
            if t > t_lo and not head_pairs:
                pipes[s].append(("commit", f"ve{pst}"))
            if do_s:
                pipes[s].append(("s", s, st, tile, t))
                pipes[s].append(("commit", f"s{s}"))
            if t < t_hi and not head_pairs:
                pipes[s].append(("commit", f"ke{st}"))
            bar[f"turn{1 - s}"].arrive()

    def softmax(s):
        for j in range(hi[s] - lo[s]):
            while not bar[f"s{s}"].done(j & 1):
                yield
            assert tmem["S"][s] == ("S", lo[s] + j)
            assert tmem["O"][s] == list(range(lo[s], lo[s] + j))  # O complete: may rescale
            tmem["S"][s] = ("P", lo[s] + j)
            for _ in range(KB):
                bar[f"p{s}"].arrive()
        if hi[s] > lo[s]:
            while not bar[f"o{s}"].done(0):
                yield
            assert tmem["O"][s] == list(range(lo[s], hi[s]))
            # the epilogue stages the output tile in the slot's Q buffer: no S MMA of
            # the slot may still be waiting to read Q
            assert not any(op[0] == "s" and op[1] == s for op in pipes[0] + pipes[1])

    def execute(op):
        if op[0] == "commit":
            bar[op[1]].arrive()
        elif op[0] == "s":
            _, s, st, tile, t = op
            assert stage["K"][st] == tile, ("S reads a K stage that does not hold its tile", op)
            assert tmem["S"][s] is None or tmem["S"][s][0] == "P", "S overwrites scores not yet turned into P"
            tmem["S"][s] = ("S", t)
        else:
            _, s, st, tile, t = op
            assert stage["V"][st] == tile, ("P V reads a V stage that does not hold its tile", op)
            assert tmem["S"][s] == ("P", t), "P V reads the wrong P"
            tmem["O"][s].append(t)

    roles = [loader(), issuer(0), issuer(1), softmax(0), softmax(1)]
    alive = list(roles)
    idle = 0
    while alive or copies or pipes[0] or pipes[1]:
        progressed = False
        for r in list(alive):
            try:
                next(r)
            except StopIteration:
                alive.remove(r)
                progressed = True
        if copies and rng.random() < 0.5:
            copies.pop(rng.randrange(len(copies)))()
            progressed = True
        pipe = pipes[rng.randrange(2)]
        if pipe and rng.random() < 0.5:
            execute(pipe.pop(0))
            progressed = True
        idle = 0 if progressed else idle + 1
        if idle > 2000:
            raise Deadlock(ranges)


def query_pair_cases():
    cases = set()
    for m in (1, 100, 128, 129, 255, 256, 257, 300, 700, 1000):
        for causal in (0, 1):
            for window in (-1, 0, 1, 127, 128, 200, 5000):
                for length in (0, 1, 50, m // 2, m):
                    for qp in range((m + 255) // 256):
                        cases.add(tuple(slot_range(m, m, length, causal, window, qp * 256 + s * KB) for s in range(2)))
    for m, n in ((100, 333), (128, 1000), (1, 77), (200, 200)):
        for length in (0, 1, n):
            for qp in range((m + 255) // 256):
                cases.add(tuple(slot_range(m, n, length, 0, -1, qp * 256 + s * KB) for s in range(2)))
    return sorted(cases)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_query_tile_pairs(seed):
    rng = random.Random(seed)
    cases = query_pair_cases()
    assert len(cases) > 30
    for ranges in cases:
        simulate(list(ranges), False, rng)


def test_head_pairs():
    rng = random.Random(4)
    for _ in range(200):
        for busy in ((1, 1), (1, 0), (0, 1), (0, 0)):
            simulate([(0, 1) if b else (0, 0) for b in busy], True, rng)


def test_model_catches_early_stage_release():
    """With a stage freed by one issuer's commit instead of both, a refill can land
    under the other issuer's MMA: the model must report it."""
    rng = random.Random(5)
    caught = 0
    for _ in range(40):
        for ranges in ([(0, 6), (0, 7)], [(2, 9), (3, 10)]):
            try:
                simulate(ranges, False, rng, release_count=1)
            except (AssertionError, Deadlock):
                caught += 1
    assert caught > 0
