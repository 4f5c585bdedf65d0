"""The tcgen05 kernel's barrier protocol, replayed on the CPU.

Each role of `w4a16_tc_kernel` (producer, the two pipelines' dequant
warpgroups and MMA warps, the epilogue) is written here as the sequence of
mbarrier waits and arrivals it performs per unit, with the same counts and
phase arithmetic as the kernel; the tensor core's completions (the
arrivals that tcgen05.commit produces) come later, in order per issuing
warp.  A random scheduler runs the roles.  A wait is checked the way the
hardware answers it (the parity of the barrier's current phase): the run
fails if a wait could be answered before its phase completed or after the
barrier moved two phases past it (parity aliasing), or if no role can move
(deadlock).  The launch shapes are those of the GPU tests and the benchmark
step (units of two 128-column groups over 128-row tiles, stream-K shares of
152 CTAs)."""
import os
import random
import re

import pytest

BOXU = 4         # units per box of eight groups
# (stages, A slots per pipeline) replayed; the kernel's own values are
# checked to be among them
CONFIGS = [(4, 2), (2, 2), (4, 1), (6, 3), (4, 3)]


class Aliasing(Exception):
    pass


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.ph = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.ph += 1
            self.pending = self.count

    def done(self, target):
        """Whether phase `target` has completed, as a parity wait sees it."""
        hw = (self.ph & 1) != (target & 1)
        real = self.ph > target
        if hw != real or self.ph >= target + 2:
            raise Aliasing("%s: wait for phase %d at phase %d" % (self.name, target, self.ph))
        return real


def roles(n_units, grp_first, G, NST, NSLOT):
    full = [Bar("full%d" % i, 1) for i in range(NST)]
    empty = [Bar("empty%d" % i, 1) for i in range(NST)]
    a_full = [[Bar("a_full%d.%d" % (w, i), 4) for i in range(NSLOT)] for w in range(2)]
    a_empty = [[Bar("a_empty%d.%d" % (w, i), 1) for i in range(NSLOT)] for w in range(2)]
    d_full = [Bar("d_full%d" % i, 2) for i in range(2)]
    d_empty = [Bar("d_empty%d" % i, 4) for i in range(2)]
    pending = {0: [], 1: []}        # commits of MMA warp w, completing in order

    def boxes():
        grp, nb = grp_first, -1
        for i in range(n_units):
            start = i == 0 or grp % BOXU == 0
            end = i == n_units - 1 or grp % BOXU == BOXU - 1
            if start:
                nb += 1
            grp = 0 if grp + 1 == G else grp + 1
            yield i, start, end, nb

    def producer():
        for i in range(n_units):
            s = i % NST
            if i >= NST:
                yield empty[s], i // NST - 1
            full[s].arrive()

    def mma(w):
        slot, lap = 0, 0
        for i, start, end, nb in boxes():
            if start and nb >= 2:
                yield d_empty[nb & 1], (nb >> 1) - 1
            if i % 2 == w:
                yield full[i % NST], i // NST
                for _ in range(2):
                    yield a_full[w][slot], lap
                    pending[w].append(a_empty[w][slot])
                    slot += 1
                    if slot == NSLOT:
                        slot, lap = 0, lap + 1
                pending[w].append(empty[i % NST])
            if end:
                pending[w].append(d_full[nb & 1])

    def dequant(w):
        slot, lap = 0, 0
        for i in range(n_units):
            if i % 2 != w:
                continue
            yield full[i % NST], i // NST
            for _ in range(2):
                if lap > 0:
                    yield a_empty[w][slot], lap - 1
                for _ in range(4):
                    a_full[w][slot].arrive()
                slot += 1
                if slot == NSLOT:
                    slot, lap = 0, lap + 1

    def epilogue():
        for i, start, end, nb in boxes():
            if end:
                yield d_full[nb & 1], nb >> 1
                for _ in range(4):
                    d_empty[nb & 1].arrive()

    main = {"producer": producer(), "mma0": mma(0), "mma1": mma(1), "dequant0": dequant(0),
            "dequant1": dequant(1), "epilogue": epilogue()}
    return main, pending


def replay(n_units, grp_first, G, seed, nst, nslot):
    rnd = random.Random(seed)
    gens, pending = roles(n_units, grp_first, G, nst, nslot)
    waiting = dict.fromkeys(gens)
    live = set(gens)
    while live or pending[0] or pending[1]:
        ready = [k for k in sorted(live) if waiting[k] is None or waiting[k][0].done(waiting[k][1])]
        tc = [w for w in (0, 1) if pending[w]]
        if not ready and not tc:
            return "deadlock: " + ", ".join("%s at %s:%d" % (k, waiting[k][0].name, waiting[k][1])
                                             for k in sorted(live))
        pick = rnd.randrange(len(ready) + len(tc))
        if pick >= len(ready):
            pending[tc[pick - len(ready)]].pop(0).arrive()
            continue
        k = ready[pick]
        try:
            waiting[k] = next(gens[k])
        except StopIteration:
            live.discard(k)
            waiting[k] = None
    return None


SHAPES = [(70, 1024), (300, 1024), (2500, 1024), (20000, 1024), (5000, 3072), (1000, 3072),
          (2000, 5120), (10240, 5120), (34816, 5120), (248320, 5120), (70, 17408), (5120, 17408)]


def kernel_constants():
    """TC_NSLOT and the stage count of a launch (TC_MAX_STAGES; shared memory
    holds more for every shape) from the kernel's source."""
    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "speculative_verify_gb300", "csrc", "w4a16_tc.cuh")).read()
    nslot = int(re.search(r"constexpr int TC_NSLOT = (\d+);", src).group(1))
    nst = int(re.search(r"constexpr int TC_MAX_STAGES = (\d+);", src).group(1))
    return nst, nslot


def test_the_kernels_configuration_is_replayed():
    assert kernel_constants() in CONFIGS


@pytest.mark.parametrize("nst,nslot", CONFIGS)
@pytest.mark.parametrize("V,K", SHAPES)
def test_protocol_has_no_deadlock_and_no_aliasing(V, K, nst, nslot):
    G = K // 128 // 2                       # units per tile
    U = ((V + 127) // 128) * G
    B = min(152, U)
    seeds = 3 if (nst, nslot) == kernel_constants() else 1
    for b in range(B):
        u0, u1 = b * U // B, (b + 1) * U // B
        for seed in range(seeds):
            r = replay(u1 - u0, u0 % G, G, seed, nst, nslot)
            assert r is None, (V, K, b, r)


def test_replay_catches_a_shared_slot_ring():
    """The check is not vacuous: the same replay with the A slots shared by
    both pipelines (three slots in unit order, the MMA warp of a unit's
    parity waiting on them) reports aliasing or a deadlock for some shape."""
    global roles
    orig = roles

    def shared_roles(n_units, grp_first, G, NST, NSLOT):
        full = [Bar("full%d" % i, 1) for i in range(NST)]
        empty = [Bar("empty%d" % i, 1) for i in range(NST)]
        a_full = [Bar("a_full%d" % i, 4) for i in range(NSLOT)]
        a_empty = [Bar("a_empty%d" % i, 1) for i in range(NSLOT)]
        pending = {0: [], 1: []}

        def producer():
            for i in range(n_units):
                if i >= NST:
                    yield empty[i % NST], i // NST - 1
                full[i % NST].arrive()

        def mma(w):
            for i in range(n_units):
                if i % 2 == w:
                    yield full[i % NST], i // NST
                    yield a_full[i % NSLOT], i // NSLOT
                    pending[w].append(a_empty[i % NSLOT])
                    pending[w].append(empty[i % NST])

        def dequant(w):
            for i in range(n_units):
                if i % 2 == w:
                    yield full[i % NST], i // NST
                    if i >= NSLOT:
                        yield a_empty[i % NSLOT], i // NSLOT - 1
                    for _ in range(4):
                        a_full[i % NSLOT].arrive()

        return {"producer": producer(), "mma0": mma(0), "mma1": mma(1), "dequant0": dequant(0),
                "dequant1": dequant(1)}, pending

    roles = shared_roles
    try:
        found = False
        for seed in range(40):
            try:
                if replay(24, 0, 20, seed, 6, 3) is not None:
                    found = True
            except Aliasing:
                found = True
            if found:
                break
        assert found
    finally:
        roles = orig
