"""Host-side model of the mbarrier protocols of the two-group dK formers (no GPU).

The dW and dY kernels run two groups of former warps on alternate tiles beside one
TMA producer and an MMA issuer, all synchronised by mbarriers that are waited on by
phase parity.  A parity wait cannot tell the phase it wants from the one two uses
back, so it is sound only for a waiter that has itself seen the barrier's previous
phase.  These tests run the kernels' protocols against a model of an mbarrier (arrival
count, transaction bytes, phase) under random schedules in which TMA copies land in any
order, and check that no tile is formed from a stage holding other data, no stage is
reloaded while still owed to a former, no dK buffer is overwritten before the MMA read
it, and nothing deadlocks.  A shared full barrier per stage (what the first two-group
version used) must fail the same checks when the ring depth is odd.
"""
import random

import pytest


class Bar:
    """An mbarrier: `count` arrivals and all expected transaction bytes complete a phase."""

    def __init__(self, count):
        self.count, self.pending, self.phase, self.tx = count, count, 0, 0

    def arrive(self, tx=0):
        self.tx += tx
        self.pending -= 1
        assert self.pending >= 0, "arrival count underflow"
        self._complete()

    def complete_tx(self, n):
        self.tx -= n
        assert self.tx >= 0, "transaction count underflow"
        self._complete()

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def passes(self, parity):
        # try_wait.parity(P) succeeds while the current phase's parity differs from P
        return (self.phase & 1) != parity


def run_dw(n, NX, per_group_full, seed):
    """dW: a producer fills an NX-deep x/grad ring; group g forms tiles i = g, g+2, ...
    into dK buffer g (first waiting on the stage's full barrier, then on the buffer's
    empty barrier); the issuer consumes the buffers in tile order and frees them later."""
    rnd = random.Random(seed)
    NL = NX if NX % 2 == 0 else 2 * NX          # tiles between two uses of one (stage, group) pair
    full = [[Bar(1) for _ in range(NX)] for _ in range(2)] if per_group_full else [[Bar(1) for _ in range(NX)]] * 2
    empty = [Bar(1) for _ in range(NX)]         # one arrival per formed tile (the group's warps as one)
    dk_full = [Bar(1), Bar(1)]
    dk_empty = [Bar(1), Bar(1)]
    stage, owner = [None] * NX, [None] * NX
    dkbuf = [None, None]
    inflight, commits = [], []
    prod, nxt, state, iss = 0, [0, 1], [0, 0], 0
    for _ in range(200000):
        if iss == n:
            return
        acts = []
        if prod < n and empty[prod % NX].passes(((prod // NX) & 1) ^ 1):
            acts.append(("prod",))
        for g in range(2):
            i = nxt[g]
            if i < n:
                par = ((i // NL) & 1) if per_group_full else ((i // NX) & 1)
                if state[g] == 0 and full[g][i % NX].passes(par):
                    acts.append(("full_seen", g))
                if state[g] == 1 and dk_empty[g].passes(((i >> 1) & 1) ^ 1):
                    acts.append(("form", g))
        if iss < n and dk_full[iss & 1].passes((iss >> 1) & 1):
            acts.append(("mma",))
        if inflight:
            acts.append(("land",))
        if commits:
            acts.append(("commit",))
        assert acts, "deadlock"
        a = rnd.choice(acts)
        if a[0] == "prod":
            s = prod % NX
            assert owner[s] is None, f"stage {s} reloaded for tile {prod} while tile {owner[s]} is not formed"
            owner[s], stage[s] = prod, None
            bar = full[prod & 1][s] if per_group_full else full[0][s]
            bar.arrive(tx=2)                     # arrive.expect_tx, then two copies
            inflight += [(prod, s, bar, False), (prod, s, bar, True)]
            prod += 1
        elif a[0] == "land":                     # copies complete in any order
            i, s, bar, last = inflight.pop(rnd.randrange(len(inflight)))
            if not any(t == i for t, *_ in inflight):
                stage[s] = i
            bar.complete_tx(1)
        elif a[0] == "full_seen":
            state[a[1]] = 1
        elif a[0] == "form":
            g = a[1]
            i = nxt[g]
            s = i % NX
            assert stage[s] == i, f"group {g} formed tile {i} from a stage holding {stage[s]}"
            assert dkbuf[g] is None, "dK buffer overwritten before the MMA read it"
            dkbuf[g] = i
            owner[s] = None
            dk_full[g].arrive()
            empty[s].arrive()
            state[g] = 0
            nxt[g] += 2
        elif a[0] == "mma":
            assert dkbuf[iss & 1] == iss, f"MMA of tile {iss} read a buffer holding {dkbuf[iss & 1]}"
            commits.append(iss & 1)
            iss += 1
        else:                                    # MMAs complete in issue order
            b = commits.pop(0)
            dkbuf[b] = None
            dk_empty[b].arrive()
    raise AssertionError("no progress")


def run_dy(nb, SUB, seed, NX=2):
    """dY: a 2-deep x/grad ring of channel blocks; with SUB = 4 sub-tiles per block both
    groups read every block (alternate sub-tiles), with SUB = 1 they take alternate blocks."""
    rnd = random.Random(seed)
    full = [Bar(1) for _ in range(NX)]
    empty = [Bar(2 if SUB > 1 else 1) for _ in range(NX)]
    dk_full, dk_empty = [Bar(1), Bar(1)], [Bar(1), Bar(1)]
    stage, readers = [None] * NX, [0] * NX
    dkbuf = [None, None]
    inflight, commits = [], []
    prod, blk, subs, iss = 0, [0, 0 if SUB > 1 else 1], [None, None], 0
    total = nb * SUB
    for _ in range(400000):
        if iss == total:
            return
        acts = []
        if prod < nb and empty[prod % NX].passes(((prod // NX) & 1) ^ 1):
            acts.append(("prod",))
        for g in range(2):
            i = blk[g]
            if i >= nb:
                continue
            if subs[g] is None and full[i % NX].passes((i // NX) & 1):
                acts.append(("full_seen", g))
            elif subs[g] is not None and dk_empty[g].passes((((i * SUB + subs[g][0]) >> 1) & 1) ^ 1):
                acts.append(("form", g))
        if iss < total and dk_full[iss & 1].passes((iss >> 1) & 1):
            acts.append(("mma",))
        if inflight:
            acts.append(("land",))
        if commits:
            acts.append(("commit",))
        assert acts, "deadlock"
        a = rnd.choice(acts)
        if a[0] == "prod":
            s = prod % NX
            assert readers[s] == 0, f"stage {s} reloaded while being read"
            stage[s], readers[s] = None, (2 if SUB > 1 else 1)
            full[s].arrive(tx=1)
            inflight.append((prod, s))
            prod += 1
        elif a[0] == "land":
            i, s = inflight.pop(rnd.randrange(len(inflight)))
            stage[s] = i
            full[s].complete_tx(1)
        elif a[0] == "full_seen":
            g = a[1]
            subs[g] = [st for st in range(SUB) if SUB == 1 or st % 2 == g]
        elif a[0] == "form":
            g = a[1]
            i = blk[g]
            s = i % NX
            kd = i * SUB + subs[g].pop(0)
            assert stage[s] == i, f"group {g} formed block {i} from a stage holding {stage[s]}"
            assert kd & 1 == g and dkbuf[g] is None, "dK buffer overwritten before the MMA read it"
            dkbuf[g] = kd
            dk_full[g].arrive()
            if not subs[g]:
                subs[g] = None
                readers[s] -= 1
                empty[s].arrive()
                blk[g] += 1 if SUB > 1 else 2
        elif a[0] == "mma":
            assert dkbuf[iss & 1] == iss, f"MMA of sub-tile {iss} read {dkbuf[iss & 1]}"
            commits.append(iss & 1)
            iss += 1
        else:
            b = commits.pop(0)
            dkbuf[b] = None
            dk_empty[b].arrive()
    raise AssertionError("no progress")


@pytest.mark.parametrize("NX", [2, 3, 4])
def test_dw_per_group_full_barriers_are_sound(NX):
    for seed in range(400):
        run_dw(1 + seed % 30, NX, per_group_full=True, seed=seed)


def test_dw_shared_full_barrier_fails_for_odd_ring_depth():
    failures = 0
    for seed in range(400):
        try:
            run_dw(1 + seed % 30, 3, per_group_full=False, seed=seed)
        except AssertionError:
            failures += 1
    assert failures > 0, "the model should catch the shared-barrier race"


@pytest.mark.parametrize("SUB", [1, 4])
def test_dy_two_group_protocol_is_sound(SUB):
    for seed in range(400):
        run_dy(1 + seed % 30, SUB, seed)
