"""Model check of the forward kernel's named-barrier variant (host-only).

With a K/V ring of four or more slots, the one-CTA forward kernel
(exact_attention_17_gb300/csrc/fa2_fwd_sm103.cuh, kNamedP) replaces the MMA
issuer's mbarrier polling by two named (hardware) barriers:

* kBarP0, one phase per key tile j of the CTA: softmax warpgroup 0 joins
  once P_0(j) is in TMEM (j < n0), a watcher warp joins once V_j and K_(j+1)
  have landed, and the issuing warp waits there before P_0(j) V and
  S_0(j+1);
* kBarP1, one phase per tile j < n1: softmax warpgroup 1 joins with
  P_1(j), the issuing warp waits before P_1(j) V and S_1(j+1).

A named barrier counts arrivals but has no phase number: an arrival meant
for the next phase, made while the current one is still open, would be
counted in the current one.  Nor does a wait on it end by timing out.  Every
role therefore waits at each phase (bar.sync) rather than only arriving:
the softmax warpgroups lose nothing by it, since their next S cannot be
ready before the issuing warp has passed the phase.  This model checks,
under random interleavings, that

* every arrival lands in the phase it is meant for (no role runs ahead);
* each phase gets exactly its expected count, with the same count given
  by every participant;
* the data protocol of test_pipeline_protocol (ring slots, TMEM S/P and O
  hazards) holds with these waits;
* after an abort raised at any point by any role (a bounded mbarrier wait
  that ran out), every role still passes every phase it owes, so that the
  CTA finishes: the softmax warpgroups go through their remaining phases
  in step with the issuing warp, the watcher skips its waits but not its
  phases, and the issuing warp keeps going.

Planted mistakes -- softmax warpgroups that only arrive (bar.arrive) and
so can run a phase ahead after an abort, a softmax warpgroup that stops at
an abort without passing its remaining phases, a watcher that stops at an
abort, and a count that leaves out the watcher -- must each end in a
reported error.
"""

import pytest

from test_pipeline_protocol import ProtocolError, Sim

P0_COUNT = 128 + 64   # softmax warpgroup 0 + issuing warp + watcher warp
P0_IDLE = 64          # issuing + watcher warps, sub-tile 0 done
P1_COUNT = 128 + 32   # softmax warpgroup 1 + issuing warp


class NamedBarrier:
    def __init__(self, name):
        self.name = name
        self.completed = 0
        self.count = None
        self.arrived = 0

    def arrive(self, phase, count, threads):
        if phase != self.completed:
            raise ProtocolError(f"{self.name}: arrival for phase {phase} while phase "
                                f"{self.completed} is open")
        if self.count is None:
            self.count = count
        elif self.count != count:
            raise ProtocolError(f"{self.name}: phase {phase} given counts {self.count} and {count}")
        self.arrived += threads
        if self.arrived > self.count:
            raise ProtocolError(f"{self.name}: phase {phase} over its count")
        if self.arrived == self.count:
            self.completed += 1
            self.count, self.arrived = None, 0

    def passed(self, phase):
        return self.completed > phase


class NamedSim(Sim):
    """The kernel's named-barrier protocol; `abort_at` = (role, step) raises
    an abort when that role reaches that many scheduling steps."""

    # planted mistakes (the kernel's protocol has none)
    softmax_stops_at_abort = False
    softmax_only_arrives = False
    watcher_stops_at_abort = False
    p0_count = P0_COUNT

    def __init__(self, stages, n0, n1, seed, abort_at=None, **kw):
        super().__init__(stages, n0, n1, seed, **kw)
        self.bp = [NamedBarrier("kBarP0"), NamedBarrier("kBarP1")]
        self.abort = False
        self.abort_at = abort_at
        self.steps = {}

    def tick(self, role):
        """One scheduling step of `role`; raises the abort if planned."""
        self.steps[role] = self.steps.get(role, 0) + 1
        if self.abort_at == (role, self.steps[role]):
            self.abort = True

    def sync(self, b, phase, count, threads):
        self.bp[b].arrive(phase, count, threads)
        while not self.bp[b].passed(phase):
            yield

    def p0_count_at(self, j):
        return self.p0_count if j < self.n[0] else P0_IDLE

    # -------------------------------------------------------- roles
    def producer(self):
        S, nmax = self.S, self.nmax
        self.q_full.arrive(tx_bytes=self.TILE)
        self.tma_load(self.q_full, None, "Q")
        for g in range(2 * nmax):
            slot, r = g % S, g // S
            if r > 0:
                # (after an abort the issuing warp's commits may run ahead of
                # this wait; the kernel's producer then stops at its next
                # check of the abort flag, or copies data nothing reads)
                while not self.abort and not self.slot_empty[slot].done(r - 1):
                    self.tick("producer")
                    yield
            if self.abort:
                return
            self.slot_full[slot].arrive(tx_bytes=self.TILE)
            self.tma_load(self.slot_full[slot], slot, g)
            self.tick("producer")
            yield

    def watcher(self):
        S, nmax = self.S, self.nmax
        ok = True
        for j in range(nmax):
            gv, gk = 2 * j + 1, 2 * j + 2
            for g in ([gv, gk] if j + 1 < nmax else [gv]):
                while ok and not self.slot_full[g % S].done(g // S):
                    if self.abort:
                        ok = False
                        break
                    self.tick("watcher")
                    yield
            if not ok and self.watcher_stops_at_abort:
                return
            yield from self.sync(0, j, self.p0_count_at(j), 32)

    def mma_checked(self, reads, tmem):
        """An MMA; after an abort it runs on whatever the buffers hold."""
        if self.abort:
            return
        self.mma(reads, tmem)

    def issuer(self):
        S, nmax = self.S, self.nmax
        n0, n1 = self.n

        def issue_s(sub, g):
            self.mma_checked([(g % S, g)], ("S", sub, g // 2))
            self.commit(self.s_full[sub])

        def issue_pv(sub, g):
            self.mma_checked([(g % S, g)], ("PV", sub, g // 2))
            if g // 2 == self.n[sub] - 1:
                self.commit(self.o_done[sub])

        while not (self.q_full.done(0) and self.slot_full[0].done(0)):
            if self.abort:
                break
            self.tick("issuer")
            yield
        if n0 > 0:
            issue_s(0, 0)
        if n1 > 0:
            issue_s(1, 0)
        for j in range(nmax):
            gv, gk = 2 * j + 1, 2 * j + 2
            nxt = j + 1 < nmax
            yield from self.sync(0, j, self.p0_count_at(j), 32)
            self.tick("issuer")
            if j < n0:
                issue_pv(0, gv)
            if nxt and j + 1 < n0:
                issue_s(0, gk)
            if j < n1:
                yield from self.sync(1, j, P1_COUNT, 32)
                issue_pv(1, gv)
                if nxt and j + 1 < n1:
                    issue_s(1, gk)
            yield
        self.commit(self.drain)
        while not self.drain.done(0):
            yield

    def softmax(self, sub):
        n = self.n[sub]
        b, count = (0, self.p0_count) if sub == 0 else (1, P1_COUNT)
        releaser = n == self.nmax and (sub == 1 or self.n[1] == 0)
        announced = 0
        ok = True
        for j in range(n):
            while not self.s_full[sub].done(j):
                if self.abort:
                    ok = False
                    break
                self.tick(f"softmax{sub}")
                yield
            if not ok:
                break
            if releaser and not self.abort:   # (after an abort the copies have stopped)
                if j > 0:
                    self.release(2 * j - 1)
                self.release(2 * j)
            if not self.abort and self.tmem_s[sub] != ("S", j):
                raise ProtocolError(f"softmax{sub}({j}) reads TMEM holding {self.tmem_s[sub]}")
            self.tick(f"softmax{sub}")
            yield
            if not self.abort:
                self.tmem_s[sub] = ("P", j)
                if j > 0 and self.rng.random() < self.rescale_prob and self.o_tiles[sub] != j - 1:
                    raise ProtocolError(f"rescale at tile {j} sees O holding tile {self.o_tiles[sub]}")
            if self.softmax_only_arrives:
                self.bp[b].arrive(j, count, 128)
            else:
                yield from self.sync(b, j, count, 128)
            announced = j + 1
        if not self.softmax_stops_at_abort:
            for j in range(announced, n):
                yield from self.sync(b, j, count, 128)
        if n > 0 and ok and not self.abort:
            while not self.o_done[sub].done(0):
                if self.abort:
                    return
                yield
            if self.abort:
                return
            if self.o_tiles[sub] != n - 1:
                raise ProtocolError(f"epilogue of sub-tile {sub} sees O holding tile {self.o_tiles[sub]}")

    def finish_one_mma(self):
        if self.abort:
            # results are not used after an abort: retire in order, no checks
            op = self.mma_queue.pop(0)
            for q in self.thread_queues.values():
                if op in q:
                    q.remove(op)
            if op[0] == "commit":
                _, bar, release = op[:3]
                if bar.pending > 0:
                    bar.pending -= 1
                    bar._maybe_complete()
            return
        super().finish_one_mma()

    def issuers(self):
        return {"issuer": self.issuer(), "watcher": self.watcher()}

    def run(self):
        super().run()
        for i, b in enumerate(self.bp):
            if b.arrived:
                raise ProtocolError(f"{b.name}: phase {b.completed} left incomplete")
        want = [self.nmax, self.n[1]]
        for b, w in zip(self.bp, want):
            if b.completed != w:
                raise ProtocolError(f"{b.name}: {b.completed} phases passed, {w} expected")


# (n0, n1) as the kernel produces them: n1 = n0 (no mask), n1 = n0 + 1 or
# n0 (causal), n1 = 0 (second sub-tile past the end, or one sub-tile per
# CTA), n0 = 0 < n1 (a key range only the second sub-tile reaches)
CASES = [(4, 3, 3), (4, 5, 6), (4, 1, 1), (4, 1, 2), (4, 4, 0), (4, 0, 2), (8, 7, 8), (5, 6, 0)]


@pytest.mark.parametrize("stages,n0,n1", CASES)
def test_named_protocol_random_interleavings(stages, n0, n1):
    for seed in range(30):
        NamedSim(stages, n0, n1, seed).run()


@pytest.mark.parametrize("stages,n0,n1", [(4, 3, 4), (4, 5, 0), (8, 2, 2)])
def test_every_role_finishes_after_an_abort_anywhere(stages, n0, n1):
    roles = ["producer", "watcher", "issuer", "softmax0", "softmax1"]
    for seed in range(6):
        for role in roles:
            for step in range(1, 30, 3):
                NamedSim(stages, n0, n1, seed, abort_at=(role, step)).run()


def _fails(cls, cases, abort=True):
    for stages, n0, n1 in cases:
        for seed in range(6):
            for role in (["softmax0", "softmax1", "watcher", "issuer"] if abort else [None]):
                for step in ([1, 2, 4, 7] if abort else [0]):
                    try:
                        cls(stages, n0, n1, seed, abort_at=(role, step) if abort else None).run()
                    except ProtocolError:
                        return True
    return False


def test_model_catches_softmax_that_only_arrives():
    class Arrives(NamedSim):
        softmax_only_arrives = True
    assert _fails(Arrives, [(4, 3, 4)])


def test_model_catches_softmax_that_stops_at_an_abort():
    class Stops(NamedSim):
        softmax_stops_at_abort = True
    assert _fails(Stops, [(4, 3, 4)])


def test_model_catches_watcher_that_stops_at_an_abort():
    class Stops(NamedSim):
        watcher_stops_at_abort = True
    assert _fails(Stops, [(4, 3, 4)])


def test_model_catches_a_count_without_the_watcher():
    class Short(NamedSim):
        p0_count = 128 + 32
    assert _fails(Short, [(4, 3, 3)], abort=False)

