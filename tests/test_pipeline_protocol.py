"""Model check of the tensor-core kernel's barrier protocol (host-only).

The forward kernel coordinates a TMA producer, one MMA-issuing thread and two
softmax warpgroups through mbarriers.  TMEM state is tracked too: S of a
sub-tile must not be overwritten before the P V product has read the P that
the softmax wrote over it, and the softmax's rescale of O and the epilogue
must see exactly the tiles accumulated so far.  This test restates that protocol in a
small discrete-event model and runs it under many random interleavings
(TMA copies finish in any order, MMAs finish in issue order, roles advance
in random order).  It fails on:

* an arrival on an mbarrier phase that has already received all of its
  expected arrivals (undefined on the hardware);
* a parity wait issued while the barrier is two or more phases past the
  phase the waiter means (the parity would be ambiguous);
* a TMA copy into a ring slot whose previous contents were not released;
* an MMA reading a slot that does not hold the load it expects;
* a TMEM hazard on S/P or on the O accumulator (see above);
* a deadlock.

The model mirrors the producer, issuer and softmax loops of the kernel in
exact_attention_17_gb300/csrc/fa2_fwd_sm103.cuh where the issuing thread
polls mbarriers: the single-buffered two-slot ring (Sim) and the
double-buffered order of head dimension 256 (DoubleSSim).  With a ring of
four or more slots the issuing warp waits on named barriers instead; that
form is modelled in test_named_barrier_protocol.py on top of this one.  A
change to the kernel's protocol must be made in the models too.
"""
import random

import pytest


class ProtocolError(AssertionError):
    pass


class MBarrier:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.completed = 0          # completed phases
        self.pending = count        # arrivals still expected in the current phase
        self.tx = 0                 # outstanding transaction bytes

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.completed += 1
            self.pending = self.count

    def arrive(self, tx_bytes=0):
        if self.pending == 0:
            raise ProtocolError(f"{self.name}: arrival beyond the expected count")
        self.pending -= 1
        self.tx += tx_bytes
        self._maybe_complete()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._maybe_complete()

    def done(self, phase):
        """Has phase number `phase` completed?  Checks the parity hazard: a
        parity wait cannot tell phase p from phase p - 2 or p + 2, so the
        barrier must be within one phase of the waiter's, on either side."""
        if self.completed > phase + 1:
            raise ProtocolError(f"{self.name}: waiter for phase {phase} sees {self.completed} "
                                "completed phases (parity aliasing)")
        if self.completed < phase:
            raise ProtocolError(f"{self.name}: waiter for phase {phase} sees only {self.completed} "
                                "completed phases (its parity wait would pass at once)")
        return self.completed == phase + 1


class Sim:
    def __init__(self, stages, n0, n1, seed, rescale_prob=0.3):
        self.rng = random.Random(seed)
        self.S, self.NG = stages, stages // 2
        self.n = (n0, n1)
        self.nmax = max(n0, n1)
        self.rescale_prob = rescale_prob
        TILE = 1
        self.TILE = TILE
        self.q_full = MBarrier("q_full", 1)
        self.slot_full = [MBarrier(f"slot_full[{i}]", 1) for i in range(stages)]
        self.group_full = [MBarrier(f"group_full[{i}]", 1) for i in range(self.NG)]
        self.slot_empty = [MBarrier(f"slot_empty[{i}]", 1) for i in range(stages)]
        self.s_full = [MBarrier(f"s_full[{i}]", 1) for i in range(2)]
        self.p_ready = [MBarrier(f"p_ready[{i}]", 1) for i in range(2)]
        self.o_done = [MBarrier(f"o_done[{i}]", 1) for i in range(2)]
        self.drain = MBarrier("mma_drain", 1)
        self.slot = [None] * stages           # ("loading"|"ready"|"free", load id)
        for i in range(stages):
            self.slot[i] = ("free", None)
        self.tma_inflight = []                # (barrier, slot or None, load id, bytes)
        self.mma_queue = []                   # ops in issue order: ("mma", reads) | ("commit", bar)
        self.released = set()
        self.tmem_s = [None, None]            # S/P columns of each sub-tile
        self.o_tiles = [-1, -1]               # last tile whose P V is in O
        self.thread_queues = {}               # issuing thread -> its ops in order
        self.current = None                   # issuing thread of the next mma/commit

    # -------------------------------------------------------- async engines
    def tma_load(self, bar, slot, g):
        if slot is not None:
            state, _ = self.slot[slot]
            if state != "free":
                raise ProtocolError(f"TMA load {g} into slot {slot} still in use ({self.slot[slot]})")
            self.slot[slot] = ("loading", g)
        self.tma_inflight.append((bar, slot, g, self.TILE))

    def finish_one_tma(self):
        bar, slot, g, nb = self.tma_inflight.pop(self.rng.randrange(len(self.tma_inflight)))
        if slot is not None:
            self.slot[slot] = ("ready", g)
        bar.complete_tx(nb)

    def mma(self, reads, tmem=None):
        """Queue an MMA reading ring slots; `tmem` = ("S", sub, j) writes S_sub of
        tile j, ("PV", sub, j) reads P_sub of tile j (checked when it executes)."""
        for slot, g in reads:
            if self.slot[slot] != ("ready", g):
                raise ProtocolError(f"MMA expects load {g} in slot {slot}, finds {self.slot[slot]}")
        op = ("mma", reads, tmem, len(self.mma_queue), self.rng.random())
        self.mma_queue.append(op)
        self.thread_queues.setdefault(self.current, []).append(op)

    def commit(self, bar, release=None):
        op = ("commit", bar, release, len(self.mma_queue), self.rng.random())
        self.mma_queue.append(op)
        self.thread_queues.setdefault(self.current, []).append(op)

    def finish_one_mma(self):
        # MMAs of one issuing thread run in order; the tensor pipe interleaves
        # the threads' streams arbitrarily (per-thread queues, random choice).
        queues = [q for q in self.thread_queues.values() if q]
        if queues:
            q = self.rng.choice(queues)
            op = q.pop(0)
            self.mma_queue.remove(op)
        else:
            op = self.mma_queue.pop(0)
        if op[0] == "mma":
            # the operands must still be in place when the MMA executes
            for slot, g in op[1]:
                if self.slot[slot] != ("ready", g):
                    raise ProtocolError(f"MMA reading load {g} executes while slot {slot} holds {self.slot[slot]}")
        if op[0] == "mma" and op[2] is not None:
            kind, sub, j = op[2]
            buf = self.s_buf(sub, j)
            state = self.tmem_s[buf]
            if kind == "S":
                # S_sub(j) overwrites the P last written into its buffer: the
                # PV that reads that P must have run
                prev = j - self.s_reuse
                if prev >= 0 and state != ("P-read", prev):
                    raise ProtocolError(f"S{sub}({j}) executes while TMEM holds {state}")
                self.tmem_s[buf] = ("S", j)
            else:
                if state != ("P", j):
                    raise ProtocolError(f"PV{sub}({j}) executes while TMEM holds {state}")
                if self.o_tiles[sub] != j - 1:
                    raise ProtocolError(f"PV{sub}({j}) accumulates onto O holding tile {self.o_tiles[sub]}")
                self.tmem_s[buf] = ("P-read", j)
                self.o_tiles[sub] = j
        if op[0] == "commit":
            _, bar, release = op[:3]
            if release is not None:
                slot, g = release
                if self.slot[slot] != ("ready", g):
                    raise ProtocolError(f"release of load {g}: slot {slot} holds {self.slot[slot]}")
                self.slot[slot] = ("free", None)
            bar.arrive()

    # The epilogue's wait for every MMA before it stages O in the ring (off
    # only in the test that checks the model rejects its absence).
    epilogue_waits_drain = True

    # Ring slots released by a softmax thread of the sub-tile that visits
    # every key tile, on seeing S of tile j complete (K_j and V_(j-1) have
    # no reader left), instead of by MMA commits; rings of four or more slots.
    @property
    def softmax_release(self):
        return self.S >= 4

    def release(self, g):
        slot = g % self.S
        if self.slot[slot] != ("ready", g):
            raise ProtocolError(f"release of load {g}: slot {slot} holds {self.slot[slot]}")
        self.slot[slot] = ("free", None)
        self.slot_empty[slot].arrive()

    # O of a sub-tile is announced (o_done) only after its last P V.
    out_done_last = True
    # With O announced after every P V: the softmax waits for P(j-1) V at the
    # last tile (off only in the test that checks the model rejects that).
    last_tile_wait = True

    def o_done_phase(self, n):
        """Phase of o_done that announces the last P V of an n-tile sub-tile."""
        return 0 if self.out_done_last else n - 1

    # S buffer of sub-tile `sub` at key tile j, and the tiles between two
    # uses of one buffer: one buffer per sub-tile here.
    s_reuse = 1

    def s_buf(self, sub, j):
        return sub

    # -------------------------------------------------------- roles
    def producer(self):
        """One full barrier per ring slot; load g (K_j for g = 2j, V_j for
        g = 2j + 1) waits for the release of load g - STAGES in its slot."""
        S, nmax = self.S, self.nmax
        self.q_full.arrive(tx_bytes=self.TILE)
        self.tma_load(self.q_full, None, "Q")
        for g in range(2 * nmax):
            slot, r = g % S, g // S
            if r > 0:
                while not self.slot_empty[slot].done(r - 1):
                    yield
            self.slot_full[slot].arrive(tx_bytes=self.TILE)
            self.tma_load(self.slot_full[slot], slot, g)
            yield

    def issuer(self):
        S, NG, nmax = self.S, self.NG, self.nmax
        n0, n1 = self.n

        def issue_s(sub, g):
            self.mma([(g % S, g)], ("S", sub, g // 2))
            self.commit(self.s_full[sub])

        def issue_pv(sub, g):
            self.mma([(g % S, g)], ("PV", sub, g // 2))
            if not self.out_done_last or g // 2 == self.n[sub] - 1:
                self.commit(self.o_done[sub])

        while not self.q_full.done(0):
            yield
        while not self.slot_full[0].done(0):
            yield
        if n0 > 0:
            issue_s(0, 0)
        if n1 > 0:
            issue_s(1, 0)
        if not self.softmax_release:
            self.commit(self.slot_empty[0], release=(0, 0))
        for j in range(nmax):
            gv, gk = 2 * j + 1, 2 * j + 2
            nxt = j + 1 < nmax
            # one combined wait for V_j, P_0(j) and (ring of four or more
            # slots) K_(j+1); with fewer slots K_(j+1) is waited for after PV_0(j)
            early_k = S >= 4
            while not (self.slot_full[gv % S].done(gv // S)
                       and (j >= n0 or self.p_ready[0].done(j))
                       and (not (early_k and nxt) or self.slot_full[gk % S].done(gk // S))):
                yield
            if j < n0:
                issue_pv(0, gv)
            if not early_k and nxt:
                while not self.slot_full[gk % S].done(gk // S):
                    yield
            if nxt and j + 1 < n0:
                issue_s(0, gk)
            if j < n1:
                while not self.p_ready[1].done(j):
                    yield
                issue_pv(1, gv)
            if not self.softmax_release:
                self.commit(self.slot_empty[gv % S], release=(gv % S, gv))
            if nxt:
                if j + 1 < n1:
                    issue_s(1, gk)
                if not self.softmax_release:
                    self.commit(self.slot_empty[gk % S], release=(gk % S, gk))
            yield
        self.commit(self.drain)
        while not self.drain.done(0):
            yield

    def s_barrier(self, sub, j):
        """(barrier, phase) announcing S_sub(j)."""
        return self.s_full[sub], j

    def p_barrier(self, sub, j):
        """(barrier, phase) announcing P_sub(j)."""
        return self.p_ready[sub], j

    def softmax(self, sub):
        n = self.n[sub]
        releaser = n == self.nmax and (sub == 1 or self.n[1] == 0)
        for j in range(n):
            bar, ph = self.s_barrier(sub, j)
            while not bar.done(ph):
                yield
            if self.softmax_release and releaser:
                if j > 0:
                    self.release(2 * j - 1)
                self.release(2 * j)
            buf = self.s_buf(sub, j)
            if self.tmem_s[buf] != ("S", j):
                raise ProtocolError(f"softmax{sub}({j}) reads TMEM holding {self.tmem_s[buf]}")
            yield
            self.tmem_s[buf] = ("P", j)
            rescale = j > 0 and self.rng.random() < self.rescale_prob
            # (with O announced only at the end, the wait for S(j) above
            # must already order the rescale after P(j-1) V; with O announced
            # after every P V the wait for P(j-1) V is also taken at the last
            # tile, so that the epilogue's parity wait is not two phases ahead)
            if not self.out_done_last and j > 0 and (rescale or (j == n - 1 and self.last_tile_wait)):
                while not self.o_done[sub].done(j - 1):
                    yield
            if rescale:
                # the rescale reads and writes O: it must hold tiles 0..j-1 exactly
                if self.o_tiles[sub] != j - 1:
                    raise ProtocolError(f"rescale at tile {j} sees O holding tile {self.o_tiles[sub]}")
            self.p_barrier(sub, j)[0].arrive()
        if n > 0:
            while not self.o_done[sub].done(self.o_done_phase(n)):
                yield
            if self.o_tiles[sub] != n - 1:
                raise ProtocolError(f"epilogue of sub-tile {sub} sees O holding tile {self.o_tiles[sub]}")
            if n == self.nmax:
                # the second epilogue round of a last-finishing sub-tile is
                # staged in ring slot `sub` once every MMA has completed: no
                # copy may still be writing the ring, no MMA still reading it
                while self.epilogue_waits_drain and not self.drain.done(0):
                    yield
                if any(slot is not None for _, slot, _, _ in self.tma_inflight):
                    raise ProtocolError("epilogue stages O in the ring while a K/V copy is in flight")
                if any(op[0] == "mma" and op[1] for op in self.mma_queue):
                    raise ProtocolError("epilogue stages O in the ring while an MMA may read it")

    # -------------------------------------------------------- scheduler
    def issuers(self):
        return {"issuer": self.issuer()}

    def run(self):
        roles = {"producer": self.producer(), "softmax0": self.softmax(0),
                 "softmax1": self.softmax(1)}
        roles.update(self.issuers())
        steps = 0
        while roles or self.tma_inflight or self.mma_queue:
            steps += 1
            if steps > 200000:
                raise ProtocolError("no progress (deadlock)")
            choices = list(roles) + (["tma"] if self.tma_inflight else []) + \
                (["mma"] if self.mma_queue else [])
            c = self.rng.choice(choices)
            if c == "tma":
                self.finish_one_tma()
            elif c == "mma":
                self.finish_one_mma()
            else:
                self.current = c
                try:
                    next(roles[c])
                except StopIteration:
                    del roles[c]
        # every load released exactly once, nothing left in flight
        for i, st in enumerate(self.slot):
            if st[0] == "loading":
                raise ProtocolError(f"slot {i} still loading at exit")


class DoubleSSim(Sim):
    """One sub-tile with two S buffers in TMEM (head dimension 256): S(j+1)
    is issued as soon as K(j+1) has landed, before P(j) V; S(j) and P(j) are
    announced on s_full[j % 2] and p_ready[j % 2]."""
    s_reuse = 2
    softmax_release = False
    out_done_last = False

    def __init__(self, stages, n0, seed, single_p_ready=False, **kw):
        super().__init__(stages, n0, 0, seed, **kw)
        self.single_p_ready = single_p_ready

    def s_buf(self, sub, j):
        return j % 2

    def s_barrier(self, sub, j):
        return self.s_full[j % 2], j // 2

    def p_barrier(self, sub, j):
        if self.single_p_ready:
            return self.p_ready[0], j
        return self.p_ready[j % 2], j // 2

    def issuer(self):
        S = self.S
        n0 = self.n[0]
        while not self.q_full.done(0):
            yield
        while not self.slot_full[0].done(0):
            yield
        if n0 > 0:
            self.mma([(0, 0)], ("S", 0, 0))
            self.commit(self.s_full[0])
        self.commit(self.slot_empty[0], release=(0, 0))
        for j in range(n0):
            gv, gk = 2 * j + 1, 2 * j + 2
            if j + 1 < n0:
                while not self.slot_full[gk % S].done(gk // S):
                    yield
                self.mma([(gk % S, gk)], ("S", 0, j + 1))
                self.commit(self.s_full[(j + 1) % 2])
                self.commit(self.slot_empty[gk % S], release=(gk % S, gk))
            bar, ph = self.p_barrier(0, j)
            while not (self.slot_full[gv % S].done(gv // S) and bar.done(ph)):
                yield
            self.mma([(gv % S, gv)], ("PV", 0, j))
            self.commit(self.o_done[0])
            self.commit(self.slot_empty[gv % S], release=(gv % S, gv))
            yield
        self.commit(self.drain)
        while not self.drain.done(0):
            yield


@pytest.mark.parametrize("n0", list(range(1, 9)) + [17])
def test_double_s_protocol_random_interleavings(n0):
    for seed in range(60):
        DoubleSSim(2, n0, seed).run()


def test_model_catches_epilogue_wait_two_phases_ahead():
    """With S double-buffered and O announced after every P V, the softmax can
    finish the last tile before P(n-2) V has completed; the epilogue's parity
    wait for P(n-1) V would then pass at once.  The wait for P(n-2) V at the
    last tile prevents it; the model must reject its absence."""

    class NoLastWait(DoubleSSim):
        last_tile_wait = False
    failures = 0
    for seed in range(100):
        try:
            NoLastWait(2, 3, seed, rescale_prob=0.0).run()
        except ProtocolError:
            failures += 1
    assert failures > 0


def test_model_catches_single_p_ready_with_double_s():
    """With S double-buffered, the softmax can finish tile j + 1 before the
    issuer has looked at P(j): a single p_ready barrier would then be two
    phases ahead of the issuer's parity wait."""
    failures = 0
    for seed in range(300):
        try:
            DoubleSSim(2, 6, seed, single_p_ready=True, rescale_prob=0.0).run()
        except ProtocolError:
            failures += 1
    assert failures > 0


def test_model_catches_ring_staging_without_drain():
    """Staging O in a ring slot as soon as the sub-tile's own last P V is done
    (without waiting for every MMA) races the other sub-tile's MMAs and the
    last copies; the model must see it."""
    class NoDrain(Sim):
        epilogue_waits_drain = False

    failures = 0
    for seed in range(200):
        try:
            NoDrain(4, 5, 5, seed).run()
        except ProtocolError:
            failures += 1
    assert failures > 0


def test_model_catches_release_by_the_wrong_sub_tile():
    """Under the causal mask the first sub-tile sees S_0(j) complete before
    P_1(j-1) V has read V_(j-1): the slots must be released by the sub-tile
    that visits every key tile, not by the first one."""
    class WrongReleaser(Sim):
        def softmax(self, sub):
            n = self.n[sub]
            for j in range(n):
                bar, ph = self.s_barrier(sub, j)
                while not bar.done(ph):
                    yield
                if sub == 0:
                    if j > 0:
                        self.release(2 * j - 1)
                    self.release(2 * j)
                if self.tmem_s[sub] != ("S", j):
                    raise ProtocolError(f"softmax{sub}({j}) reads TMEM holding {self.tmem_s[sub]}")
                yield
                self.tmem_s[sub] = ("P", j)
                self.p_ready[sub].arrive()
            if n > 0:
                while not self.o_done[sub].done(self.o_done_phase(n)):
                    yield

    failures = 0
    for seed in range(300):
        try:
            WrongReleaser(4, 5, 6, seed).run()
        except ProtocolError:
            failures += 1
    assert failures > 0


def test_model_catches_rescale_before_pv_when_s_comes_first():
    """Without per-tile o_done the rescale relies on S(j) being issued after
    P(j-1) V; in the double-buffered order (S(j+1) ahead of P(j) V) that does
    not hold, and the model must see the rescale racing P V."""
    class DoubleNoDone(DoubleSSim):
        out_done_last = True

        def issuer(self):
            S = self.S
            n0 = self.n[0]
            while not (self.q_full.done(0) and self.slot_full[0].done(0)):
                yield
            self.mma([(0, 0)], ("S", 0, 0))
            self.commit(self.s_full[0])
            self.commit(self.slot_empty[0], release=(0, 0))
            for j in range(n0):
                gv, gk = 2 * j + 1, 2 * j + 2
                if j + 1 < n0:
                    while not self.slot_full[gk % S].done(gk // S):
                        yield
                    self.mma([(gk % S, gk)], ("S", 0, j + 1))
                    self.commit(self.s_full[(j + 1) % 2])
                    self.commit(self.slot_empty[gk % S], release=(gk % S, gk))
                bar, ph = self.p_barrier(0, j)
                while not (self.slot_full[gv % S].done(gv // S) and bar.done(ph)):
                    yield
                self.mma([(gv % S, gv)], ("PV", 0, j))
                if j == n0 - 1:
                    self.commit(self.o_done[0])
                self.commit(self.slot_empty[gv % S], release=(gv % S, gv))
                yield
            self.commit(self.drain)
            while not self.drain.done(0):
                yield

    failures = 0
    for seed in range(300):
        try:
            DoubleNoDone(2, 6, seed, rescale_prob=0.5).run()
        except ProtocolError:
            failures += 1
    assert failures > 0


CASES = []
for stages in (2, 4, 5, 8):
    for nmax in list(range(1, 11)) + [17]:
        CASES.append((stages, nmax, nmax))          # non-causal: both sub-tiles, same range
        CASES.append((stages, nmax - 1, nmax) if nmax > 1 else (stages, 1, 1))  # causal pair
        CASES.append((stages, nmax, 0))             # second sub-tile past the end
    CASES.append((stages, 0, 1))   # causal key range that only the second sub-tile reaches


@pytest.mark.parametrize("stages,n0,n1", CASES)
def test_protocol_random_interleavings(stages, n0, n1):
    for seed in range(40):
        Sim(stages, n0, n1, seed).run()


def test_model_catches_early_rearm():
    """A grouped variant of the protocol (V_(t-1) and K_t landing on one
    barrier, STAGES/2 barriers reused in turn) whose producer only waited for
    its own slots re-armed a barrier before its previous phase had been
    consumed when the last group held only V.  That ordering faulted the GPU;
    the model must reject it."""

    class GroupedSim(Sim):
        softmax_release = False
        out_done_last = False

        def producer(self):
            S, NG, nmax = self.S, self.NG, self.nmax
            self.q_full.arrive(tx_bytes=self.TILE)
            self.tma_load(self.q_full, None, "Q")
            for t in range(nmax + 1):
                g_first = 0 if t == 0 else 2 * t - 1
                g_last = 2 * t if t < nmax else 2 * t - 1
                for g in range(g_first, g_last + 1):
                    r = g // S
                    if r > 0:
                        while not self.slot_empty[g % S].done(r - 1):
                            yield
                full = self.group_full[t % NG]
                full.arrive(tx_bytes=(g_last - g_first + 1) * self.TILE)
                for g in range(g_first, g_last + 1):
                    self.tma_load(full, g % S, g)
                yield

        def issuer(self):
            S, NG, nmax = self.S, self.NG, self.nmax
            n0, n1 = self.n
            while not self.q_full.done(0):
                yield
            while not self.group_full[0].done(0):
                yield
            for sub in (0, 1):
                if self.n[sub] > 0:
                    self.mma([(0, 0)])
                    self.commit(self.s_full[sub])
            self.commit(self.slot_empty[0], release=(0, 0))
            for j in range(nmax):
                t = j + 1
                gv, gk = 2 * j + 1, 2 * j + 2
                nxt = j + 1 < nmax
                while not self.group_full[t % NG].done(t // NG):
                    yield
                for sub in (0, 1):
                    if j < self.n[sub]:
                        while not self.p_ready[sub].done(j):
                            yield
                        self.mma([(gv % S, gv)])
                        self.commit(self.o_done[sub])
                    if nxt and j + 1 < self.n[sub]:
                        self.mma([(gk % S, gk)])
                        self.commit(self.s_full[sub])
                self.commit(self.slot_empty[gv % S], release=(gv % S, gv))
                if nxt:
                    self.commit(self.slot_empty[gk % S], release=(gk % S, gk))
                yield
            self.commit(self.drain)
            while not self.drain.done(0):
                yield

    failures = 0
    for seed in range(200):
        try:
            GroupedSim(4, 1, 2, seed).run()
        except ProtocolError:
            failures += 1
    assert failures > 0


def test_model_catches_commits_from_another_lane_than_the_mmas():
    """tcgen05.commit makes its mbarrier track only the tensor-core operations
    issued by the thread that executes it.  The kernel issues every MMA and
    every commit from one thread (lane 0 of the MMA warp).  A variant that
    picks the issuing lane afresh for each group of MMAs and for each commit
    (the PTX description of elect.sync does not promise which active lane it
    elects) can issue a commit from a lane that issued none of the MMAs it
    is meant to cover: its arrival then does not wait for them, and the
    softmax or the epilogue reads TMEM before the MMA has written it --
    wrong values, with no fault and no timed-out wait.  The model must
    reject that variant."""
    class LaneSwitching(Sim):
        def mma(self, reads, tmem=None):
            self.current = ("issuer", self.rng.randrange(2))
            super().mma(reads, tmem)

        def commit(self, bar, release=None):
            self.current = ("issuer", self.rng.randrange(2))
            super().commit(bar, release)

    failures = 0
    for seed in range(200):
        try:
            LaneSwitching(4, 5, 5, seed).run()
        except ProtocolError:
            failures += 1
    assert failures > 0


def test_one_issuing_lane_passes_the_same_interleavings():
    """The same seeds with every MMA and commit from one lane are clean."""
    class OneLane(Sim):
        def mma(self, reads, tmem=None):
            self.current = ("issuer", 0)
            super().mma(reads, tmem)

        def commit(self, bar, release=None):
            self.current = ("issuer", 0)
            super().commit(bar, release)

    for seed in range(200):
        OneLane(4, 5, 5, seed).run()
