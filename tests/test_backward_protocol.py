"""Model check of the backward kernel's barrier protocol (host-only).

The backward kernel (exact_attention_17_gb300/csrc/fa2_bwd_sm103.cuh) keeps
one key block's K and V in shared memory and streams the query tiles' Q and
dO through a ring.  A TMA producer, one MMA-issuing thread and two
elementwise warpgroups (each owning half of a tile's query columns)
coordinate through mbarriers:

  issuer, tile t:  wait Q/dO(t) landed; dP^T(t); wait dq_free(t-1); S^T(t);
                   commit s_full; wait p_ready; dV(t); wait ds_ready; dK(t);
                   dQ(t); commit dq_full
  warpgroup w:     wait s_full; read S^T, write P^T; arrive p_ready; release
                   the ring slot of tile t-1 once its dQ reduction has read
                   its staging; read dP^T, write dS^T (TMEM and shared
                   memory); arrive ds_ready; wait dq_full; read dQ; arrive
                   dq_free; stage dQ in its half of tile t's ring slot and
                   start the TMA reduction from it
  producer:        Q/dO(t) into slot t % STAGES after both warpgroups
                   released the slot's previous tile

TMEM holds S^T (then P^T, then the dQ partial) and dP^T (then dS^T) in
column halves per warpgroup.  This restates that protocol in a small
discrete-event model (copies and reductions finish in any order, MMAs in
issue order, roles advance in random order) and fails on: an arrival past
a barrier's expected count, an ambiguous parity wait, a copy into a slot
whose previous contents are still in use, an MMA reading operands that are
not (or no longer) in place when it executes, dQ staged over operands an
MMA has yet to read, a TMEM read or overwrite out of order, and a deadlock.
"""
import random

import pytest

from test_pipeline_protocol import MBarrier, ProtocolError


class BwdSim:
    def __init__(self, stages, n, seed, release_before_read=False, early_stage=False):
        self.rng = random.Random(seed)
        self.S, self.n = stages, n
        self.release_before_read = release_before_read   # mutant: slot released before the reduction read it
        self.early_stage = early_stage                   # mutant: dQ staged before dq_full
        self.kv_full = MBarrier("kv_full", 1)
        self.q_full = [MBarrier(f"q_full[{i}]", 1) for i in range(stages)]
        self.q_empty = [MBarrier(f"q_empty[{i}]", 2) for i in range(stages)]
        self.s_full = MBarrier("s_full", 1)
        self.p_ready = MBarrier("p_ready", 2)
        self.ds_ready = MBarrier("ds_ready", 2)
        self.dq_full = MBarrier("dq_full", 1)
        self.dq_free = MBarrier("dq_free", 2)
        self.drain = MBarrier("mma_drain", 1)
        # ring slot halves: [slot][w] (w = 0: the Q tile, w = 1: the dO tile)
        self.part = [[("free", None), ("free", None)] for _ in range(stages)]
        self.kv = "loading"
        self.tma = []          # (barrier, slot or None, tile)
        self.reduce = []       # (w, slot, tile): TMA reductions still reading their staging
        self.queue = []        # MMAs and commits in issue order
        self.tS = [None, None]     # TMEM S^T columns, per warpgroup half
        self.tDP = [None, None]    # TMEM dP^T columns, per warpgroup half
        self.dS = [None, None]     # dS staged in shared memory, per half

    # ----------------------------------------------------------- engines
    def finish_tma(self):
        bar, slot, t = self.tma.pop(self.rng.randrange(len(self.tma)))
        if slot is None:
            self.kv = "ready"
        else:
            self.part[slot] = [("ready", t), ("ready", t)]
        bar.complete_tx(1)

    def finish_reduce(self):
        self.reduce.pop(self.rng.randrange(len(self.reduce)))

    def mma(self, reads, effect):
        """reads: (slot, w, t) ring halves; effect(): TMEM / staging checks at execution."""
        for slot, w, t in reads:
            if self.part[slot][w] != ("ready", t):
                raise ProtocolError(f"MMA issued for tile {t} finds slot {slot}/{w} holding {self.part[slot][w]}")
        self.queue.append(("mma", reads, effect))

    def commit(self, bar):
        self.queue.append(("commit", bar))

    def finish_mma(self):
        op = self.queue.pop(0)
        if op[0] == "commit":
            op[1].arrive()
            return
        for slot, w, t in op[1]:
            if self.part[slot][w] != ("ready", t):
                raise ProtocolError(f"MMA for tile {t} executes while slot {slot}/{w} holds {self.part[slot][w]}")
        op[2]()

    def pending_reads(self, slot, w):
        return any(op[0] == "mma" and any(s == slot and ww == w for s, ww, _ in op[1]) for op in self.queue)

    # ----------------------------------------------------------- roles
    def producer(self):
        S = self.S
        self.kv_full.arrive(tx_bytes=1)
        self.tma.append((self.kv_full, None, -1))
        for t in range(self.n):
            slot, lap = t % S, t // S
            if lap > 0:
                while not self.q_empty[slot].done(lap - 1):
                    yield
            if self.part[slot] != [("free", None), ("free", None)]:
                raise ProtocolError(f"copy of tile {t} into slot {slot} still in use ({self.part[slot]})")
            if any(r[1] == slot for r in self.reduce):
                raise ProtocolError(f"copy of tile {t} into slot {slot} while a dQ reduction reads it")
            self.part[slot] = [("loading", t), ("loading", t)]
            self.q_full[slot].arrive(tx_bytes=1)
            self.tma.append((self.q_full[slot], slot, t))
            yield

    def issuer(self):
        S = self.S
        while not self.kv_full.done(0):
            yield
        for t in range(self.n):
            slot = t % S
            while not self.q_full[slot].done(t // S):
                yield

            def dp(t=t):
                for w in (0, 1):
                    if t > 0 and self.tDP[w] != ("dS-read", t - 1):
                        raise ProtocolError(f"dP^T({t}) overwrites {self.tDP[w]}")
                    self.tDP[w] = ("dP", t)
            self.mma([(slot, 1, t)], dp)
            if t > 0:
                while not self.dq_free.done(t - 1):
                    yield

            def s(t=t):
                for w in (0, 1):
                    if t > 0 and self.tS[w] != ("dQ-read", t - 1):
                        raise ProtocolError(f"S^T({t}) overwrites {self.tS[w]}")
                    self.tS[w] = ("S", t)
            self.mma([(slot, 0, t)], s)
            self.commit(self.s_full)
            while not self.p_ready.done(t):
                yield

            def dv(t=t):
                for w in (0, 1):
                    if self.tS[w] != ("P", t):
                        raise ProtocolError(f"dV({t}) reads {self.tS[w]}")
                    self.tS[w] = ("P-read", t)
            self.mma([(slot, 1, t)], dv)
            while not self.ds_ready.done(t):
                yield

            def dk(t=t):
                for w in (0, 1):
                    if self.tDP[w] != ("dS", t):
                        raise ProtocolError(f"dK({t}) reads {self.tDP[w]}")
                    self.tDP[w] = ("dS-read", t)
            self.mma([(slot, 0, t)], dk)

            def dq(t=t):
                for w in (0, 1):
                    if self.dS[w] != ("dS", t):
                        raise ProtocolError(f"dQ({t}) reads staged dS {self.dS[w]}")
                    if self.tS[w] != ("P-read", t):
                        raise ProtocolError(f"dQ({t}) overwrites {self.tS[w]}")
                    self.tS[w] = ("dQ", t)
                    self.dS[w] = ("dS-read", t)
            self.mma([], dq)
            self.commit(self.dq_full)
            yield
        self.commit(self.drain)
        while not self.drain.done(0):
            yield

    def warpgroup(self, w):
        S = self.S
        for t in range(self.n):
            slot = t % S
            while not self.s_full.done(t):
                yield
            if self.tS[w] != ("S", t):
                raise ProtocolError(f"P phase {t}/{w} reads {self.tS[w]}")
            yield
            self.tS[w] = ("P", t)
            self.p_ready.arrive()
            if t > 0:
                prev = (t - 1) % S
                if not self.release_before_read:
                    while any(r[0] == w for r in self.reduce):
                        yield
                self.part[prev][w] = ("free", None)
                self.q_empty[prev].arrive()
            # dP^T(t) was issued before S^T(t): complete once s_full(t) is
            if self.tDP[w] != ("dP", t):
                raise ProtocolError(f"dS phase {t}/{w} reads {self.tDP[w]}")
            # the previous tile's dQ MMA must have read the staged dS
            if t > 0 and self.dS[w] != ("dS-read", t - 1):
                raise ProtocolError(f"dS staging of tile {t}/{w} overwrites {self.dS[w]}")
            yield
            self.tDP[w] = ("dS", t)
            self.dS[w] = ("dS", t)
            self.ds_ready.arrive()
            if not self.early_stage:
                while not self.dq_full.done(t):
                    yield
                if self.tS[w] != ("dQ", t):
                    raise ProtocolError(f"dQ read-out {t}/{w} finds {self.tS[w]}")
                self.tS[w] = ("dQ-read", t)
                self.dq_free.arrive()
            # stage dQ in this warpgroup's half of the tile's slot
            if self.pending_reads(slot, w) or self.part[slot][w] != ("ready", t):
                raise ProtocolError(f"dQ staging {t}/{w} over slot {slot} still read ({self.part[slot][w]})")
            self.part[slot][w] = ("staged", t)
            self.reduce.append((w, slot, t))
            if self.early_stage:
                while not self.dq_full.done(t):
                    yield
                self.tS[w] = ("dQ-read", t)
                self.dq_free.arrive()
            yield
        while any(r[0] == w for r in self.reduce):
            yield

    def run(self):
        roles = {"producer": self.producer(), "issuer": self.issuer(),
                 "wg0": self.warpgroup(0), "wg1": self.warpgroup(1)}
        steps = 0
        while roles or self.tma or self.queue or self.reduce:
            steps += 1
            if steps > 300000:
                raise ProtocolError("no progress (deadlock)")
            choices = list(roles) + (["tma"] if self.tma else []) + (["mma"] if self.queue else []) + \
                (["reduce"] if self.reduce else [])
            c = self.rng.choice(choices)
            if c == "tma":
                self.finish_tma()
            elif c == "mma":
                self.finish_mma()
            elif c == "reduce":
                self.finish_reduce()
            else:
                try:
                    next(roles[c])
                except StopIteration:
                    del roles[c]


@pytest.mark.parametrize("stages", [2, 4])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 9, 16])
def test_backward_protocol_random_interleavings(stages, n):
    for seed in range(40):
        BwdSim(stages, n, seed).run()


def test_model_catches_slot_release_before_the_reduction_read():
    """Releasing a ring slot before the dQ reduction has read the staging in
    it lets the producer copy the next Q/dO tile over data still in use."""
    failures = 0
    for seed in range(300):
        try:
            BwdSim(2, 6, seed, release_before_read=True).run()
        except ProtocolError:
            failures += 1
    assert failures > 0


def test_model_catches_staging_before_dq_full():
    """Staging dQ in the ring slot before dq_full (the completion of every
    MMA of the tile) writes over Q or dO while dK or dV may still read them."""
    failures = 0
    for seed in range(300):
        try:
            BwdSim(2, 6, seed, early_stage=True).run()
        except ProtocolError:
            failures += 1
    assert failures > 0
