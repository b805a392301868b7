"""Model check of the two-tile backward kernel's barrier protocol (host-only).

The two-tile backward kernel (exact_attention_17_gb300/csrc/fa2_bwd2_sm103.cuh)
streams query tiles of 64 rows past one block of 128 keys and keeps two of
them in flight: TMEM holds S^T and dP^T for two tiles (buffer t % 2), and
the two elementwise warpgroups take the tiles in turn (warpgroup g owns the
tiles t with t % 2 == g, buffer g, its own barriers and its own dS tile in
shared memory), so one warpgroup's phases overlap the other's and the
tensor core runs the scores of one tile while the other tile's dV, dK and
dQ MMAs wait for their operands.  dQ^T(t) = K^T dS^T(t) lands in tile t's
S^T buffer once dV(t) has read P^T(t) from it.

  issuer, tile t:  wait p_ready[t%2]; dV(t); wait Q/dO(t+1) landed and
                   dq_free[(t+1)%2] (the read-out of tile t-1); dP^T(t+1),
                   S^T(t+1); commit s_full[(t+1)%2]; wait ds_ready[t%2];
                   dK(t); dQ^T(t); commit dq_full[t%2]
  warpgroup g, its tile t:  wait s_full[g]; S^T -> P^T; arrive p_ready[g];
                   release the ring slot of its previous tile t-2 once that
                   tile's dQ reduction has read its staging; dP^T -> dS^T
                   (TMEM and its dS tile); arrive ds_ready[g]; wait
                   dq_full[g]; read dQ^T(t); arrive dq_free[g]; stage it in
                   tile t's ring slot and start the TMA reduction; after its
                   last tile, wait for the drain commit before reading dK
                   and dV
  producer:        Q/dO(t) into slot t % STAGES after the owning warpgroup
                   released the slot's previous tile

This restates that protocol as a discrete-event model (copies and
reductions finish in any order, MMAs in issue order, roles advance in
random order) and fails on: an arrival past a barrier's expected count, an
ambiguous parity wait, a copy into a slot still in use, an MMA reading
operands not (or no longer) in place when it executes, dQ staged over
operands an MMA has yet to read, a TMEM buffer read or overwritten out of
order, a dS tile overwritten before dQ^T read it, dK and dV read out while
an MMA may still accumulate into them, and a deadlock.
"""
import random

import pytest

from test_pipeline_protocol import MBarrier, ProtocolError


class Bwd2Sim:
    def __init__(self, stages, n, seed, no_dq_free_wait=False, stage_too_early=False, shared_ds=False,
                 no_drain_wait=False):
        self.rng = random.Random(seed)
        self.S, self.n = stages, n
        self.no_dq_free_wait = no_dq_free_wait    # mutant: S^T(t+1) issued without waiting dq_free
        self.stage_too_early = stage_too_early    # mutant: dQ staged in the slot before dq_full
        self.shared_ds = shared_ds                # mutant: one dS tile for both warpgroups
        self.no_drain_wait = no_drain_wait        # mutant: dK/dV read out without waiting for the drain
        self.kv_full = MBarrier("kv_full", 1)
        self.q_full = [MBarrier(f"q_full[{i}]", 1) for i in range(stages)]
        self.q_empty = [MBarrier(f"q_empty[{i}]", 1) for i in range(stages)]
        self.s_full = [MBarrier(f"s_full[{g}]", 1) for g in range(2)]
        self.p_ready = [MBarrier(f"p_ready[{g}]", 1) for g in range(2)]
        self.ds_ready = [MBarrier(f"ds_ready[{g}]", 1) for g in range(2)]
        self.dq_full = [MBarrier(f"dq_full[{g}]", 1) for g in range(2)]
        self.dq_free = [MBarrier(f"dq_free[{g}]", 1) for g in range(2)]
        self.drain = MBarrier("mma_drain", 1)
        self.part = [("free", None) for _ in range(stages)]   # ring slot: Q and dO of a tile, or its dQ staging
        self.tma, self.reduce, self.queue = [], [], []
        self.tS = [None, None]        # TMEM S^T buffer b (P^T, then dQ^T)
        self.tDP = [None, None]       # TMEM dP^T buffer b (then dS^T)
        self.dS = [None, None]        # dS tile of warpgroup g in shared memory

    def ds_tile(self, g):
        return 0 if self.shared_ds else g

    # ----------------------------------------------------------- engines
    def finish_tma(self):
        bar, slot, t = self.tma.pop(self.rng.randrange(len(self.tma)))
        if slot is not None:
            self.part[slot] = ("ready", t)
        bar.complete_tx(1)

    def finish_reduce(self):
        self.reduce.pop(self.rng.randrange(len(self.reduce)))

    def mma(self, reads, effect):
        for slot, t in reads:
            if self.part[slot] != ("ready", t):
                raise ProtocolError(f"MMA issued for tile {t} finds slot {slot} holding {self.part[slot]}")
        self.queue.append(("mma", reads, effect))

    def commit(self, bar):
        self.queue.append(("commit", bar))

    def finish_mma(self):
        op = self.queue.pop(0)
        if op[0] == "commit":
            op[1].arrive()
            return
        for slot, t in op[1]:
            if self.part[slot] != ("ready", t):
                raise ProtocolError(f"MMA for tile {t} executes while slot {slot} holds {self.part[slot]}")
        op[2]()

    def pending_reads(self, slot):
        return any(op[0] == "mma" and any(s == slot for s, _ in op[1]) for op in self.queue)

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
            if self.part[slot] != ("free", None):
                raise ProtocolError(f"copy of tile {t} into slot {slot} still in use ({self.part[slot]})")
            if any(r[0] == slot for r in self.reduce):
                raise ProtocolError(f"copy of tile {t} into slot {slot} while a dQ reduction reads it")
            self.part[slot] = ("loading", t)
            self.q_full[slot].arrive(tx_bytes=1)
            self.tma.append((self.q_full[slot], slot, t))
            yield

    def issue_sp(self, t):
        """dP^T(t) then S^T(t) into buffer t % 2, then the s_full commit."""
        b, slot = t % 2, t % self.S

        def sp(t=t, b=b):
            if t >= 2 and self.tDP[b] != ("dS-read", t - 2):
                raise ProtocolError(f"dP^T({t}) overwrites {self.tDP[b]}")
            if t >= 2 and self.tS[b] != ("dQ-read", t - 2):
                raise ProtocolError(f"S^T({t}) overwrites {self.tS[b]}")
            self.tDP[b] = ("dP", t)
            self.tS[b] = ("S", t)
        self.mma([(slot, t)], sp)
        self.commit(self.s_full[b])

    def issuer(self):
        S, n = self.S, self.n
        while not self.kv_full.done(0):
            yield
        while not self.q_full[0].done(0):
            yield
        self.issue_sp(0)
        for t in range(n):
            slot, b = t % S, t % 2
            while not self.p_ready[b].done(t // 2):
                yield

            def dv(t=t, b=b):
                if self.tS[b] != ("P", t):
                    raise ProtocolError(f"dV({t}) reads {self.tS[b]}")
                self.tS[b] = ("P-read", t)
            self.mma([(slot, t)], dv)
            if t + 1 < n:
                s1, b1 = (t + 1) % S, (t + 1) % 2
                while not self.q_full[s1].done((t + 1) // S):
                    yield
                if t >= 1 and not self.no_dq_free_wait:
                    while not self.dq_free[b1].done((t - 1) // 2):
                        yield
                self.issue_sp(t + 1)
            while not self.ds_ready[b].done(t // 2):
                yield

            def dk(t=t, b=b):
                if self.tDP[b] != ("dS", t):
                    raise ProtocolError(f"dK({t}) reads {self.tDP[b]}")
                self.tDP[b] = ("dS-read", t)
            self.mma([(slot, t)], dk)

            def dq(t=t, b=b):
                d = self.ds_tile(b)
                if self.dS[d] != ("dS", t):
                    raise ProtocolError(f"dQ^T({t}) reads a dS tile holding {self.dS[d]}")
                if self.tS[b] != ("P-read", t):
                    raise ProtocolError(f"dQ^T({t}) overwrites {self.tS[b]}")
                self.tS[b] = ("dQ", t)
                self.dS[d] = ("dS-read", t)
            self.mma([], dq)
            self.commit(self.dq_full[b])
            yield
        self.commit(self.drain)
        while not self.drain.done(0):
            yield

    def warpgroup(self, g):
        S, n = self.S, self.n
        for t in range(g, n, 2):
            k, slot = t // 2, t % S
            while not self.s_full[g].done(k):
                yield
            if self.tS[g] != ("S", t):
                raise ProtocolError(f"P phase {t} reads {self.tS[g]}")
            yield
            self.tS[g] = ("P", t)
            self.p_ready[g].arrive()
            if t >= 2:
                # its previous tile's reduction has had a whole P phase to read the staging
                while any(r[1] == t - 2 for r in self.reduce):
                    yield
                prev = (t - 2) % S
                self.part[prev] = ("free", None)
                self.q_empty[prev].arrive()
            if self.tDP[g] != ("dP", t):
                raise ProtocolError(f"dS phase {t} reads {self.tDP[g]}")
            d = self.ds_tile(g)
            if self.dS[d] is not None and self.dS[d][0] == "dS":
                raise ProtocolError(f"dS tile of {t} overwrites {self.dS[d]} before dQ^T read it")
            yield
            self.tDP[g] = ("dS", t)
            self.dS[d] = ("dS", t)
            self.ds_ready[g].arrive()
            if self.stage_too_early:
                if self.pending_reads(slot) or self.part[slot] != ("ready", t):
                    raise ProtocolError(f"dQ staging {t} over slot {slot} still read ({self.part[slot]})")
            while not self.dq_full[g].done(k):
                yield
            if self.tS[g] != ("dQ", t):
                raise ProtocolError(f"dQ read-out {t} finds {self.tS[g]}")
            self.tS[g] = ("dQ-read", t)
            self.dq_free[g].arrive()
            if self.pending_reads(slot) or self.part[slot] != ("ready", t):
                raise ProtocolError(f"dQ staging {t} over slot {slot} still read ({self.part[slot]})")
            self.part[slot] = ("staged", t)
            self.reduce.append((slot, t))
            yield
        while any(r[1] % 2 == g for r in self.reduce):
            yield
        # dK and dV are read out of TMEM once every MMA has completed: the
        # warpgroup that does not own the last tile gets there first
        if n > 0:
            while not self.no_drain_wait and not self.drain.done(0):
                yield
            if any(op[0] == "mma" for op in self.queue):
                raise ProtocolError(f"warpgroup {g} reads dK/dV while an MMA may still accumulate into them")

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


@pytest.mark.parametrize("stages", [3, 4])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8, 13])
def test_two_tile_backward_protocol_random_interleavings(stages, n):
    for seed in range(30):
        Bwd2Sim(stages, n, seed).run()


def _fails(**kw):
    for seed in range(200):
        try:
            Bwd2Sim(4, 7, seed, **kw).run()
        except ProtocolError:
            return True
    return False


def test_model_catches_one_ds_tile_for_both_warpgroups():
    """The warpgroups' dS phases overlap: with one dS tile in shared memory,
    one warpgroup would overwrite the other's dS before dQ^T has read it."""
    assert _fails(shared_ds=True)


def test_model_catches_scores_over_an_unread_dq():
    """S^T(t+1) overwrites buffer (t+1) % 2, which holds dQ^T(t-1) until its
    warpgroup has read it out."""
    assert _fails(no_dq_free_wait=True)


def test_model_catches_dq_staged_before_the_tile_completes():
    """Staging dQ in the tile's ring slot before dq_full writes over Q or dO
    while dK or dV may still read them."""
    assert _fails(stage_too_early=True)


def test_model_catches_dk_dv_read_before_the_last_mma():
    """The warpgroup that does not own the last tile finishes its own tiles
    first: reading dK and dV then, without the drain commit, can read them
    before the last tile's dV and dK MMAs have completed."""
    assert _fails(no_drain_wait=True)
