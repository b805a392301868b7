"""Model check of the two-tile backward kernel's barrier protocol (host-only).

The two-tile backward kernel (exact_attention_17_gb300/csrc/fa2_bwd2_sm103.cuh)
streams query tiles of 64 rows past one block of 128 keys and keeps two of
them in flight: TMEM holds S^T and dP^T for two tiles (buffer t % 2), so the
scores of tile t + 1 are computed while tile t's elementwise phases and its
dV, dK and dQ MMAs run.  dQ^T(t) = K^T dS^T(t) lands in tile t's S^T buffer
once dV(t) has read P^T(t) from it.

  issuer, tile t:  wait p_ready(t); dV(t); wait Q/dO(t+1) landed and
                   dq_free(t-1); dP^T(t+1), S^T(t+1); commit s_full;
                   wait ds_ready(t); dK(t); dQ^T(t); commit dq_full
  warpgroup w:     wait s_full; S^T -> P^T; arrive p_ready; release the
                   ring slot of tile t-2 once its dQ reduction has read its
                   staging; wait dq_full(t-1); read dQ^T(t-1); arrive
                   dq_free; stage it in its half of tile t-1's ring slot and
                   start the TMA reduction; dP^T -> dS^T (TMEM and shared
                   memory); arrive ds_ready
  producer:        Q/dO(t) into slot t % STAGES after both warpgroups
                   released the slot's previous tile

This restates that protocol as a discrete-event model (copies and
reductions finish in any order, MMAs in issue order, roles advance in
random order) and fails on: an arrival past a barrier's expected count, an
ambiguous parity wait, a copy into a slot still in use, an MMA reading
operands not (or no longer) in place when it executes, dQ staged over
operands an MMA has yet to read, a TMEM buffer read or overwritten out of
order, the shared dS tile overwritten before dQ^T read it, and a deadlock.
"""
import random

import pytest

from test_pipeline_protocol import MBarrier, ProtocolError


class Bwd2Sim:
    def __init__(self, stages, n, seed, no_dq_free_wait=False, stage_too_early=False, ds_before_readout=False):
        self.rng = random.Random(seed)
        self.S, self.n = stages, n
        self.no_dq_free_wait = no_dq_free_wait    # mutant: S^T(t+1) issued without waiting dq_free(t-1)
        self.stage_too_early = stage_too_early    # mutant: dQ staged in the slot before dq_full
        self.ds_before_readout = ds_before_readout  # mutant: dS(t) written before dQ^T(t-1) is read out
        self.kv_full = MBarrier("kv_full", 1)
        self.q_full = [MBarrier(f"q_full[{i}]", 1) for i in range(stages)]
        self.q_empty = [MBarrier(f"q_empty[{i}]", 2) for i in range(stages)]
        # One s_full barrier serves both buffers: S^T(t+1) is issued only
        # after dq_free(t-1), which the warpgroups arrive on after they have
        # waited for S^T(t), so phase t+1 never completes before phase t is seen.
        self.s_full = MBarrier("s_full", 1)
        self.p_ready = MBarrier("p_ready", 2)
        self.ds_ready = MBarrier("ds_ready", 2)
        self.dq_full = MBarrier("dq_full", 1)
        self.dq_free = MBarrier("dq_free", 2)
        self.drain = MBarrier("mma_drain", 1)
        self.part = [[("free", None), ("free", None)] for _ in range(stages)]   # [slot][0: Q, 1: dO]
        self.tma, self.reduce, self.queue = [], [], []
        # TMEM buffers b = 0, 1; per warpgroup column half w
        self.tS = [[None, None], [None, None]]
        self.tDP = [[None, None], [None, None]]
        self.dS = [None, None]        # the shared dS tile, per warpgroup half

    # ----------------------------------------------------------- engines
    def finish_tma(self):
        bar, slot, t = self.tma.pop(self.rng.randrange(len(self.tma)))
        if slot is not None:
            self.part[slot] = [("ready", t), ("ready", t)]
        bar.complete_tx(1)

    def finish_reduce(self):
        self.reduce.pop(self.rng.randrange(len(self.reduce)))

    def mma(self, reads, effect):
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

    def issue_sp(self, t):
        """dP^T(t) then S^T(t) into buffer t % 2, then the s_full commit."""
        b, slot = t % 2, t % self.S

        def sp(t=t, b=b):
            for w in (0, 1):
                if t >= 2 and self.tDP[b][w] != ("dS-read", t - 2):
                    raise ProtocolError(f"dP^T({t}) overwrites {self.tDP[b][w]}")
                if t >= 2 and self.tS[b][w] != ("dQ-read", t - 2):
                    raise ProtocolError(f"S^T({t}) overwrites {self.tS[b][w]}")
                self.tDP[b][w] = ("dP", t)
                self.tS[b][w] = ("S", t)
        self.mma([(slot, 0, t), (slot, 1, t)], sp)
        self.commit(self.s_full)

    def issuer(self):
        S, n = self.S, self.n
        while not self.kv_full.done(0):
            yield
        while not self.q_full[0].done(0):
            yield
        self.issue_sp(0)
        for t in range(n):
            slot, b = t % S, t % 2
            while not self.p_ready.done(t):
                yield

            def dv(t=t, b=b):
                for w in (0, 1):
                    if self.tS[b][w] != ("P", t):
                        raise ProtocolError(f"dV({t}) reads {self.tS[b][w]}")
                    self.tS[b][w] = ("P-read", t)
            self.mma([(slot, 1, t)], dv)
            if t + 1 < n:
                s1 = (t + 1) % S
                while not self.q_full[s1].done((t + 1) // S):
                    yield
                if t >= 1 and not self.no_dq_free_wait:
                    while not self.dq_free.done(t - 1):
                        yield
                self.issue_sp(t + 1)
            while not self.ds_ready.done(t):
                yield

            def dk(t=t, b=b):
                for w in (0, 1):
                    if self.tDP[b][w] != ("dS", t):
                        raise ProtocolError(f"dK({t}) reads {self.tDP[b][w]}")
                    self.tDP[b][w] = ("dS-read", t)
            self.mma([(slot, 0, t)], dk)

            def dq(t=t, b=b):
                for w in (0, 1):
                    if self.dS[w] != ("dS", t):
                        raise ProtocolError(f"dQ^T({t}) reads the dS tile holding {self.dS[w]}")
                    if self.tS[b][w] != ("P-read", t):
                        raise ProtocolError(f"dQ^T({t}) overwrites {self.tS[b][w]}")
                    self.tS[b][w] = ("dQ", t)
                    self.dS[w] = ("dS-read", t)
            self.mma([], dq)
            self.commit(self.dq_full)
            yield
        self.commit(self.drain)
        while not self.drain.done(0):
            yield

    def readout(self, w, t):
        """Wait for dQ^T(t), read it, free its buffer, stage it in tile t's slot."""
        S, b, slot = self.S, t % 2, t % self.S
        if self.stage_too_early:
            if self.pending_reads(slot, w) or self.part[slot][w] != ("ready", t):
                raise ProtocolError(f"dQ staging {t}/{w} over slot {slot} still read ({self.part[slot][w]})")
        while not self.dq_full.done(t):
            yield
        if self.tS[b][w] != ("dQ", t):
            raise ProtocolError(f"dQ read-out {t}/{w} finds {self.tS[b][w]}")
        self.tS[b][w] = ("dQ-read", t)
        self.dq_free.arrive()
        if self.pending_reads(slot, w) or self.part[slot][w] != ("ready", t):
            raise ProtocolError(f"dQ staging {t}/{w} over slot {slot} still read ({self.part[slot][w]})")
        self.part[slot][w] = ("staged", t)
        self.reduce.append((w, slot, t))

    def warpgroup(self, w):
        S, n = self.S, self.n
        for t in range(n):
            b = t % 2
            while not self.s_full.done(t):
                yield
            if self.tS[b][w] != ("S", t):
                raise ProtocolError(f"P phase {t}/{w} reads {self.tS[b][w]}")
            yield
            self.tS[b][w] = ("P", t)
            self.p_ready.arrive()
            if t >= 2:
                # tile t-2's reduction has had a whole P phase to read its staging
                while any(r[0] == w and r[2] == t - 2 for r in self.reduce):
                    yield
                prev = (t - 2) % S
                self.part[prev][w] = ("free", None)
                self.q_empty[prev].arrive()
            if t >= 1 and not self.ds_before_readout:
                yield from self.readout(w, t - 1)
            if self.tDP[b][w] != ("dP", t):
                raise ProtocolError(f"dS phase {t}/{w} reads {self.tDP[b][w]}")
            if t >= 1 and self.dS[w] != ("dS-read", t - 1):
                raise ProtocolError(f"dS tile of {t}/{w} overwrites {self.dS[w]}")
            yield
            self.tDP[b][w] = ("dS", t)
            self.dS[w] = ("dS", t)
            self.ds_ready.arrive()
            if t >= 1 and self.ds_before_readout:
                yield from self.readout(w, t - 1)
        if n >= 1:
            yield from self.readout(w, n - 1)
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


def test_model_catches_ds_written_before_the_previous_dq_is_read():
    """The shared dS tile holds dS(t-1) until dQ^T(t-1) has executed: the
    warpgroups may overwrite it only after they have seen dq_full(t-1)."""
    assert _fails(ds_before_readout=True)


def test_model_catches_scores_over_an_unread_dq():
    """S^T(t+1) overwrites buffer (t+1) % 2, which holds dQ^T(t-1) until the
    warpgroups have read it out."""
    assert _fails(no_dq_free_wait=True)


def test_model_catches_dq_staged_before_the_tile_completes():
    """Staging dQ in the tile's ring slot before dq_full writes over Q or dO
    while dK or dV may still read them."""
    assert _fails(stage_too_early=True)
