"""Model check of the two-SM forward kernel's barrier protocol (host-only).

The two-SM variant of the forward kernel runs a cluster of two CTAs (the
leader, rank 0, and its peer, rank 1).  Each CTA holds its own query rows
and one half of every K and V tile in its own shared-memory ring; one
thread of the leader issues every tensor-core MMA for both SMs
(tcgen05.mma.cta_group::2 reads A and B from both CTAs' shared memory and
writes each CTA's rows into that CTA's TMEM) and every commit, which arrives
on the barrier of that name in both CTAs (multicast).  The peer's loads
complete on the peer's own barriers; a forwarding thread of the peer waits
for each and then arrives on the leader's barrier of the same slot, so that
the leader's issuer sees a slot full only when both halves have landed.
Each softmax warpgroup arrives on the leader's p_ready barrier (the peer's
remotely).  Each CTA's ring slots are released by its own softmax thread of
the sub-tile that visits every key tile, on seeing that sub-tile's S
complete.

This test restates that protocol as a discrete-event model and runs it
under many random interleavings (copies finish in any order, MMAs in issue
order, roles advance in random order).  It fails on an arrival beyond a
phase's expected count, a parity wait that could alias, a copy into a slot
still in use, an MMA reading a slot (in either CTA) that does not hold the
load it expects, a TMEM hazard on S/P or O in either CTA, a CTA that exits
while a signal to it may still be in flight, or a deadlock.  The model
mirrors exact_attention_17_gb300/csrc/fa2_fwd_pair_sm103.cuh.
"""
import random

import pytest

from test_pipeline_protocol import MBarrier, ProtocolError

LEADER, PEER = 0, 1


class PairSim:
    def __init__(self, stages, n0, n1, seed, rescale_prob=0.3, forward_before_landing=False,
                 unicast_commits=False, peer_skips_drain=False):
        self.rng = random.Random(seed)
        self.S = stages
        self.n = (n0, n1)
        self.nmax = max(n0, n1)
        self.rescale_prob = rescale_prob
        self.forward_before_landing = forward_before_landing
        self.unicast_commits = unicast_commits
        self.peer_skips_drain = peer_skips_drain
        mk = MBarrier
        self.q_full = [mk("q_full[L]", 2), mk("q_full[P]", 1)]
        self.kv_full = [[mk(f"kv_full[{r}][{i}]", 2 if r == LEADER else 1) for i in range(stages)]
                        for r in (LEADER, PEER)]
        self.kv_empty = [[mk(f"kv_empty[{r}][{i}]", 1) for i in range(stages)] for r in (LEADER, PEER)]
        self.s_full = [[mk(f"s_full[{r}][{i}]", 1) for i in range(2)] for r in (LEADER, PEER)]
        self.o_done = [[mk(f"o_done[{r}][{i}]", 1) for i in range(2)] for r in (LEADER, PEER)]
        self.drain = [mk("drain[L]", 1), mk("drain[P]", 1)]
        self.p_ready = [mk(f"p_ready[L][{i}]", 2) for i in range(2)]   # both CTAs' warpgroups
        self.slot = [[("free", None)] * stages for _ in (LEADER, PEER)]
        self.q_loaded = [False, False]
        self.tma_inflight = []        # (cta, barrier, slot or None, load id)
        self.mma_queue = []           # issue order
        self.deliveries = []          # multicast arrivals in flight: (cta, barrier)
        self.tmem_s = [[None, None], [None, None]]
        self.o_tiles = [[-1, -1], [-1, -1]]
        self.exited = [False, False]
        self.teardown_arrived = [False, False]

    # -------------------------------------------------------- async engines
    def tma_load(self, cta, bar, slot, g):
        if slot is not None:
            if self.slot[cta][slot][0] != "free":
                raise ProtocolError(f"CTA {cta}: load {g} into slot {slot} still in use {self.slot[cta][slot]}")
            self.slot[cta][slot] = ("loading", g)
        self.tma_inflight.append((cta, bar, slot, g))

    def finish_one_tma(self):
        cta, bar, slot, g = self.tma_inflight.pop(self.rng.randrange(len(self.tma_inflight)))
        if self.exited[cta]:
            raise ProtocolError(f"a copy lands in CTA {cta} after it exited")
        if slot is None:
            self.q_loaded[cta] = True
        else:
            self.slot[cta][slot] = ("ready", g)
        bar.complete_tx(1)

    def signal(self, cta, bar):
        if self.exited[cta]:
            raise ProtocolError(f"{bar.name}: signal to CTA {cta} after it exited")
        bar.arrive()

    def mma(self, slot, g, tmem):
        for cta in (LEADER, PEER):
            if slot is not None and self.slot[cta][slot] != ("ready", g):
                raise ProtocolError(f"MMA expects load {g} in CTA {cta} slot {slot}, finds {self.slot[cta][slot]}")
            if not self.q_loaded[cta]:
                raise ProtocolError(f"MMA issued before CTA {cta}'s Q landed")
        self.mma_queue.append(("mma", slot, g, tmem))

    def commit(self, bars):
        """bars: one barrier per CTA (multicast) or only the leader's (unicast variant)."""
        if self.unicast_commits:
            bars = bars[:1]
        self.mma_queue.append(("commit", bars))

    def finish_one_mma(self):
        op = self.mma_queue.pop(0)
        if op[0] == "mma":
            _, slot, g, (kind, sub, j) = op
            for cta in (LEADER, PEER):
                if slot is not None and self.slot[cta][slot] != ("ready", g):
                    raise ProtocolError(f"MMA reading load {g} runs while CTA {cta} slot {slot} holds "
                                        f"{self.slot[cta][slot]}")
                state = self.tmem_s[cta][sub]
                if kind == "S":
                    if j > 0 and state != ("P-read", j - 1):
                        raise ProtocolError(f"S{sub}({j}) runs while CTA {cta} TMEM holds {state}")
                    self.tmem_s[cta][sub] = ("S", j)
                else:
                    if state != ("P", j):
                        raise ProtocolError(f"PV{sub}({j}) runs while CTA {cta} TMEM holds {state}")
                    if self.o_tiles[cta][sub] != j - 1:
                        raise ProtocolError(f"PV{sub}({j}) accumulates onto CTA {cta} O holding "
                                            f"{self.o_tiles[cta][sub]}")
                    self.tmem_s[cta][sub] = ("P-read", j)
                    self.o_tiles[cta][sub] = j
        else:
            # a multicast commit's arrivals reach the two CTAs independently
            for cta, bar in enumerate(op[1]):
                self.deliveries.append((cta, bar))

    def deliver_one(self):
        cta, bar = self.deliveries.pop(self.rng.randrange(len(self.deliveries)))
        self.signal(cta, bar)

    # -------------------------------------------------------- roles
    def producer(self, cta):
        """Q and the K/V halves of this CTA into its own ring.  The leader's
        full barriers expect two arrivals (its own, with the bytes, and the
        peer's forwarded one); the peer's expect one."""
        S = self.S
        self.q_full[cta].arrive(tx_bytes=1)
        self.tma_load(cta, self.q_full[cta], None, "Q")
        for g in range(2 * self.nmax):
            slot, lap = g % S, g // S
            if lap > 0:
                while not self.kv_empty[cta][slot].done(lap - 1):
                    yield
            self.kv_full[cta][slot].arrive(tx_bytes=1)
            self.tma_load(cta, self.kv_full[cta][slot], slot, g)
            yield
        # before the CTA may exit, its own copies must have landed
        while any(c == cta for c, _, _, _ in self.tma_inflight):
            yield

    def forwarder(self):
        """Peer: once a copy of the peer has landed, arrive on the leader's
        barrier of the same slot (or Q)."""
        if not self.forward_before_landing:
            while not self.q_full[PEER].done(0):
                yield
        self.signal(LEADER, self.q_full[LEADER])
        for g in range(2 * self.nmax):
            slot, lap = g % self.S, g // self.S
            while not self.forward_before_landing and not self.kv_full[PEER][slot].done(lap):
                yield
            self.signal(LEADER, self.kv_full[LEADER][slot])
            yield
        # the leader's last commit (drain) must have reached the peer before it exits
        while not self.peer_skips_drain and self.nmax > 0 and not self.drain[PEER].done(0):
            yield

    def issuer(self):
        S, nmax = self.S, self.nmax
        n0, n1 = self.n
        kvf = self.kv_full[LEADER]
        if nmax == 0:
            return
        while not (self.q_full[LEADER].done(0) and kvf[0].done(0)):
            yield
        if n0 > 0:
            self.mma(0, 0, ("S", 0, 0))
            self.commit([self.s_full[LEADER][0], self.s_full[PEER][0]])
        if n1 > 0:
            self.mma(0, 0, ("S", 1, 0))
            self.commit([self.s_full[LEADER][1], self.s_full[PEER][1]])
        for j in range(nmax):
            gv, gk = 2 * j + 1, 2 * j + 2
            nxt = j + 1 < nmax
            while not (kvf[gv % S].done(gv // S)
                       and (j >= n0 or self.p_ready[0].done(j))
                       and (not nxt or kvf[gk % S].done(gk // S))):
                yield
            if j < n0:
                self.mma(gv % S, gv, ("PV", 0, j))
                if j + 1 == n0:
                    self.commit([self.o_done[LEADER][0], self.o_done[PEER][0]])
            if nxt and j + 1 < n0:
                self.mma(gk % S, gk, ("S", 0, j + 1))
                self.commit([self.s_full[LEADER][0], self.s_full[PEER][0]])
            if j < n1:
                while not self.p_ready[1].done(j):
                    yield
                self.mma(gv % S, gv, ("PV", 1, j))
                if j + 1 == n1:
                    self.commit([self.o_done[LEADER][1], self.o_done[PEER][1]])
            if nxt and j + 1 < n1:
                self.mma(gk % S, gk, ("S", 1, j + 1))
                self.commit([self.s_full[LEADER][1], self.s_full[PEER][1]])
            yield
        self.commit([self.drain[LEADER], self.drain[PEER]])
        while not self.drain[LEADER].done(0):
            yield

    def release(self, cta, g):
        slot = g % self.S
        if self.slot[cta][slot] != ("ready", g):
            raise ProtocolError(f"CTA {cta}: release of load {g}: slot {slot} holds {self.slot[cta][slot]}")
        self.slot[cta][slot] = ("free", None)
        self.kv_empty[cta][slot].arrive()

    def softmax(self, cta, sub):
        n = self.n[sub]
        releaser = n == self.nmax and (sub == 1 or self.n[1] == 0)
        for j in range(n):
            while not self.s_full[cta][sub].done(j):
                yield
            if releaser:
                if j > 0:
                    self.release(cta, 2 * j - 1)
                self.release(cta, 2 * j)
            if self.tmem_s[cta][sub] != ("S", j):
                raise ProtocolError(f"CTA {cta} softmax{sub}({j}) reads TMEM holding {self.tmem_s[cta][sub]}")
            yield
            self.tmem_s[cta][sub] = ("P", j)
            if j > 0 and self.rng.random() < self.rescale_prob:
                # the wait for S(j) must already order the rescale after P(j-1) V
                if self.o_tiles[cta][sub] != j - 1:
                    raise ProtocolError(f"CTA {cta} rescale at tile {j} sees O holding {self.o_tiles[cta][sub]}")
            self.signal(LEADER, self.p_ready[sub])
        if n > 0:
            while not self.o_done[cta][sub].done(0):
                yield
            if self.o_tiles[cta][sub] != n - 1:
                raise ProtocolError(f"CTA {cta} epilogue of sub-tile {sub} sees O holding {self.o_tiles[cta][sub]}")
            if n == self.nmax:
                # second epilogue round staged in ring slots once every MMA has completed
                while not self.drain[cta].done(0):
                    yield
                if any(c == cta and slot is not None for c, _, slot, _ in self.tma_inflight):
                    raise ProtocolError(f"CTA {cta} stages O in the ring while a copy is in flight")
                if any(op[0] == "mma" for op in self.mma_queue):
                    raise ProtocolError(f"CTA {cta} stages O in the ring while an MMA may read it")

    # -------------------------------------------------------- scheduler
    def run(self):
        roles = {("producer", LEADER): self.producer(LEADER), ("producer", PEER): self.producer(PEER),
                 ("forwarder", PEER): self.forwarder(), ("issuer", LEADER): self.issuer()}
        for cta in (LEADER, PEER):
            for sub in (0, 1):
                roles[("softmax", cta, sub)] = self.softmax(cta, sub)
        alive = {LEADER: set(k for k in roles if k[1] == LEADER), PEER: set(k for k in roles if k[1] == PEER)}
        steps = 0
        while roles or self.tma_inflight or self.mma_queue or self.deliveries:
            steps += 1
            if steps > 300000:
                raise ProtocolError("no progress (deadlock)")
            choices = list(roles) + (["tma"] if self.tma_inflight else []) + \
                (["mma"] if self.mma_queue else []) + (["arrival"] if self.deliveries else [])
            c = self.rng.choice(choices)
            if c == "tma":
                self.finish_one_tma()
            elif c == "mma":
                self.finish_one_mma()
            elif c == "arrival":
                self.deliver_one()
            else:
                try:
                    next(roles[c])
                except StopIteration:
                    del roles[c]
                    alive[c[1]].discard(c)
                    # teardown: a CTA exits once both CTAs' roles have all
                    # finished (the cluster-wide barrier before TMEM is freed)
                    if not alive[LEADER] and not alive[PEER]:
                        self.exited = [True, True]
        for cta in (LEADER, PEER):
            for i, st in enumerate(self.slot[cta]):
                if st[0] == "loading":
                    raise ProtocolError(f"CTA {cta} slot {i} still loading at exit")


CASES = []
for stages in (4, 8):
    for nmax in (1, 2, 3, 4, 5, 7, 13):
        CASES.append((stages, nmax, nmax))                            # non-causal
        CASES.append((stages, max(nmax - 2, 1), nmax))                 # causal: sub-tile 0 stops two tiles earlier
        CASES.append((stages, nmax, 0))                                # second pair sub-tile past the end
    CASES.append((stages, 0, 2))                                       # only the second sub-tile has rows


@pytest.mark.parametrize("stages,n0,n1", CASES)
def test_pair_protocol_random_interleavings(stages, n0, n1):
    for seed in range(10):
        PairSim(stages, n0, n1, seed).run()


def _fails(**kw):
    """Does some interleaving of the variant fail a check?"""
    for seed in range(60):
        try:
            PairSim(8, 4, 6, seed, **kw).run()
        except ProtocolError:
            return True
    return False


def test_model_catches_forwarding_before_the_peer_half_landed():
    """An arrival on the leader's barrier before the peer's half is in its
    shared memory lets the MMA read a slot still loading."""
    assert _fails(forward_before_landing=True)


def test_model_catches_commits_to_the_leader_only():
    """S, O and the drain must be announced in both CTAs: with commits
    arriving only on the leader's barriers the peer's softmax never sees its
    S and the pair deadlocks."""
    assert _fails(unicast_commits=True)


def test_model_catches_peer_exit_before_the_last_commit():
    """The peer must see the drain commit before the pair's teardown: if it
    does not wait for it, its roles can all finish while the multicast
    arrival is still in flight."""
    class NoEpilogueDrain(PairSim):
        def softmax(self, cta, sub):
            # epilogue without the ring staging (so no drain wait there)
            n = self.n[sub]
            releaser = n == self.nmax and (sub == 1 or self.n[1] == 0)
            for j in range(n):
                while not self.s_full[cta][sub].done(j):
                    yield
                if releaser:
                    if j > 0:
                        self.release(cta, 2 * j - 1)
                    self.release(cta, 2 * j)
                yield
                self.tmem_s[cta][sub] = ("P", j)
                self.signal(LEADER, self.p_ready[sub])
            if n > 0:
                while not self.o_done[cta][sub].done(0):
                    yield

    failures = 0
    for seed in range(300):
        try:
            NoEpilogueDrain(8, 1, 1, seed, peer_skips_drain=True).run()
        except ProtocolError:
            failures += 1
    assert failures > 0
