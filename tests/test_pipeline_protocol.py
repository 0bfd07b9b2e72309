"""Race detection for the barrier protocol of the tensor-core prefill's tile
pipeline (CPU, a model of the protocol, not of the arithmetic).

Every role of one CTA (Q/K producer, the two Q.K^T issuers, the deciders, the
exponential warps, the V producer, the P.V issuer) is written out as the
sequence of mbarrier arrivals and parity waits it performs per traversed block,
following the kernel's protocol.  A random scheduler interleaves the roles with
the asynchronous events: tensor-core products complete in issue order (one
pipe per SM) and fire the commits issued after them; TMA loads complete in any
order.  Each parity wait is checked against the phase it means: passing before
that phase has completed, or blocking after it completed (the parity then
points two phases ahead), is reported, and so are deadlocks and reads of a
buffer that no longer holds the block read.

mbarrier parity semantics used: after n completed phases a wait on parity p
succeeds iff n % 2 != p (right after init, parity 1 counts as completed).
"""
import random

import pytest


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.arrived, self.tx, self.n = name, count, 0, 0, 0

    def _check(self):
        if self.arrived == self.count and self.tx == 0:
            self.n += 1
            self.arrived = 0

    def arrive(self, tx=0):
        self.arrived += 1
        self.tx += tx
        self._check()

    def complete_tx(self, tx):
        self.tx -= tx
        self._check()


class ProtocolError(AssertionError):
    pass


def simulate(nblk, keep, rescale, seed, NK=4, NV=2, NS=3, NDEC=4, pv_slots=None):
    """Run one CTA's protocol once; raises ProtocolError on any violation.

    Block c is issued after one wait, on slot c % NK of the "ready" ring (two
    arrivals: the key producer's, with the tile's bytes, and the S buffer's
    release by block c - NS: its decision if skipped, its P.V commit if kept;
    the first NS slots get the release at set-up).  Slot c % NK of "qk_done"
    is block c's Q.K^T commit: the deciders' scores and the key stage's
    release in one."""
    rng = random.Random(seed)
    pv_slots = NS if pv_slots is None else pv_slots
    B = {}

    def bar(name, count=1):
        B[name] = Bar(name, count)

    bar("q_full")
    for i in range(NK):
        bar(("ready", i), 2), bar(("qk_done", i))
    for i in range(NS):
        B[("ready", i % NK)].arrive()  # S buffers free at set-up
    for i in range(NV):
        bar(("v_full", i)), bar(("v_empty", i))
    for i in range(NS):
        bar(("p_full", i))
    for i in range(pv_slots):
        bar(("pv_done", i))
    for i in range(NDEC):
        bar(("dec_full", i)), bar(("dec_read", i), 3)  # V producer, P.V issuer, exponential warps
    bar("l_full")

    def free_bar(b):  # the slot that block b's S buffer release goes to: block b + NS's
        return ("ready", (b + NS) % NK)

    kstage = [None] * NK    # block whose keys a K stage holds (None: loading / empty)
    vstage = [None] * NV
    sbuf = [None] * NS      # block whose scores / P an S buffer holds
    dec = [None] * NDEC
    pv_done_count = [0]
    pipe = []               # in-order tensor pipe: completion callbacks of issued products
    tma = []                # TMA loads in flight: their landing callbacks

    def wait(name, phase):
        b = B[name]
        ok = (b.n % 2) != (phase % 2)
        if ok and b.n <= phase:
            raise ProtocolError(f"{name}: wait for phase {phase} passed after {b.n} phases")
        if not ok and b.n > phase:
            raise ProtocolError(f"{name}: phase {phase} completed but the parity wait blocks "
                                f"({b.n} phases)")
        return ok

    def expect(cond, msg):
        if not cond:
            raise ProtocolError(msg)

    # -- roles as generators: yield ("wait", name, phase) or None (a step) ----------
    def kprod():
        B["q_full"].arrive(tx=1)
        tma.append(lambda: B["q_full"].complete_tx(1))
        yield None
        for c in range(nblk):
            s = c % NK
            if c >= NK:
                yield ("wait", ("qk_done", s), c // NK - 1)
            kstage[s] = None
            B[("ready", s)].arrive(tx=1)

            def land(s=s, c=c):
                kstage[s] = c
                B[("ready", s)].complete_tx(1)
            tma.append(land)
            yield None

    def qk(par):
        yield ("wait", "q_full", 0)
        for c in range(par, nblk, 2):
            s, sb = c % NK, c % NS
            yield ("wait", ("ready", s), c // NK)
            expect(kstage[s] == c, f"Q.K^T of block {c} reads K stage {s} holding {kstage[s]}")
            expect(sbuf[sb] is None, f"Q.K^T of block {c} overwrites S buffer {sb} "
                                     f"still holding block {sbuf[sb]}")
            sbuf[sb] = ("writing", c)

            def done(c=c, s=s, sb=sb):
                sbuf[sb] = c
                B[("qk_done", s)].arrive()
            pipe.append(done)
            yield None

    def deciders():
        for c in range(nblk):
            sb = c % NS
            yield ("wait", ("qk_done", c % NK), c // NK)
            expect(sbuf[sb] == c, f"deciders read S buffer {sb} for block {c}: {sbuf[sb]}")
            k = keep[c]
            if not k:
                sbuf[sb] = None
                B[free_bar(c)].arrive()
            if c >= NDEC:
                yield ("wait", ("dec_read", c % NDEC), c // NDEC - 1)
            dec[c % NDEC] = (c, k)
            B[("dec_full", c % NDEC)].arrive()
            yield None

    def read_dec(c):
        d = dec[c % NDEC]
        expect(d is not None and d[0] == c, f"decision slot {c % NDEC} holds {d}, not block {c}")
        B[("dec_read", c % NDEC)].arrive()
        return d[1]

    def exps():
        kc = 0
        for c in range(nblk):
            yield ("wait", ("dec_full", c % NDEC), c // NDEC)
            if not read_dec(c):
                continue
            sb = c % NS
            expect(sbuf[sb] == c, f"exponential warps read S buffer {sb} for block {c}: {sbuf[sb]}")
            if rescale[c] and kc >= 1:
                yield ("wait", ("pv_done", (kc - 1) % pv_slots), (kc - 1) // pv_slots)
                expect(pv_done_count[0] >= kc, f"O rescaled before P.V {kc - 1} completed")
            B[("p_full", kc % NS)].arrive()
            kc += 1
            yield None
        if kc:
            yield ("wait", ("pv_done", (kc - 1) % pv_slots), (kc - 1) // pv_slots)
            expect(pv_done_count[0] == kc, f"epilogue reads O with {pv_done_count[0]} of {kc} "
                                           f"P.V products complete")
        B["l_full"].arrive()

    def vprod():
        vi = 0
        for c in range(nblk):
            yield ("wait", ("dec_full", c % NDEC), c // NDEC)
            if not read_dec(c):
                continue
            s = vi % NV
            if vi >= NV:
                yield ("wait", ("v_empty", s), vi // NV - 1)
            vstage[s] = None
            B[("v_full", s)].arrive(tx=1)

            def land(s=s, c=c):
                vstage[s] = c
                B[("v_full", s)].complete_tx(1)
            tma.append(land)
            vi += 1
            yield None

    def pv():
        kc = vi = 0
        for c in range(nblk):
            yield ("wait", ("dec_full", c % NDEC), c // NDEC)
            if not read_dec(c):
                continue
            vs = vi % NV
            yield ("wait", ("p_full", kc % NS), kc // NS)
            yield ("wait", ("v_full", vs), vi // NV)
            expect(sbuf[c % NS] == c, f"P.V of block {c} reads P from S buffer {c % NS}: "
                                      f"{sbuf[c % NS]}")
            expect(vstage[vs] == c, f"P.V of block {c} reads V stage {vs} holding {vstage[vs]}")

            def done(c=c, vs=vs, kc=kc):
                B[("v_empty", vs)].arrive()
                sbuf[c % NS] = None
                B[free_bar(c)].arrive()
                pv_done_count[0] += 1
                B[("pv_done", kc % pv_slots)].arrive()
            pipe.append(done)
            kc += 1
            vi += 1
            yield None

    roles = {"K": kprod(), "QK0": qk(0), "QK1": qk(1), "D": deciders(), "E": exps(),
             "V": vprod(), "PV": pv()}
    pending = {name: None for name in roles}  # a wait the role is blocked on
    live = set(roles)
    while live or pipe or tma:
        runnable = []
        for name in live:
            w = pending[name]
            if w is None or wait(w[1], w[2]):
                runnable.append(name)
        events = (["pipe"] if pipe else []) + (["tma"] if tma else [])
        choices = runnable + events
        if not choices:
            blocked = {n: pending[n] for n in live}
            raise ProtocolError(f"deadlock: {blocked}")
        pick = rng.choice(choices)
        if pick == "pipe":
            pipe.pop(0)()
        elif pick == "tma":
            tma.pop(rng.randrange(len(tma)))()
        else:
            try:
                pending[pick] = next(roles[pick])
            except StopIteration:
                live.discard(pick)
                pending[pick] = None


def _run_many(n_runs, nblk=14, **kw):
    rng = random.Random(12345)
    for run in range(n_runs):
        frac = rng.choice([0.0, 0.3, 0.7, 0.95])
        keep = [True] + [rng.random() > frac for _ in range(nblk - 1)]  # block 0 is always kept
        rescale = [rng.random() < 0.2 for _ in range(nblk)]
        simulate(nblk, keep, rescale, seed=run, **kw)


@pytest.mark.parametrize("NK,NV", [(4, 2), (6, 2), (8, 2)])
def test_prefill_protocol_has_no_parity_race_or_deadlock(NK, NV):
    """The shipped protocol (one "ready" wait per block on an even ring longer
    than the S buffer ring, one Q.K^T commit per block, one P.V completion
    slot per S buffer) under random interleavings, keep patterns and
    rescales."""
    _run_many(400, NK=NK, NV=NV)


def test_model_catches_a_ready_ring_as_short_as_the_s_buffers():
    """Self-check of the model: with a ready ring of 3 slots and 3 S buffers,
    the release of block c's buffer (meant for block c + 3, the same slot)
    can reach the slot while block c's own phase is still pending, and an
    issuer's parity wait passes on it; the model must report it."""
    with pytest.raises(ProtocolError):
        _run_many(400, nblk=20, NK=3, NV=2)


def test_model_catches_two_pv_completion_slots():
    """Self-check of the model: two P.V completion slots with three S buffers
    let the end-of-tile wait pass while products are still in flight."""
    with pytest.raises(ProtocolError):
        _run_many(400, NK=4, NV=2, pv_slots=2)
