"""Race detection for the barrier protocol of the absorbed-MLA decode kernel
(CPU, a model of the protocol, not of the arithmetic); the barrier model and
the checks are those of the prefill protocol test.

Roles of one CTA: the producer (Q, whose TMEM part is staged in latent slot 1,
then the latent blocks into a two-slot ring), the Q.K^T issuer, the softmax
warps (copy of Q's TMEM part, scores, decision, P over S, the in-place fp16
conversion of the value half in the latent slot), and the P.V issuer.  A
latent slot is empty again after two arrivals: the Q.K^T commit and either the
P.V commit (kept) or the P.V issuer's arrival for a skipped block.  The
decision ring has no "slot read" barrier: a decision slot is reused only after
its block's latent slot was released, which needs the P.V issuer to have
read the decision.
"""
import random

import pytest

from tests.test_pipeline_protocol import Bar, ProtocolError


def simulate_mla(nb, keep, rescale, seed, NDEC=4, skip_arrival=True):
    rng = random.Random(seed)
    B = {}

    def bar(name, count=1):
        B[name] = Bar(name, count)

    bar("q_full"), bar("qt_ready")
    for i in range(2):
        bar(("k_full", i)), bar(("k_empty", i), 2)
        bar(("s_full", i)), bar(("s_free", i)), bar(("p_full", i)), bar(("pv_done", i))
    for i in range(NDEC):
        bar(("dec_full", i))

    slot = ["-", "Q"]  # latent slot contents: a block index, "Q" (staging) or None (loading)
    conv = [None, None]  # block whose value half was converted to fp16 in the slot
    sbuf = [None, None]
    dec = [None] * NDEC
    pv_count = [0]
    pipe, tma = [], []

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

    def producer():
        B["q_full"].arrive(tx=1)
        tma.append(lambda: B["q_full"].complete_tx(1))
        yield None
        for j in range(nb):
            s = j & 1
            if j == 1:
                yield ("wait", "qt_ready", 0)
            if j >= 2:
                yield ("wait", ("k_empty", s), (j >> 1) - 1)
            slot[s] = None
            conv[s] = None
            B[("k_full", s)].arrive(tx=1)

            def land(s=s, j=j):
                slot[s] = j
                B[("k_full", s)].complete_tx(1)
            tma.append(land)
            yield None

    def qk():
        yield ("wait", "q_full", 0)
        yield ("wait", "qt_ready", 0)
        for j in range(nb):
            s = j & 1
            yield ("wait", ("k_full", s), j >> 1)
            if j >= 2:
                yield ("wait", ("s_free", s), (j >> 1) - 1)
            expect(slot[s] == j and conv[s] is None,
                   f"Q.K^T of block {j} reads latent slot {s}: {slot[s]} (converted: {conv[s]})")
            expect(sbuf[s] is None, f"Q.K^T of block {j} overwrites S buffer {s}: {sbuf[s]}")
            sbuf[s] = ("writing", j)

            def done(j=j, s=s):
                sbuf[s] = j
                B[("s_full", s)].arrive()
                B[("k_empty", s)].arrive()
            pipe.append(done)
            yield None

    def softmax():
        yield ("wait", "q_full", 0)
        expect(slot[1] == "Q", f"Q staging in latent slot 1 overwritten: {slot[1]}")
        B["qt_ready"].arrive()
        kc = 0
        for j in range(nb):
            s = j & 1
            yield ("wait", ("s_full", s), j >> 1)
            expect(sbuf[s] == j, f"softmax reads S buffer {s} for block {j}: {sbuf[s]}")
            k = keep[j]
            if not k:
                sbuf[s] = None
                B[("s_free", s)].arrive()
            d = dec[j % NDEC]
            expect(d is None or d[0] == j - NDEC, f"decision slot {j % NDEC} still holds {d}")
            dec[j % NDEC] = (j, k)
            B[("dec_full", j % NDEC)].arrive()
            yield None
            if not k:
                continue
            expect(slot[s] == j, f"fp16 conversion of block {j} in latent slot {s}: {slot[s]}")
            conv[s] = j
            if rescale[j] and kc >= 1:
                yield ("wait", ("pv_done", (kc - 1) & 1), (kc - 1) >> 1)
                expect(pv_count[0] >= kc, f"O rescaled before P.V {kc - 1} completed")
            B[("p_full", kc & 1)].arrive()
            kc += 1
            yield None
        if kc:
            yield ("wait", ("pv_done", (kc - 1) & 1), (kc - 1) >> 1)
            expect(pv_count[0] == kc, f"epilogue reads O with {pv_count[0]} of {kc} products")

    def pv():
        kc = 0
        for i in range(nb):
            s = i & 1
            yield ("wait", ("dec_full", i % NDEC), i // NDEC)
            d = dec[i % NDEC]
            expect(d is not None and d[0] == i, f"decision slot {i % NDEC} holds {d}, not {i}")
            dec[i % NDEC] = None  # read
            if not d[1]:
                if skip_arrival:
                    B[("k_empty", s)].arrive()
                continue
            yield ("wait", ("p_full", kc & 1), kc >> 1)
            expect(sbuf[s] == i, f"P.V of block {i} reads P from S buffer {s}: {sbuf[s]}")
            expect(slot[s] == i and conv[s] == i,
                   f"P.V of block {i} reads values in slot {s}: {slot[s]} (converted: {conv[s]})")

            def done(s=s, kc=kc):
                sbuf[s] = None
                B[("s_free", s)].arrive()
                pv_count[0] += 1
                B[("pv_done", kc & 1)].arrive()
                B[("k_empty", s)].arrive()
            pipe.append(done)
            kc += 1
            yield None

    roles = {"P": producer(), "QK": qk(), "SM": softmax(), "PV": pv()}
    pending = {n: None for n in roles}
    live = set(roles)
    while live or pipe or tma:
        runnable = [n for n in live if pending[n] is None or wait(pending[n][1], pending[n][2])]
        choices = runnable + (["pipe"] if pipe else []) + (["tma"] if tma else [])
        if not choices:
            raise ProtocolError(f"deadlock: { {n: pending[n] for n in live} }")
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


def _run_many(n_runs, nb=16, **kw):
    rng = random.Random(4242)
    for run in range(n_runs):
        frac = rng.choice([0.0, 0.3, 0.7, 0.95])
        n = rng.choice([nb, nb - 3, 1, 2])
        keep = [True] + [rng.random() > frac for _ in range(n - 1)]
        rescale = [rng.random() < 0.2 for _ in range(n)]
        simulate_mla(n, keep, rescale, seed=run, **kw)


def test_mla_decode_protocol_has_no_parity_race_or_deadlock():
    _run_many(400)


def test_model_catches_a_missing_skip_arrival():
    """Self-check of the model: without the P.V issuer's arrival for a skipped
    block, the latent slot is never released; the model must report it."""
    with pytest.raises(ProtocolError):
        _run_many(400, skip_arrival=False)


def test_mla_decision_ring_bound():
    """The implicit bound on the decision ring: two slots already suffice
    (a decision two blocks later needs its latent slot, released only after
    the P.V issuer read the decision); one slot does not."""
    _run_many(300, NDEC=2)
    with pytest.raises(ProtocolError):
        _run_many(300, NDEC=1)
