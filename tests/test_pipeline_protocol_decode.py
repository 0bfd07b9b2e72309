"""Race detection for the barrier protocol of the GQA split-KV decode kernel
(CPU, a model of the protocol, not of the arithmetic); the barrier model and
the checks are those of the prefill protocol test.

Roles of one CTA: the K producer, the Q.K^T issuer, the softmax warp (scores
into registers, S buffer freed at once, decision, P of a kept block into one
of two TMEM P buffers, O rescale, epilogue), the V producer (kept blocks) and
the P.V issuer.  Decisions go through a ring read by the V producer and the
P.V issuer; P buffers are released by the P.V commits.
"""
import random

import pytest

from tests.test_pipeline_protocol import Bar, ProtocolError


def simulate_decode(nb, keep, rescale, seed, NK=4, NV=2, NS=2, NP=2, NDEC=8, pv_slots=2):
    rng = random.Random(seed)
    B = {}

    def bar(name, count=1):
        B[name] = Bar(name, count)

    for i in range(NK):
        bar(("k_full", i)), bar(("k_empty", i))
    for i in range(NV):
        bar(("v_full", i)), bar(("v_empty", i))
    for i in range(NS):
        bar(("s_full", i)), bar(("s_free", i))
    for i in range(NP):
        bar(("p_full", i)), bar(("p_free", i))
    for i in range(pv_slots):
        bar(("pv_done", i))
    for i in range(NDEC):
        bar(("dec_full", i)), bar(("dec_empty", i), 2)

    kst, vst, sbuf, pbuf, dec = [None] * NK, [None] * NV, [None] * NS, [None] * NP, [None] * NDEC
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

    def kprod():
        for j in range(nb):
            s = j % NK
            if j >= NK:
                yield ("wait", ("k_empty", s), j // NK - 1)
            kst[s] = None
            B[("k_full", s)].arrive(tx=1)

            def land(s=s, j=j):
                kst[s] = j
                B[("k_full", s)].complete_tx(1)
            tma.append(land)
            yield None

    def qk():
        for j in range(nb):
            s, sb = j % NK, j % NS
            yield ("wait", ("k_full", s), j // NK)
            if j >= NS:
                yield ("wait", ("s_free", sb), j // NS - 1)
            expect(kst[s] == j, f"Q.K^T of block {j} reads K stage {s} holding {kst[s]}")
            expect(sbuf[sb] is None, f"Q.K^T of block {j} overwrites S buffer {sb}: {sbuf[sb]}")
            sbuf[sb] = ("writing", j)

            def done(j=j, s=s, sb=sb):
                sbuf[sb] = j
                B[("s_full", sb)].arrive()
                B[("k_empty", s)].arrive()
            pipe.append(done)
            yield None

    def softmax():
        kc = 0
        for j in range(nb):
            sb = j % NS
            yield ("wait", ("s_full", sb), j // NS)
            expect(sbuf[sb] == j, f"softmax reads S buffer {sb} for block {j}: {sbuf[sb]}")
            sbuf[sb] = None  # scores in registers
            B[("s_free", sb)].arrive()
            if j >= NDEC:
                yield ("wait", ("dec_empty", j % NDEC), j // NDEC - 1)
            dec[j % NDEC] = (j, keep[j])
            B[("dec_full", j % NDEC)].arrive()
            yield None
            if not keep[j]:
                continue
            pb = kc % NP
            if kc >= NP:
                yield ("wait", ("p_free", pb), kc // NP - 1)
            expect(pbuf[pb] is None, f"P of block {j} overwrites P buffer {pb}: {pbuf[pb]}")
            pbuf[pb] = j
            if rescale[j] and kc >= 1:
                yield ("wait", ("pv_done", (kc - 1) % pv_slots), (kc - 1) // pv_slots)
                expect(pv_count[0] >= kc, f"O rescaled before P.V {kc - 1} completed")
            B[("p_full", pb)].arrive()
            kc += 1
            yield None
        if kc:
            yield ("wait", ("pv_done", (kc - 1) % pv_slots), (kc - 1) // pv_slots)
            expect(pv_count[0] == kc, f"epilogue reads O with {pv_count[0]} of {kc} products")

    def read_dec(j):
        d = dec[j % NDEC]
        expect(d is not None and d[0] == j, f"decision slot {j % NDEC} holds {d}, not block {j}")
        B[("dec_empty", j % NDEC)].arrive()
        return d[1]

    def vprod():
        vi = 0
        for j in range(nb):
            yield ("wait", ("dec_full", j % NDEC), j // NDEC)
            if not read_dec(j):
                continue
            s = vi % NV
            if vi >= NV:
                yield ("wait", ("v_empty", s), vi // NV - 1)
            vst[s] = None
            B[("v_full", s)].arrive(tx=1)

            def land(s=s, j=j):
                vst[s] = j
                B[("v_full", s)].complete_tx(1)
            tma.append(land)
            vi += 1
            yield None

    def pv():
        kc = vi = 0
        for j in range(nb):
            yield ("wait", ("dec_full", j % NDEC), j // NDEC)
            if not read_dec(j):
                continue
            pb, vs = kc % NP, vi % NV
            yield ("wait", ("p_full", pb), kc // NP)
            yield ("wait", ("v_full", vs), vi // NV)
            expect(pbuf[pb] == j, f"P.V of block {j} reads P buffer {pb} holding {pbuf[pb]}")
            expect(vst[vs] == j, f"P.V of block {j} reads V stage {vs} holding {vst[vs]}")

            def done(pb=pb, vs=vs, kc=kc):
                B[("v_empty", vs)].arrive()
                pbuf[pb] = None
                B[("p_free", pb)].arrive()
                pv_count[0] += 1
                B[("pv_done", kc % pv_slots)].arrive()
            pipe.append(done)
            kc += 1
            vi += 1
            yield None

    roles = {"K": kprod(), "QK": qk(), "SM": softmax(), "V": vprod(), "PV": pv()}
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


def _run_many(n_runs, nb=32, **kw):
    rng = random.Random(99)
    for run in range(n_runs):
        frac = rng.choice([0.0, 0.3, 0.7, 0.95])
        n = rng.choice([nb, nb - 5, 1, 2])
        keep = [True] + [rng.random() > frac for _ in range(n - 1)]  # split-local first block
        rescale = [rng.random() < 0.2 for _ in range(n)]
        simulate_decode(n, keep, rescale, seed=run, **kw)


def test_gqa_decode_protocol_has_no_parity_race_or_deadlock():
    """As shipped: two P buffers, so at most two products in flight and the
    two P.V completion slots are unambiguous."""
    _run_many(300)


def test_model_catches_three_p_buffers_with_two_completion_slots():
    """Self-check of the model: a third P buffer with the same two completion
    slots lets the end-of-split wait pass with a product in flight."""
    with pytest.raises(ProtocolError):
        _run_many(300, NP=3)
