"""Race detection for the barrier protocol of the FP8-cache decode kernel
(CPU, a model of the protocol, not of the arithmetic); the barrier model and
the checks are those of the prefill protocol test.

Roles of one CTA: the K producer (E4M3 key tiles), the S^T issuer, the score
warps (blocks in pairs: both S^T buffers read and freed, both decisions
published, then P^T of each kept block), the V producer (E4M3 value tiles of
kept blocks), the converter warps (E4M3 -> fp16 value tiles) and the O^T
issuer.  Decisions go through a ring read by the V producer, the converters
and the O^T issuer; the P^T buffers are released by the O^T commits, which
also serve the O^T rescale and the end-of-split waits.
"""
import random

import pytest

from tests.test_pipeline_protocol import Bar, ProtocolError


def simulate_fp8(nb, keep, rescale, seed, NKF=7, NVF=2, NVH=2, NS=4, NPT=3, NDEC=32,
                 wait_ring_slot=True):
    rng = random.Random(seed)
    B = {}

    def bar(name, count=1):
        B[name] = Bar(name, count)

    for i in range(NKF):
        bar(("kf_full", i)), bar(("kf_empty", i))
    for i in range(NVF):
        bar(("vf_full", i)), bar(("vf_empty", i))
    for i in range(NVH):
        bar(("vh_full", i)), bar(("vh_empty", i))
    for i in range(NS):
        bar(("s_full", i)), bar(("s_free", i))
    for i in range(NPT):
        bar(("p_full", i)), bar(("p_free", i))
    for i in range(NDEC):
        bar(("dec_full", i)), bar(("dec_empty", i), 3)  # V producer, converters, O^T issuer

    kf = [None] * NKF
    vf = [None] * NVF
    vh = [None] * NVH
    sbuf = [None] * NS
    pt = [None] * NPT
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

    def kprod():
        for j in range(nb):
            f = j % NKF
            if j >= NKF:
                yield ("wait", ("kf_empty", f), j // NKF - 1)
            kf[f] = None
            B[("kf_full", f)].arrive(tx=1)

            def land(f=f, j=j):
                kf[f] = j
                B[("kf_full", f)].complete_tx(1)
            tma.append(land)
            yield None

    def qk():
        for j in range(nb):
            f, sb = j % NKF, j % NS
            yield ("wait", ("kf_full", f), j // NKF)
            if j >= NS:
                yield ("wait", ("s_free", sb), j // NS - 1)
            expect(kf[f] == j, f"S^T of block {j} reads key stage {f} holding {kf[f]}")
            expect(sbuf[sb] is None, f"S^T of block {j} overwrites buffer {sb} holding {sbuf[sb]}")
            sbuf[sb] = ("writing", j)

            def done(j=j, f=f, sb=sb):
                sbuf[sb] = j
                B[("s_full", sb)].arrive()
                B[("kf_empty", f)].arrive()
            pipe.append(done)
            yield None

    def scores():
        kc = 0
        for j in range(0, nb, 2):
            two = j + 1 < nb
            blocks = [j, j + 1] if two else [j]
            for b in blocks:
                yield ("wait", ("s_full", b % NS), b // NS)
            for b in blocks:
                expect(sbuf[b % NS] == b, f"score warps read buffer {b % NS} for block {b}: "
                                          f"{sbuf[b % NS]}")
            for b in blocks:
                sbuf[b % NS] = None
                B[("s_free", b % NS)].arrive()
            for b in blocks:  # publication by thread 0
                if b >= NDEC and wait_ring_slot:
                    yield ("wait", ("dec_empty", b % NDEC), b // NDEC - 1)
                dec[b % NDEC] = (b, keep[b])
                B[("dec_full", b % NDEC)].arrive()
                yield None
            for b in blocks:
                if not keep[b]:
                    continue
                pb = kc % NPT
                if kc >= NPT:
                    yield ("wait", ("p_free", pb), kc // NPT - 1)
                expect(pt[pb] is None, f"P^T of block {b} overwrites buffer {pb} holding {pt[pb]}")
                pt[pb] = b
                if rescale[b] and kc >= 1:
                    yield ("wait", ("p_free", (kc - 1) % NPT), (kc - 1) // NPT)
                    expect(pv_count[0] >= kc, f"O^T rescaled before product {kc - 1} completed")
                B[("p_full", pb)].arrive()
                kc += 1
                yield None
        if kc:
            yield ("wait", ("p_free", (kc - 1) % NPT), (kc - 1) // NPT)
            expect(pv_count[0] == kc, f"epilogue reads O^T with {pv_count[0]} of {kc} products")

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
            f = vi % NVF
            if vi >= NVF:
                yield ("wait", ("vf_empty", f), vi // NVF - 1)
            vf[f] = None
            B[("vf_full", f)].arrive(tx=1)

            def land(f=f, j=j):
                vf[f] = j
                B[("vf_full", f)].complete_tx(1)
            tma.append(land)
            vi += 1
            yield None

    def converters():
        vi = 0
        for j in range(nb):
            yield ("wait", ("dec_full", j % NDEC), j // NDEC)
            if not read_dec(j):
                continue
            f, hs = vi % NVF, vi % NVH
            yield ("wait", ("vf_full", f), vi // NVF)
            if vi >= NVH:
                yield ("wait", ("vh_empty", hs), vi // NVH - 1)
            expect(vf[f] == j, f"converters read value stage {f} for block {j}: {vf[f]}")
            expect(vh[hs] is None, f"converters overwrite fp16 stage {hs} holding {vh[hs]}")
            vh[hs] = j
            B[("vf_empty", f)].arrive()
            B[("vh_full", hs)].arrive()
            vi += 1
            yield None

    def ot():
        kc = 0
        for j in range(nb):
            yield ("wait", ("dec_full", j % NDEC), j // NDEC)
            if not read_dec(j):
                continue
            pb, hs = kc % NPT, kc % NVH
            yield ("wait", ("p_full", pb), kc // NPT)
            yield ("wait", ("vh_full", hs), kc // NVH)
            expect(pt[pb] == j, f"O^T of block {j} reads P^T buffer {pb} holding {pt[pb]}")
            expect(vh[hs] == j, f"O^T of block {j} reads fp16 stage {hs} holding {vh[hs]}")

            def done(pb=pb, hs=hs):
                vh[hs] = None
                B[("vh_empty", hs)].arrive()
                pt[pb] = None
                pv_count[0] += 1
                B[("p_free", pb)].arrive()
            pipe.append(done)
            kc += 1
            yield None

    roles = {"K": kprod(), "QK": qk(), "S": scores(), "V": vprod(), "C": converters(),
             "OT": ot()}
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


def _run_many(n_runs, nb=40, **kw):
    rng = random.Random(777)
    for run in range(n_runs):
        frac = rng.choice([0.0, 0.3, 0.7, 0.95])
        n = rng.choice([nb, nb - 1, 1, 2, 3])  # odd counts leave a single last block
        keep = [True] + [rng.random() > frac for _ in range(n - 1)]  # first block kept
        rescale = [rng.random() < 0.2 for _ in range(n)]
        simulate_fp8(n, keep, rescale, seed=run, **kw)


def test_fp8_decode_protocol_has_no_parity_race_or_deadlock():
    _run_many(300)


def test_fp8_decode_protocol_with_a_short_decision_ring():
    """The ring bound exercised: 4 decision slots instead of 32."""
    _run_many(300, NDEC=4)


def test_model_catches_a_decision_published_over_an_unread_slot():
    """Self-check of the model: publishing without waiting for the slot's
    previous decision to be read by all three readers must be reported."""
    with pytest.raises(ProtocolError):
        _run_many(300, NDEC=4, wait_ring_slot=False)
