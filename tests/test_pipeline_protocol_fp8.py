"""Race detection for the barrier protocol of the FP8-cache decode kernel
(CPU, a model of the protocol, not of the arithmetic); the barrier model and
the checks are those of the prefill protocol test.

Roles of one CTA: the K producer (E4M3 key tiles, two blocks per stage and
barrier), the S^T issuer (one pair per key barrier, one S^T pair buffer of two
adjacent buffers per barrier), the score warps (blocks in pairs: the pair
buffer read and freed, both decisions published under one ring barrier, then
P^T of each kept block), the V producer (E4M3 value tiles of kept blocks), the
converter warps (E4M3 -> fp16 value tiles) and the O^T issuer.  Decisions go
through a ring of block pairs read by the V producer, the converters and the
O^T issuer (each reads a pair's slot once); the P^T buffers are released by
the O^T commits, which also serve the O^T rescale and the end-of-split waits.
"""
import random

import pytest

from tests.test_pipeline_protocol import Bar, ProtocolError


def simulate_fp8(nb, keep, rescale, seed, NKP=3, NVF=2, NVH=2, NPT=3, NDP=16,
                 wait_ring_slot=True):
    rng = random.Random(seed)
    B = {}

    def bar(name, count=1):
        B[name] = Bar(name, count)

    for i in range(NKP):
        bar(("kf_full", i)), bar(("kf_empty", i))
    for i in range(NVF):
        bar(("vf_full", i)), bar(("vf_empty", i))
    for i in range(NVH):
        bar(("vh_full", i)), bar(("vh_empty", i))
    for i in range(2):  # pair buffers
        bar(("s_full", i)), bar(("s_free", i))
    for i in range(NPT):
        bar(("p_full", i)), bar(("p_free", i))
    for i in range(NDP):
        bar(("dec_full", i)), bar(("dec_empty", i), 3)  # V producer, converters, O^T issuer

    npair = (nb + 1) // 2
    kf = [None] * NKP
    vf = [None] * NVF
    vh = [None] * NVH
    sbuf = [None] * 2
    pt = [None] * NPT
    dec = [None] * NDP
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
        for q in range(npair):
            f = q % NKP
            n = 2 if 2 * q + 1 < nb else 1
            if q >= NKP:
                yield ("wait", ("kf_empty", f), q // NKP - 1)
            kf[f] = None
            B[("kf_full", f)].arrive(tx=n)
            got = []

            def land(f=f, q=q, got=got, n=n):  # one tile of the pair; the stage holds
                got.append(1)                   # the pair once both have landed
                if len(got) == n:
                    kf[f] = q
                B[("kf_full", f)].complete_tx(1)
            for _ in range(n):
                tma.append(land)
            yield None

    def qk():
        for q in range(npair):
            f, pb = q % NKP, q % 2
            yield ("wait", ("kf_full", f), q // NKP)
            if q >= 2:
                yield ("wait", ("s_free", pb), q // 2 - 1)
            expect(kf[f] == q, f"S^T of pair {q} reads key stage {f} holding {kf[f]}")
            expect(sbuf[pb] is None, f"S^T of pair {q} overwrites buffer {pb} holding {sbuf[pb]}")
            sbuf[pb] = ("writing", q)

            def done(q=q, f=f, pb=pb):
                sbuf[pb] = q
                B[("s_full", pb)].arrive()
                B[("kf_empty", f)].arrive()
            pipe.append(done)
            yield None

    def scores():
        kc = 0
        for j in range(0, nb, 2):
            two = j + 1 < nb
            blocks = [j, j + 1] if two else [j]
            q, pb = j // 2, (j // 2) % 2
            yield ("wait", ("s_full", pb), q // 2)
            expect(sbuf[pb] == q, f"score warps read pair buffer {pb} for pair {q}: {sbuf[pb]}")
            sbuf[pb] = None
            B[("s_free", pb)].arrive()
            # publication of the pair by thread 0
            if q >= NDP and wait_ring_slot:
                yield ("wait", ("dec_empty", q % NDP), q // NDP - 1)
            dec[q % NDP] = (q, [keep[b] for b in blocks])
            B[("dec_full", q % NDP)].arrive()
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
        q = j // 2
        d = dec[q % NDP]
        expect(d is not None and d[0] == q, f"decision slot {q % NDP} holds {d}, not pair {q}")
        keep_j = d[1][j % 2]
        if j % 2 == 1 or j == nb - 1:  # the pair's slot is read
            B[("dec_empty", q % NDP)].arrive()
        return keep_j

    def wait_dec(j):  # the readers wait once per pair, at its first block
        return [("wait", ("dec_full", (j // 2) % NDP), (j // 2) // NDP)] if j % 2 == 0 else []

    def vprod():
        vi = 0
        for j in range(nb):
            for w in wait_dec(j):
                yield w
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
            for w in wait_dec(j):
                yield w
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
            for w in wait_dec(j):
                yield w
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
    """The ring bound exercised: 2 pair slots instead of 16."""
    _run_many(300, NDP=2)


def test_fp8_decode_protocol_with_one_key_stage():
    _run_many(200, NKP=1)


def test_model_catches_a_decision_published_over_an_unread_slot():
    """Self-check of the model: publishing without waiting for the slot's
    previous pair to be read by all three readers must be reported."""
    with pytest.raises(ProtocolError):
        _run_many(300, NDP=2, wait_ring_slot=False)
