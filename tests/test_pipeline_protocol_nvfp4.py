"""Race detection for the barrier protocol of the NVFP4-cache decode kernel
(CPU, a model of the protocol, not of the arithmetic); the barrier model and
the checks are those of the prefill protocol test.

Roles of one CTA: the key producer (code tile and block scales of one block
per stage), four score warps (blocks in pairs: each warp reads its rows of
both stages into registers and releases them, the four meet on a named
barrier, warp 0 publishes both decisions through the decision ring, then each
warp writes its part of P^T of every kept block), the value producer (value
codes of kept blocks), and four value warps (each reads every decision, widens
its own columns of a kept block's codes, then reads the block's P^T buffer;
the buffer is free again once all four have read it).  The score warps'
named barrier is modelled as a rendezvous of the four roles once per pair.
"""
import random

import pytest

from tests.test_pipeline_protocol import Bar, ProtocolError


def simulate_nvfp4(nb, keep, seed, NKF=5, NVF=2, NP=4, NDEC=16, p_free_count=4,
                   wait_ring_slot=True):
    rng = random.Random(seed)
    B = {}

    def bar(name, count=1):
        B[name] = Bar(name, count)

    for i in range(NKF):
        bar(("kc_full", i)), bar(("kc_empty", i), 4)
    for i in range(NVF):
        bar(("vc_full", i)), bar(("vc_empty", i), 4)
    for i in range(NP):
        bar(("p_full", i), 4), bar(("p_free", i), p_free_count)
    for i in range(NDEC):
        bar(("dec_full", i)), bar(("dec_empty", i), 1 + 4)  # value producer, value warps
    bar("l_full", 4)

    kstage = [None] * NKF       # block whose codes a key stage holds (None: loading)
    kreaders = [set() for _ in range(NKF)]
    vstage = [None] * NVF
    vreaders = [set() for _ in range(NVF)]
    pbuf = [None] * NP          # kept block whose P^T a buffer holds
    pwriters = [set() for _ in range(NP)]
    preaders = [set() for _ in range(NP)]
    dec = [None] * NDEC
    rendezvous = {}             # pair -> score warps arrived
    tma = []

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
                yield ("wait", ("kc_empty", f), j // NKF - 1)
            expect(not kreaders[f], f"key stage {f} reloaded while score warps "
                                    f"{sorted(kreaders[f])} read it")
            kstage[f] = None
            B[("kc_full", f)].arrive(tx=1)

            def land(f=f, j=j):
                kstage[f] = j
                kreaders[f].update(range(4))
                B[("kc_full", f)].complete_tx(1)
            tma.append(land)
            yield None

    def score(w):
        kc = 0
        for j in range(0, nb, 2):
            blocks = [j, j + 1] if j + 1 < nb else [j]
            for jj in blocks:
                f = jj % NKF
                yield ("wait", ("kc_full", f), jj // NKF)
                expect(kstage[f] == jj, f"score warp {w} reads key stage {f} for block {jj}: "
                                        f"{kstage[f]}")
                kreaders[f].discard(w)  # the rows are in registers
                B[("kc_empty", f)].arrive()
                yield None
            # the four score warps' named barrier, once per pair
            rendezvous.setdefault(j, set()).add(w)
            yield ("rendezvous", j)
            if w == 0:  # warp 0's thread 0 publishes both decisions
                for jj in blocks:
                    ds = jj % NDEC
                    if jj >= NDEC and wait_ring_slot:
                        yield ("wait", ("dec_empty", ds), jj // NDEC - 1)
                    dec[ds] = (jj, keep[jj])
                    B[("dec_full", ds)].arrive()
            for jj in blocks:
                if not keep[jj]:
                    continue
                pb = kc % NP
                if kc >= NP:
                    yield ("wait", ("p_free", pb), kc // NP - 1)
                expect(not preaders[pb], f"score warp {w} writes P^T buffer {pb} for block {jj} "
                                         f"while value warps {sorted(preaders[pb])} read block "
                                         f"{pbuf[pb]}")
                if not pwriters[pb]:
                    pbuf[pb] = jj
                expect(pbuf[pb] == jj, f"P^T buffer {pb} holds {pbuf[pb]}, warp {w} writes {jj}")
                pwriters[pb].add(w)
                B[("p_full", pb)].arrive()
                kc += 1
                yield None
        B["l_full"].arrive()

    def read_dec(j, who):
        d = dec[j % NDEC]
        expect(d is not None and d[0] == j, f"{who} reads decision slot {j % NDEC}: {d}, "
                                            f"not block {j}")
        B[("dec_empty", j % NDEC)].arrive()
        return d[1]

    def vprod():
        vi = 0
        for j in range(nb):
            yield ("wait", ("dec_full", j % NDEC), j // NDEC)
            if not read_dec(j, "value producer"):
                continue
            f = vi % NVF
            if vi >= NVF:
                yield ("wait", ("vc_empty", f), vi // NVF - 1)
            expect(not vreaders[f], f"value stage {f} reloaded while value warps "
                                    f"{sorted(vreaders[f])} read it")
            vstage[f] = None
            B[("vc_full", f)].arrive(tx=1)

            def land(f=f, j=j):
                vstage[f] = j
                vreaders[f].update(range(4))
                B[("vc_full", f)].complete_tx(1)
            tma.append(land)
            vi += 1
            yield None

    def value(w):
        kc = 0
        for j in range(nb):
            yield ("wait", ("dec_full", j % NDEC), j // NDEC)
            if not read_dec(j, f"value warp {w}"):
                continue
            f, pb = kc % NVF, kc % NP
            yield ("wait", ("vc_full", f), kc // NVF)
            expect(vstage[f] == j, f"value warp {w} widens stage {f} for block {j}: {vstage[f]}")
            vreaders[f].discard(w)
            B[("vc_empty", f)].arrive()
            yield ("wait", ("p_full", pb), kc // NP)
            expect(pbuf[pb] == j and len(pwriters[pb]) == 4,
                   f"value warp {w} reads P^T buffer {pb} for block {j}: block {pbuf[pb]}, "
                   f"written by {sorted(pwriters[pb])}")
            preaders[pb].add(w)
            yield None  # the products read the buffer
            preaders[pb].discard(w)
            B[("p_free", pb)].arrive()
            if B[("p_free", pb)].arrived == 0:  # the phase completed: the buffer is free
                pwriters[pb].clear()
            kc += 1
            yield None
        yield ("wait", "l_full", 0)

    roles = {"K": kprod(), "V": vprod()}
    for w in range(4):
        roles[f"S{w}"] = score(w)
        roles[f"W{w}"] = value(w)
    pending = {n: None for n in roles}
    live = set(roles)

    def ready(n):
        p = pending[n]
        if p is None:
            return True
        if p[0] == "rendezvous":
            return len(rendezvous.get(p[1], ())) == 4
        return wait(p[1], p[2])

    while live or tma:
        runnable = [n for n in live if ready(n)]
        choices = runnable + (["tma"] if tma else [])
        if not choices:
            raise ProtocolError(f"deadlock: { {n: pending[n] for n in live} }")
        pick = rng.choice(choices)
        if pick == "tma":
            tma.pop(rng.randrange(len(tma)))()
        else:
            try:
                pending[pick] = next(roles[pick])
            except StopIteration:
                live.discard(pick)
                pending[pick] = None


def _run_many(n_runs, nb=24, **kw):
    rng = random.Random(4242)
    for run in range(n_runs):
        frac = rng.choice([0.0, 0.3, 0.7, 0.95])
        n = rng.choice([nb, nb - 1, 1, 2, 3])  # odd counts leave a single last block
        keep = [True] + [rng.random() > frac for _ in range(n - 1)]  # first block kept
        simulate_nvfp4(n, keep, seed=run, **kw)


def test_nvfp4_decode_protocol_has_no_parity_race_or_deadlock():
    _run_many(200)


def test_nvfp4_decode_protocol_with_short_rings():
    """The ring bounds exercised: 2 decision slots, 1 key stage, 1 value stage,
    1 P^T buffer."""
    _run_many(150, NDEC=2, NKF=1, NVF=1, NP=1)


def test_model_catches_a_decision_published_over_an_unread_slot():
    """Self-check: publishing without waiting for the slot's previous
    decision to be read by all five readers must be reported."""
    with pytest.raises(ProtocolError):
        _run_many(300, NDEC=2, wait_ring_slot=False)


def test_model_catches_a_p_buffer_freed_by_one_value_warp():
    """Self-check: if the first value warp's read alone freed a P^T buffer,
    the score warps could overwrite it under the other three."""
    with pytest.raises(ProtocolError):
        _run_many(300, NP=1, p_free_count=1)
