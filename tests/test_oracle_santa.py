"""Pins for the oracle's sampled decode output (CPU only).

The sampler follows the page "Stochastic Sparse Attention for Memory-Bound
Inference" (SANTA), section "关键设计": the attention weights of a query are a
categorical distribution, the estimate of p V is the mean of the value rows at
S inverse-CDF samples, drawn i.i.d., one per equal-mass stratum, or on one
shifted lattice (systematic).  Each test checks the oracle against something
other than itself: exact closed forms (equal scores, a dominant key), numpy's
own softmax / cumulative sum / sorted search on tiny inputs, the lattice count
of the systematic sampler, its deterministic error bound, and unbiasedness
(the mean over offsets or draws equals dense attention).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _inputs(B, Hq, Hkv, L, d, seed, q_scale=1.0, peaked=True):
    rng = np.random.default_rng(seed)
    q = (q_scale * rng.standard_normal((B, Hq, d))).astype(np.float32)
    k = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
    if peaked:
        # A few heavy keys, as in long-context attention (sink + salient keys).
        G = Hq // Hkv
        for b in range(B):
            for hk in range(Hkv):
                dirn = q[b, hk * G:(hk + 1) * G].mean(axis=0)
                dirn /= np.linalg.norm(dirn) + 1e-9
                heavy = rng.choice(L, size=max(1, L // 16), replace=False)
                k[b, hk, heavy] += (3.0 * dirn).astype(np.float32)
                k[b, hk, 0] += (5.0 * dirn).astype(np.float32)
    v = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
    return q, k, v


def _softmax_cdf(q, k, scale):
    """numpy: p [B,Hq,L] and its cumulative sum (fp64)."""
    G = q.shape[1] // k.shape[1]
    kk = np.repeat(k.astype(np.float64), G, axis=1)
    s = scale * np.einsum("bhd,bhld->bhl", q.astype(np.float64), kk)
    p = np.exp(s - s.max(axis=-1, keepdims=True))
    p /= p.sum(axis=-1, keepdims=True)
    return p, np.cumsum(p, axis=-1)


def _dense(q, k, v, scale):
    p, _ = _softmax_cdf(q, k, scale)
    G = q.shape[1] // k.shape[1]
    return np.einsum("bhl,bhle->bhe", p, np.repeat(v.astype(np.float64), G, axis=1))


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["sys", "strat", "iid"])
@pytest.mark.parametrize("L,S", [(96, 8), (96, 32), (50, 16), (7, 64)])
def test_equal_scores_closed_form(mode, L, S):
    """q = 0: every key weighs 1/L, so J_m = floor(T_m L) and the gap is the
    distance of T_m L from the nearer integer, over L (exact rationals)."""
    B, Hq, d = 1, 3, 8
    rng = np.random.default_rng(L * 1000 + S)
    q = np.zeros((B, Hq, d), np.float32)
    k = rng.standard_normal((B, 1, L, d)).astype(np.float32)
    v = rng.standard_normal((B, 1, L, d)).astype(np.float32)
    shape = (B, Hq) if mode == "sys" else (B, Hq, S)
    u = rng.random(shape, dtype=np.float32)
    r = oracle.santa_decode(q, k, v, 0.5, S, mode, u)
    for h in range(Hq):
        for m in range(S):
            if mode == "sys":
                T = (m + Fraction(float(u[0, h]))) / S
            elif mode == "strat":
                T = (m + Fraction(float(u[0, h, m]))) / S
            else:
                T = Fraction(float(u[0, h, m]))
            x = T * L
            J = int(x)  # floor
            assert r["idx"][0, h, m] == J
            frac = x - J
            assert r["gap"][0, h, m] == pytest.approx(float(min(frac, 1 - frac) / L), abs=1e-12)
        want = v[0, 0, r["idx"][0, h]].astype(np.float64).mean(axis=0)
        np.testing.assert_allclose(r["y"][0, h], want, rtol=0, atol=1e-12)
        # the closed form directly, not through the oracle's indices
        Js = [int(((m + Fraction(float(u[0, h]))) / S if mode == "sys" else
                   (m + Fraction(float(u[0, h, m]))) / S if mode == "strat" else
                   Fraction(float(u[0, h, m]))) * L) for m in range(S)]
        np.testing.assert_allclose(r["y"][0, h], v[0, 0, Js].astype(np.float64).mean(axis=0),
                                   rtol=0, atol=1e-12)


@pytest.mark.parametrize("mode", ["sys", "strat", "iid"])
def test_dominant_key_takes_every_sample(mode):
    """One key 40 nats above the rest holds all but e^-40 L of the mass: every
    threshold away from 0 and 1 lands on it and the estimate is its value row."""
    B, Hq, Hkv, L, d, S = 2, 4, 2, 300, 16, 32
    rng = np.random.default_rng(5)
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = (0.1 * rng.standard_normal((B, Hkv, L, d))).astype(np.float32)
    star = [[17, 250], [0, 299]]
    G = Hq // Hkv
    for b in range(B):
        for hk in range(Hkv):
            k[b, hk, star[b][hk]] = 40.0 * q[b, hk * G:(hk + 1) * G].mean(axis=0) / np.linalg.norm(
                q[b, hk * G:(hk + 1) * G].mean(axis=0)) * 1.5
    v = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
    shape = (B, Hq) if mode == "sys" else (B, Hq, S)
    u = (0.01 + 0.98 * rng.random(shape)).astype(np.float32)
    r = oracle.santa_decode(q, k, v, 1.0, S, mode, u)
    p, _ = _softmax_cdf(q, k, 1.0)
    for b in range(B):
        for h in range(Hq):
            j = star[b][h // G]
            assert p[b, h, j] > 1 - 1e-12
            assert (r["idx"][b, h] == j).all()
            np.testing.assert_allclose(r["y"][b, h], v[b, h // G, j], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# numpy's inverse CDF on tiny inputs
# --------------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["strat", "iid", "sys"])
def test_indices_are_numpy_inverse_cdf(mode):
    """J_m = the first index whose cumulative weight exceeds T_m, found by
    numpy's sorted search over numpy's cumulative sum; stratified sample m
    stays inside stratum m; the systematic and stratified indices never
    decrease."""
    B, Hq, Hkv, L, d, S = 2, 8, 2, 257, 32, 64
    q, k, v = _inputs(B, Hq, Hkv, L, d, seed=11)
    scale = d ** -0.5
    rng = np.random.default_rng(12)
    shape = (B, Hq) if mode == "sys" else (B, Hq, S)
    u = rng.random(shape, dtype=np.float32)
    r = oracle.santa_decode(q, k, v, scale, S, mode, u, with_cdf=True)
    _, F = _softmax_cdf(q, k, scale)
    np.testing.assert_allclose(r["cdf"], F, rtol=0, atol=1e-12)
    m = np.arange(S)
    for b in range(B):
        for h in range(Hq):
            if mode == "sys":
                T = (m + np.float64(u[b, h])) / S
            elif mode == "strat":
                T = (m + u[b, h].astype(np.float64)) / S
            else:
                T = u[b, h].astype(np.float64)
            J = np.searchsorted(F[b, h], T, side="right")
            clear = r["gap"][b, h] > 1e-12
            assert clear.mean() > 0.9
            np.testing.assert_array_equal(r["idx"][b, h][clear], J[clear])
            if mode != "iid":
                assert (np.diff(r["idx"][b, h]) >= 0).all()
            if mode == "strat":
                lo = np.concatenate([[0.0], F[b, h]])[r["idx"][b, h]]
                hi = F[b, h][r["idx"][b, h]]
                # sample m's interval meets stratum [m/S, (m+1)/S)
                assert (lo < (m + 1) / S + 1e-12).all() and (hi > m / S - 1e-12).all()


# --------------------------------------------------------------------------
# The systematic sampler: lattice counts and the deterministic error bound
# --------------------------------------------------------------------------

@pytest.mark.parametrize("S", [16, 128, 1000])
def test_systematic_counts_are_lattice_counts(S):
    """Key i is picked once per lattice point (m + u)/S inside its CDF interval
    [F_{i-1}, F_i): ceil(S F_i - u) - ceil(S F_{i-1} - u) times, which is
    floor(S p_i) or ceil(S p_i)."""
    B, Hq, Hkv, L, d = 2, 4, 2, 333, 32
    q, k, v = _inputs(B, Hq, Hkv, L, d, seed=21 + S)
    scale = d ** -0.5
    u = np.random.default_rng(22).random((B, Hq), dtype=np.float32)
    r = oracle.santa_decode(q, k, v, scale, S, "sys", u)
    p, F = _softmax_cdf(q, k, scale)
    for b in range(B):
        for h in range(Hq):
            cnt = np.bincount(r["idx"][b, h], minlength=L)
            Fl = np.concatenate([[0.0], F[b, h]])
            x = S * Fl - np.float64(u[b, h])
            want = np.diff(np.ceil(x))
            # a lattice point within rounding of a boundary may fall either side
            near = np.abs(x - np.round(x)) < 1e-9
            ok = ~(near[1:] | near[:-1])
            np.testing.assert_array_equal(cnt[ok], want[ok])
            assert cnt.sum() == S
            sp = S * p[b, h]
            assert (cnt >= np.floor(sp - 1e-9)).all() and (cnt <= np.ceil(sp + 1e-9)).all()


def test_systematic_error_bound():
    """Every count is within 1 of S p_i, so |y - p V| <= (1/S) sum_i |V_i| per
    output column, for any offset."""
    B, Hq, Hkv, L, d, S = 1, 8, 2, 64, 16, 4096
    q, k, v = _inputs(B, Hq, Hkv, L, d, seed=31)
    scale = d ** -0.5
    u = np.random.default_rng(32).random((B, Hq), dtype=np.float32)
    r = oracle.santa_decode(q, k, v, scale, S, "sys", u)
    ref = _dense(q, k, v, scale)
    G = Hq // Hkv
    for h in range(Hq):
        bound = np.abs(v[0, h // G].astype(np.float64)).sum(axis=0) / S
        assert (np.abs(r["y"][0, h] - ref[0, h]) <= bound + 1e-12).all()


# --------------------------------------------------------------------------
# Unbiasedness: E[y] = p V
# --------------------------------------------------------------------------

def test_systematic_mean_over_offset_grid_is_dense_attention():
    """y(u) is piecewise constant in u with at most L + S jumps of size at
    most max|V_a - V_b| / S; the midpoint rule over N offsets is within
    (L + S) max|V_a - V_b| / (2 S N) of the integral, which is p V."""
    L, d, S, N = 40, 16, 4, 20000
    rng = np.random.default_rng(41)
    q1 = rng.standard_normal((1, 1, d)).astype(np.float32)
    k = rng.standard_normal((1, 1, L, d)).astype(np.float32)
    v = rng.standard_normal((1, 1, L, d)).astype(np.float32)
    q = np.repeat(q1, N, axis=1)  # N query heads on one KV head: one offset each
    u = ((np.arange(N) + 0.5) / N).astype(np.float32)[None]
    r = oracle.santa_decode(q, k, v, 0.5, S, "sys", u)
    ref = _dense(q1, k, v, 0.5)[0, 0]
    spread = (v[0, 0].max(axis=0) - v[0, 0].min(axis=0)).astype(np.float64)
    tol = (L + S) * spread / (2 * S * N) + 1e-6  # + float32 rounding of the grid
    assert (np.abs(r["y"][0].mean(axis=0) - ref) <= tol).all()


@pytest.mark.parametrize("mode", ["strat", "iid"])
def test_random_draws_average_to_dense_attention(mode):
    """The mean over N independent draws is within 5 standard errors of p V,
    and the stratified draws have lower variance than the i.i.d. ones at the
    same S (variance reduction)."""
    L, d, S, N = 60, 8, 8, 20000
    rng = np.random.default_rng(51)
    q1 = (1.5 * rng.standard_normal((1, 1, d))).astype(np.float32)
    k = rng.standard_normal((1, 1, L, d)).astype(np.float32)
    v = rng.standard_normal((1, 1, L, d)).astype(np.float32)
    q = np.repeat(q1, N, axis=1)
    ref = _dense(q1, k, v, 1.0)[0, 0]
    ys = {}
    for md in ("strat", "iid"):
        u = np.random.default_rng(52 if md == "strat" else 53).random((1, N, S), dtype=np.float32)
        ys[md] = oracle.santa_decode(q, k, v, 1.0, S, md, u)["y"][0]
    y = ys[mode]
    se = y.std(axis=0) / np.sqrt(N)
    assert (np.abs(y.mean(axis=0) - ref) <= 5 * se + 1e-9).all()
    assert ys["strat"].var(axis=0).sum() < 0.7 * ys["iid"].var(axis=0).sum()


# --------------------------------------------------------------------------
# Arguments
# --------------------------------------------------------------------------

def test_rejects_offsets_outside_unit_interval():
    q, k, v = _inputs(1, 2, 1, 10, 8, seed=61)
    for bad in (1.0, -0.25, np.nan):
        u = np.array([[0.5, bad]], np.float32)
        with pytest.raises(ValueError):
            oracle.santa_decode(q, k, v, 0.3, 4, "sys", u)
    with pytest.raises(ValueError):
        oracle.santa_decode(q, k, v, 0.3, 4, "strat", np.zeros((1, 2), np.float32))
