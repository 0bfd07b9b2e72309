"""Host-side threshold calibration helpers (section "校准算法：一次前向，一个指数模型"
of the BLASST page) against plain numpy, and the property they rest on: the
block statistic does not depend on lambda (checked with the oracle)."""
import math

import numpy as np
import pytest

import oracle
from block_sparse_attention_online_gb300 import binding as bs
from block_sparse_attention_online_gb300 import workloads as W


def _margins(rng, n, frac_nan=0.1, frac_ninf=0.05, frac_zero=0.2):
    m = -rng.exponential(3.0, n).astype(np.float32)
    u = rng.random(n)
    m[u < frac_zero] = 0.0
    m[(u >= frac_zero) & (u < frac_zero + frac_ninf)] = -np.inf
    m[(u >= frac_zero + frac_ninf) & (u < frac_zero + frac_ninf + frac_nan)] = np.nan
    return m


def _brute_sparsity(m, lam):
    t = m[~np.isnan(m)]
    if lam == 0.0 or t.size == 0:
        return 0.0
    return float((t.astype(np.float64) < math.log(lam)).mean())


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_sparsity_at_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    m = _margins(rng, 5000)
    for lam in (0.0, 1e-9, 1e-3, 0.05, 0.5, 0.999):
        assert bs.attn_skip_sparsity_at(m, lam) == pytest.approx(_brute_sparsity(m, lam), abs=0)


@pytest.mark.parametrize("target", [0.0, 0.1, 0.3, 0.5, 0.7])
def test_lambda_for_sparsity_hits_the_target(target):
    rng = np.random.default_rng(7)
    m = _margins(rng, 4001)
    lam = bs.attn_skip_lambda_for_sparsity(m, target)
    assert 0.0 <= lam < 1.0
    trav = int((~np.isnan(m)).sum())
    want = round(target * trav) / trav
    assert _brute_sparsity(m, lam) == pytest.approx(want, abs=0.5 / trav)


def test_lambda_for_sparsity_caps_at_the_negative_fraction():
    """A statistic of 0 (some row found a new max) is skipped by no lambda < 1."""
    m = np.array([0, 0, 0, -1, -2, np.nan], dtype=np.float32)
    lam = bs.attn_skip_lambda_for_sparsity(m, 0.9)
    assert lam < 1.0 and _brute_sparsity(m, lam) == pytest.approx(2 / 5)
    m0 = np.zeros(4, dtype=np.float32)
    assert bs.attn_skip_lambda_for_sparsity(m0, 0.5) == 0.0


def test_lambda_for_sparsity_rejects_bad_input():
    with pytest.raises(bs.AttnSkipError):
        bs.attn_skip_lambda_for_sparsity(np.full(3, np.nan, dtype=np.float32), 0.5)
    with pytest.raises(bs.AttnSkipError):
        bs.attn_skip_lambda_for_sparsity(np.zeros(3, dtype=np.float32), 1.5)


def test_fit_recovers_the_exponential_model():
    alpha, beta = 950.0, 4.2
    L = [4096, 8192, 16384, 32768, 65536] * 3
    s = [0.3] * 5 + [0.5] * 5 + [0.7] * 5
    lam = [alpha * math.exp(beta * si) / Li for Li, si in zip(L, s)]
    a, b = bs.attn_skip_fit_lambda_model(L, s, lam)
    assert a == pytest.approx(alpha, rel=1e-9) and b == pytest.approx(beta, rel=1e-9)
    # noisy points: the same least-squares line as numpy's
    rng = np.random.default_rng(3)
    lam_n = [x * math.exp(0.1 * rng.standard_normal()) for x in lam]
    a2, b2 = bs.attn_skip_fit_lambda_model(L, s, lam_n)
    y = np.log(np.array(lam_n) * np.array(L))
    bb, aa = np.polyfit(np.array(s), y, 1)
    assert b2 == pytest.approx(bb, rel=1e-9) and math.log(a2) == pytest.approx(aa, rel=1e-9)


def test_fit_rejects_degenerate_points():
    with pytest.raises(bs.AttnSkipError):
        bs.attn_skip_fit_lambda_model([4096, 8192], [0.5, 0.5], [0.1, 0.05])
    with pytest.raises(bs.AttnSkipError):
        bs.attn_skip_fit_lambda_model([4096], [0.5], [0.1])
    with pytest.raises(bs.AttnSkipError):
        bs.attn_skip_fit_lambda_model([4096, 8192], [0.5, 0.7], [0.0, 0.05])


def test_lambda_for_target_rule():
    assert bs.attn_skip_lambda_for_target(1000.0, 2.0, 0.7, 8192) == pytest.approx(
        1000.0 * math.exp(1.4) / 8192, rel=1e-15)
    assert bs.attn_skip_lambda_for_target(1e9, 2.0, 0.7, 10) < 1.0
    assert bs.attn_skip_lambda_for_target(-1.0, 2.0, 0.7, 10) == 0.0


def test_oracle_statistic_does_not_depend_on_lambda():
    """The header's premise: one pass gives the statistic for every lambda, and
    the bitmap at any lambda is {statistic < ln lambda} (lambda > 0)."""
    cfg = W.temperate(W.TINY_PREFILL.with_(T=512, seed=71))
    q, k, v = W.prefill_inputs(cfg)
    base = oracle.prefill(q, k, v, cfg.scale, 0.0, 128, 128, True)["margin"]
    for lam in (1e-3, 0.2, 0.9):
        r = oracle.prefill(q, k, v, cfg.scale, lam, 128, 128, True)
        np.testing.assert_array_equal(r["margin"], base)
        trav = ~np.isnan(base)
        assert ((base < math.log(lam))[trav] == r["skip"][trav].astype(bool)).all()
    dcfg = W.temperate(W.GQA_DECODE_32K.with_(B=2, L=1500, n_splits=3, seed=72))
    q, k, v = W.decode_inputs(dcfg)
    base = oracle.decode(q, k, v, dcfg.scale, 0.0, dcfg.Bc, 3)["margin"]
    r = oracle.decode(q, k, v, dcfg.scale, 0.3, dcfg.Bc, 3)
    np.testing.assert_array_equal(r["margin"], base)
