"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: a brute-force
numpy softmax, torch's fp64 scaled_dot_product_attention, hand-worked cases
(tests/golden/blasst_hand_cases.json), the numbers the BLASST page prints
(tests/golden/blasst_worked_numbers.json), closed forms (lambda = 0 is dense
attention; the output is the softmax restricted to the kept tokens) and the
invariants the page states (a block holding a row's maximum is never skipped;
every skipped token has softmax weight below lambda; the output error bound of
the page's Appendix B, in its rigorous first-order form).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_online_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# Independent brute force (numpy, whole score matrix at once)
# --------------------------------------------------------------------------

def scores_full(q, k, scale, causal):
    """[B,Hq,T,T] scaled scores with -inf where masked (fp64)."""
    q = q.astype(np.float64)
    k = k.astype(np.float64)
    G = q.shape[1] // k.shape[1]
    kk = np.repeat(k, G, axis=1)
    s = scale * np.einsum("bhrd,bhcd->bhrc", q, kk)
    if causal:
        T = q.shape[2]
        s = np.where(np.tril(np.ones((T, T), dtype=bool))[None, None], s, -np.inf)
    return s


def softmax_rows(s):
    m = s.max(axis=-1, keepdims=True)
    p = np.exp(s - m)
    return p / p.sum(axis=-1, keepdims=True), (m[..., 0] + np.log(p.sum(axis=-1)))


def brute_dense(q, k, v, scale, causal):
    s = scores_full(q, k, scale, causal)
    p, lse = softmax_rows(s)
    G = q.shape[1] // k.shape[1]
    vv = np.repeat(v.astype(np.float64), G, axis=1)
    return np.einsum("bhrc,bhce->bhre", p, vv), lse, p


def visible_block_mask(T, Br, Bc, causal):
    """[n_t, n_b] True where the tile traverses the block."""
    n_t, n_b = -(-T // Br), -(-T // Bc)
    m = np.ones((n_t, n_b), dtype=bool)
    if causal:
        for t in range(n_t):
            last = min(T, (t + 1) * Br) - 1
            m[t, last // Bc + 1:] = False
    return m


def kept_token_mask(skip, T, Br, Bc, causal):
    """[B,Hq,T,T] True for tokens of blocks the row's tile keeps (and visible)."""
    B, Hq, n_t, n_b = skip.shape
    trav = visible_block_mask(T, Br, Bc, causal)
    keep_blk = (~skip.astype(bool)) & trav[None, None]
    rows_t = np.arange(T) // Br
    cols_b = np.arange(T) // Bc
    km = keep_blk[:, :, rows_t][:, :, :, cols_b]
    if causal:
        km &= np.tril(np.ones((T, T), dtype=bool))[None, None]
    return km


def rand_prefill(B, Hq, Hkv, T, d, seed, dv=None, spread=1.0):
    g = np.random.default_rng(seed)
    dv = dv or d
    q = (g.standard_normal((B, Hq, T, d)) * spread).astype(np.float32)
    k = (g.standard_normal((B, Hkv, T, d)) * spread).astype(np.float32)
    v = g.standard_normal((B, Hkv, T, dv)).astype(np.float32)
    return q, k, v


# --------------------------------------------------------------------------
# Dense attention
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [True, False])
def test_dense_prefill_matches_bruteforce(causal):
    q, k, v = rand_prefill(2, 4, 2, 37, 8, seed=1, dv=5)
    y, lse = oracle.dense_prefill(q, k, v, 0.3, causal=causal)
    yb, lseb, _ = brute_dense(q, k, v, 0.3, causal)
    np.testing.assert_allclose(y, yb, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lseb, rtol=1e-12, atol=1e-13)


def test_dense_prefill_matches_torch_sdpa_fp64():
    q, k, v = rand_prefill(1, 4, 2, 70, 16, seed=2)
    y, _ = oracle.dense_prefill(q, k, v, 1 / 4.0, causal=True)
    tq, tk, tv = (torch.from_numpy(x).double() for x in (q, k, v))
    tk = tk.repeat_interleave(2, dim=1)
    tv = tv.repeat_interleave(2, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True,
                                                           scale=1 / 4.0)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-11, atol=1e-12)


def test_dense_prefill_row_subset():
    q, k, v = rand_prefill(1, 2, 1, 40, 8, seed=3)
    rows = [0, 17, 39, 40 + 5, 79]
    y, lse = oracle.dense_prefill(q, k, v, 0.5, causal=True, rows=rows)
    yb, lseb, _ = brute_dense(q, k, v, 0.5, True)
    yf, lf = y.reshape(-1, 8), lse.reshape(-1)
    np.testing.assert_allclose(yf[rows], yb.reshape(-1, 8)[rows], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lf[rows], lseb.reshape(-1)[rows], rtol=1e-12)


def test_dense_decode_matches_bruteforce_and_latent_alias():
    g = np.random.default_rng(4)
    B, Hq, Hkv, L, dk, dv = 2, 6, 2, 50, 12, 8
    q = g.standard_normal((B, Hq, dk)).astype(np.float32)
    k = g.standard_normal((B, Hkv, L, dk)).astype(np.float32)
    v = g.standard_normal((B, Hkv, L, dv)).astype(np.float32)
    y, lse = oracle.dense_decode(q, k, v, 0.25)
    yb, lseb, _ = brute_dense(q[:, :, None], k, v, 0.25, False)
    np.testing.assert_allclose(y, yb[:, :, 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lseb[:, :, 0], rtol=1e-12)
    # latent cache: values are the first dv columns of the keys
    y2, _ = oracle.dense_decode(q, k, None, 0.25, dv=dv)
    yb2, _, _ = brute_dense(q[:, :, None], k, k[..., :dv].copy(), 0.25, False)
    np.testing.assert_allclose(y2, yb2[:, :, 0], rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# Hand-worked fixtures
# --------------------------------------------------------------------------

def _hand_cases():
    with open(os.path.join(GOLDEN, "blasst_hand_cases.json")) as f:
        return json.load(f)


def _lam(case):
    return case["lambda"] if case.get("ln_lambda") is None else math.exp(case["ln_lambda"])


def _softmax_over(scores_row, keys):
    s = np.array([scores_row[c] for c in keys], dtype=np.float64)
    m = s.max()
    p = np.exp(s - m)
    return p / p.sum(), m + math.log(p.sum())


@pytest.mark.parametrize("fx", _hand_cases()["prefill"], ids=lambda f: f["name"])
def test_hand_prefill_cases(fx):
    S = np.array(fx["scores"], dtype=np.float32)
    T = fx["T"]
    q = np.eye(T, dtype=np.float32)[None, None]             # q_r = e_r
    k = np.ascontiguousarray(S.T)[None, None]                # key c = column c of S
    v = np.eye(T, dtype=np.float32)[None, None]              # v_c = e_c
    for case in fx["cases"]:
        r = oracle.prefill(q, k, v, 1.0, _lam(case), fx["Br"], fx["Bc"], fx["causal"])
        np.testing.assert_array_equal(r["skip"][0, 0], np.array(case["skip"]))
        np.testing.assert_allclose(r["margin"][0, 0], np.array(case["margin"]), atol=0)
        for row, keys in enumerate(case["kept"]):
            p, lse = _softmax_over(fx["scores"][row], keys)
            expect = np.zeros(T)
            expect[keys] = p
            np.testing.assert_allclose(r["o"][0, 0, row], expect, rtol=1e-13, atol=1e-15)
            assert abs(r["lse"][0, 0, row] - lse) < 1e-13
        for key, val in case.get("spot", {}).items():
            name, idx = key.split("[", 1)
            ix = tuple(int(x) for x in idx.replace("]", "").split("[") if x)
            got = r["o"][0, 0][ix] if name == "o" else r["lse"][0, 0][ix]
            assert abs(got - val) < 1e-13, key


@pytest.mark.parametrize("fx", _hand_cases()["decode"], ids=lambda f: f["name"])
def test_hand_decode_cases(fx):
    S = np.array(fx["scores"], dtype=np.float32)  # [G, L]
    G, L = S.shape
    q = np.eye(G, dtype=np.float32)[None]          # [1, G, dk=G]
    k = np.ascontiguousarray(S.T)[None, None]      # [1, 1, L, G]
    v = np.eye(L, dtype=np.float32)[None, None]    # [1, 1, L, L]
    for case in fx["cases"]:
        n = case["n_splits"]
        r = oracle.decode(q, k, v, 1.0, _lam(case), fx["Bc"], n)
        np.testing.assert_array_equal(r["skip"][0, 0], np.array(case["skip_positions"]))
        np.testing.assert_allclose(r["margin"][0, 0], np.array(case["margin"]), atol=0)
        o, lse = oracle.combine(r["o_part"], r["lse_part"])
        for h, keys in enumerate(case["kept"]):
            p, l_ = _softmax_over(fx["scores"][h], keys)
            expect = np.zeros(L)
            expect[keys] = p
            np.testing.assert_allclose(o[0, h], expect, rtol=1e-13, atol=1e-15)
            assert abs(lse[0, h] - l_) < 1e-13


# --------------------------------------------------------------------------
# Thresholded prefill: closed forms and invariants
# --------------------------------------------------------------------------

PREFILL_SHAPES = [
    # B, Hq, Hkv, T, d, Br, Bc, causal
    (1, 4, 2, 300, 16, 64, 64, True),    # several tiles and a ragged tail
    (2, 2, 2, 200, 8, 64, 32, True),     # Br != Bc: rows with no visible key in a block
    (1, 3, 1, 130, 8, 32, 64, False),    # non-causal, Br < Bc
]


@pytest.mark.parametrize("shape", PREFILL_SHAPES)
def test_prefill_lambda0_is_dense(shape):
    B, Hq, Hkv, T, d, Br, Bc, causal = shape
    q, k, v = rand_prefill(B, Hq, Hkv, T, d, seed=5, spread=1.5)
    r = oracle.prefill(q, k, v, 0.4, 0.0, Br, Bc, causal)
    yb, lseb, _ = brute_dense(q, k, v, 0.4, causal)
    assert not r["skip"].any()
    np.testing.assert_allclose(r["o"], yb, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(r["lse"], lseb, rtol=1e-12, atol=1e-12)


def _planted_small(T=512, d=32, Hq=4, Hkv=2, temperate=False, seed=11, band=0.0):
    cfg = W.PrefillConfig("t", 1, Hq, Hkv, T, d, "f32", Br=64, Bc=64, seed=seed, band_a=band)
    if temperate:
        cfg = W.temperate(cfg)
    q, k, v = W.prefill_inputs(cfg)
    return cfg, q.numpy(), k.numpy(), v.numpy()


@pytest.mark.parametrize("temperate", [False, True])
@pytest.mark.parametrize("lam", [1e-6, 1e-3, 3e-2])
def test_prefill_output_is_softmax_over_kept_tokens(temperate, lam):
    cfg, q, k, v = _planted_small(temperate=temperate)
    r = oracle.prefill(q, k, v, cfg.scale, lam, cfg.Br, cfg.Bc, True)
    s = scores_full(q, k, cfg.scale, True)
    km = kept_token_mask(r["skip"], cfg.T, cfg.Br, cfg.Bc, True)
    sk = np.where(km, s, -np.inf)
    p, lse = softmax_rows(sk)
    vv = np.repeat(v.astype(np.float64), cfg.G, axis=1)
    np.testing.assert_allclose(r["o"], np.einsum("bhrc,bhce->bhre", p, vv), rtol=1e-10,
                               atol=1e-11)
    np.testing.assert_allclose(r["lse"], lse, rtol=1e-12, atol=1e-11)


def _prefix_margins(s, T, Br, Bc, causal):
    """Brute-force tile statistic max_r(rowmax_j - max over blocks <= j) from the
    full score matrix: the running max after block j is the prefix max of all
    traversed scores, whatever was skipped."""
    B, Hq = s.shape[:2]
    n_t, n_b = -(-T // Br), -(-T // Bc)
    trav = visible_block_mask(T, Br, Bc, causal)
    out = np.full((B, Hq, n_t, n_b), np.nan)
    for t in range(n_t):
        rows = s[:, :, t * Br:min(T, (t + 1) * Br)]
        for j in range(n_b):
            if not trav[t, j]:
                continue
            blk = rows[..., j * Bc:min(T, (j + 1) * Bc)].max(-1)
            pre = rows[..., :min(T, (j + 1) * Bc)].max(-1)
            diff = np.where(np.isneginf(blk), -np.inf, blk - pre)
            out[:, :, t, j] = diff.max(-1)
    return out


@pytest.mark.parametrize("shape", PREFILL_SHAPES[:2])
def test_prefill_skip_bits_are_a_function_of_scores(shape):
    B, Hq, Hkv, T, d, Br, Bc, causal = shape
    q, k, v = rand_prefill(B, Hq, Hkv, T, d, seed=6, spread=2.0)
    s = scores_full(q, k, 0.5, causal)
    mu = _prefix_margins(s, T, Br, Bc, causal)
    for lam in (1e-4, 1e-2, 0.2):
        r = oracle.prefill(q, k, v, 0.5, lam, Br, Bc, causal)
        np.testing.assert_allclose(r["margin"], mu, rtol=0, atol=1e-12)
        expect = np.nan_to_num(mu, nan=np.inf) < math.log(lam)
        np.testing.assert_array_equal(r["skip"].astype(bool), expect)


@pytest.mark.parametrize("lam", [1e-4, 1e-2, 0.3])
def test_prefill_champion_block_never_skipped(lam):
    cfg, q, k, v = _planted_small(temperate=True, seed=12)
    r = oracle.prefill(q, k, v, cfg.scale, lam, cfg.Br, cfg.Bc, True)
    s = scores_full(q, k, cfg.scale, True)
    arg = s.argmax(-1)  # [B,Hq,T] key index of each row's global max
    for b in range(cfg.B):
        for h in range(cfg.Hq):
            for row in range(cfg.T):
                assert r["skip"][b, h, row // cfg.Br, arg[b, h, row] // cfg.Bc] == 0


def _skipped_token_weights(r, q, k, v, cfg, causal=True):
    _, _, p = brute_dense(q, k, v, cfg.scale, causal)
    s = scores_full(q, k, cfg.scale, causal)
    trav = visible_block_mask(cfg.T, cfg.Br, cfg.Bc, causal)
    skipped_blk = r["skip"].astype(bool) & trav[None, None]
    rows_t = np.arange(cfg.T) // cfg.Br
    cols_b = np.arange(cfg.T) // cfg.Bc
    sm = skipped_blk[:, :, rows_t][:, :, :, cols_b] & np.isfinite(s)
    return p, sm


@pytest.mark.parametrize("lam", [1e-5, 1e-3, 1e-2, 0.1])
def test_prefill_skipped_tokens_weigh_less_than_lambda(lam):
    cfg, q, k, v = _planted_small(temperate=True, seed=13)
    r = oracle.prefill(q, k, v, cfg.scale, lam, cfg.Br, cfg.Bc, True)
    p, sm = _skipped_token_weights(r, q, k, v, cfg)
    assert sm.any() or lam < 1e-3  # non-vacuous from 1e-3 up
    assert (p[sm] < lam).all()


@pytest.mark.parametrize("temperate", [False, True])
@pytest.mark.parametrize("lam", [1e-3, 1e-2, 0.1])
def test_prefill_error_bound(temperate, lam):
    """Appendix B: with delta the skipped softmax mass of a row, the output moves
    by delta * (y_kept - y_skipped), so |y_hat - y| <= 2 delta V_max, and
    delta < (#skipped tokens) * lambda <= |S| * Bc * lambda."""
    cfg, q, k, v = _planted_small(temperate=temperate, seed=14)
    r = oracle.prefill(q, k, v, cfg.scale, lam, cfg.Br, cfg.Bc, True)
    y, _, p = brute_dense(q, k, v, cfg.scale, True)
    _, sm = _skipped_token_weights(r, q, k, v, cfg)
    delta = np.where(sm, p, 0.0).sum(-1)
    n_skipped_blocks = r["skip"].sum(-1)[:, :, np.arange(cfg.T) // cfg.Br]
    vmax = np.linalg.norm(v.astype(np.float64), axis=-1).max()
    err = np.linalg.norm(r["o"] - y, axis=-1)
    assert (err <= 2 * delta * vmax * (1 + 1e-9) + 1e-12).all()
    assert (delta <= sm.sum(-1) * lam + 1e-15).all()
    assert (delta <= n_skipped_blocks * cfg.Bc * lam + 1e-15).all()


def test_worked_numbers_from_the_page():
    """lambda = 1e-3, Bc = 128: a skipped token weighs < 1e-3 and a skipped
    128-token block carries < 0.128 of its row's mass."""
    with open(os.path.join(GOLDEN, "blasst_worked_numbers.json")) as f:
        wn = json.load(f)
    assert wn["lambda"] * wn["Bc"] == pytest.approx(wn["max_block_mass"])
    cfg = W.TINY_PREFILL.with_(T=512, Bc=wn["Bc"], Br=128)
    q, k, v = (x.numpy() for x in W.prefill_inputs(cfg))
    r = oracle.prefill(q, k, v, cfg.scale, wn["lambda"], cfg.Br, cfg.Bc, True)
    p, sm = _skipped_token_weights(r, q, k, v, cfg)
    assert sm.any()
    assert p[sm].max() < wn["max_token_weight"]
    blk = np.where(sm, p, 0.0).reshape(1, 1, cfg.T, cfg.T // cfg.Bc, cfg.Bc).sum(-1)
    assert blk.max() < wn["max_block_mass"]


def test_prefill_unit_subset_matches_full():
    cfg, q, k, v = _planted_small(seed=15)
    full = oracle.prefill(q, k, v, cfg.scale, 1e-3, cfg.Br, cfg.Bc, True)
    units = [0, 5, 7, 8 * 3 + 7]  # flat (b, h, t) indices into [1, 4, 8]
    sub = oracle.prefill(q, k, v, cfg.scale, 1e-3, cfg.Br, cfg.Bc, True, units=units)
    for u in units:
        h, t = divmod(u, cfg.n_t)
        np.testing.assert_array_equal(sub["skip"][0, h, t], full["skip"][0, h, t])
        rs = slice(t * cfg.Br, (t + 1) * cfg.Br)
        np.testing.assert_array_equal(sub["o"][0, h, rs], full["o"][0, h, rs])


# --------------------------------------------------------------------------
# Split-KV decode and the merge
# --------------------------------------------------------------------------

def _small_decode(B=2, Hq=8, Hkv=2, L=1000, dk=32, dv=32, latent=False, temperate=False,
                  seed=21):
    cfg = W.DecodeConfig("t", B, Hq, Hkv, L, dk, dv, "f32", Bc=64, n_splits=4, latent=latent,
                         seed=seed)
    if temperate:
        cfg = W.temperate(cfg)
    q, k, v = W.decode_inputs(cfg)
    return cfg, q.numpy(), k.numpy(), (None if v is None else v.numpy())


@pytest.mark.parametrize("n_splits", [1, 3, 4, 16, 20])
def test_decode_lambda0_merged_is_dense(n_splits):
    cfg, q, k, v = _small_decode(temperate=True)
    r = oracle.decode(q, k, v, cfg.scale, 0.0, cfg.Bc, n_splits)
    o, lse = oracle.combine(r["o_part"], r["lse_part"])
    yb, lseb, _ = brute_dense(q[:, :, None], k, v, cfg.scale, False)
    np.testing.assert_allclose(o, yb[:, :, 0], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, lseb[:, :, 0], rtol=1e-12)
    assert not r["skip"].any()
    n_b = -(-cfg.L // cfg.Bc)
    empty = [s for s in range(n_splits) if (s * n_b) // n_splits == ((s + 1) * n_b) // n_splits]
    for s in empty:  # splits with no block: LSE -inf, zero output, zero weight in the merge
        assert np.isneginf(r["lse_part"][:, :, s]).all()
        assert not r["o_part"][:, :, s].any()


def test_combine_single_split_is_identity():
    g = np.random.default_rng(7)
    o_part = g.standard_normal((3, 5, 1, 9))
    lse_part = g.standard_normal((3, 5, 1)) * 10
    o, lse = oracle.combine(o_part, lse_part)
    np.testing.assert_array_equal(o, o_part[:, :, 0])
    np.testing.assert_array_equal(lse, lse_part[:, :, 0])


def test_combine_is_lse_weighted_mixture():
    g = np.random.default_rng(8)
    o_part = g.standard_normal((2, 3, 5, 7))
    lse_part = g.standard_normal((2, 3, 5)) * 20
    lse_part[0, 0, 2] = -np.inf
    o, lse = oracle.combine(o_part, lse_part)
    w = np.exp(lse_part - lse_part.max(-1, keepdims=True))
    np.testing.assert_allclose(lse, np.log(w.sum(-1)) + lse_part.max(-1), rtol=1e-13)
    np.testing.assert_allclose(o, (w[..., None] * o_part).sum(2) / w.sum(-1)[..., None],
                               rtol=1e-12, atol=1e-13)


def _decode_kept_mask(r, cfg, n_splits):
    """[B,Hq,L] True for tokens of kept blocks (per KV head, broadcast to its heads)."""
    n_b = -(-cfg.L // cfg.Bc)
    keep = np.ones((cfg.B, cfg.Hkv, n_b), dtype=bool)
    for s in range(n_splits):
        j0, j1 = s * n_b // n_splits, (s + 1) * n_b // n_splits
        keep[:, :, j0:j1] = ~r["skip"][:, :, s, :j1 - j0].astype(bool)
    tok = np.repeat(keep, cfg.Bc, axis=-1)[..., :cfg.L]
    return np.repeat(tok, cfg.G, axis=1)


@pytest.mark.parametrize("latent", [False, True])
@pytest.mark.parametrize("lam", [1e-4, 1e-2, 0.2])
def test_decode_closed_form_and_invariants(latent, lam):
    dv = 24 if latent else 32
    cfg, q, k, v = _small_decode(latent=latent, dv=dv, temperate=True, seed=22)
    vv = k[..., :dv].copy() if latent else v
    n_splits = 4
    r = oracle.decode(q, k, v, cfg.scale, lam, cfg.Bc, n_splits, dv=dv)
    o, lse = oracle.combine(r["o_part"], r["lse_part"])
    s = scores_full(q[:, :, None], k, cfg.scale, False)[:, :, 0]  # [B,Hq,L]
    km = _decode_kept_mask(r, cfg, n_splits)
    p_kept, lse_kept = softmax_rows(np.where(km, s, -np.inf))
    G = cfg.G
    vrep = np.repeat(vv.astype(np.float64), G, axis=1)
    # closed form: merged output is the softmax over the kept tokens
    np.testing.assert_allclose(o, np.einsum("bhc,bhce->bhe", p_kept, vrep), rtol=1e-10,
                               atol=1e-11)
    np.testing.assert_allclose(lse, lse_kept, rtol=1e-12, atol=1e-11)
    # every skipped token weighs < lambda against the dense normaliser
    p, _ = softmax_rows(s)
    assert (p[~km] < lam).all()
    # the block holding each head's global max is never skipped
    arg = s.argmax(-1)
    assert km[np.arange(cfg.B)[:, None], np.arange(cfg.Hq)[None, :], arg].all()
    # error bound
    y = np.einsum("bhc,bhce->bhe", p, vrep)
    delta = np.where(km, 0.0, p).sum(-1)
    vmax = np.linalg.norm(vv.astype(np.float64), axis=-1).max()
    assert (np.linalg.norm(o - y, axis=-1) <= 2 * delta * vmax * (1 + 1e-9) + 1e-12).all()


def test_decode_split_local_first_block_never_skipped():
    cfg, q, k, v = _small_decode(seed=23)
    for n_splits in (2, 5, 8):
        r = oracle.decode(q, k, v, cfg.scale, 0.5, cfg.Bc, n_splits)
        n_b = -(-cfg.L // cfg.Bc)
        for s in range(n_splits):
            if (s * n_b) // n_splits < ((s + 1) * n_b) // n_splits:
                assert (r["skip"][:, :, s, 0] == 0).all()
                assert (r["margin"][:, :, s, 0] == 0).all()


def test_decode_group_and_vote():
    """A block is skipped for a KV head only when all G heads of the group vote
    skip: recompute the per-head votes by brute force and AND them."""
    cfg, q, k, v = _small_decode(temperate=True, seed=24)
    n_splits, lam = 2, 0.05
    r = oracle.decode(q, k, v, cfg.scale, lam, cfg.Bc, n_splits)
    s = scores_full(q[:, :, None], k, cfg.scale, False)[:, :, 0]
    n_b = -(-cfg.L // cfg.Bc)
    for sp in range(n_splits):
        j0, j1 = sp * n_b // n_splits, (sp + 1) * n_b // n_splits
        for j in range(j0, j1):
            blk = s[..., j * cfg.Bc:min(cfg.L, (j + 1) * cfg.Bc)].max(-1)
            pre = s[..., j0 * cfg.Bc:min(cfg.L, (j + 1) * cfg.Bc)].max(-1)
            vote = (blk - pre) < math.log(lam)
            skip = vote.reshape(cfg.B, cfg.Hkv, cfg.G).all(-1)
            np.testing.assert_array_equal(r["skip"][:, :, sp, j - j0].astype(bool), skip)


# --------------------------------------------------------------------------
# Argument checks and generator determinism
# --------------------------------------------------------------------------

def test_oracle_rejects_bad_lambda():
    q, k, v = rand_prefill(1, 1, 1, 8, 4, seed=9)
    for lam in (-0.1, 1.0, float("nan")):
        with pytest.raises(ValueError):
            oracle.prefill(q, k, v, 1.0, lam, 4, 4, True)


def test_generator_is_deterministic_and_head_restricted_draw_matches():
    cfg = W.GQA_PREFILL_16K.with_(T=300, Hq=8, Hkv=4, seed=99)
    a = W.prefill_inputs(cfg)
    b = W.prefill_inputs(cfg)
    c = W.prefill_inputs(cfg, heads=[2])
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert torch.equal(a[1][:, 2], c[1][:, 2]) and torch.equal(a[2][:, 2], c[2][:, 2])
    assert torch.equal(a[0][:, 4:6], c[0][:, 4:6])
    assert a[0].dtype == torch.bfloat16
    dcfg = W.GQA_DECODE_32K.with_(B=3, L=256)
    d1, d2 = W.decode_inputs(dcfg), W.decode_inputs(dcfg, batches=[1])
    assert torch.equal(d1[1][1], d2[1][1]) and torch.equal(d1[0][1], d2[0][1])


def test_generator_plants_sink_and_salient_keys():
    cfg = W.GQA_PREFILL_16K.with_(T=2048, Hq=2, Hkv=1)
    q, k, v = (x.float() for x in W.prefill_inputs(cfg))
    u_dir = q[0, 0].mean(0)
    u_dir = u_dir / u_dir.norm()
    proj = k[0, 0] @ u_dir  # about a_j * sqrt(d) plus noise
    d = cfg.d
    assert proj[0] > 5 * math.sqrt(d)                        # sink, a_0 = 6
    n_sal = int(((proj > 2 * math.sqrt(d)) & (proj < 4 * math.sqrt(d))).sum())
    assert abs(n_sal - round(0.02 * (cfg.T - 1))) <= 3       # 2 % salient at a = 3


# --------------------------------------------------------------------------
# Explicit block sets (the SparDA page, section 2.1: an access set per query
# tile, composed with the threshold test inside it)
# --------------------------------------------------------------------------

def _random_block_set(B, Hq, T, Br, Bc, density, seed, drop_diagonal=False):
    g = np.random.default_rng(seed)
    n_t, n_b = -(-T // Br), -(-T // Bc)
    allow = g.random((B, Hq, n_t, n_b)) < density
    allow[..., 0] = True  # an "init" block
    if drop_diagonal:
        allow[:, :, 1, :] = False  # tile 1 selects nothing at all
    return allow.astype(np.uint8)


def test_block_set_all_ones_is_the_plain_loop():
    cfg, q, k, v = _planted_small(temperate=True, seed=21)
    allow = np.ones((1, cfg.Hq, cfg.n_t, cfg.n_b), dtype=np.uint8)
    for lam in (0.0, 1e-3):
        a = oracle.prefill(q, k, v, cfg.scale, lam, cfg.Br, cfg.Bc, True)
        b = oracle.prefill(q, k, v, cfg.scale, lam, cfg.Br, cfg.Bc, True, allow=allow)
        for key in ("o", "lse", "skip", "margin"):
            np.testing.assert_array_equal(a[key], b[key])


@pytest.mark.parametrize("lam", [0.0, 1e-4, 2e-2])
def test_block_set_output_is_softmax_over_selected_kept_tokens(lam):
    """Closed form: O is the softmax over the visible tokens of the selected,
    kept blocks; rows whose tile selected no visible key get O = 0, LSE = -inf;
    blocks outside the set are untraversed (bit 0, statistic NaN)."""
    cfg, q, k, v = _planted_small(temperate=True, seed=22)
    allow = _random_block_set(1, cfg.Hq, cfg.T, cfg.Br, cfg.Bc, 0.5, seed=5, drop_diagonal=True)
    r = oracle.prefill(q, k, v, cfg.scale, lam, cfg.Br, cfg.Bc, True, allow=allow)
    out = ~allow.astype(bool)
    assert (r["skip"][out] == 0).all() and np.isnan(r["margin"][out]).all()
    s = scores_full(q, k, cfg.scale, True)
    km = kept_token_mask(r["skip"], cfg.T, cfg.Br, cfg.Bc, True)
    sel = allow.astype(bool)[:, :, np.arange(cfg.T) // cfg.Br][:, :, :, np.arange(cfg.T) // cfg.Bc]
    km &= sel
    empty = ~km.any(axis=-1)
    assert empty[:, :, cfg.Br:2 * cfg.Br].all()  # the tile that selected nothing
    sk = np.where(km, s, -np.inf)
    with np.errstate(invalid="ignore", divide="ignore"):
        p, lse = softmax_rows(np.where(empty[..., None], 0.0, sk))
    vv = np.repeat(v.astype(np.float64), cfg.G, axis=1)
    want = np.einsum("bhrc,bhce->bhre", p, vv)
    want[empty] = 0.0
    lse[empty] = -np.inf
    np.testing.assert_allclose(r["o"], want, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(r["lse"], lse, rtol=1e-12, atol=1e-11)
    if lam > 0:  # every skipped selected block lies below ln(lambda)
        sk_ = r["skip"].astype(bool)
        assert (r["margin"][sk_] < np.log(lam)).all()


# --------------------------------------------------------------------------
# Per-head decode decisions (each query head of a GQA group decides alone)
# --------------------------------------------------------------------------

def _decode_kept_mask_per_head(r, cfg, n_splits):
    """[B,Hq,L] True for tokens of the blocks each head keeps."""
    n_b = -(-cfg.L // cfg.Bc)
    keep = np.ones((cfg.B, cfg.Hq, n_b), dtype=bool)
    for s in range(n_splits):
        j0, j1 = s * n_b // n_splits, (s + 1) * n_b // n_splits
        keep[:, :, j0:j1] = ~r["skip"][:, :, s, :j1 - j0].astype(bool)
    return np.repeat(keep, cfg.Bc, axis=-1)[..., :cfg.L]


def test_per_head_decode_with_one_head_per_group_is_the_group_decode():
    cfg, q, k, v = _small_decode(Hq=4, Hkv=4, temperate=True, seed=41)
    for lam in (0.0, 1e-2, 0.3):
        a = oracle.decode(q, k, v, cfg.scale, lam, cfg.Bc, 4)
        b = oracle.decode(q, k, v, cfg.scale, lam, cfg.Bc, 4, per_head=True)
        for key in ("o_part", "lse_part", "skip", "margin"):
            np.testing.assert_array_equal(a[key], b[key])


@pytest.mark.parametrize("lam", [1e-3, 5e-2, 0.3])
def test_per_head_decode_closed_form_and_group_relation(lam):
    """Merged output of each head = softmax over the tokens that head keeps;
    the group statistic is the max of its heads' statistics, so the group
    skips a block exactly when every head of it skips."""
    cfg, q, k, v = _small_decode(temperate=True, seed=42)
    n_splits = 4
    r = oracle.decode(q, k, v, cfg.scale, lam, cfg.Bc, n_splits, per_head=True)
    o, lse = oracle.combine(r["o_part"], r["lse_part"])
    s = scores_full(q[:, :, None], k, cfg.scale, False)[:, :, 0]
    km = _decode_kept_mask_per_head(r, cfg, n_splits)
    p_kept, lse_kept = softmax_rows(np.where(km, s, -np.inf))
    vrep = np.repeat(v.astype(np.float64), cfg.G, axis=1)
    np.testing.assert_allclose(o, np.einsum("bhc,bhce->bhe", p_kept, vrep), rtol=1e-10,
                               atol=1e-11)
    np.testing.assert_allclose(lse, lse_kept, rtol=1e-12, atol=1e-11)
    g = oracle.decode(q, k, v, cfg.scale, lam, cfg.Bc, n_splits)
    hm = r["margin"].reshape(cfg.B, cfg.Hkv, cfg.G, n_splits, -1)
    np.testing.assert_array_equal(np.nanmax(hm, axis=2), g["margin"])
    hs = r["skip"].reshape(cfg.B, cfg.Hkv, cfg.G, n_splits, -1).astype(bool)
    np.testing.assert_array_equal(hs.all(axis=2), g["skip"].astype(bool))
    assert hs.any(axis=2).sum() > hs.all(axis=2).sum()  # heads do disagree here
