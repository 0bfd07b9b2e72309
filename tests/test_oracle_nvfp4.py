"""Pins of the NVFP4 key/value-cache decode oracle (CPU only).

The oracle decodes E2M1 codes from the format's bit fields, unpacks two codes
per byte, scales 16-element blocks by E4M3 codes, folds the per-(sequence, KV
head) key scale into the score scale and the value scale into the output.
Those steps are checked against routes the oracle does not take: the FP4
value table of the OCP Microscaling (MX) formats specification, the
generator's own packing, and brute-force fp64 attention over rows decoded
here from that table with non-power-of-two scales.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_online_gb300 import workloads as W
from tests.test_oracle import _decode_kept_mask, softmax_rows
from tests.test_oracle_fp8 import decoded as e4m3_decoded

# FP4 (E2M1) values of codes 0..15, as tabulated in the OCP Microscaling
# Formats (MX) specification v1.0 (section "FP4"): positive codes 0-7, then
# the same magnitudes negated (code 8 is -0).
FP4_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
             -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def table_rows(x4, bs8):
    """Rows decoded through FP4_TABLE (element 2i in the low nibble) and the
    E4M3 table of the FP8 pins."""
    x4 = np.asarray(x4, dtype=np.uint8)
    lo, hi = np.array(FP4_TABLE)[x4 & 0xF], np.array(FP4_TABLE)[x4 >> 4]
    el = np.stack([lo, hi], axis=-1).reshape(x4.shape[:-1] + (2 * x4.shape[-1],))
    return el * np.repeat(e4m3_decoded(np.asarray(bs8, dtype=np.uint8)), 16, axis=-1)


def test_e2m1_decoding_matches_the_mx_table():
    got = oracle.e2m1_decode(np.arange(16))
    assert (got == np.array(FP4_TABLE)).all()
    assert np.signbit(got[8]) and not np.signbit(got[0])


def _small(seed=41, L=1000, B=2, Hq=8, Hkv=2, d=32):
    cfg = W.temperate(W.GQA_DECODE_32K.with_(B=B, Hq=Hq, Hkv=Hkv, L=L, dk=d, dv=d, seed=seed))
    g = np.random.default_rng(seed)
    q, _, _ = W.decode_inputs(cfg)
    k4 = g.integers(0, 256, size=(B, Hkv, L, d // 2), dtype=np.uint8)
    v4 = g.integers(0, 256, size=(B, Hkv, L, d // 2), dtype=np.uint8)
    kbs = g.integers(0, 0x7E, size=(B, Hkv, L, d // 16), dtype=np.uint8)  # positive, finite
    vbs = g.integers(0, 0x7E, size=(B, Hkv, L, d // 16), dtype=np.uint8)
    ks = g.uniform(0.001, 0.02, size=(B, Hkv)).astype(np.float32)  # not powers of two
    vs = g.uniform(0.5, 3.0, size=(B, Hkv)).astype(np.float32)
    return cfg, q, k4, v4, kbs, vbs, ks, vs


def _brute(cfg, q, k4, v4, kbs, vbs, ks, vs):
    kd = table_rows(k4, kbs) * ks.astype(np.float64)[:, :, None, None]
    vd = table_rows(v4, vbs) * vs.astype(np.float64)[:, :, None, None]
    kd, vd = np.repeat(kd, cfg.G, axis=1), np.repeat(vd, cfg.G, axis=1)
    s = cfg.scale * np.einsum("bhd,bhcd->bhc", q.double().numpy(), kd)
    return s, vd


@pytest.mark.parametrize("n_splits", [1, 3, 8])
def test_nvfp4_decode_lambda0_is_scaled_dense_attention(n_splits):
    cfg, q, k4, v4, kbs, vbs, ks, vs = _small()
    r = oracle.decode_nvfp4(q, k4, v4, kbs, vbs, ks, vs, cfg.scale, 0.0, cfg.Bc, n_splits)
    o, lse = oracle.combine(r["o_part"], r["lse_part"])
    s, vd = _brute(cfg, q, k4, v4, kbs, vbs, ks, vs)
    p, lse_b = softmax_rows(s)
    np.testing.assert_allclose(o, np.einsum("bhc,bhce->bhe", p, vd), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(lse, lse_b, rtol=1e-12, atol=1e-10)
    assert r["skip"].sum() == 0


@pytest.mark.parametrize("lam", [1e-4, 1e-2, 0.2])
def test_nvfp4_decode_output_is_softmax_over_kept_tokens(lam):
    cfg = W.temperate(W.GQA_DECODE_NVFP4_32K.with_(B=2, Hq=8, Hkv=2, L=3000, dk=32, dv=32,
                                                   seed=42))
    q, k4, v4, kbs, vbs, ks, vs = (x.numpy() if i else x for i, x in
                                   enumerate(W.decode_inputs_nvfp4(cfg)))
    n_splits = 3
    r = oracle.decode_nvfp4(q, k4, v4, kbs, vbs, ks, vs, cfg.scale, lam, cfg.Bc, n_splits)
    o, lse = oracle.combine(r["o_part"], r["lse_part"])
    s, vd = _brute(cfg, q, k4, v4, kbs, vbs, ks, vs)
    km = _decode_kept_mask(r, cfg, n_splits)
    p, lse_k = softmax_rows(np.where(km, s, -np.inf))
    np.testing.assert_allclose(o, np.einsum("bhc,bhce->bhe", p, vd), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(lse, lse_k, rtol=1e-12, atol=1e-10)
    pd, _ = softmax_rows(s)
    assert (pd[~km] < lam).all()


def test_nvfp4_generator_rows_lie_within_half_an_e2m1_step():
    """Dequantised rows (oracle route) against the bf16 draws: each element
    within half the E2M1 grid spacing at its magnitude (0.5 below 2, 1 up to 4,
    2 up to 6) times its block's scale, none past the grid; block scales are
    E4M3 codes of at most 448 and every (sequence, KV head) slice reaches the
    upper part of the grid."""
    cfg = W.GQA_DECODE_NVFP4_32K.with_(B=2, L=700)
    q, k4, v4, kbs, vbs, ks, vs = W.decode_inputs_nvfp4(cfg)
    _, k, v = W.decode_inputs(cfg)
    for x4, bs, sc, x in ((k4, kbs, ks, k), (v4, vbs, vs, v)):
        rows = oracle.nvfp4_rows(x4.numpy(), bs.numpy()).astype(np.float64)
        unit = np.repeat(e4m3_decoded(bs.numpy()), 16, axis=-1) * sc.double().numpy()[:, :, None, None]
        xr = x.double().numpy()
        y = np.abs(xr) / unit
        half = np.where(y < 2, 0.25, np.where(y < 4, 0.5, 1.0))
        err = np.abs(rows * sc.double().numpy()[:, :, None, None] - xr)
        # block scales are rounded up: no element exceeds the grid (up to the
        # fp32 rounding of x / unit in the generator)
        assert (y <= 6.0 * (1 + 1e-6)).all()
        # the generator rounds x / unit computed in fp32: a tie there may sit
        # 1e-7 off the tie in fp64
        assert (err <= half * unit * (1 + 1e-6)).all()
        assert (e4m3_decoded(bs.numpy()) <= 448).all()
        assert (np.abs(table_rows(x4.numpy(), bs.numpy())).max(axis=(2, 3)) >= 6 * 224).all()
