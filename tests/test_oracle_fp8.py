"""Pins of the FP8 (E4M3) key/value-cache decode oracle (CPU only).

The oracle decodes E4M3 codes through torch and folds the per-(sequence, KV
head) key scale into the score scale and the value scale into the output.
Those steps are checked against routes the oracle does not take: a bit-level
E4M3 decoder written from the format's definition, and brute-force fp64
attention over rows dequantised here with non-power-of-two scales.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_online_gb300 import workloads as W
from tests.test_oracle import _decode_kept_mask, softmax_rows


def e4m3_value(code: int) -> float:
    """E4M3 (bias 7, no infinities, S.1111.111 = NaN) from its bits."""
    s = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def decoded(codes: np.ndarray) -> np.ndarray:
    table = np.array([e4m3_value(c) for c in range(256)])
    return table[codes]


def test_e4m3_decoding_matches_the_format_definition():
    codes = torch.arange(256, dtype=torch.uint8)
    got = codes.view(torch.float8_e4m3fn).double().numpy()
    want = decoded(np.arange(256))
    nan = np.isnan(want)
    assert (np.isnan(got) == nan).all() and nan.sum() == 2
    assert (got[~nan] == want[~nan]).all()
    assert want[0x7E] == 448.0 and want[0x01] == 2.0 ** -9


def _small(seed=31, L=1000, B=2, Hq=8, Hkv=2, d=32, temperate=True):
    cfg = W.GQA_DECODE_32K.with_(B=B, Hq=Hq, Hkv=Hkv, L=L, dk=d, dv=d, seed=seed)
    if temperate:
        cfg = W.temperate(cfg)
    g = np.random.default_rng(seed)
    q, _, _ = W.decode_inputs(cfg)
    k8 = g.integers(0, 256, size=(B, Hkv, L, d), dtype=np.uint8)
    v8 = g.integers(0, 256, size=(B, Hkv, L, d), dtype=np.uint8)
    k8[(k8 & 0x7F) == 0x7F] ^= 1  # no NaN codes
    v8[(v8 & 0x7F) == 0x7F] ^= 1
    ks = g.uniform(0.001, 0.02, size=(B, Hkv)).astype(np.float32)  # not powers of two
    vs = g.uniform(0.5, 3.0, size=(B, Hkv)).astype(np.float32)
    return cfg, q, k8, v8, ks, vs


def _brute(cfg, q, k8, v8, ks, vs):
    """Scaled fp64 scores [B,Hq,L] of the given query against rows
    dequantised here (bit-level decoder times the scale), and the
    dequantised values [B,Hq,L,d]."""
    kd = decoded(k8) * ks.astype(np.float64)[:, :, None, None]
    vd = decoded(v8) * vs.astype(np.float64)[:, :, None, None]
    kd, vd = np.repeat(kd, cfg.G, axis=1), np.repeat(vd, cfg.G, axis=1)
    s = cfg.scale * np.einsum("bhd,bhcd->bhc", q.double().numpy(), kd)
    return s, vd


@pytest.mark.parametrize("n_splits", [1, 3, 8])
def test_fp8_decode_lambda0_is_scaled_dense_attention(n_splits):
    cfg, q, k8, v8, ks, vs = _small()
    r = oracle.decode_fp8(q, k8, v8, ks, vs, cfg.scale, 0.0, cfg.Bc, n_splits)
    o, lse = oracle.combine(r["o_part"], r["lse_part"])
    s, vd = _brute(cfg, q, k8, v8, ks, vs)
    p, lse_b = softmax_rows(s)
    np.testing.assert_allclose(o, np.einsum("bhc,bhce->bhe", p, vd), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(lse, lse_b, rtol=1e-12, atol=1e-10)
    assert r["skip"].sum() == 0


@pytest.mark.parametrize("lam", [1e-4, 1e-2, 0.2])
def test_fp8_decode_output_is_softmax_over_kept_tokens(lam):
    """Planted inputs quantised with scales amax / 448 (not powers of two)."""
    cfg = W.temperate(W.GQA_DECODE_FP8_32K.with_(B=2, Hq=8, Hkv=2, L=3000, dk=32, dv=32,
                                                 seed=32))
    q, k8, v8, ks, vs = W.decode_inputs_fp8(cfg, pow2_scales=False)
    k8, v8, ks, vs = k8.numpy(), v8.numpy(), ks.numpy(), vs.numpy()
    n_splits = 3
    r = oracle.decode_fp8(q, k8, v8, ks, vs, cfg.scale, lam, cfg.Bc, n_splits)
    o, lse = oracle.combine(r["o_part"], r["lse_part"])
    s, vd = _brute(cfg, q, k8, v8, ks, vs)
    km = _decode_kept_mask(r, cfg, n_splits)
    p, lse_k = softmax_rows(np.where(km, s, -np.inf))
    np.testing.assert_allclose(o, np.einsum("bhc,bhce->bhe", p, vd), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(lse, lse_k, rtol=1e-12, atol=1e-10)
    assert r["skip"].sum() > 0 or lam < 1e-3  # a weak threshold may skip nothing here
    pd, _ = softmax_rows(s)
    assert (pd[~km] < lam).all()


def test_fp8_generator_quantises_within_half_a_step():
    cfg = W.GQA_DECODE_FP8_32K.with_(B=2, L=700)
    q, k8, v8, ks, vs = W.decode_inputs_fp8(cfg)
    _, k, v = W.decode_inputs(cfg)
    for x8, sc, x in ((k8, ks, k), (v8, vs, v)):
        xd = decoded(x8.numpy()) * sc.double().numpy()[:, :, None, None]
        xr = x.double().numpy()
        # E4M3 keeps 3 fraction bits: a relative step of 2^-3 for normals, an
        # absolute step of 2^-9 * scale below 2^-6 * scale
        step = np.maximum(np.abs(xr) * 2.0 ** -3, 2.0 ** -9 * sc.double().numpy()[:, :, None, None])
        assert (np.abs(xd - xr) <= 0.5 * step * (1 + 1e-12)).all()
        # power-of-two scales and the upper half of the code range used
        lg = np.log2(sc.double().numpy())
        assert (lg == np.round(lg)).all()
        amax = np.abs(decoded(x8.numpy())).max(axis=(2, 3))
        assert (amax >= 224).all() and (amax <= 448).all()
