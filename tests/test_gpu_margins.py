"""Statistics mode (one-pass threshold calibration) on the GPU against the fp64
oracle's block statistic max_r(rowmax - m_new), and its consistency with the
skip bitmaps of ordinary runs (section "校准算法：一次前向，一个指数模型")."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_online_gb300 import binding as bs
from block_sparse_attention_online_gb300 import workloads as W
from tests.parity import MARGIN_BAND

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
# fp32 scores from the same bf16 inputs: the statistic agrees to well under
# the margin band used for the bitmaps.
TOL = {"bf16": 1e-3, "f32": 1e-4}


def _lambda(cfg_name, target):
    with open(os.path.join(GOLDEN, "lambdas.json")) as f:
        return json.load(f)[cfg_name][str(target)]["lambda"]


def _compare(g, r, dtype, sel=None):
    """Same NaN (not traversed) and -inf patterns; finite values within TOL."""
    if sel is not None:
        g, r = g[sel], r[sel]
    assert (np.isnan(g) == np.isnan(r)).all(), "traversal pattern differs"
    assert (np.isneginf(g) == np.isneginf(r)).all(), "-inf pattern differs"
    fin = np.isfinite(r)
    err = np.abs(g[fin] - r[fin]).max() if fin.any() else 0.0
    assert err <= TOL[dtype], f"statistic max-abs error {err}"


def _prefill_margins(q, k, Br=128, Bc=128, causal=True):
    dev = torch.device("cuda")
    m = bs.attn_skip_prefill_margins(q.to(dev), k.to(dev), Br, Bc, causal)
    bs.attn_skip_last_device_error()
    return m.cpu().numpy()


def test_prefill_f32_tiny_margins():
    cfg = W.temperate(W.TINY_PREFILL.with_(seed=81))
    q, k, v = W.prefill_inputs(cfg)
    for Br, Bc in ((128, 128), (64, 128), (128, 64)):
        g = _prefill_margins(q, k, Br, Bc)
        r = oracle.prefill(q, k, v, cfg.scale, 0.0, Br, Bc, True)["margin"]
        _compare(g, r, "f32")


@pytest.mark.parametrize("T", [640, 1000])
def test_prefill_tc_margins(T):
    cfg = W.temperate(W.GQA_PREFILL_16K.with_(B=1, Hq=4, Hkv=2, T=T, seed=82))
    q, k, v = W.prefill_inputs(cfg)
    g = _prefill_margins(q, k)
    r = oracle.prefill(q, k, v, cfg.scale, 0.0, 128, 128, True)["margin"]
    _compare(g, r, "bf16")


def test_prefill_tc_margins_noncausal_ragged():
    cfg = W.temperate(W.GQA_PREFILL_16K.with_(B=1, Hq=2, Hkv=1, T=700, seed=83))
    q, k, v = W.prefill_inputs(cfg)
    g = _prefill_margins(q, k, causal=False)
    r = oracle.prefill(q, k, v, cfg.scale, 0.0, 128, 128, False)["margin"]
    _compare(g, r, "bf16")


def test_prefill_margins_full_size_match_bitmap_and_calibrate():
    """T=16384: sampled tiles against the oracle; every traversed bit of a run
    at the ~70 % threshold is {statistic < ln lambda} outside the margin band;
    a lambda computed from the statistics for a 70 % target reaches it."""
    cfg = W.GQA_PREFILL_16K
    q, k, v = W.prefill_inputs(cfg)
    g = _prefill_margins(q, k)
    units = sorted({h * cfg.n_t + t for h in (3, 17) for t in (0, 1, cfg.n_t // 2, cfg.n_t - 1)})
    r = oracle.prefill(q, k, v, cfg.scale, 0.0, 128, 128, True, units=units)["margin"]
    sel = np.zeros(g.shape[:3], dtype=bool)
    sel.reshape(-1)[units] = True
    _compare(g, r, "bf16", sel)

    dev = torch.device("cuda")
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    lam = _lambda(cfg.name, "0.7")
    _, _, bits = bs.attn_skip_prefill(dq, dk, dv, lam, 128, 128, True)
    skip = bs.unpack_bits(bits, cfg.n_t).numpy()
    trav = ~np.isnan(g)
    pred = g < math.log(lam)
    near = np.abs(g - math.log(lam)) < MARGIN_BAND
    assert ((pred == skip) | near | ~trav).all()

    lam70 = bs.attn_skip_lambda_for_sparsity(g, 0.7)
    _, _, bits = bs.attn_skip_prefill(dq, dk, dv, lam70, 128, 128, True)
    got = bs.unpack_bits(bits, cfg.n_t).numpy()[trav].mean()
    assert abs(got - 0.7) < 0.005, got


def _decode_margins(q, k, Bc, n_splits):
    dev = torch.device("cuda")
    m = bs.attn_skip_decode_margins(q.to(dev), k.to(dev), Bc, n_splits)
    bs.attn_skip_last_device_error()
    return m.cpu().numpy()


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("L,n_splits", [(2048, 4), (1999, 3), (1500, 20)])
def test_decode_margins(G, L, n_splits):
    cfg = W.temperate(W.GQA_DECODE_32K.with_(B=2, Hq=2 * G, Hkv=2, L=L, n_splits=n_splits,
                                             seed=84))
    q, k, v = W.decode_inputs(cfg)
    g = _decode_margins(q, k, cfg.Bc, n_splits)
    r = oracle.decode(q, k, v, cfg.scale, 0.0, cfg.Bc, n_splits)["margin"]
    _compare(g, r, "bf16")


def test_decode_margins_full_size_match_bitmap():
    cfg = W.GQA_DECODE_32K
    q, k, v = W.decode_inputs(cfg)
    g = _decode_margins(q, k, cfg.Bc, cfg.n_splits)
    units = [0, 5, 63, 64 * 7 + 3, 127]  # flat (b, hk, split) units
    r = oracle.decode(q, k, v, cfg.scale, 0.0, cfg.Bc, cfg.n_splits, units=units)["margin"]
    sel = np.zeros(g.shape[:3], dtype=bool)
    sel.reshape(-1)[units] = True
    _compare(g, r, "bf16", sel)
    lam = _lambda(cfg.name, "0.7")
    dev = torch.device("cuda")
    _, _, bits = bs.attn_skip_decode(q.to(dev), k.to(dev), v.to(dev), lam, cfg.Bc, cfg.n_splits)
    n_b = -(-cfg.L // cfg.Bc)
    skip = bs.unpack_bits(bits, -(-n_b // cfg.n_splits)).numpy()
    trav = ~np.isnan(g)
    near = np.abs(g - math.log(lam)) < MARGIN_BAND
    assert (((g < math.log(lam)) == skip) | near | ~trav).all()


@pytest.mark.parametrize("L,n_splits", [(1000, 4), (200, 6)])
def test_mla_margins(L, n_splits):
    cfg = W.MLA_DECODE_16K.with_(B=2, L=L, n_splits=n_splits, seed=85)
    q, k, _ = W.decode_inputs(cfg)
    g = _decode_margins(q, k, cfg.Bc, n_splits)
    r = oracle.decode(q, k, None, cfg.scale, 0.0, cfg.Bc, n_splits, dv=cfg.dv)["margin"]
    _compare(g, r, "bf16")
