"""Split-KV decode + LSE merge on the GPU against the fp64 oracle."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_online_gb300 import binding as bs
from block_sparse_attention_online_gb300 import workloads as W
from tests.parity import check_outputs, compare_bits

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _lambda(cfg_name, target):
    with open(os.path.join(GOLDEN, "lambdas.json")) as f:
        return json.load(f)[cfg_name][str(target)]["lambda"]


def run_decode(cfg, q, k, v, lam, n_splits=None, units=None):
    n_splits = n_splits or cfg.n_splits
    dev = torch.device("cuda")
    op, lp, bits = bs.attn_skip_decode(q.to(dev), k.to(dev), None if v is None else v.to(dev),
                                       lam, cfg.Bc, n_splits, dv=cfg.dv)
    o, lse = bs.attn_skip_decode_combine(op, lp, torch.bfloat16)
    bs.attn_skip_last_device_error()
    n_b = -(-cfg.L // cfg.Bc)
    bps = -(-n_b // n_splits)
    return dict(o_part=op.cpu().numpy(), lse_part=lp.cpu().numpy(),
                skip=bs.unpack_bits(bits, bps).numpy(), o=o.float().cpu().numpy(),
                lse=lse.cpu().numpy())


def check_decode(cfg, q, k, v, lam, n_splits=None):
    n_splits = n_splits or cfg.n_splits
    g = run_decode(cfg, q, k, v, lam, n_splits)
    r = oracle.decode(q, k, v, cfg.scale, lam, cfg.Bc, n_splits, dv=cfg.dv)
    n_bad, flips = compare_bits(g["skip"], r["skip"], r["margin"], lam)
    assert n_bad == 0, f"{n_bad} skip bits differ outside the margin band"
    if flips.any():
        r = oracle.decode(q, k, v, cfg.scale, lam, cfg.Bc, n_splits, dv=cfg.dv,
                          force_skip=g["skip"].astype(np.uint8))
    ro, rl = oracle.combine(r["o_part"], r["lse_part"])
    # partials of non-empty splits
    ne = np.isfinite(r["lse_part"])
    assert (np.isneginf(g["lse_part"]) == ~ne).all()
    check_outputs(g["o_part"][ne], r["o_part"][ne], g["lse_part"][ne], r["lse_part"][ne],
                  "bf16", "o_part")
    check_outputs(g["o"], ro, g["lse"], rl, "bf16", "merged")
    trav = np.isfinite(r["margin"])
    return float(g["skip"][trav].mean()), int(flips.sum())


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("L", [2048, 1999])
def test_decode_small(G, L):
    cfg = W.GQA_DECODE_32K.with_(B=3, Hq=2 * G, Hkv=2, L=L, n_splits=4, seed=31)
    q, k, v = W.decode_inputs(cfg)
    for lam in (0.0, 1e-12, 1e-9):
        check_decode(cfg, q, k, v, lam)


@pytest.mark.parametrize("n_splits", [1, 3, 20])
def test_decode_split_counts_and_empty_splits(n_splits):
    cfg = W.GQA_DECODE_32K.with_(B=2, L=1500, n_splits=n_splits, seed=32)
    q, k, v = W.decode_inputs(cfg)
    check_decode(cfg, q, k, v, 1e-10, n_splits)


@pytest.mark.parametrize("L", [1, 127, 129])
@pytest.mark.parametrize("n_splits", [1, 4])
def test_decode_shortest_caches(L, n_splits):
    """A cache of one key, one ragged block, and one key past a block; with
    four splits some splits own no block (LSE -inf, O 0, merged away)."""
    cfg = W.GQA_DECODE_32K.with_(B=3, L=L, seed=66)
    q, k, v = W.decode_inputs(cfg)
    for lam in (0.0, 0.5):
        check_decode(cfg, q, k, v, lam, n_splits)


@pytest.mark.parametrize("lam", [1e-3, 1e-2, 0.2, 0.999])
def test_decode_temperate_mixtures(lam):
    cfg = W.temperate(W.GQA_DECODE_32K.with_(B=2, L=4096, seed=33))
    q, k, v = W.decode_inputs(cfg)
    check_decode(cfg, q, k, v, lam)


@pytest.mark.parametrize("target", ["0.0", "0.7"])
def test_decode_full_size(target):
    """B=16, 32/8 heads, L=32768, 8 splits: the configuration the benchmark times."""
    cfg = W.GQA_DECODE_32K
    q, k, v = W.decode_inputs(cfg)
    lam = 0.0 if target == "0.0" else _lambda(cfg.name, target)
    sparsity, flips = check_decode(cfg, q, k, v, lam)
    if target == "0.7":
        assert 0.6 <= sparsity <= 0.8, sparsity
