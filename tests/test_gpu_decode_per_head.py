"""Split-KV decode with per-head decisions (each query head of a GQA group
decides for itself) on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_online_gb300 import binding as bs
from block_sparse_attention_online_gb300 import workloads as W
from tests.parity import check_outputs, compare_bits
from tests.test_gpu_decode import _lambda

pytestmark = pytest.mark.gpu


def check_per_head(cfg, q, k, v, lam, n_splits=None, units=None):
    n_splits = n_splits or cfg.n_splits
    dev = torch.device("cuda")
    op, lp, bits = bs.attn_skip_decode_per_head(q.to(dev), k.to(dev), v.to(dev), lam, cfg.Bc,
                                                n_splits)
    o, lse = bs.attn_skip_decode_combine(op, lp, torch.float32)
    bs.attn_skip_last_device_error()
    n_b = -(-cfg.L // cfg.Bc)
    bps = -(-n_b // n_splits)
    skip = bs.unpack_bits(bits, bps).numpy()
    r = oracle.decode(q, k, v, cfg.scale, lam, cfg.Bc, n_splits, per_head=True, units=units)
    sel = np.zeros((cfg.B, cfg.Hkv, n_splits), dtype=bool)
    if units is None:
        sel[:] = True
    else:
        sel.reshape(-1)[np.asarray(units)] = True
    hsel = np.repeat(sel, cfg.G, axis=1)  # [B,Hq,S]
    n_bad, flips = compare_bits(skip[hsel], r["skip"][hsel], r["margin"][hsel], lam)
    assert n_bad == 0, f"{n_bad} per-head skip bits differ outside the margin band"
    if flips.any():
        forced = np.zeros_like(r["skip"])
        forced[hsel] = skip[hsel]
        r = oracle.decode(q, k, v, cfg.scale, lam, cfg.Bc, n_splits, per_head=True, units=units,
                          force_skip=forced)
    ne = np.isfinite(r["lse_part"]) & hsel
    check_outputs(op.cpu().numpy()[ne], r["o_part"][ne], lp.cpu().numpy()[ne],
                  r["lse_part"][ne], "bf16", "o_part")
    if units is None:
        ro, rl = oracle.combine(r["o_part"], r["lse_part"])
        check_outputs(o.cpu().numpy(), ro, lse.cpu().numpy(), rl, "bf16", "merged")
    trav = np.isfinite(r["margin"][hsel])
    return float(skip[hsel][trav].mean())


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("L", [2048, 1999])
def test_per_head_small(G, L):
    cfg = W.temperate(W.GQA_DECODE_32K.with_(B=3, Hq=2 * G, Hkv=2, L=L, n_splits=4, seed=111))
    q, k, v = W.decode_inputs(cfg)
    for lam in (0.0, 1e-3, 0.2):
        check_per_head(cfg, q, k, v, lam)


def test_per_head_empty_splits():
    cfg = W.temperate(W.GQA_DECODE_32K.with_(B=2, L=1500, n_splits=20, seed=112))
    q, k, v = W.decode_inputs(cfg)
    check_per_head(cfg, q, k, v, 1e-2, 20)


def test_per_head_with_one_head_per_group_equals_group_decode():
    cfg = W.temperate(W.GQA_DECODE_32K.with_(B=2, Hq=4, Hkv=4, L=3000, n_splits=4, seed=113))
    q, k, v = W.decode_inputs(cfg)
    dev = torch.device("cuda")
    a = bs.attn_skip_decode_per_head(q.to(dev), k.to(dev), v.to(dev), 1e-2, cfg.Bc, 4)
    b = bs.attn_skip_decode(q.to(dev), k.to(dev), v.to(dev), 1e-2, cfg.Bc, 4)
    for x, y in zip(a, b):
        assert torch.equal(x.cpu(), y.cpu())


def test_per_head_full_size_sampled_and_group_is_and_of_heads():
    """B=16, 32/8 heads, L=32768, 8 splits at the group's ~70 % threshold:
    sampled units against the oracle, and over the whole launch the group
    call skips a block exactly when every head of the per-head call does."""
    cfg = W.GQA_DECODE_32K
    q, k, v = W.decode_inputs(cfg)
    lam = _lambda(cfg.name, "0.7")
    check_per_head(cfg, q, k, v, lam, units=[0, 9, 63, 300, 1023])
    dev = torch.device("cuda")
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    n_b = -(-cfg.L // cfg.Bc)
    bps = -(-n_b // cfg.n_splits)
    hb = bs.unpack_bits(bs.attn_skip_decode_per_head(dq, dk, dv, lam, cfg.Bc, cfg.n_splits)[2],
                        bps).numpy()
    gb = bs.unpack_bits(bs.attn_skip_decode(dq, dk, dv, lam, cfg.Bc, cfg.n_splits)[2],
                        bps).numpy()
    hb = hb.reshape(cfg.B, cfg.Hkv, cfg.G, cfg.n_splits, bps)
    np.testing.assert_array_equal(hb.all(axis=2), gb)
    assert hb.mean() > gb.mean()  # heads that would keep a block alone are rarer


def check_mla_per_head(cfg, q, k, lam):
    """Absorbed MLA (128 heads on one latent row, values = its first 512
    columns) with per-head decisions, against the oracle's per-head decode."""
    dev = torch.device("cuda")
    op, lp, bits = bs.attn_skip_decode_per_head(q.to(dev), k.to(dev), None, lam, cfg.Bc,
                                                cfg.n_splits, dv=cfg.dv)
    bs.attn_skip_last_device_error()
    n_b = -(-cfg.L // cfg.Bc)
    bps = -(-n_b // cfg.n_splits)
    skip = bs.unpack_bits(bits, bps).numpy()
    r = oracle.decode(q, k, None, cfg.scale, lam, cfg.Bc, cfg.n_splits, dv=cfg.dv,
                      per_head=True)
    n_bad, flips = compare_bits(skip, r["skip"], r["margin"], lam, label="mla per-head")
    assert n_bad == 0, f"{n_bad} per-head skip bits differ outside the margin band"
    if flips.any():
        r = oracle.decode(q, k, None, cfg.scale, lam, cfg.Bc, cfg.n_splits, dv=cfg.dv,
                          per_head=True, force_skip=skip)
    ne = np.isfinite(r["lse_part"])
    check_outputs(op.cpu().numpy()[ne], r["o_part"][ne], lp.cpu().numpy()[ne],
                  r["lse_part"][ne], "bf16", "mla o_part")
    trav = np.isfinite(r["margin"])
    return float(skip[trav].mean())


@pytest.mark.parametrize("lam", [0.0, 1e-3, 0.05])
def test_mla_per_head(lam):
    """Per-head decisions on the MLA shape: ragged last block, 4 splits; the
    per-head sparsity exceeds the group AND's on the same inputs."""
    cfg = W.temperate(W.MLA_DECODE_16K.with_(B=2, L=3000, n_splits=4, seed=171))
    q, k, _ = W.decode_inputs(cfg)
    sp = check_mla_per_head(cfg, q, k, lam)
    if lam > 0:
        dev = torch.device("cuda")
        _, _, gbits = bs.attn_skip_decode(q.to(dev), k.to(dev), None, lam, cfg.Bc, cfg.n_splits,
                                          dv=cfg.dv)
        n_b = -(-cfg.L // cfg.Bc)
        bps = -(-n_b // cfg.n_splits)
        gskip = bs.unpack_bits(gbits, bps).numpy()
        r = oracle.decode(q, k, None, cfg.scale, lam, cfg.Bc, cfg.n_splits, dv=cfg.dv)
        gsp = float(gskip[np.isfinite(r["margin"])].mean())
        assert sp >= gsp


def test_mla_per_head_empty_splits():
    """More splits than blocks: empty splits give LSE -inf and zero bitmap rows."""
    cfg = W.temperate(W.MLA_DECODE_16K.with_(B=1, L=300, n_splits=8, seed=172))
    q, k, _ = W.decode_inputs(cfg)
    check_mla_per_head(cfg, q, k, 1e-3)
