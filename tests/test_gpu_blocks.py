"""Prefill restricted to an explicit block set per query tile (the SparDA page,
section 2.1: an access set such as B_init u B_local u B_topk), composed with the
threshold test, on the GPU against the fp64 oracle."""
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


def random_set(B, Hq, n_t, n_b, density, seed, empty_tile=None):
    g = np.random.default_rng(seed)
    allow = g.random((B, Hq, n_t, n_b)) < density
    allow[..., 0] = True
    if empty_tile is not None:
        allow[:, :, empty_tile, :] = False
    return allow


def infllm_set(B, Hq, n_t, n_b, topk, seed):
    """B_init (block 0) u B_local (the tile's diagonal block and the one before)
    u B_topk (topk blocks drawn at random among the rest of the causal range)."""
    g = np.random.default_rng(seed)
    allow = np.zeros((B, Hq, n_t, n_b), dtype=bool)
    allow[..., 0] = True
    for t in range(n_t):
        allow[:, :, t, t] = True
        if t > 0:
            allow[:, :, t, t - 1] = True
        rest = np.arange(1, max(t - 1, 1))
        if rest.size:
            for b in range(B):
                for h in range(Hq):
                    allow[b, h, t, g.choice(rest, min(topk, rest.size), replace=False)] = True
    return allow


def run_blocks(q, k, v, lam, allow, Br, Bc, causal=True):
    dev = torch.device("cuda")
    words = bs.pack_block_set(torch.from_numpy(allow)).to(dev)
    o, lse, bits = bs.attn_skip_prefill_blocks(q.to(dev), k.to(dev), v.to(dev), lam, words, Br,
                                               Bc, causal)
    bs.attn_skip_last_device_error()
    return o.float().cpu().numpy(), lse.cpu().numpy(), bits


def check_blocks(cfg, q, k, v, lam, allow, kind, Br=128, Bc=128, units=None, causal=True):
    o, lse, bits = run_blocks(q, k, v, lam, allow, Br, Bc, causal)
    n_t, n_b = -(-cfg.T // Br), -(-cfg.T // Bc)
    skip = bs.unpack_bits(bits, n_b).numpy()
    r = oracle.prefill(q, k, v, cfg.scale, lam, Br, Bc, causal, units=units, allow=allow)
    sel = np.zeros((cfg.B, cfg.Hq, n_t), dtype=bool)
    if units is None:
        sel[:] = True
    else:
        sel.reshape(-1)[np.asarray(units)] = True
    assert not (skip[sel] & ~allow[sel]).any(), "a block outside the set reads skipped"
    n_bad, flips = compare_bits(skip[sel], r["skip"][sel], r["margin"][sel], lam)
    assert n_bad == 0, f"{n_bad} skip bits differ outside the margin band"
    if flips.any():
        forced = np.zeros_like(r["skip"])
        forced[sel] = skip[sel]
        r = oracle.prefill(q, k, v, cfg.scale, lam, Br, Bc, causal, units=units,
                           force_skip=forced, allow=allow)
    rows = np.repeat(sel, Br, axis=2)[:, :, :cfg.T]
    empty = np.isneginf(r["lse"]) & rows
    assert (np.isneginf(lse) == np.isneginf(r["lse"]))[rows].all()
    assert (o[empty] == 0).all()
    live = rows & ~empty
    check_outputs(o[live], r["o"][live], lse[live], r["lse"][live], kind, "blocks")
    return int(flips.sum())


def test_blocks_f32_tiny():
    cfg = W.temperate(W.TINY_PREFILL.with_(seed=101))
    q, k, v = W.prefill_inputs(cfg)
    for Br, Bc in ((128, 128), (64, 64)):
        n_t, n_b = -(-cfg.T // Br), -(-cfg.T // Bc)
        allow = random_set(1, 1, n_t, n_b, 0.5, seed=Br, empty_tile=2)
        for lam in (0.0, 1e-3, 1e-1):
            check_blocks(cfg, q, k, v, lam, allow, "f32", Br, Bc)


@pytest.mark.parametrize("T", [640, 1000])
def test_blocks_tc_random_sets(T):
    cfg = W.temperate(W.GQA_PREFILL_16K.with_(B=2, Hq=4, Hkv=2, T=T, seed=102))
    q, k, v = W.prefill_inputs(cfg)
    allow = random_set(cfg.B, cfg.Hq, cfg.n_t, cfg.n_b, 0.5, seed=T, empty_tile=1)
    for lam in (0.0, 1e-3, 0.3):
        check_blocks(cfg, q, k, v, lam, allow, "bf16")


def test_blocks_tc_noncausal():
    cfg = W.temperate(W.GQA_PREFILL_16K.with_(B=1, Hq=2, Hkv=1, T=700, seed=103))
    q, k, v = W.prefill_inputs(cfg)
    allow = random_set(cfg.B, cfg.Hq, cfg.n_t, cfg.n_b, 0.4, seed=9)
    check_blocks(cfg, q, k, v, 1e-2, allow, "bf16", causal=False)


def test_blocks_all_ones_equal_plain_prefill_bitwise():
    cfg = W.temperate(W.GQA_PREFILL_16K.with_(B=1, Hq=4, Hkv=2, T=1000, seed=104))
    q, k, v = W.prefill_inputs(cfg)
    dev = torch.device("cuda")
    allow = np.ones((cfg.B, cfg.Hq, cfg.n_t, cfg.n_b), dtype=bool)
    o1, l1, b1 = run_blocks(q, k, v, 1e-2, allow, 128, 128)
    o2, l2, b2 = bs.attn_skip_prefill(q.to(dev), k.to(dev), v.to(dev), 1e-2, 128, 128, True)
    np.testing.assert_array_equal(o1, o2.float().cpu().numpy())
    np.testing.assert_array_equal(l1, l2.cpu().numpy())
    assert torch.equal(b1.cpu(), b2.cpu())


def test_blocks_full_size_infllm_like_set():
    """T=16384, 32/8 heads: init + local + 8 random top-k blocks per tile at the
    ~70 % threshold, sampled tiles against the oracle."""
    cfg = W.GQA_PREFILL_16K
    q, k, v = W.prefill_inputs(cfg)
    allow = infllm_set(cfg.B, cfg.Hq, cfg.n_t, cfg.n_b, 8, seed=105)
    units = sorted({h * cfg.n_t + t for h in (2, 29) for t in (0, 1, 2, 70, cfg.n_t - 1)})
    check_blocks(cfg, q, k, v, _lambda(cfg.name, "0.7"), allow, "bf16", units=units)


def test_blocks_tc_many_tiles_per_cta():
    """1024 (b, h, t) tiles, several waves of CTAs per SM: random sets with a
    fifth of the tiles empty (their CTAs issue no key load), sampled tiles
    against the oracle, and every empty tile's rows O = 0, LSE = -inf."""
    cfg = W.temperate(W.GQA_PREFILL_16K.with_(B=2, Hq=32, Hkv=8, T=2048, seed=106))
    q, k, v = W.prefill_inputs(cfg)
    allow = random_set(cfg.B, cfg.Hq, cfg.n_t, cfg.n_b, 0.3, seed=106)
    g = np.random.default_rng(107)
    empty = g.random((cfg.B, cfg.Hq, cfg.n_t)) < 0.2
    allow[empty] = False
    units = sorted(int(u) for u in g.choice(cfg.B * cfg.Hq * cfg.n_t, 48, replace=False))
    for lam in (0.0, 1e-3):
        check_blocks(cfg, q, k, v, lam, allow, "bf16", units=units)
    o, lse, _ = run_blocks(q, k, v, 1e-3, allow, 128, 128)
    rows = np.repeat(empty, 128, axis=2)[:, :, :cfg.T]
    assert (o[rows] == 0).all() and np.isneginf(lse[rows]).all()
