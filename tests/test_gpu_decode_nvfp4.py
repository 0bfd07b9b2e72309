"""Split-KV decode over an NVFP4 key/value cache on the GPU against the fp64
oracle, which takes the query as given and the rows as head scale x E4M3
block scale x E2M1 code: bits exact outside the margin band (widened by the
kernel's derived fp16 query bound), partials and merged output within the
bf16 tolerances."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_online_gb300 import binding as bs
from block_sparse_attention_online_gb300 import workloads as W
from tests.parity import check_outputs, compare_bits, nvfp4_query_band

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run_nvfp4(cfg, inputs, lam, n_splits):
    dev = torch.device("cuda")
    o, lse, bits = bs.attn_skip_decode_nvfp4(*(x.to(dev) for x in inputs), lam, cfg.Bc,
                                             n_splits)
    bs.attn_skip_last_device_error()
    return o, lse, bits


def _oracle(cfg, q, np_in, lam, n_splits, force_skip=None):
    return oracle.decode_nvfp4(q, *np_in, cfg.scale, lam, cfg.Bc, n_splits,
                               force_skip=force_skip)


def check_nvfp4(cfg, inputs, lam, n_splits, slices=None):
    """Compare every (sequence, KV head) slice, or the listed ones (the oracle
    then runs on those slices' inputs alone: each slice is independent)."""
    q, k4, v4, kbs, vbs, ks, vs = inputs
    o, lse, bits = run_nvfp4(cfg, inputs, lam, n_splits)
    n_b = -(-cfg.L // cfg.Bc)
    bps = -(-n_b // n_splits)
    skip = bs.unpack_bits(bits, bps).numpy()
    op, lp = o.cpu().numpy(), lse.cpu().numpy()
    mo, ml = bs.attn_skip_decode_combine(o, lse, out_dtype=torch.float32)
    mo, ml = mo.cpu().numpy(), ml.cpu().numpy()
    G = cfg.G
    if slices is None:
        parts = [(slice(None), slice(None), slice(None))]
    else:
        parts = [(slice(b, b + 1), slice(h, h + 1), slice(h * G, (h + 1) * G))
                 for b, h in slices]
    skipped = traversed = n_flips = 0
    for sb, sh, sq in parts:
        qq = q[sb, sq]
        np_in = [x[sb, sh].numpy() for x in (k4, v4, kbs, vbs, ks, vs)]
        r = _oracle(cfg, qq, np_in, lam, n_splits)
        gs = skip[sb, sh]
        band = np.broadcast_to(nvfp4_query_band(qq, np_in[0], np_in[2], np_in[4], cfg.scale,
                                                cfg.Bc, n_splits, G), gs.shape)
        n_bad, flips = compare_bits(gs, r["skip"], r["margin"], lam, extra_band=band,
                                    label=f"nvfp4 decode L={cfg.L} lambda={lam:.4g}")
        assert n_bad == 0, f"{n_bad} skip bits differ outside the margin band"
        if flips.any():
            r = _oracle(cfg, qq, np_in, lam, n_splits, force_skip=gs.astype(np.uint8))
        fin = np.isfinite(r["lse_part"])  # empty splits: -inf on both sides
        assert (np.isfinite(lp[sb, sq]) == fin).all()
        check_outputs(op[sb, sq][fin], r["o_part"][fin], lp[sb, sq][fin], r["lse_part"][fin],
                      "bf16", "nvfp4 decode partials")
        ro, rl = oracle.combine(r["o_part"], r["lse_part"])
        check_outputs(mo[sb, sq], ro, ml[sb, sq], rl, "bf16", "nvfp4 decode merged")
        trav = np.isfinite(r["margin"])
        skipped += int(gs[trav].sum())
        traversed += int(trav.sum())
        n_flips += int(flips.sum())
    return skipped / max(traversed, 1), n_flips


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_nvfp4_decode_small(G):
    cfg = W.temperate(W.GQA_DECODE_NVFP4_32K.with_(B=2, Hq=2 * G, Hkv=2, L=3000, seed=81))
    inputs = W.decode_inputs_nvfp4(cfg)
    for lam, n_splits in ((0.0, 2), (1e-4, 3), (1e-2, 4), (0.2, 1)):
        check_nvfp4(cfg, inputs, lam, n_splits)


@pytest.mark.parametrize("L,n_splits", [(129, 1), (1, 1), (1000, 16), (4097, 5)])
def test_nvfp4_decode_ragged_and_empty_splits(L, n_splits):
    cfg = W.temperate(W.GQA_DECODE_NVFP4_32K.with_(B=2, Hq=8, Hkv=2, L=L, seed=82))
    inputs = W.decode_inputs_nvfp4(cfg)
    for lam in (0.0, 3e-2):
        check_nvfp4(cfg, inputs, lam, n_splits)


def test_nvfp4_decode_every_code_and_scale():
    """Random bytes for every code nibble and block scales over the whole
    finite E4M3 range (no NaN codes), non-power-of-two head scales: the
    widening must be exact for all of them."""
    cfg = W.temperate(W.GQA_DECODE_NVFP4_32K.with_(B=2, Hq=8, Hkv=2, L=700, seed=83))
    g = np.random.default_rng(83)
    q = W.decode_inputs(cfg)[0]
    shp = (cfg.B, cfg.Hkv, cfg.L)
    k4 = torch.from_numpy(g.integers(0, 256, size=shp + (64,), dtype=np.uint8))
    v4 = torch.from_numpy(g.integers(0, 256, size=shp + (64,), dtype=np.uint8))

    def scales():
        b = g.integers(0, 256, size=shp + (8,), dtype=np.uint8)
        b[(b & 0x7F) == 0x7F] ^= 1  # no NaN codes
        return torch.from_numpy(b)
    kbs, vbs = scales(), scales()
    # head scales keep the rows within a few units (|E4M3 x E2M1| <= 2688)
    ks = torch.from_numpy(g.uniform(5e-4, 1e-3, size=(cfg.B, cfg.Hkv)).astype(np.float32))
    vs = torch.from_numpy(g.uniform(2e-4, 7e-4, size=(cfg.B, cfg.Hkv)).astype(np.float32))
    for lam in (0.0, 0.05):
        check_nvfp4(cfg, (q, k4, v4, kbs, vbs, ks, vs), lam, 3)


def test_nvfp4_decode_full_size_at_70_percent():
    """B=16, 32/8 heads, L=32768, 8 splits at the oracle's ~70 % threshold;
    sampled (sequence, KV head) slices against the oracle, the sparsity of the
    whole launch against the oracle's figure."""
    cfg = W.GQA_DECODE_NVFP4_32K
    with open(os.path.join(GOLDEN, "lambdas.json")) as f:
        lam = json.load(f)[cfg.name]["0.7"]["lambda"]
    inputs = W.decode_inputs_nvfp4(cfg)
    slices = [divmod(u, cfg.Hkv) for u in (0, 37, 77, 127)]
    sp, _ = check_nvfp4(cfg, inputs, lam, cfg.n_splits, slices=slices)
    _, _, bits = run_nvfp4(cfg, inputs, lam, cfg.n_splits)
    total = float(bs.unpack_bits(bits, 32).float().mean())
    assert abs(total - 0.70) < 0.01
    assert sp > 0.5
