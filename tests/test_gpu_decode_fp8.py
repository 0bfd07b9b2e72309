"""Split-KV decode over an FP8 (E4M3) key/value cache on the GPU against the
fp64 oracle, which takes the query as given (bits exact outside the margin
band widened by the kernel's derived query-pair bound, partials and merged
output within the bf16 tolerances)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_online_gb300 import binding as bs
from block_sparse_attention_online_gb300 import workloads as W
from tests.parity import check_outputs, compare_bits, fp8_query_pair_band

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run_fp8(cfg, q, k8, v8, ks, vs, lam, n_splits):
    dev = torch.device("cuda")
    o, lse, bits = bs.attn_skip_decode_fp8(q.to(dev), k8.to(dev), v8.to(dev), ks.to(dev),
                                           vs.to(dev), lam, cfg.Bc, n_splits)
    bs.attn_skip_last_device_error()
    return o, lse, bits


def check_fp8(cfg, q, k8, v8, ks, vs, lam, n_splits, units=None):
    o, lse, bits = run_fp8(cfg, q, k8, v8, ks, vs, lam, n_splits)
    n_b = -(-cfg.L // cfg.Bc)
    bps = -(-n_b // n_splits)
    skip = bs.unpack_bits(bits, bps).numpy()
    r = oracle.decode_fp8(q, k8.numpy(), v8.numpy(), ks.numpy(), vs.numpy(), cfg.scale, lam,
                          cfg.Bc, n_splits, units=units)
    sel = np.ones((cfg.B, cfg.Hkv), dtype=bool)
    if units is not None:
        sel[:] = False
        for u in np.asarray(units).ravel():
            sel.reshape(-1)[int(u) // n_splits] = True
    band = np.broadcast_to(fp8_query_pair_band(q, k8.numpy(), ks.numpy(), cfg.scale, cfg.Bc,
                                               n_splits, cfg.G), skip.shape)
    n_bad, flips = compare_bits(skip[sel], r["skip"][sel], r["margin"][sel], lam,
                                extra_band=band[sel], label=f"fp8 decode L={cfg.L} lambda={lam:.4g}")
    assert n_bad == 0, f"{n_bad} skip bits differ outside the margin band"
    if flips.any():
        forced = r["skip"].copy()
        forced[sel] = skip[sel]
        r = oracle.decode_fp8(q, k8.numpy(), v8.numpy(), ks.numpy(), vs.numpy(), cfg.scale, lam,
                              cfg.Bc, n_splits, units=units, force_skip=forced)
    hsel = np.repeat(sel, cfg.G, axis=1)
    op, lp = o.cpu().numpy(), lse.cpu().numpy()
    # empty splits (n_splits > blocks) have LSE -inf on both sides
    fin = np.isfinite(r["lse_part"][hsel])
    assert (np.isfinite(lp[hsel]) == fin).all()
    check_outputs(op[hsel][fin], r["o_part"][hsel][fin], lp[hsel][fin], r["lse_part"][hsel][fin],
                  "bf16", "fp8 decode partials")
    # merged output
    mo, ml = bs.attn_skip_decode_combine(o, lse, out_dtype=torch.float32)
    ro, rl = oracle.combine(r["o_part"], r["lse_part"])
    check_outputs(mo.cpu().numpy()[hsel], ro[hsel], ml.cpu().numpy()[hsel], rl[hsel], "bf16",
                  "fp8 decode merged")
    return float(skip[sel].mean()), int(flips.sum())


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_fp8_decode_small(G):
    cfg = W.temperate(W.GQA_DECODE_FP8_32K.with_(B=2, Hq=2 * G, Hkv=2, L=3000, seed=71))
    q, k8, v8, ks, vs = W.decode_inputs_fp8(cfg)
    for lam, n_splits in ((0.0, 2), (1e-4, 3), (1e-2, 4), (0.2, 1)):
        check_fp8(cfg, q, k8, v8, ks, vs, lam, n_splits)


@pytest.mark.parametrize("L,n_splits", [(129, 1), (1, 1), (1000, 16), (4097, 5)])
def test_fp8_decode_ragged_and_empty_splits(L, n_splits):
    cfg = W.temperate(W.GQA_DECODE_FP8_32K.with_(B=2, Hq=8, Hkv=2, L=L, seed=72))
    q, k8, v8, ks, vs = W.decode_inputs_fp8(cfg, pow2_scales=False)
    for lam in (0.0, 3e-2):
        check_fp8(cfg, q, k8, v8, ks, vs, lam, n_splits)


def test_fp8_decode_full_size_at_70_percent():
    """B=16, 32/8 heads, L=32768, 8 splits at the oracle's ~70 % threshold;
    sampled (sequence, KV head) slices against the oracle, the sparsity of
    the whole launch against the oracle's statistics."""
    cfg = W.GQA_DECODE_FP8_32K
    with open(os.path.join(GOLDEN, "lambdas.json")) as f:
        lam = json.load(f)[cfg.name]["0.7"]["lambda"]
    q, k8, v8, ks, vs = W.decode_inputs_fp8(cfg)
    units = [u * cfg.n_splits + s for u in (0, 37, 77, 127) for s in range(cfg.n_splits)]
    sp, _ = check_fp8(cfg, q, k8, v8, ks, vs, lam, cfg.n_splits, units=units)
    _, _, bits = run_fp8(cfg, q, k8, v8, ks, vs, lam, cfg.n_splits)
    total = float(bs.unpack_bits(bits, 32).float().mean())
    assert abs(total - 0.70) < 0.01
    assert sp > 0.5
