"""Sampled decode output (SANTA estimator) on the GPU against the fp64 oracle.

Comparison rule.  The sample indices are integers decided by floating point:
the kernel places threshold T_m on the CDF in fp32, the oracle in fp64.  They
must agree exactly wherever the oracle's threshold lies more than GAP_TOL
(probability units) from both ends of its key's CDF interval.  Closer than
that, the kernel's key must still be admissible: its CDF interval, widened by
GAP_TOL, contains T_m.  The output must be the mean of the value rows at the
kernel's own indices (fp32 accumulation), and equals the oracle's output on
every head whose indices all agree.

GAP_TOL: the kernel's CDF differs from the exact one by the fp32 error of the
scores (bf16 products accumulated in fp32 over d = 128: relative ~1e-6 of the
score scale, i.e. ~1e-5 relative on a weight), of ex2 (2 ulp) and of the fp32
prefix sums (at most ~100 sequential additions at 2^-24 each); together below
2e-5 in probability units.  GAP_TOL = 5e-5 leaves a factor 2.5.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_online_gb300 import binding as bs
from block_sparse_attention_online_gb300 import workloads as W

pytestmark = pytest.mark.gpu
GAP_TOL = 5e-5


def run_santa(cfg, q, k, v, S, mode, u, n_tiles, out_dtype=torch.float32, workspace=None):
    dev = torch.device("cuda")
    o, idx = bs.attn_skip_santa_decode(q.to(dev), k.to(dev), v.to(dev), S, mode, u.to(dev),
                                       n_tiles=n_tiles, out_dtype=out_dtype, with_idx=True,
                                       workspace=workspace)
    bs.attn_skip_last_device_error()  # raises on a device-side error
    return o.float().cpu().numpy().astype(np.float64), idx.cpu().numpy()


def thresholds(u, S, mode):
    u = u.double().numpy()
    m = np.arange(S)
    if mode == "sys":
        return (m[None, None, :] + u[:, :, None]) / S
    if mode == "iid":
        return u
    return (m[None, None, :] + u) / S


def check_santa(cfg, q, k, v, S, mode, u, n_tiles):
    y, idx = run_santa(cfg, q, k, v, S, mode, u, n_tiles)
    r = oracle.santa_decode(q, k, v, cfg.scale, S, mode, u, with_cdf=True)
    B, Hq = q.shape[0], q.shape[1]
    G = Hq // k.shape[1]
    assert idx.shape == (B, Hq, S)
    assert ((idx >= 0) & (idx < cfg.L)).all()
    clear = r["gap"] > GAP_TOL
    bad = clear & (idx != r["idx"])
    assert not bad.any(), f"{int(bad.sum())} sample indices differ away from CDF boundaries"
    # Near a boundary: the kernel's key is admissible within GAP_TOL.
    T = thresholds(u, S, mode)
    cdf = r["cdf"]
    lo = np.where(idx > 0, np.take_along_axis(cdf, np.maximum(idx - 1, 0), axis=-1), 0.0)
    hi = np.take_along_axis(cdf, idx, axis=-1)
    assert ((lo - GAP_TOL <= T) & (T < hi + GAP_TOL)).all()
    # The output is the mean of the kernel's own sampled rows ...
    vf = v.float().numpy().astype(np.float64)
    mine = np.stack([np.stack([vf[b, h // G][idx[b, h]].mean(axis=0) for h in range(Hq)])
                     for b in range(B)])
    vmax = float(np.abs(vf).max())
    assert np.abs(y - mine).max() <= 1e-6 * vmax * max(1.0, np.log2(S)) + 1e-7
    # ... and the oracle's output wherever every index agrees; elsewhere it is
    # off by at most (number of moved samples) x (value spread) / S.
    diff_n = (idx != r["idx"]).sum(axis=-1)
    same = diff_n == 0
    if same.any():
        assert np.abs(y[same] - r["y"][same]).max() <= 1e-5
    spread = float(vf.max() - vf.min())
    bound = diff_n[..., None] * spread / S + 1e-5
    assert (np.abs(y - r["y"]) <= bound).all()
    return float((~clear).mean()), float(same.mean())


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("mode", ["sys", "strat", "iid"])
def test_santa_small(G, mode):
    cfg = W.SANTA_DECODE_32K.with_(B=2, Hq=2 * G, Hkv=2, L=2048, seed=41)
    q, k, v = W.decode_inputs(cfg)
    for S, n_tiles in ((128, 4), (1, 1), (2048, 16), (100, 3)):
        u = W.santa_offsets(cfg, S, mode, seed=S)
        check_santa(cfg, q, k, v, S, mode, u, n_tiles)


@pytest.mark.parametrize("L,n_tiles", [(1999, 2), (130, 1), (1, 1), (300, 5), (4097, 33),
                                       (5000, 3)])
def test_santa_ragged_lengths_and_empty_tiles(L, n_tiles):
    """Ragged last block (keys past L stashed as -inf), a single key, tiles
    with no block (n_tiles > number of blocks)."""
    cfg = W.SANTA_DECODE_32K.with_(B=2, Hq=8, Hkv=2, L=L, seed=42)
    q, k, v = W.decode_inputs(cfg)
    for mode in ("sys", "strat", "iid"):
        u = W.santa_offsets(cfg, 64, mode, seed=L)
        check_santa(cfg, q, k, v, 64, mode, u, n_tiles)


def test_santa_flat_attention():
    """Flatter attention still: the samples spread over many keys and tiles."""
    cfg = W.SANTA_DECODE_32K.with_(B=2, L=8192, sink_a=0.5, salient_a=0.3, seed=43)
    q, k, v = W.decode_inputs(cfg)
    for mode in ("sys", "strat", "iid"):
        u = W.santa_offsets(cfg, 256, mode, seed=1)
        check_santa(cfg, q, k, v, 256, mode, u, 8)


def test_santa_bf16_output_and_workspace_reuse():
    """Two calls in a row on one workspace give identical results; the bf16
    output is the fp32 output rounded to nearest."""
    cfg = W.SANTA_DECODE_32K.with_(B=2, L=4096, seed=44)
    q, k, v = W.decode_inputs(cfg)
    u = W.santa_offsets(cfg, 128, "sys")
    ns, nt = bs.attn_skip_santa_workspace(cfg.B, cfg.Hq, cfg.L, 8)
    ws = (torch.empty(ns, device="cuda"), torch.empty(nt, device="cuda"))
    y1, i1 = run_santa(cfg, q, k, v, 128, "sys", u, 8, workspace=ws)
    y2, i2 = run_santa(cfg, q, k, v, 128, "sys", u, 8, workspace=ws)
    yb, ib = run_santa(cfg, q, k, v, 128, "sys", u, 8, out_dtype=torch.bfloat16, workspace=ws)
    assert (i1 == i2).all() and (y1 == y2).all() and (ib == i1).all()
    want = torch.from_numpy(y1).float().to(torch.bfloat16).double().numpy()
    assert (yb == want).all()


def test_santa_sink_dominated():
    """The BLASST decode recipe: the sink holds all but e^-30 of the mass, so
    every sample lands on key 0 and the output is its value row."""
    cfg = W.GQA_DECODE_32K.with_(B=2)
    q, k, v = W.decode_inputs(cfg)
    u = W.santa_offsets(cfg, 128, "sys")
    y, idx = run_santa(cfg, q, k, v, 128, "sys", u, 16)
    assert (idx == 0).mean() > 0.99
    check_santa(cfg, q, k, v, 128, "sys", u, 16)


@pytest.mark.parametrize("mode", ["sys", "strat", "iid"])
def test_santa_full_size(mode):
    """B=16, 32/8 heads, L=32768, S=128 samples, 16 key tiles, spread
    attention: the configuration the benchmark times."""
    cfg = W.SANTA_DECODE_32K
    q, k, v = W.decode_inputs(cfg)
    u = W.santa_offsets(cfg, 128, mode)
    near, same = check_santa(cfg, q, k, v, 128, mode, u, 16)
    assert near < 0.3
