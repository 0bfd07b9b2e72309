"""Comparison rules between the CUDA path and the fp64 oracle.

* Skip bitmaps are bit-exact except on blocks whose tile statistic lies within
  ``MARGIN_BAND`` of ln(lambda) (there fp32 and fp64 may round to different
  sides); such flips are counted and returned, never silently accepted
  elsewhere.  Untraversed positions must read 0.
* When a flip happened, the outputs are compared against the oracle re-run with
  the GPU's decisions (both decision sets are valid within rounding).
* bf16: O max-abs <= 2e-2 and relative L2 <= 5e-3; LSE max-abs <= 1e-2.
  fp32: O max-abs <= 1e-4; LSE max-abs <= 1e-4.
"""
import math

import numpy as np

MARGIN_BAND = 1e-3
TOL = {
    "bf16": dict(o_abs=2e-2, o_rel_l2=5e-3, lse_abs=1e-2),
    "f32": dict(o_abs=1e-4, o_rel_l2=1e-5, lse_abs=1e-4),
}


def compare_bits(gpu_skip: np.ndarray, ora_skip: np.ndarray, ora_margin: np.ndarray,
                 lam: float):
    """gpu_skip/ora_skip/ora_margin share a shape; returns (n_bad, flips_mask)."""
    gpu_skip = gpu_skip.astype(bool)
    ora = ora_skip.astype(bool)
    trav = np.isfinite(ora_margin)
    ln_lam = math.log(lam) if lam > 0 else -math.inf
    if math.isfinite(ln_lam):
        near = trav & (np.abs(np.nan_to_num(ora_margin, nan=0.0) - ln_lam) < MARGIN_BAND)
    else:
        near = np.zeros_like(trav)
    diff = gpu_skip != ora
    bad = (diff & ~near) | (gpu_skip & ~trav)
    return int(bad.sum()), diff & near


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-300))


def check_outputs(o_gpu, o_ref, lse_gpu, lse_ref, kind: str, what: str = ""):
    t = TOL[kind]
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    err = np.abs(o_gpu - o_ref)
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite output"
    assert err.max() <= t["o_abs"], f"{what}: O max-abs {err.max():.3g} > {t['o_abs']}"
    rl = rel_l2(o_gpu, o_ref)
    assert rl <= t["o_rel_l2"], f"{what}: O rel-L2 {rl:.3g} > {t['o_rel_l2']}"
    if lse_gpu is not None:
        le = np.abs(np.asarray(lse_gpu, dtype=np.float64) - lse_ref)
        assert le.max() <= t["lse_abs"], f"{what}: LSE max-abs {le.max():.3g}"
    return float(err.max()), rl
