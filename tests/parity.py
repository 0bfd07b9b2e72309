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


# Every compare_bits call appends (label, flips, blocks in the band, traversed
# blocks); the session's terminal summary prints them (tests/conftest.py).
FLIP_LOG = []


def compare_bits(gpu_skip: np.ndarray, ora_skip: np.ndarray, ora_margin: np.ndarray,
                 lam: float, extra_band=0.0, label: str = ""):
    """gpu_skip/ora_skip/ora_margin share a shape; returns (n_bad, flips_mask).

    A traversed block is in the band when its oracle statistic lies within
    MARGIN_BAND + ``extra_band`` of ln(lambda) (``extra_band`` a scalar or an
    array of the same shape, for a kernel whose scores differ from the
    oracle's by a derived amount); only there may the bits differ.  Flips are
    counted, checked against the number of blocks in the band, and logged."""
    gpu_skip = gpu_skip.astype(bool)
    ora = ora_skip.astype(bool)
    trav = np.isfinite(ora_margin)
    ln_lam = math.log(lam) if lam > 0 else -math.inf
    if math.isfinite(ln_lam):
        band = MARGIN_BAND + np.asarray(extra_band, dtype=np.float64)
        near = trav & (np.abs(np.nan_to_num(ora_margin, nan=0.0) - ln_lam) < band)
    else:
        near = np.zeros_like(trav)
    diff = gpu_skip != ora
    bad = (diff & ~near) | (gpu_skip & ~trav)
    flips = diff & near
    assert flips.sum() <= near.sum()
    FLIP_LOG.append((label or f"lambda={lam:.6g}", int(flips.sum()), int(near.sum()),
                     int(trav.sum())))
    return int(bad.sum()), flips


def _split_band(eps, Bc, n_splits):
    """From per-(b, query head, key) score deviations eps [B, Hkv, G, L]: twice
    the largest over the split's keys and the group's heads, per (b, KV head,
    split); shape [B, Hkv, n_splits, 1]."""
    eps = eps.max(axis=2)
    B, Hkv, L = eps.shape
    n_b = -(-L // Bc)
    out = np.zeros((B, Hkv, n_splits, 1))
    for s in range(n_splits):
        b0, b1 = (s * n_b) // n_splits, ((s + 1) * n_b) // n_splits
        if b1 > b0:
            out[:, :, s, 0] = 2.0 * eps[:, :, b0 * Bc:min(b1 * Bc, L)].max(axis=-1)
    return out


def _pow2_exponent(q, top):
    """Per head: e = top - ceil(log2 max|q|) (0 for a zero row)."""
    import torch
    qf = q.detach().to("cpu", torch.float64).numpy()
    amax = np.abs(qf).max(axis=-1)
    frac, ex = np.frexp(np.where(amax > 0, amax, 1.0))
    return np.where(amax > 0, top - np.where(frac == 0.5, ex - 1, ex), 0).astype(np.float64)


def fp8_query_pair_band(q, k8, k_scale, scale: float, Bc: int, n_splits: int, G: int):
    """Extra bit band of the E4M3-cache decode kernel, per (b, KV head, split).

    The kernel multiplies the E4M3 key codes with the query written as the
    exact pair hi + lo of E4M3 values after a per-head power-of-two scale
    sigma = 2^e, the largest with max|q| sigma <= 256 (an E4M3 x E4M3 product
    needs both operands in E4M3).  For a bf16 element x = q sigma with |x| >=
    2^-6 the remainder x - hi is a multiple of x's last place with at most four
    significant bits, exact in E4M3 when |x| >= 2^-2 (its last place is then
    at least E4M3's subnormal step 2^-9); below 2^-2 rounding lo to that step
    moves x by at most 2^-10.  So query element d of head h moves by at most
    2^-10 / sigma_h, and only if |q_hd sigma_h| < 2^-2.  A score of key c then
    moves by at most eps_hc = scale * k_scale * 2^-10 / sigma_h * (sum of
    |code_cd| over those d), and a block statistic max_r(rowmax_r - m_new_r)
    by at most twice the largest eps over the split's keys and the group's
    heads.  Returns that bound, shape [B, Hkv, n_splits, 1]."""
    import torch
    e = _pow2_exponent(q, 8)                                          # [B, Hq]
    qf = q.detach().to("cpu", torch.float64).numpy()
    moved = (np.abs(qf) * np.exp2(e)[..., None] < 0.25).astype(np.float32)  # [B, Hq, dk]
    kd = torch.as_tensor(np.ascontiguousarray(k8, dtype=np.uint8)).view(
        torch.float8_e4m3fn).float().abs()                            # [B, Hkv, L, dk]
    B, Hq, dk = moved.shape
    Hkv = Hq // G
    m = torch.from_numpy(moved.reshape(B, Hkv, G, dk))
    ksum = torch.einsum("bhgd,bhld->bhgl", m, kd).double().numpy()    # [B, Hkv, G, L]
    coef = (scale * np.asarray(k_scale, dtype=np.float64)[:, :, None]
            * (2.0 ** -10) * np.exp2(-e).reshape(B, Hkv, G))
    return _split_band(coef[..., None] * ksum, Bc, n_splits)


# E2M1 magnitudes by the code's low three bits (OCP MX FP4).
_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def nvfp4_query_band(q, k4, k_bs, k_scale, scale: float, Bc: int, n_splits: int, G: int):
    """Extra bit band of the NVFP4-cache decode kernel, per (b, KV head, split).

    The kernel's key products are fp16 x fp16: each query head enters as
    fp16(q sigma), sigma = 2^e the largest power of two with max|q| sigma <=
    2^15.  A bf16 element keeps its eight significant bits in fp16 unless
    |q sigma| < 2^-17, where fp16's subnormal step 2^-24 rounds it by at most
    2^-25: each query element moves by at most 2^-25 / sigma.  The widened keys
    are exact, so a score moves by at most scale * k_scale * 2^-25 / sigma *
    sum_d |k_d| and a block statistic by twice the largest such amount over
    the split's keys and the group's heads.  Returns [B, Hkv, n_splits, 1]."""
    import torch
    e = _pow2_exponent(q, 15)                                         # [B, Hq]
    k4 = np.ascontiguousarray(k4, dtype=np.uint8)
    mag = _E2M1[k4 & 7] + _E2M1[(k4 >> 4) & 7]                       # per byte: two elements
    bs = torch.as_tensor(np.ascontiguousarray(k_bs, dtype=np.uint8)).view(
        torch.float8_e4m3fn).double().abs().numpy()                   # [B, Hkv, L, d/16]
    ksum = (mag.reshape(*mag.shape[:-1], bs.shape[-1], 8).sum(-1) * bs).sum(-1)  # [B, Hkv, L]
    B, Hq = e.shape
    Hkv = Hq // G
    coef = (scale * np.asarray(k_scale, dtype=np.float64)[:, :, None]
            * (2.0 ** -25) * np.exp2(-e).reshape(B, Hkv, G))
    return _split_band(coef[..., None] * ksum[:, :, None, :], Bc, n_splits)


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
