"""fp64 CPU oracle for softmax-threshold block-skipping attention.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
library under ``block_sparse_attention_online_gb300`` never does.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over independent
query tiles or decode splits); this module only marshals numpy arrays.  It
follows the BLASST page ("BLASST：一个标量阈值实现的动态块稀疏注意力", sections
"铺垫：FlashAttention 的在线 softmax" and "BLASST 的判定准则") step by step.

Parity status of each function (what pins it, in ``tests/test_oracle.py``):

* ``dense_prefill`` / ``dense_decode``: brute-force numpy softmax on tiny
  inputs, and torch's fp64 ``scaled_dot_product_attention`` on CPU.
* ``prefill`` / ``decode``: lambda = 0 equals dense attention; the closed form
  "softmax restricted to the kept tokens"; the champion rule (the block holding
  a row's maximum is never skipped); every skipped token has softmax weight
  below lambda; the output error bound; hand-worked fixtures under
  ``tests/golden/``; brute-force recomputation of each skip bit.
* ``combine``: lambda = 0 merged decode equals dense single-pass attention;
  one split is the identity.
* ``decode_fp8``: the E4M3 decoding it relies on equals an independent
  bit-level decoder over all 256 codes; at lambda = 0 and with thresholds the
  merged output equals a brute-force fp64 softmax of the given query against
  the scaled decoded rows (key scale in the scores, value scale on the
  output), for scales that are not powers of two.
* ``decode_nvfp4`` / ``nvfp4_rows`` / ``e2m1_decode``: the E2M1 decoding
  equals the FP4 value table of the OCP Microscaling formats specification
  over all 16 codes; rows dequantised from the seeded generator lie within
  half an E2M1 step of the drawn values (which pins the nibble order and the
  block-scale indexing against the generator's independent packing); at
  lambda = 0 and with thresholds the output equals brute-force fp64 attention
  over rows decoded from that table, with non-power-of-two scales.
* ``prefill_varlen``: each packed sequence at lambda = 0 equals torch's fp64
  SDPA on that sequence alone; with thresholds, each sequence's output is the
  softmax over its own kept tokens, a larger lambda skips a superset of
  blocks, and empty sequences leave their rows untouched.
* ``santa_decode`` (the page "Stochastic Sparse Attention for Memory-Bound
  Inference", section "关键设计"): the closed form of equal scores (every
  sample index and gap known exactly); a dominant key takes every sample; the
  systematic sampler picks each key floor(S p_i) or ceil(S p_i) times and its
  stratified form keeps sample m inside stratum m; the mean over a fine grid
  of offsets, and the mean over many i.i.d. or stratified draws, equal dense
  attention (unbiasedness).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libbsa_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc (fp64, no fast-math, no FMA contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i, d, i64 = ctypes.c_int, ctypes.c_double, ctypes.c_int64
        lib.bsa_oracle_dense_prefill.argtypes = [P, P, P, i, i, i, i, i, i, d, i, P, i64, P, P]
        lib.bsa_oracle_dense_decode.argtypes = [P, P, P, i, i, i, i, i, i, i64, i64, d, P, P]
        lib.bsa_oracle_prefill.argtypes = [P, P, P, i, i, i, i, i, i, d, d, i, i, i, P, i64,
                                           P, P, P, P, P, P]
        lib.bsa_oracle_decode.argtypes = [P, P, P, i, i, i, i, i, i, i64, i64, d, d, i, i, P,
                                          i64, P, i, P, P, P, P]
        lib.bsa_oracle_combine.argtypes = [P, P, i, i, i, i, P, P]
        lib.bsa_oracle_santa_decode.argtypes = [P, P, P, i, i, i, i, i, i, i64, i64, d, i, i, P,
                                                P, P, P, P]
        for f in ("bsa_oracle_dense_prefill", "bsa_oracle_dense_decode", "bsa_oracle_prefill",
                  "bsa_oracle_decode", "bsa_oracle_combine", "bsa_oracle_num_threads",
                  "bsa_oracle_santa_decode"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    return _load().bsa_oracle_num_threads()


def _f32(x) -> np.ndarray:
    """Exact fp32 numpy copy of a torch tensor (bf16 widens exactly) or array."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu", torch.float32).numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _units(units):
    if units is None:
        return None, 0
    u = np.ascontiguousarray(np.asarray(units, dtype=np.int64).ravel())
    return u, u.size


def dense_prefill(q, k, v, scale, causal=True, rows=None):
    """Exact softmax attention; q [B,Hq,T,dk], k [B,Hkv,T,dk], v [B,Hkv,T,dv].

    Returns ``(y [B,Hq,T,dv], lse [B,Hq,T])`` in fp64 (only ``rows`` — flat
    indices into [B,Hq,T] — are filled when given)."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, Hq, T, dk = q.shape
    Hkv, dv = k.shape[1], v.shape[3]
    y = np.zeros((B, Hq, T, dv))
    lse = np.full((B, Hq, T), np.nan)
    r, nr = _units(rows)
    rc = _load().bsa_oracle_dense_prefill(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, T, dk, dv,
                                          float(scale), int(bool(causal)),
                                          None if r is None else _ptr(r), nr, _ptr(y), _ptr(lse))
    if rc:
        raise ValueError("bsa_oracle_dense_prefill: invalid arguments")
    return y, lse


def dense_decode(q, k, v, scale, dv=None):
    """Exact softmax attention for one query token per sequence.

    q [B,Hq,dk]; k [B,Hkv,L,dk]; v [B,Hkv,L,dv] or ``None`` for a latent cache
    whose values are the first ``dv`` columns of k."""
    q, k = _f32(q), _f32(k)
    B, Hq, dk = q.shape
    _, Hkv, L, kstride = k.shape
    if v is None:
        vv, vstride = k, kstride
    else:
        vv = _f32(v)
        dv, vstride = vv.shape[3], vv.shape[3]
    y = np.zeros((B, Hq, dv))
    lse = np.zeros((B, Hq))
    rc = _load().bsa_oracle_dense_decode(_ptr(q), _ptr(k), _ptr(vv), B, Hq, Hkv, L, dk, dv,
                                         kstride, vstride, float(scale), _ptr(y), _ptr(lse))
    if rc:
        raise ValueError("bsa_oracle_dense_decode: invalid arguments")
    return y, lse


def _forced(force_skip, shape):
    if force_skip is None:
        return None
    f = np.ascontiguousarray(np.asarray(force_skip, dtype=np.uint8))
    if f.shape != shape:
        raise ValueError(f"force_skip has shape {f.shape}, expected {shape}")
    return f


def prefill(q, k, v, scale, lam, Br=128, Bc=128, causal=True, units=None, force_skip=None,
            allow=None):
    """Thresholded online-softmax prefill in fp64.

    Returns a dict with ``o`` [B,Hq,T,dv], ``lse`` [B,Hq,T], ``skip``
    [B,Hq,n_t,n_b] (uint8, 1 = skipped) and ``margin`` [B,Hq,n_t,n_b] (the tile
    statistic max_r(rowmax - m_new); NaN where not traversed).  ``units`` are
    flat indices into [B,Hq,n_t]; only those tiles are computed.
    ``force_skip`` ([B,Hq,n_t,n_b]) replaces the skip decisions by given ones
    (the loop's arithmetic is unchanged).  ``allow`` ([B,Hq,n_t,n_b], nonzero =
    in the set) restricts each tile to an explicit block set: blocks outside it
    are not traversed; a row with no visible key in its set gets O = 0 and
    LSE = -inf."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, Hq, T, dk = q.shape
    Hkv, dv = k.shape[1], v.shape[3]
    n_t, n_b = -(-T // Br), -(-T // Bc)
    o = np.zeros((B, Hq, T, dv))
    lse = np.full((B, Hq, T), np.nan)
    skip = np.zeros((B, Hq, n_t, n_b), dtype=np.uint8)
    margin = np.full((B, Hq, n_t, n_b), np.nan)
    u, nu = _units(units)
    f = _forced(force_skip, skip.shape)
    al = None if allow is None else _forced(np.asarray(allow) != 0, skip.shape)
    rc = _load().bsa_oracle_prefill(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, T, dk, dv,
                                    float(scale), float(lam), Br, Bc, int(bool(causal)),
                                    None if u is None else _ptr(u), nu,
                                    None if f is None else _ptr(f),
                                    None if al is None else _ptr(al), _ptr(o), _ptr(lse),
                                    _ptr(skip), _ptr(margin))
    if rc:
        raise ValueError("bsa_oracle_prefill: invalid arguments")
    return {"o": o, "lse": lse, "skip": skip, "margin": margin}


def decode(q, k, v, scale, lam, Bc, n_splits, dv=None, units=None, force_skip=None,
           per_head=False):
    """Split-KV thresholded decode in fp64 (partials, before the merge).

    Returns ``o_part`` [B,Hq,S,dv], ``lse_part`` [B,Hq,S], ``skip`` and
    ``margin`` [B,Hkv,S,bps] with bps = ceil(n_b / S).  ``units`` are flat
    indices into [B,Hkv,S]; ``force_skip`` ([B,Hkv,S,bps]) replaces the skip
    decisions by given ones.  ``per_head``: each query head decides for
    itself; ``skip``, ``margin`` and ``force_skip`` are then [B,Hq,S,bps]."""
    q, k = _f32(q), _f32(k)
    B, Hq, dk = q.shape
    _, Hkv, L, kstride = k.shape
    if v is None:
        vv, vstride = k, kstride
    else:
        vv = _f32(v)
        dv, vstride = vv.shape[3], vv.shape[3]
    n_b = -(-L // Bc)
    bps = -(-n_b // n_splits)
    o_part = np.zeros((B, Hq, n_splits, dv))
    lse_part = np.full((B, Hq, n_splits), np.nan)
    rows = Hq if per_head else Hkv
    skip = np.zeros((B, rows, n_splits, bps), dtype=np.uint8)
    margin = np.full((B, rows, n_splits, bps), np.nan)
    u, nu = _units(units)
    f = _forced(force_skip, skip.shape)
    rc = _load().bsa_oracle_decode(_ptr(q), _ptr(k), _ptr(vv), B, Hq, Hkv, L, dk, dv, kstride,
                                   vstride, float(scale), float(lam), Bc, n_splits,
                                   None if u is None else _ptr(u), nu,
                                   None if f is None else _ptr(f), int(bool(per_head)),
                                   _ptr(o_part), _ptr(lse_part), _ptr(skip), _ptr(margin))
    if rc:
        raise ValueError("bsa_oracle_decode: invalid arguments")
    return {"o_part": o_part, "lse_part": lse_part, "skip": skip, "margin": margin}


def decode_fp8(q, k8, v8, k_scale, v_scale, scale, lam, Bc, n_splits, units=None,
               force_skip=None):
    """Split-KV thresholded decode over an FP8 (E4M3) key/value cache, fp64.

    Reading (the pages name FP8/NVFP4 models but define no cache format): the
    cache holds E4M3 codes ``k8``, ``v8`` ``[B,Hkv,L,d]`` (uint8 bit patterns)
    and one fp32 scale per (sequence, KV head); the key and value rows are
    ``k_scale[b,h] * decode(k8)`` and ``v_scale[b,h] * decode(v8)``.  The
    scale of a key row multiplies its scores, so it is folded into the score
    scale (``scale * k_scale``, exact in double); the value scale multiplies
    the split outputs.  The query is used as given (bf16, widened exactly):
    the dequantised cache rows meet the caller's query.  Each (b, h) slice
    then runs :func:`decode` on the decoded codes, which are exact in fp32.
    ``units`` / ``force_skip`` as for :func:`decode`.  Returns the same dict."""
    import torch
    q = _f32(q)
    B, Hq, dk = q.shape
    k8 = torch.as_tensor(np.ascontiguousarray(k8, dtype=np.uint8))
    v8 = torch.as_tensor(np.ascontiguousarray(v8, dtype=np.uint8))
    kf = k8.view(torch.float8_e4m3fn).float().numpy()
    vf = v8.view(torch.float8_e4m3fn).float().numpy()
    _, Hkv, L, _ = kf.shape
    dv = vf.shape[3]
    ks = np.asarray(k_scale, dtype=np.float32).reshape(B, Hkv)
    vs = np.asarray(v_scale, dtype=np.float32).reshape(B, Hkv)
    G = Hq // Hkv
    n_b = -(-L // Bc)
    bps = -(-n_b // n_splits)
    o_part = np.zeros((B, Hq, n_splits, dv))
    lse_part = np.full((B, Hq, n_splits), np.nan)
    skip = np.zeros((B, Hkv, n_splits, bps), dtype=np.uint8)
    margin = np.full((B, Hkv, n_splits, bps), np.nan)
    want = None if units is None else set(int(x) // n_splits for x in np.asarray(units).ravel())
    for b in range(B):
        for h in range(Hkv):
            if want is not None and (b * Hkv + h) not in want:
                continue
            fs = None if force_skip is None else np.asarray(force_skip)[b:b + 1, h:h + 1]
            r = decode(q[b:b + 1, h * G:(h + 1) * G], kf[b:b + 1, h:h + 1], vf[b:b + 1, h:h + 1],
                       float(scale) * float(ks[b, h]), lam, Bc, n_splits, force_skip=fs)
            o_part[b, h * G:(h + 1) * G] = r["o_part"][0] * float(vs[b, h])
            lse_part[b, h * G:(h + 1) * G] = r["lse_part"][0]
            skip[b, h] = r["skip"][0, 0]
            margin[b, h] = r["margin"][0, 0]
    return {"o_part": o_part, "lse_part": lse_part, "skip": skip, "margin": margin}


def e2m1_decode(codes):
    """Values of E2M1 (FP4) codes: bit 3 the sign, bits 2-1 the exponent (bias
    1), bit 0 the mantissa; exponent 0 is subnormal (0 or 0.5)."""
    c = np.asarray(codes).astype(np.int64)
    sgn = np.where(c & 8, -1.0, 1.0)
    e, m = (c >> 1) & 3, c & 1
    mag = np.where(e == 0, 0.5 * m, np.exp2(e - 1.0) * (1.0 + 0.5 * m))
    return sgn * mag


def nvfp4_rows(x4, bs8):
    """Rows of an NVFP4 cache without its per-(sequence, head) scale: the two
    E2M1 codes of each byte of ``x4`` [..., d/2] (element 2i in the low
    nibble) times the E4M3 scale ``bs8`` [..., d/16] of their 16-element
    block; exact in fp32 (two by four significant bits)."""
    import torch
    x4 = np.ascontiguousarray(x4, dtype=np.uint8)
    codes = np.empty(x4.shape[:-1] + (2 * x4.shape[-1],), dtype=np.uint8)
    codes[..., 0::2] = x4 & 0xF
    codes[..., 1::2] = x4 >> 4
    bs = torch.as_tensor(np.ascontiguousarray(bs8, dtype=np.uint8)).view(
        torch.float8_e4m3fn).double().numpy()
    return (e2m1_decode(codes) * np.repeat(bs, 16, axis=-1)).astype(np.float32)


def decode_nvfp4(q, k4, v4, k_bs, v_bs, k_scale, v_scale, scale, lam, Bc, n_splits,
                 units=None, force_skip=None):
    """Split-KV thresholded decode over an NVFP4 key/value cache, fp64.

    Reading (the pages name NVFP4 models but define no cache format): a row
    element is ``s * E4M3(block scale) * E2M1(code)`` with one fp32 ``s`` per
    (sequence, KV head) and one E4M3 block scale per 16 consecutive elements
    (:func:`nvfp4_rows`).  As for the FP8 cache, the key scale ``s`` is folded
    into the score scale and the value scale multiplies the split outputs; the
    query is used as given (bf16).  Each (b, h) slice then runs
    :func:`decode`.  ``units`` / ``force_skip`` as for :func:`decode`."""
    q = _f32(q)
    B, Hq, dk = q.shape
    kf, vf = nvfp4_rows(k4, k_bs), nvfp4_rows(v4, v_bs)
    _, Hkv, L, _ = kf.shape
    dv = vf.shape[3]
    ks = np.asarray(k_scale, dtype=np.float32).reshape(B, Hkv)
    vs = np.asarray(v_scale, dtype=np.float32).reshape(B, Hkv)
    G = Hq // Hkv
    n_b = -(-L // Bc)
    bps = -(-n_b // n_splits)
    o_part = np.zeros((B, Hq, n_splits, dv))
    lse_part = np.full((B, Hq, n_splits), np.nan)
    skip = np.zeros((B, Hkv, n_splits, bps), dtype=np.uint8)
    margin = np.full((B, Hkv, n_splits, bps), np.nan)
    want = None if units is None else set(int(x) // n_splits for x in np.asarray(units).ravel())
    for b in range(B):
        for h in range(Hkv):
            if want is not None and (b * Hkv + h) not in want:
                continue
            fs = None if force_skip is None else np.asarray(force_skip)[b:b + 1, h:h + 1]
            r = decode(q[b:b + 1, h * G:(h + 1) * G], kf[b:b + 1, h:h + 1], vf[b:b + 1, h:h + 1],
                       float(scale) * float(ks[b, h]), lam, Bc, n_splits, force_skip=fs)
            o_part[b, h * G:(h + 1) * G] = r["o_part"][0] * float(vs[b, h])
            lse_part[b, h * G:(h + 1) * G] = r["lse_part"][0]
            skip[b, h] = r["skip"][0, 0]
            margin[b, h] = r["margin"][0, 0]
    return {"o_part": o_part, "lse_part": lse_part, "skip": skip, "margin": margin}


def combine(o_part, lse_part):
    """LSE merge of split partials: returns ``(o [B,Hq,dv], lse [B,Hq])``."""
    o_part = np.ascontiguousarray(o_part, dtype=np.float64)
    lse_part = np.ascontiguousarray(lse_part, dtype=np.float64)
    B, Hq, S, dv = o_part.shape
    o = np.zeros((B, Hq, dv))
    lse = np.zeros((B, Hq))
    rc = _load().bsa_oracle_combine(_ptr(o_part), _ptr(lse_part), B, Hq, S, dv, _ptr(o), _ptr(lse))
    if rc:
        raise ValueError("bsa_oracle_combine: invalid arguments")
    return o, lse


def prefill_varlen(q, k, v, cu_seqlens, scale, lambdas, Br=128, Bc=128, causal=True,
                   max_seqlen=None):
    """Batched variable-length prefill in fp64: every sequence is its own
    thresholded prefill (the loop of :func:`prefill` with B = 1) with its own
    threshold ``lambdas[s]`` (the BLASST page, section "λ = a/L：反比关系的直觉与
    依据": the threshold of a sequence scales as a / L with its length).

    q ``[total, Hq, dk]``, k ``[total, Hkv, dk]``, v ``[total, Hkv, dv]``
    (token-major, sequence s at tokens ``[cu[s], cu[s+1])``).  Returns ``o``
    ``[total, Hq, dv]``, ``lse`` ``[Hq, total]``, ``skip`` and ``margin``
    ``[n_seq, Hq, n_t, n_t]`` with ``n_t = ceil(max_seqlen / Br)`` (blocks a
    sequence does not have read 0 and NaN)."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    lam = np.asarray(lambdas, dtype=np.float64)
    n_seq = len(cu) - 1
    total, Hq, _ = q.shape
    dv = v.shape[2]
    lens = np.diff(cu)
    mx = int(lens.max()) if max_seqlen is None else int(max_seqlen)
    if Br != Bc:
        raise ValueError("prefill_varlen: Br must equal Bc")
    n_t = -(-mx // Br)
    o = np.zeros((total, Hq, dv))
    lse = np.full((Hq, total), np.nan)
    skip = np.zeros((n_seq, Hq, n_t, n_t), dtype=np.uint8)
    margin = np.full((n_seq, Hq, n_t, n_t), np.nan)
    for s in range(n_seq):
        c0, c1 = int(cu[s]), int(cu[s + 1])
        if c1 == c0:
            continue
        qs = np.ascontiguousarray(q[c0:c1].transpose(1, 0, 2)[None])
        ks = np.ascontiguousarray(k[c0:c1].transpose(1, 0, 2)[None])
        vs = np.ascontiguousarray(v[c0:c1].transpose(1, 0, 2)[None])
        r = prefill(qs, ks, vs, scale, float(lam[s]), Br, Bc, causal)
        o[c0:c1] = r["o"][0].transpose(1, 0, 2)
        lse[:, c0:c1] = r["lse"][0]
        nt = r["skip"].shape[2]
        skip[s, :, :nt, :nt] = r["skip"][0]
        margin[s, :, :nt, :nt] = r["margin"][0]
    return {"o": o, "lse": lse, "skip": skip, "margin": margin}


SANTA_MODES = {"iid": 0, "sys": 1, "strat": 2}


def santa_decode(q, k, v, scale, n_samples, mode, u, with_cdf=False):
    """Sampled decode output (SANTA estimator) in fp64.

    q [B,Hq,dk]; k [B,Hkv,L,dk]; v [B,Hkv,L,dv].  ``mode`` is ``"iid"``
    (thresholds T_m = u[b,h,m]), ``"sys"`` (T_m = (m + u[b,h]) / S) or
    ``"strat"`` (T_m = (m + u[b,h,m]) / S); every u lies in [0, 1).  Returns
    ``y`` [B,Hq,dv] (mean of the sampled value rows), ``idx`` [B,Hq,S] (int32
    sample indices), ``gap`` [B,Hq,S] (distance of each threshold from the
    nearer end of its key's CDF interval) and, with ``with_cdf``, ``cdf``
    [B,Hq,L]."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, Hq, dk = q.shape
    _, Hkv, L, kstride = k.shape
    dv, vstride = v.shape[3], v.shape[3]
    S = int(n_samples)
    md = SANTA_MODES[mode]
    uu = _f32(u)
    want = (B, Hq) if md == 1 else (B, Hq, S)
    if uu.shape != want:
        raise ValueError(f"u has shape {uu.shape}, expected {want}")
    y = np.zeros((B, Hq, dv))
    idx = np.zeros((B, Hq, S), dtype=np.int32)
    gap = np.zeros((B, Hq, S))
    cdf = np.zeros((B, Hq, L)) if with_cdf else None
    rc = _load().bsa_oracle_santa_decode(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, L, dk, dv,
                                         kstride, vstride, float(scale), S, md, _ptr(uu),
                                         _ptr(y), _ptr(idx), _ptr(gap),
                                         None if cdf is None else _ptr(cdf))
    if rc:
        raise ValueError("bsa_oracle_santa_decode: invalid arguments")
    out = {"y": y, "idx": idx, "gap": gap}
    if with_cdf:
        out["cdf"] = cdf
    return out


def ln_lambda(lam: float) -> float:
    return math.log(lam) if lam > 0 else -math.inf
