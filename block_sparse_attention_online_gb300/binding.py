"""ctypes binding of ``libattn_skip.so`` (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: it checks tensor placement, allocates the outputs with
torch (device memory is plumbing), passes raw pointers and the current CUDA
stream, and raises :class:`AttnSkipError` on a non-OK status.  There is no CPU
fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build",
                         "libattn_skip.so")
_lib = None

ATTN_OK, ATTN_EINVAL, ATTN_EUNSUPPORTED, ATTN_ECUDA, ATTN_ETIMEOUT, ATTN_EINTERNAL = range(6)
ATTN_BF16, ATTN_F32 = 0, 1

#: Every symbol include/attn_skip.h declares.
EXPORTED = ("attn_skip_prefill", "attn_skip_prefill_from_host", "attn_skip_prefill_blocks",
            "attn_skip_prefill_varlen",
            "attn_skip_decode", "attn_skip_decode_fp8", "attn_skip_decode_nvfp4",
            "attn_skip_decode_per_head", "attn_skip_decode_combine",
            "attn_skip_prefill_margins", "attn_skip_decode_margins", "attn_skip_sparsity_at",
            "attn_skip_lambda_for_sparsity", "attn_skip_fit_lambda_model",
            "attn_skip_lambda_for_target", "attn_skip_selftest_wait_timeout",
            "attn_skip_last_device_error", "attn_skip_status_string",
            "attn_skip_santa_workspace", "attn_skip_santa_decode",
            "attn_skip_santa_decode_noalloc")

#: Samplers of attn_skip_santa_decode.
SANTA_MODES = {"iid": 0, "sys": 1, "strat": 2}


class AttnSkipError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


def library_path() -> str:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load the library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                           "`python -m block_sparse_attention_online_gb300.build`")
    lib = ctypes.CDLL(_LIB_PATH)
    P, i, f, d, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_int64
    lib.attn_skip_prefill.argtypes = [P, P, P, i, i, i, i, i, i, i, f, d, i, i, i, P, P, P, P]
    lib.attn_skip_prefill_from_host.argtypes = [P, P, P, P, P, P, i, i, i, i, i, i, i, f, d, i, i,
                                                i, P, P, P, P, P, i, P, P, P]
    lib.attn_skip_prefill_blocks.argtypes = [P, P, P, i, i, i, i, i, i, i, f, d, i, i, i, P, P, P,
                                             P, P]
    lib.attn_skip_prefill_varlen.argtypes = [P, P, P, i, i, P, i, i, i, i, i, i, f, P, i, i, i,
                                             P, P, P, P]
    lib.attn_skip_decode_fp8.argtypes = [P, P, P, P, P, i, i, i, i, i, i, i64, i64, f, d, i, i,
                                         P, P, P, P]
    lib.attn_skip_decode_nvfp4.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, i, i64, i64, f,
                                           d, i, i, P, P, P, P]
    lib.attn_skip_decode.argtypes = [P, P, P, i, i, i, i, i, i, i, i64, i64, f, d, i, i, P, P, P,
                                     P]
    lib.attn_skip_decode_combine.argtypes = [P, P, i, i, i, i, i, P, P, P]
    lib.attn_skip_decode_per_head.argtypes = [P, P, P, i, i, i, i, i, i, i, i64, i64, f, d, i,
                                              i, P, P, P, P]
    lib.attn_skip_prefill_margins.argtypes = [P, P, i, i, i, i, i, i, f, i, i, i, P, P]
    lib.attn_skip_decode_margins.argtypes = [P, P, i, i, i, i, i, i, i64, f, i, i, P, P]
    lib.attn_skip_sparsity_at.argtypes = [P, i64, d]
    lib.attn_skip_sparsity_at.restype = d
    lib.attn_skip_lambda_for_sparsity.argtypes = [P, i64, d, P]
    lib.attn_skip_fit_lambda_model.argtypes = [P, P, P, i, P, P]
    lib.attn_skip_lambda_for_target.argtypes = [d, d, d, d]
    lib.attn_skip_lambda_for_target.restype = d
    lib.attn_skip_last_device_error.argtypes = [P]
    lib.attn_skip_selftest_wait_timeout.argtypes = [P]
    lib.attn_skip_santa_workspace.argtypes = [i, i, i, i, P, P]
    lib.attn_skip_santa_decode.argtypes = [P, P, P, i, i, i, i, i, i, i, i64, i64, f, i, i, P, i,
                                           P, P, i, P, P, P]
    lib.attn_skip_santa_decode_noalloc.argtypes = [P, P, P, i, i, i, i, i, i, i, i64, i64, f, i,
                                                   i, P, i, i, P, P, P]
    lib.attn_skip_status_string.argtypes = [i]
    lib.attn_skip_status_string.restype = ctypes.c_char_p
    for fn in ("attn_skip_prefill", "attn_skip_prefill_blocks", "attn_skip_prefill_varlen",
               "attn_skip_decode", "attn_skip_decode_fp8", "attn_skip_decode_nvfp4",
               "attn_skip_decode_per_head", "attn_skip_decode_combine",
               "attn_skip_prefill_margins", "attn_skip_decode_margins",
               "attn_skip_lambda_for_sparsity", "attn_skip_fit_lambda_model",
               "attn_skip_selftest_wait_timeout", "attn_skip_last_device_error",
               "attn_skip_santa_workspace", "attn_skip_santa_decode",
               "attn_skip_santa_decode_noalloc"):
        getattr(lib, fn).restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().attn_skip_status_string(int(status)).decode()


attn_skip_status_string = status_string


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float32:
        return ATTN_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr() if t.numel() else None)


def _check(fn: str, status: int):
    if status != ATTN_OK:
        raise AttnSkipError(fn, status)


def _cuda_contig(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def prefill_bitmap_shape(B, Hq, T, Br, Bc):
    n_t, n_b = -(-T // Br), -(-T // Bc)
    return (B, Hq, n_t, -(-n_b // 32))


def decode_bitmap_shape(B, Hkv, L, Bc, n_splits):
    n_b = -(-L // Bc)
    bps = -(-n_b // n_splits)
    return (B, Hkv, n_splits, -(-bps // 32))


def attn_skip_prefill(q, k, v, lam, Br=128, Bc=128, causal=True, scale=0.0, out=None,
                      stream=None):
    """q [B,Hq,T,dk], k [B,Hkv,T,dk], v [B,Hkv,T,dv] on one CUDA device.

    Returns ``(o, lse, skip_bits)``; ``out`` may pass preallocated
    ``(o, lse, skip_bits)`` tensors."""
    _cuda_contig(q, k, v)
    B, Hq, T, dk = q.shape
    Hkv, dv = k.shape[1], v.shape[3]
    if out is None:
        o = torch.empty(B, Hq, T, dv, dtype=q.dtype, device=q.device)
        lse = torch.empty(B, Hq, T, dtype=torch.float32, device=q.device)
        bits = torch.empty(prefill_bitmap_shape(B, Hq, T, Br, Bc), dtype=torch.int32,
                           device=q.device)
    else:
        o, lse, bits = out
    st = load().attn_skip_prefill(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), B, Hq, Hkv, T, dk,
                                  dv, float(scale), float(lam), Br, Bc, int(bool(causal)),
                                  _ptr(o), _ptr(lse), _ptr(bits), _stream(stream, q.device))
    _check("attn_skip_prefill", st)
    return o, lse, bits


def attn_skip_prefill_from_host(q, k, v, lam, dev, out_host, Br=128, Bc=128, causal=True,
                                scale=0.0, n_groups=0, stream=None, copy_streams=(None, None)):
    """The prefill with host-resident inputs and outputs, the copies overlapped
    with the computation over groups of KV heads.

    ``q, k, v`` are CPU tensors (pinned for asynchronous copies) in the
    layouts of :func:`attn_skip_prefill`; ``dev`` holds the device tensors
    ``(q_dev, k_dev, v_dev, o_dev, lse_dev, skip_bits)``; ``out_host`` the CPU
    tensors ``(o, lse)`` written once ``stream`` has reached the end of the
    call.  ``copy_streams`` are the CUDA streams of the copies in and out
    (None: ``stream``).  Returns ``out_host``."""
    for x in (q, k, v, *out_host):
        if x.is_cuda or not x.is_contiguous():
            raise ValueError("host tensors must be contiguous CPU tensors")
    qd, kd, vd, od, ld, bd = dev
    _cuda_contig(qd, kd, vd, od, ld, bd)
    B, Hq, T, dk = q.shape
    Hkv, dv = k.shape[1], v.shape[3]
    o, lse = out_host
    cs = tuple(None if c is None else _stream(c, qd.device) for c in copy_streams)
    st = load().attn_skip_prefill_from_host(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        _ptr(qd), _ptr(kd), _ptr(vd), _dtype_code(q), B, Hq, Hkv, T, dk, dv, float(scale),
        float(lam), Br, Bc, int(bool(causal)), _ptr(od), _ptr(ld), _ptr(bd),
        ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()), int(n_groups),
        _stream(stream, qd.device), cs[0], cs[1])
    _check("attn_skip_prefill_from_host", st)
    return out_host


def pack_block_set(allow: torch.Tensor) -> torch.Tensor:
    """Pack a bool tensor [..., n_b] (True = block in the set) into uint32 words
    [..., ceil(n_b/32)], stored as int32, on the tensor's device."""
    n = allow.shape[-1]
    w = -(-n // 32)
    a = torch.zeros(*allow.shape[:-1], w * 32, dtype=torch.int64, device=allow.device)
    a[..., :n] = allow.to(torch.int64)
    a = a.reshape(*allow.shape[:-1], w, 32)
    words = (a << torch.arange(32, dtype=torch.int64, device=allow.device)).sum(-1)
    return torch.where(words >= (1 << 31), words - (1 << 32), words).to(torch.int32)


def attn_skip_prefill_blocks(q, k, v, lam, block_set, Br=128, Bc=128, causal=True, scale=0.0,
                             out=None, stream=None):
    """Prefill restricted to a block set: ``block_set`` is the packed uint32
    mask [B,Hq,n_t,words] (see :func:`pack_block_set`) on the inputs' device.
    Returns ``(o, lse, skip_bits)``."""
    _cuda_contig(q, k, v, block_set)
    B, Hq, T, dk = q.shape
    Hkv, dv = k.shape[1], v.shape[3]
    if tuple(block_set.shape) != prefill_bitmap_shape(B, Hq, T, Br, Bc):
        raise ValueError(f"block_set has shape {tuple(block_set.shape)}, expected "
                         f"{prefill_bitmap_shape(B, Hq, T, Br, Bc)}")
    if out is None:
        o = torch.empty(B, Hq, T, dv, dtype=q.dtype, device=q.device)
        lse = torch.empty(B, Hq, T, dtype=torch.float32, device=q.device)
        bits = torch.empty(prefill_bitmap_shape(B, Hq, T, Br, Bc), dtype=torch.int32,
                           device=q.device)
    else:
        o, lse, bits = out
    st = load().attn_skip_prefill_blocks(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), B, Hq, Hkv,
                                         T, dk, dv, float(scale), float(lam), Br, Bc,
                                         int(bool(causal)), _ptr(block_set), _ptr(o), _ptr(lse),
                                         _ptr(bits), _stream(stream, q.device))
    _check("attn_skip_prefill_blocks", st)
    return o, lse, bits


def varlen_bitmap_shape(n_seq, Hq, max_seqlen, Br=128):
    n_t = -(-int(max_seqlen) // Br)
    return (int(n_seq), int(Hq), n_t, -(-n_t // 32))


def attn_skip_prefill_varlen(q, k, v, cu_seqlens, max_seqlen, lambdas, causal=True, scale=0.0,
                             Br=128, Bc=128, out=None, stream=None):
    """Batched variable-length prefill.  q [total,Hq,dk], k/v [total,Hkv,d]
    token-major; ``cu_seqlens`` int32 [n_seq+1] and ``lambdas`` fp32 [n_seq]
    on the inputs' device.  Returns ``(o [total,Hq,dv], lse [Hq,total],
    skip_bits [n_seq,Hq,n_t,words])``."""
    _cuda_contig(q, k, v, cu_seqlens, lambdas)
    if cu_seqlens.dtype != torch.int32 or lambdas.dtype != torch.float32:
        raise TypeError("cu_seqlens must be int32 and lambdas float32")
    total, Hq, dk = q.shape
    Hkv, dv = k.shape[1], v.shape[2]
    n_seq = cu_seqlens.numel() - 1
    if lambdas.numel() != n_seq:
        raise ValueError(f"lambdas has {lambdas.numel()} entries, expected {n_seq}")
    if out is None:
        o = torch.empty(total, Hq, dv, dtype=q.dtype, device=q.device)
        lse = torch.empty(Hq, total, dtype=torch.float32, device=q.device)
        bits = torch.empty(varlen_bitmap_shape(n_seq, Hq, max_seqlen, Br), dtype=torch.int32,
                           device=q.device)
    else:
        o, lse, bits = out
    st = load().attn_skip_prefill_varlen(
        _ptr(q), _ptr(k), _ptr(v), _dtype_code(q), n_seq, _ptr(cu_seqlens), int(max_seqlen),
        total, Hq, Hkv, dk, dv, float(scale), _ptr(lambdas), Br, Bc, int(bool(causal)), _ptr(o),
        _ptr(lse), _ptr(bits), _stream(stream, q.device))
    _check("attn_skip_prefill_varlen", st)
    return o, lse, bits


def attn_skip_decode(q, k, v, lam, Bc=128, n_splits=8, dv=None, scale=0.0, out=None,
                     stream=None):
    """q [B,Hq,dk], k [B,Hkv,L,dk], v [B,Hkv,L,dv] or ``None`` (values are the
    first ``dv`` columns of each key row).  Returns fp32 ``(o_part, lse_part,
    skip_bits)``."""
    _cuda_contig(q, k)
    B, Hq, dk = q.shape
    _, Hkv, L, kstride = k.shape
    if v is None:
        vv, vstride = k, kstride
        if dv is None:
            raise ValueError("dv is required when values alias the keys")
    else:
        _cuda_contig(v)
        vv, dv, vstride = v, v.shape[3], v.shape[3]
    if out is None:
        o_part = torch.empty(B, Hq, n_splits, dv, dtype=torch.float32, device=q.device)
        lse_part = torch.empty(B, Hq, n_splits, dtype=torch.float32, device=q.device)
        bits = torch.empty(decode_bitmap_shape(B, Hkv, L, Bc, n_splits), dtype=torch.int32,
                           device=q.device)
    else:
        o_part, lse_part, bits = out
    st = load().attn_skip_decode(_ptr(q), _ptr(k), _ptr(vv), _dtype_code(q), B, Hq, Hkv, L, dk,
                                 dv, kstride, vstride, float(scale), float(lam), Bc, n_splits,
                                 _ptr(o_part), _ptr(lse_part), _ptr(bits),
                                 _stream(stream, q.device))
    _check("attn_skip_decode", st)
    return o_part, lse_part, bits


def attn_skip_decode_per_head(q, k, v, lam, Bc=128, n_splits=8, dv=None, scale=0.0, out=None,
                              stream=None):
    """Decode with per-head decisions (GQA shape, or MLA with ``v=None`` and
    ``dv``): returns fp32 ``(o_part, lse_part, skip_bits)`` with bits per
    query head [B,Hq,S,words]."""
    _cuda_contig(q, k)
    B, Hq, dk = q.shape
    _, Hkv, L, kstride = k.shape
    if v is None:
        v, vstride = k, kstride
        if dv is None:
            raise ValueError("dv is required when values alias the keys")
    else:
        _cuda_contig(v)
        dv, vstride = v.shape[3], v.shape[3]
    if out is None:
        o_part = torch.empty(B, Hq, n_splits, dv, dtype=torch.float32, device=q.device)
        lse_part = torch.empty(B, Hq, n_splits, dtype=torch.float32, device=q.device)
        bits = torch.empty(decode_bitmap_shape(B, Hq, L, Bc, n_splits), dtype=torch.int32,
                           device=q.device)
    else:
        o_part, lse_part, bits = out
    st = load().attn_skip_decode_per_head(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), B, Hq, Hkv,
                                          L, dk, dv, kstride, vstride, float(scale), float(lam),
                                          Bc, n_splits, _ptr(o_part), _ptr(lse_part),
                                          _ptr(bits), _stream(stream, q.device))
    _check("attn_skip_decode_per_head", st)
    return o_part, lse_part, bits


def attn_skip_decode_fp8(q, k8, v8, k_scale, v_scale, lam, Bc=128, n_splits=8, scale=0.0,
                         out=None, stream=None):
    """Decode over an FP8 cache: q [B,Hq,128] bf16, k8/v8 [B,Hkv,L,128] uint8
    E4M3 codes, k_scale/v_scale [B,Hkv] fp32, all on one device.  Returns
    fp32 ``(o_part, lse_part, skip_bits)`` like :func:`attn_skip_decode`."""
    _cuda_contig(q, k8, v8, k_scale, v_scale)
    if k8.dtype != torch.uint8 or v8.dtype != torch.uint8:
        raise TypeError("k8 and v8 must be uint8 E4M3 codes")
    if k_scale.dtype != torch.float32 or v_scale.dtype != torch.float32:
        raise TypeError("scales must be float32")
    B, Hq, dk = q.shape
    _, Hkv, L, dv = v8.shape
    if out is None:
        o = torch.empty(B, Hq, n_splits, dv, dtype=torch.float32, device=q.device)
        lse = torch.empty(B, Hq, n_splits, dtype=torch.float32, device=q.device)
        bits = torch.empty(decode_bitmap_shape(B, Hkv, L, Bc, n_splits), dtype=torch.int32,
                           device=q.device)
    else:
        o, lse, bits = out
    st = load().attn_skip_decode_fp8(_ptr(q), _ptr(k8), _ptr(v8), _ptr(k_scale), _ptr(v_scale),
                                     B, Hq, Hkv, L, dk, dv, k8.shape[3], v8.shape[3],
                                     float(scale), float(lam), Bc, n_splits, _ptr(o), _ptr(lse),
                                     _ptr(bits), _stream(stream, q.device))
    _check("attn_skip_decode_fp8", st)
    return o, lse, bits


def attn_skip_decode_nvfp4(q, k4, v4, k_bs, v_bs, k_scale, v_scale, lam, Bc=128, n_splits=8,
                           scale=0.0, out=None, stream=None):
    """Decode over an NVFP4 cache: q [B,Hq,128] bf16; k4/v4 [B,Hkv,L,64] uint8
    (two E2M1 codes per byte, element 2i in the low nibble); k_bs/v_bs
    [B,Hkv,L,8] uint8 E4M3 block scales; k_scale/v_scale [B,Hkv] fp32; all on
    one device.  Returns fp32 ``(o_part, lse_part, skip_bits)`` like
    :func:`attn_skip_decode`."""
    _cuda_contig(q, k4, v4, k_bs, v_bs, k_scale, v_scale)
    for t in (k4, v4, k_bs, v_bs):
        if t.dtype != torch.uint8:
            raise TypeError("codes and block scales must be uint8")
    if k_scale.dtype != torch.float32 or v_scale.dtype != torch.float32:
        raise TypeError("scales must be float32")
    B, Hq, dk = q.shape
    _, Hkv, L, half = v4.shape
    dv = 2 * half
    if k_bs.shape != (B, Hkv, L, dk // 16) or v_bs.shape != (B, Hkv, L, dv // 16):
        raise ValueError("block scales must be [B, Hkv, L, d/16]")
    if out is None:
        o = torch.empty(B, Hq, n_splits, dv, dtype=torch.float32, device=q.device)
        lse = torch.empty(B, Hq, n_splits, dtype=torch.float32, device=q.device)
        bits = torch.empty(decode_bitmap_shape(B, Hkv, L, Bc, n_splits), dtype=torch.int32,
                           device=q.device)
    else:
        o, lse, bits = out
    st = load().attn_skip_decode_nvfp4(_ptr(q), _ptr(k4), _ptr(v4), _ptr(k_bs), _ptr(v_bs),
                                       _ptr(k_scale), _ptr(v_scale), B, Hq, Hkv, L, dk, dv,
                                       k4.shape[3], v4.shape[3], float(scale), float(lam), Bc,
                                       n_splits, _ptr(o), _ptr(lse), _ptr(bits),
                                       _stream(stream, q.device))
    _check("attn_skip_decode_nvfp4", st)
    return o, lse, bits


def attn_skip_decode_combine(o_part, lse_part, out_dtype=torch.bfloat16, out=None, stream=None):
    """Merge ``o_part`` [B,Hq,S,dv] / ``lse_part`` [B,Hq,S] into ``(o, lse)``."""
    _cuda_contig(o_part, lse_part)
    B, Hq, S, dv = o_part.shape
    if out is None:
        o = torch.empty(B, Hq, dv, dtype=out_dtype, device=o_part.device)
        lse = torch.empty(B, Hq, dtype=torch.float32, device=o_part.device)
    else:
        o, lse = out
    st = load().attn_skip_decode_combine(_ptr(o_part), _ptr(lse_part), B, Hq, S, dv,
                                         _dtype_code(o), _ptr(o), _ptr(lse),
                                         _stream(stream, o_part.device))
    _check("attn_skip_decode_combine", st)
    return o, lse


def prefill_margin_shape(B, Hq, T, Br, Bc):
    return (B, Hq, -(-T // Br), -(-T // Bc))


def decode_margin_shape(B, Hkv, L, Bc, n_splits):
    n_b = -(-L // Bc)
    return (B, Hkv, n_splits, -(-n_b // n_splits))


def attn_skip_prefill_margins(q, k, Br=128, Bc=128, causal=True, scale=0.0, out=None,
                              stream=None):
    """Statistics pass of the prefill kernel: fp32 ``margin`` [B,Hq,n_t,n_b]
    (NaN = not traversed) on the inputs' device."""
    _cuda_contig(q, k)
    B, Hq, T, dk = q.shape
    Hkv = k.shape[1]
    margin = out if out is not None else torch.empty(
        prefill_margin_shape(B, Hq, T, Br, Bc), dtype=torch.float32, device=q.device)
    st = load().attn_skip_prefill_margins(_ptr(q), _ptr(k), _dtype_code(q), B, Hq, Hkv, T, dk,
                                          float(scale), Br, Bc, int(bool(causal)), _ptr(margin),
                                          _stream(stream, q.device))
    _check("attn_skip_prefill_margins", st)
    return margin


def attn_skip_decode_margins(q, k, Bc=128, n_splits=8, scale=0.0, out=None, stream=None):
    """Statistics pass of the decode kernels: fp32 ``margin``
    [B,Hkv,n_splits,bps] (NaN past a split's last block)."""
    _cuda_contig(q, k)
    B, Hq, dk = q.shape
    _, Hkv, L, kstride = k.shape
    margin = out if out is not None else torch.empty(
        decode_margin_shape(B, Hkv, L, Bc, n_splits), dtype=torch.float32, device=q.device)
    st = load().attn_skip_decode_margins(_ptr(q), _ptr(k), _dtype_code(q), B, Hq, Hkv, L, dk,
                                         kstride, float(scale), Bc, n_splits, _ptr(margin),
                                         _stream(stream, q.device))
    _check("attn_skip_decode_margins", st)
    return margin


def _host_f32(margin):
    """A contiguous host fp32 copy of ``margin`` (torch tensor or numpy array)."""
    if isinstance(margin, torch.Tensor):
        m = margin.detach().to("cpu", torch.float32).contiguous()
    else:
        m = torch.from_numpy(np.ascontiguousarray(margin, dtype=np.float32))
    return m, ctypes.c_void_p(m.data_ptr()), m.numel()


def attn_skip_sparsity_at(margin, lam):
    """Fraction of the traversed blocks that ``lam`` skips (host computation)."""
    m, p, n = _host_f32(margin)
    r = load().attn_skip_sparsity_at(p, n, float(lam))
    if r < 0:
        raise AttnSkipError("attn_skip_sparsity_at", ATTN_EINVAL)
    return r


def attn_skip_lambda_for_sparsity(margin, target):
    """A lambda in [0, 1) that skips the fraction ``target`` of the traversed
    blocks of ``margin`` (host computation)."""
    m, p, n = _host_f32(margin)
    out = ctypes.c_double()
    st = load().attn_skip_lambda_for_sparsity(p, n, float(target), ctypes.byref(out))
    _check("attn_skip_lambda_for_sparsity", st)
    return out.value


def attn_skip_fit_lambda_model(lengths, sparsities, lambdas):
    """Least-squares ``(alpha, beta)`` of lambda * L = alpha * exp(beta * s)."""
    n = len(lengths)
    if len(sparsities) != n or len(lambdas) != n:
        raise ValueError("lengths, sparsities and lambdas must have equal length")
    arr = ctypes.c_double * n
    a_, b_ = ctypes.c_double(), ctypes.c_double()
    st = load().attn_skip_fit_lambda_model(arr(*map(float, lengths)), arr(*map(float, sparsities)),
                                           arr(*map(float, lambdas)), n, ctypes.byref(a_),
                                           ctypes.byref(b_))
    _check("attn_skip_fit_lambda_model", st)
    return a_.value, b_.value


def attn_skip_lambda_for_target(alpha, beta, sparsity, L):
    """lambda = alpha * exp(beta * S) / L, capped below 1."""
    return load().attn_skip_lambda_for_target(float(alpha), float(beta), float(sparsity),
                                              float(L))


def attn_skip_santa_workspace(B, Hq, L, n_tiles):
    """Sizes, in floats, of the score stash and the tile statistics."""
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    _check("attn_skip_santa_workspace",
           load().attn_skip_santa_workspace(int(B), int(Hq), int(L), int(n_tiles),
                                            ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def attn_skip_santa_decode(q, k, v, n_samples, mode, u, n_tiles=16, scale=0.0,
                           out_dtype=torch.float32, with_idx=False, workspace=None, out=None,
                           idx_out=None, stream=None):
    """Sampled decode output (SANTA estimator).  q [B,Hq,128], k/v
    [B,Hkv,L,128] bf16; ``mode`` ``"sys"`` (u [B,Hq]) or ``"strat"`` (u
    [B,Hq,S]), u fp32 in [0, 1) on the device.  Returns ``o`` [B,Hq,128] and,
    with ``with_idx``, the int32 sample indices [B,Hq,S].  ``workspace`` is
    an optional ``(scores, tile_stats)`` pair of fp32 device tensors of the
    sizes attn_skip_santa_workspace gives; ``out`` and ``idx_out`` optional
    preallocated outputs."""
    _cuda_contig(q, k, v, u)
    B, Hq, dk = q.shape
    _, Hkv, L, kstride = k.shape
    dv, vstride = v.shape[3], v.shape[3]
    if u.dtype != torch.float32:
        raise TypeError("u must be float32")
    if workspace is None:
        ns, nt = attn_skip_santa_workspace(B, Hq, L, n_tiles)
        workspace = (torch.empty(ns, dtype=torch.float32, device=q.device),
                     torch.empty(nt, dtype=torch.float32, device=q.device))
    scores, stats = workspace
    _cuda_contig(scores, stats)
    o = out if out is not None else torch.empty(B, Hq, dv, dtype=out_dtype, device=q.device)
    idx = idx_out
    if idx is None and with_idx:
        idx = torch.empty(B, Hq, int(n_samples), dtype=torch.int32, device=q.device)
    st = load().attn_skip_santa_decode(
        _ptr(q), _ptr(k), _ptr(v), _dtype_code(q), B, Hq, Hkv, L, dk, dv, kstride, vstride,
        float(scale), int(n_samples), SANTA_MODES[mode], _ptr(u), int(n_tiles), _ptr(scores),
        _ptr(stats), _dtype_code(o), _ptr(o), None if idx is None else _ptr(idx),
        _stream(stream, q.device))
    _check("attn_skip_santa_decode", st)
    return (o, idx) if with_idx else o


# Sizes of the library's built-in sampled-decode scratch, in floats.
NOALLOC_SCORE_FLOATS = 4 << 20
NOALLOC_STAT_FLOATS = 64 << 10


def attn_skip_santa_decode_noalloc(q, k, v, n_samples, mode, u, o, idx=None, n_tiles=16,
                                   scale=0.0, stream=None):
    """attn_skip_santa_decode with both workspaces in the library's own
    device memory, for callers that cannot allocate when they decode.  The
    caller passes the outputs: ``o`` [B,Hq,128] fp32 or bf16 and optionally
    ``idx`` [B,Hq,S] int32; nothing is allocated here or in the library.
    Sizes: B*Hq*ceil(L/128)*128 <= 4,194,304 and B*Hq*n_tiles*2 <= 65,536.
    Calls that overlap on the GPU share the scratch and race."""
    _cuda_contig(q, k, v, u, o)
    if idx is not None:
        _cuda_contig(idx)
        if idx.dtype != torch.int32:
            raise TypeError("idx must be int32")
    B, Hq, dk = q.shape
    _, Hkv, L, kstride = k.shape
    dv, vstride = v.shape[3], v.shape[3]
    if u.dtype != torch.float32:
        raise TypeError("u must be float32")
    st = load().attn_skip_santa_decode_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _dtype_code(q), B, Hq, Hkv, L, dk, dv, kstride, vstride,
        float(scale), int(n_samples), SANTA_MODES[mode], _ptr(u), int(n_tiles), _dtype_code(o),
        _ptr(o), None if idx is None else _ptr(idx), _stream(stream, q.device))
    over = (B * Hq * (-(-L // 128)) * 128 > NOALLOC_SCORE_FLOATS
            or B * Hq * int(n_tiles) * 2 > NOALLOC_STAT_FLOATS)
    if st == ATTN_EINVAL and over:
        raise AttnSkipError("attn_skip_santa_decode_noalloc (the built-in scratch holds "
                            f"B*Hq*ceil(L/128)*128 <= {NOALLOC_SCORE_FLOATS} score floats and "
                            f"B*Hq*n_tiles*2 <= {NOALLOC_STAT_FLOATS} statistics floats)", st)
    _check("attn_skip_santa_decode_noalloc", st)
    return o


def attn_skip_selftest_wait_timeout(stream=None, device=None):
    """Launch the diagnostic CTA whose bounded wait runs out (see the header)."""
    st = load().attn_skip_selftest_wait_timeout(_stream(stream, device))
    _check("attn_skip_selftest_wait_timeout", st)


def attn_skip_last_device_error(stream=None, device=None):
    st = load().attn_skip_last_device_error(_stream(stream, device))
    _check("attn_skip_last_device_error", st)


def unpack_bits(bits: torch.Tensor, n: int) -> torch.Tensor:
    """Expand uint32 bitmap words [..., W] into a bool tensor [..., n] (CPU)."""
    w = bits.to("cpu").to(torch.int64) & 0xFFFFFFFF
    shifts = torch.arange(32, dtype=torch.int64)
    b = ((w[..., :, None] >> shifts) & 1).reshape(*w.shape[:-1], w.shape[-1] * 32)
    return b[..., :n].bool()
