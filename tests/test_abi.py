"""The C-ABI library loads, exports every declared symbol, and validates its
arguments on the host (CPU only: no call here reaches a kernel launch)."""
import ctypes
import os
import re

import pytest

from block_sparse_attention_online_gb300 import binding as bs
from block_sparse_attention_online_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return bs.load()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "attn_skip.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_skip_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    syms = declared_symbols()
    assert "attn_skip_prefill" in syms and "attn_skip_decode_combine" in syms
    for s in syms:
        assert hasattr(lib, s), s
    assert set(syms) == set(bs.EXPORTED)


def test_status_strings(lib):
    for code in range(5):
        assert bs.status_string(code)
    assert "invalid" in bs.status_string(bs.ATTN_EINVAL)


FAKE = ctypes.c_void_p(0x10000)  # aligned, never dereferenced: validation fails first


def _prefill(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dt=0, B=1, Hq=4, Hkv=2, T=256, dk=128, dv=128, scale=0.0,
             lam=0.01, Br=128, Bc=128, causal=1, o=FAKE, lse=FAKE, bits=FAKE, stream=None)
    a.update(kw)
    return lib.attn_skip_prefill(*a.values())


@pytest.mark.parametrize("kw", [
    dict(q=None), dict(o=None), dict(bits=None), dict(B=0), dict(T=-1), dict(Hq=3),
    dict(lam=-0.1), dict(lam=1.0), dict(lam=float("nan")), dict(scale=float("nan")),
    dict(dt=7), dict(q=ctypes.c_void_p(0x10004)), dict(Br=0),
])
def test_prefill_rejects_invalid_arguments(lib, kw):
    assert _prefill(lib, **kw) == bs.ATTN_EINVAL


def _prefill_host(lib, **kw):
    a = dict(qh=FAKE, kh=FAKE, vh=FAKE, qd=FAKE, kd=FAKE, vd=FAKE, dt=0, B=1, Hq=4, Hkv=2, T=256,
             dk=128, dv=128, scale=0.0, lam=0.01, Br=128, Bc=128, causal=1, o=FAKE, lse=FAKE,
             bits=FAKE, oh=FAKE, lh=FAKE, n_groups=2, stream=None, si=None, so=None)
    a.update(kw)
    return lib.attn_skip_prefill_from_host(*a.values())


@pytest.mark.parametrize("kw", [
    dict(qh=None), dict(vh=None), dict(oh=None), dict(lh=None), dict(qd=None), dict(o=None),
    dict(bits=None), dict(n_groups=-1), dict(n_groups=3), dict(Hq=3), dict(lam=1.0),
    dict(kd=ctypes.c_void_p(0x10004)),
])
def test_prefill_from_host_rejects_invalid_arguments(lib, kw):
    """Argument errors are found before any copy or event (n_groups must lie
    in 1 .. B * Hkv; here B * Hkv = 2)."""
    assert _prefill_host(lib, **kw) == bs.ATTN_EINVAL


def test_prefill_from_host_unsupported_shape(lib):
    assert _prefill_host(lib, dk=64, dv=64) == bs.ATTN_EUNSUPPORTED


def _decode(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dt=0, B=2, Hq=8, Hkv=2, L=1024, dk=128, dv=128, ks=128,
             vs=128, scale=0.0, lam=0.01, Bc=128, n=4, op=FAKE, lp=FAKE, bits=FAKE, stream=None)
    a.update(kw)
    return lib.attn_skip_decode(*a.values())


@pytest.mark.parametrize("kw", [
    dict(k=None), dict(lp=None), dict(n=0), dict(L=0), dict(Hq=6, Hkv=4), dict(lam=1.5),
    dict(ks=64), dict(bits=None), dict(v=ctypes.c_void_p(0x10002)),
])
def test_decode_rejects_invalid_arguments(lib, kw):
    assert _decode(lib, **kw) == bs.ATTN_EINVAL


def _prefill_blocks(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dt=0, B=1, Hq=4, Hkv=2, T=256, dk=128, dv=128, scale=0.0,
             lam=0.01, Br=128, Bc=128, causal=1, set=FAKE, o=FAKE, lse=FAKE, bits=FAKE,
             stream=None)
    a.update(kw)
    return lib.attn_skip_prefill_blocks(*a.values())


@pytest.mark.parametrize("kw", [
    dict(set=None), dict(set=ctypes.c_void_p(0x10004)), dict(o=None), dict(q=None),
    dict(lam=1.0), dict(Hq=3), dict(T=0),
])
def test_prefill_blocks_rejects_invalid_arguments(lib, kw):
    assert _prefill_blocks(lib, **kw) == bs.ATTN_EINVAL


def test_decode_per_head_rejects_invalid_arguments(lib):
    f = lib.attn_skip_decode_per_head
    base = [FAKE, FAKE, FAKE, 0, 2, 8, 2, 1024, 128, 128, 128, 128, 0.0, 0.01, 128, 4, FAKE, FAKE,
            FAKE, None]
    for i, bad in ((0, None), (16, None), (18, None), (4, 0), (13, 1.0), (15, 0)):
        args = list(base)
        args[i] = bad
        assert f(*args) == bs.ATTN_EINVAL


def _prefill_margins(lib, **kw):
    a = dict(q=FAKE, k=FAKE, dt=0, B=1, Hq=4, Hkv=2, T=256, dk=128, scale=0.0, Br=128, Bc=128,
             causal=1, m=FAKE, stream=None)
    a.update(kw)
    return lib.attn_skip_prefill_margins(*a.values())


@pytest.mark.parametrize("kw", [
    dict(q=None), dict(k=None), dict(m=None), dict(m=ctypes.c_void_p(0x10008)), dict(B=0),
    dict(Hq=3), dict(scale=float("nan")), dict(dt=5), dict(Bc=0),
])
def test_prefill_margins_rejects_invalid_arguments(lib, kw):
    assert _prefill_margins(lib, **kw) == bs.ATTN_EINVAL


def _decode_margins(lib, **kw):
    a = dict(q=FAKE, k=FAKE, dt=0, B=2, Hq=8, Hkv=2, L=1024, dk=128, ks=128, scale=0.0, Bc=128,
             n=4, m=FAKE, stream=None)
    a.update(kw)
    return lib.attn_skip_decode_margins(*a.values())


@pytest.mark.parametrize("kw", [
    dict(q=None), dict(m=None), dict(n=0), dict(L=0), dict(Hq=6, Hkv=4), dict(ks=64),
    dict(k=ctypes.c_void_p(0x10002)),
])
def test_decode_margins_rejects_invalid_arguments(lib, kw):
    assert _decode_margins(lib, **kw) == bs.ATTN_EINVAL


def test_combine_rejects_invalid_arguments(lib):
    f = lib.attn_skip_decode_combine
    assert f(None, FAKE, 1, 1, 1, 128, 0, FAKE, FAKE, None) == bs.ATTN_EINVAL
    assert f(FAKE, FAKE, 1, 1, 0, 128, 0, FAKE, FAKE, None) == bs.ATTN_EINVAL
    assert f(FAKE, FAKE, 1, 1, 4, 128, 5, FAKE, FAKE, None) == bs.ATTN_EINVAL


def test_bitmap_shapes():
    assert bs.prefill_bitmap_shape(1, 32, 16384, 128, 128) == (1, 32, 128, 4)
    assert bs.decode_bitmap_shape(16, 8, 32768, 128, 8) == (16, 8, 8, 1)
    assert bs.decode_bitmap_shape(32, 1, 16384, 64, 16) == (32, 1, 16, 1)


def test_unpack_bits_roundtrip():
    import torch
    w = torch.tensor([[0b1011, -1]], dtype=torch.int32)
    u = bs.unpack_bits(w, 40)
    assert u[0, :4].tolist() == [True, True, False, True]
    assert u[0, 4:32].sum() == 0 and u[0, 32:40].all()


def _santa(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dt=0, B=2, Hq=8, Hkv=2, L=4096, dk=128, dv=128, ks=128,
             vs=128, scale=0.0, S=128, mode=1, u=FAKE, T=4, scores=FAKE, stats=FAKE, odt=1,
             o=FAKE, idx=None, stream=None)
    a.update(kw)
    return lib.attn_skip_santa_decode(*a.values())


@pytest.mark.parametrize("kw", [
    dict(q=None), dict(u=None), dict(scores=None), dict(stats=None), dict(o=None), dict(B=0),
    dict(L=0), dict(S=0), dict(T=0), dict(Hq=6, Hkv=4), dict(mode=3), dict(mode=-1),
    dict(odt=9), dict(dt=4), dict(ks=64), dict(scale=float("nan")),
    dict(u=ctypes.c_void_p(0x10004)), dict(idx=ctypes.c_void_p(0x10008)),
])
def test_santa_rejects_invalid_arguments(lib, kw):
    assert _santa(lib, **kw) == bs.ATTN_EINVAL


@pytest.mark.parametrize("kw", [
    dict(dk=64, ks=64), dict(dt=1), dict(S=4096), dict(L=32768, T=8),
    dict(Hq=6, Hkv=2), dict(T=2000),
])
def test_santa_unsupported_shapes(lib, kw):
    assert _santa(lib, **kw) == bs.ATTN_EUNSUPPORTED


def test_santa_workspace_sizes(lib):
    assert bs.attn_skip_santa_workspace(16, 32, 32768, 16) == (16 * 32 * 32768, 16 * 32 * 16 * 2)
    assert bs.attn_skip_santa_workspace(1, 1, 1, 1) == (128, 2)
    with pytest.raises(bs.AttnSkipError):
        bs.attn_skip_santa_workspace(1, 0, 10, 1)


def _varlen(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dt=0, n=3, cu=FAKE, mx=512, total=900, Hq=8, Hkv=2, dk=128,
             dv=128, scale=0.0, lam=FAKE, Br=128, Bc=128, causal=1, o=FAKE, lse=FAKE, bits=FAKE,
             stream=None)
    a.update(kw)
    return lib.attn_skip_prefill_varlen(*a.values())


@pytest.mark.parametrize("kw", [
    dict(cu=None), dict(lam=None), dict(q=None), dict(o=None), dict(lse=None), dict(bits=None),
    dict(n=0), dict(mx=-1), dict(total=-5), dict(Hq=6, Hkv=4), dict(dt=3),
    dict(scale=float("nan")), dict(q=ctypes.c_void_p(0x10008)), dict(cu=ctypes.c_void_p(0x10002)),
])
def test_varlen_rejects_invalid_arguments(lib, kw):
    assert _varlen(lib, **kw) == bs.ATTN_EINVAL


@pytest.mark.parametrize("kw", [dict(dt=1), dict(dk=64, dv=64), dict(Br=64), dict(Bc=64)])
def test_varlen_unsupported_shapes(lib, kw):
    assert _varlen(lib, **kw) == bs.ATTN_EUNSUPPORTED


def test_varlen_nothing_to_do_without_tiles(lib):
    # max_seqlen = 0: every sequence is empty, no tile row exists, nothing launches
    assert _varlen(lib, mx=0, total=0, q=None, k=None, v=None, o=None, lse=None,
                   bits=None) == bs.ATTN_OK
