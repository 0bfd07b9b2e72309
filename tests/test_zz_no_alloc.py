"""attn_skip_santa_decode_noalloc: the sampled decode output with both
workspaces in the library's own device memory.

It is meant for callers that cannot allocate device memory at the point where
they decode (a plugin interface that hands over only input and output
pointers, an engine whose device memory is reserved up front, a loop that
cannot take cudaMalloc's device-wide synchronisation).  Its results must be
those of attn_skip_santa_decode with caller workspaces, call after call,
whatever an earlier call left in the shared scratch.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_sparse_attention_online_gb300 import binding as bs
from block_sparse_attention_online_gb300 import build as B
from block_sparse_attention_online_gb300 import workloads as W

FAKE = ctypes.c_void_p(0x10000)  # aligned, never dereferenced: the size check fails first


def _noalloc(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dt=0, B=4, Hq=32, Hkv=8, L=32768, dk=128, dv=128, ks=128,
             vs=128, scale=0.0, S=128, mode=1, u=FAKE, T=16, odt=1, o=FAKE, idx=None,
             stream=None)
    a.update(kw)
    return lib.attn_skip_santa_decode_noalloc(*a.values())


@pytest.mark.parametrize("kw", [
    dict(B=5),                      # 5 * 32 * 32768 score floats > 4,194,304
    dict(L=32769),                  # one more 128-key block per head
    dict(B=32, L=128, T=64),        # 32 * 32 * 64 * 2 statistics floats > 65,536
    dict(B=1 << 20, Hq=1 << 20),    # a product that would wrap in 32 bits
    dict(B=0), dict(L=0), dict(T=0),
])
def test_noalloc_rejects_sizes_beyond_the_scratch(kw):
    """Checked on the host before any CUDA call (runs without a GPU)."""
    B.build()
    assert _noalloc(bs.load(), **kw) == bs.ATTN_EINVAL


def _inputs(cfg, S, mode, seed):
    q, k, v = W.decode_inputs(cfg)
    u = W.santa_offsets(cfg, S, mode, seed=seed)
    dev = torch.device("cuda")
    return q.to(dev), k.to(dev), v.to(dev), u.to(dev)


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point_on_calls_in_a_row():
    # At the score-stash limit (4 * 32 * 32768 floats), then a ragged length
    # with stratified samples, then the first case again over what the second
    # left in the scratch.
    case_a = (W.SANTA_DECODE_32K.with_(B=4), 128, "sys", 16, 1)
    case_b = (W.SANTA_DECODE_32K.with_(B=2, Hq=8, Hkv=2, L=5000, seed=45), 256, "strat", 5, 2)
    want = {}
    for name, (cfg, S, mode, n_tiles, seed) in (("a", case_a), ("b", case_b)):
        q, k, v, u = _inputs(cfg, S, mode, seed)
        o, idx = bs.attn_skip_santa_decode(q, k, v, S, mode, u, n_tiles=n_tiles, with_idx=True)
        bs.attn_skip_last_device_error()
        want[name] = (o.cpu(), idx.cpu(), float(v.float().abs().max()))
        del q, k, v, u, o, idx
    torch.cuda.synchronize()

    calls = 0
    for name, (cfg, S, mode, n_tiles, seed) in (("a", case_a), ("b", case_b), ("a", case_a)):
        q, k, v, u = _inputs(cfg, S, mode, seed)
        torch.cuda.synchronize()
        o = torch.full((cfg.B, cfg.Hq, 128), float("nan"), device="cuda")
        idx = torch.full((cfg.B, cfg.Hq, S), -1, dtype=torch.int32, device="cuda")
        before = torch.cuda.memory_allocated()
        free_before = torch.cuda.mem_get_info()[0]
        bs.attn_skip_santa_decode_noalloc(q, k, v, S, mode, u, o, idx, n_tiles=n_tiles)
        bs.attn_skip_last_device_error()
        # torch's counter sees its own caching allocator; the driver's free
        # bytes also see a cudaMalloc made inside the library.  The first call
        # may load the library's device code (the scratch array included), so
        # the driver figure is compared from the second call on.
        assert torch.cuda.memory_allocated() == before
        if calls:
            assert torch.cuda.mem_get_info()[0] == free_before
        calls += 1
        o_ref, idx_ref, vmax = want[name]
        assert torch.equal(idx.cpu(), idx_ref)
        err = (o.cpu().double() - o_ref.double()).abs().max().item()
        assert np.isfinite(err) and err <= 1e-6 * vmax
        del q, k, v, u


@pytest.mark.gpu
def test_noalloc_binding_reports_the_limit():
    cfg = W.SANTA_DECODE_32K.with_(B=1, Hq=8, Hkv=2, L=600, seed=46)
    q, k, v, u = _inputs(cfg, 32, "sys", 3)
    o = torch.empty(cfg.B, cfg.Hq, 128, device="cuda")
    with pytest.raises(bs.AttnSkipError, match="scratch"):
        bs.attn_skip_santa_decode_noalloc(q, k, v, 32, "sys", u, o, n_tiles=4200)
    # within the limits, an invalid argument of the sampled decode itself is
    # not reported as the scratch limit
    k3 = torch.zeros(cfg.B, 3, cfg.L, 128, dtype=k.dtype, device="cuda")  # 8 % 3 != 0
    with pytest.raises(bs.AttnSkipError) as e:
        bs.attn_skip_santa_decode_noalloc(q, k3, k3, 32, "sys", u, o, n_tiles=4)
    assert e.value.status == bs.ATTN_EINVAL and "scratch" not in str(e.value)
