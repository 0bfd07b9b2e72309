"""The FP8- and NVFP4-cache decodes over caches whose rows are padded: the C
ABI's row strides (bytes, multiples of 16) larger than a row.  The results
must be those of the same call over the dense cache, bit for bit: the
kernels read the same values.  The padding holds large codes, so any read of
it would change the scores."""
import pytest
import torch

from block_sparse_attention_online_gb300 import binding as bs
from block_sparse_attention_online_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _padded(x, row_bytes, fill):
    B, H, L, r = x.shape
    p = torch.full((B, H, L, row_bytes), fill, dtype=torch.uint8, device=x.device)
    p[..., :r] = x
    return p


def _outs(cfg, n_splits, dev):
    o = torch.empty(cfg.B, cfg.Hq, n_splits, 128, dtype=torch.float32, device=dev)
    lse = torch.empty(cfg.B, cfg.Hq, n_splits, dtype=torch.float32, device=dev)
    bits = torch.empty(bs.decode_bitmap_shape(cfg.B, cfg.Hkv, cfg.L, 128, n_splits),
                       dtype=torch.int32, device=dev)
    return o, lse, bits


@pytest.mark.parametrize("L,n_splits", [(3000, 4), (1000, 16)])
def test_nvfp4_decode_padded_rows(L, n_splits):
    cfg = W.temperate(W.GQA_DECODE_NVFP4_32K.with_(B=2, Hq=8, Hkv=2, L=L, seed=91))
    dev = torch.device("cuda")
    q, k4, v4, kbs, vbs, ks, vs = (x.to(dev) for x in W.decode_inputs_nvfp4(cfg))
    lam = 0.05
    ref = bs.attn_skip_decode_nvfp4(q, k4, v4, kbs, vbs, ks, vs, lam, 128, n_splits)
    kp, vp = _padded(k4, 96, 0x77), _padded(v4, 128, 0x77)  # E2M1 code 7 = 6.0
    o, lse, bits = _outs(cfg, n_splits, dev)
    st = bs.load().attn_skip_decode_nvfp4(
        bs._ptr(q), bs._ptr(kp), bs._ptr(vp), bs._ptr(kbs), bs._ptr(vbs), bs._ptr(ks),
        bs._ptr(vs), cfg.B, cfg.Hq, cfg.Hkv, L, 128, 128, 96, 128, 0.0, lam, 128, n_splits,
        bs._ptr(o), bs._ptr(lse), bs._ptr(bits), bs._stream(None, dev))
    assert st == bs.ATTN_OK
    torch.cuda.synchronize()
    bs.attn_skip_last_device_error()
    for got, want in zip((o, lse, bits), ref):
        assert torch.equal(got, want)


@pytest.mark.parametrize("L,n_splits", [(3000, 4), (1000, 16)])
def test_fp8_decode_padded_rows(L, n_splits):
    cfg = W.temperate(W.GQA_DECODE_FP8_32K.with_(B=2, Hq=8, Hkv=2, L=L, seed=92))
    dev = torch.device("cuda")
    q, k8, v8, ks, vs = (x.to(dev) for x in W.decode_inputs_fp8(cfg))
    lam = 0.05
    ref = bs.attn_skip_decode_fp8(q, k8, v8, ks, vs, lam, 128, n_splits)
    kp, vp = _padded(k8, 144, 0x7E), _padded(v8, 256, 0x7E)  # E4M3 0x7E = 448
    o, lse, bits = _outs(cfg, n_splits, dev)
    st = bs.load().attn_skip_decode_fp8(
        bs._ptr(q), bs._ptr(kp), bs._ptr(vp), bs._ptr(ks), bs._ptr(vs), cfg.B, cfg.Hq,
        cfg.Hkv, L, 128, 128, 144, 256, 0.0, lam, 128, n_splits, bs._ptr(o), bs._ptr(lse),
        bs._ptr(bits), bs._stream(None, dev))
    assert st == bs.ATTN_OK
    torch.cuda.synchronize()
    bs.attn_skip_last_device_error()
    for got, want in zip((o, lse, bits), ref):
        assert torch.equal(got, want)
