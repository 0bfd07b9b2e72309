"""The host-buffer prefill (copies in and out pipelined with the computation
over groups of KV heads): its outputs equal the device call's bit for bit, and
the device call is the one checked against the oracle elsewhere."""
import pytest
import torch

from block_sparse_attention_online_gb300 import binding as bs

pytestmark = pytest.mark.gpu


def _inputs(B, Hq, Hkv, T, seed):
    g = torch.Generator().manual_seed(seed)
    # every query leans on key 0 (a sink: its score ~22 against ~3 for the
    # rest), so a threshold skips most later blocks
    q = (torch.randn(B, Hq, T, 128, generator=g) + 0.5).to(torch.bfloat16)
    k = torch.randn(B, Hkv, T, 128, generator=g)
    k[:, :, 0] = 4.0
    v = torch.randn(B, Hkv, T, 128, generator=g).to(torch.bfloat16)
    return q, k.to(torch.bfloat16), v


@pytest.mark.parametrize("B,Hq,Hkv,T,n_groups,pinned,streams", [
    (2, 8, 2, 1100, 0, True, True),    # default grouping, ragged tail
    (2, 8, 2, 1100, 4, True, True),    # one KV head per group
    (2, 8, 2, 1100, 1, False, False),  # one group, pageable memory, one stream
    (1, 4, 4, 384, 3, True, False),    # G = 1, uneven groups
])
def test_prefill_from_host_matches_the_device_call(B, Hq, Hkv, T, n_groups, pinned, streams):
    dev = torch.device("cuda")
    q, k, v = _inputs(B, Hq, Hkv, T, seed=T + Hq)
    lam = 0.02
    o_ref, lse_ref, bits_ref = bs.attn_skip_prefill(q.to(dev), k.to(dev), v.to(dev), lam)
    if pinned:
        q, k, v = (x.pin_memory() for x in (q, k, v))
    o_h = torch.full((B, Hq, T, 128), float("nan"), dtype=torch.bfloat16)
    lse_h = torch.full((B, Hq, T), float("nan"), dtype=torch.float32)
    if pinned:
        o_h, lse_h = o_h.pin_memory(), lse_h.pin_memory()
    devbuf = (torch.empty_like(q, device=dev), torch.empty_like(k, device=dev),
              torch.empty_like(v, device=dev), torch.empty_like(o_ref), torch.empty_like(lse_ref),
              torch.empty_like(bits_ref))
    cs = (torch.cuda.Stream(), torch.cuda.Stream()) if streams else (None, None)
    for _ in range(2):  # twice: the second call reuses the staging buffers
        bs.attn_skip_prefill_from_host(q, k, v, lam, devbuf, (o_h, lse_h), n_groups=n_groups,
                                       copy_streams=cs)
    torch.cuda.current_stream().synchronize()
    bs.attn_skip_last_device_error()
    assert torch.equal(o_h, o_ref.cpu())
    assert torch.equal(lse_h, lse_ref.cpu())
    assert torch.equal(devbuf[5], bits_ref)
    skipped = int(bs.unpack_bits(bits_ref, -(-T // 128)).sum())
    assert skipped > 0  # the threshold did skip blocks
