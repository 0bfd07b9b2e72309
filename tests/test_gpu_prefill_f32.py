"""fp32 CUDA-core prefill on the GPU against the fp64 oracle (tiny workload and
edge cases: ragged tails, Br != Bc, GQA, non-causal, lambda near 1)."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_online_gb300 import binding as bs
from block_sparse_attention_online_gb300 import workloads as W
from tests.parity import check_outputs, compare_bits

pytestmark = pytest.mark.gpu


def check_prefill(cfg, q, k, v, lam, kind):
    dev = torch.device("cuda")
    o, lse, bits = bs.attn_skip_prefill(q.to(dev), k.to(dev), v.to(dev), lam, cfg.Br, cfg.Bc,
                                        cfg.causal)
    bs.attn_skip_last_device_error()
    skip = bs.unpack_bits(bits, cfg.n_b).numpy()
    r = oracle.prefill(q, k, v, cfg.scale, lam, cfg.Br, cfg.Bc, cfg.causal)
    n_bad, flips = compare_bits(skip, r["skip"], r["margin"], lam)
    assert n_bad == 0, f"{n_bad} skip bits differ outside the margin band"
    if flips.any():
        r = oracle.prefill(q, k, v, cfg.scale, lam, cfg.Br, cfg.Bc, cfg.causal,
                           force_skip=skip.astype(np.uint8))
    check_outputs(o.float().cpu().numpy(), r["o"], lse.cpu().numpy(), r["lse"], kind, "prefill")
    trav = np.isfinite(r["margin"])
    return float(skip[trav].mean())


@pytest.mark.parametrize("lam", [0.0, 1e-3, 1e-2])
def test_tiny_prefill_f32(lam):
    """batch 1, one head, d=64, T=1024, causal, fp32, Br=Bc=128."""
    cfg = W.TINY_PREFILL
    q, k, v = W.prefill_inputs(cfg)
    s = check_prefill(cfg, q, k, v, lam, "f32")
    if lam == 0.0:
        assert s == 0.0
    else:
        assert s > 0.3


@pytest.mark.parametrize("T,Br,Bc", [(1000, 128, 128), (300, 64, 64), (333, 128, 64),
                                     (257, 64, 128)])
def test_prefill_f32_ragged_and_tiles(T, Br, Bc):
    cfg = W.temperate(W.TINY_PREFILL.with_(T=T, Br=Br, Bc=Bc, Hq=4, Hkv=2, seed=41))
    q, k, v = W.prefill_inputs(cfg)
    for lam in (0.0, 1e-2, 0.3):
        check_prefill(cfg, q, k, v, lam, "f32")


def test_prefill_f32_noncausal_d32_and_lambda_near_one():
    cfg = W.temperate(W.TINY_PREFILL.with_(T=500, d=32, causal=False, Br=64, Bc=64, seed=42))
    q, k, v = W.prefill_inputs(cfg)
    for lam in (1e-3, 0.999):
        check_prefill(cfg, q, k, v, lam, "f32")
