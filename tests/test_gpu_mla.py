"""Absorbed-MLA split-KV decode (128 heads, 576-column latent, values = first
512 columns) on the GPU against the fp64 oracle."""
import json
import os

import pytest

from block_sparse_attention_online_gb300 import workloads as W
from tests.test_gpu_decode import check_decode

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _lambda(cfg_name, target):
    with open(os.path.join(GOLDEN, "lambdas.json")) as f:
        return json.load(f)[cfg_name][str(target)]["lambda"]


@pytest.mark.parametrize("L,n_splits", [(1000, 4), (2048, 16), (200, 6)])
def test_mla_small(L, n_splits):
    """Ragged last block (1000 = 15*64 + 40), one block per split, and empty splits."""
    cfg = W.MLA_DECODE_16K.with_(B=2, L=L, n_splits=n_splits, seed=61)
    q, k, _ = W.decode_inputs(cfg)
    for lam in (0.0, 1e-9, 1e-4):
        check_decode(cfg, q, k, None, lam, n_splits)


@pytest.mark.parametrize("lam", [1e-2, 0.3, 0.999])
def test_mla_temperate_mixtures(lam):
    cfg = W.temperate(W.MLA_DECODE_16K.with_(B=2, L=3000, n_splits=4, seed=62))
    q, k, _ = W.decode_inputs(cfg)
    check_decode(cfg, q, k, None, lam)


@pytest.mark.parametrize("target", ["0.0", "max"])
def test_mla_full_size(target):
    """B=32, 128 heads, L=16384, Bc=64, 16 splits.  On this workload about 65 %
    of the (split, block) pairs raise some head's running max, so ~35 % is the
    largest block sparsity any lambda < 1 reaches; "max" is that threshold."""
    cfg = W.MLA_DECODE_16K
    q, k, _ = W.decode_inputs(cfg)
    lam = 0.0 if target == "0.0" else _lambda(cfg.name, target)
    sparsity, _ = check_decode(cfg, q, k, None, lam)
    if target == "max":
        with open(os.path.join(GOLDEN, "lambdas.json")) as f:
            expect = json.load(f)[cfg.name]["max"]["sparsity"]
        assert abs(sparsity - expect) < 0.01, (sparsity, expect)


def test_mla_long_split_uses_the_two_cta_kernel():
    """A split of more than 2048 blocks (one split over 131,136 keys) runs the
    two-CTA kernel the cluster kernel hands over to; the same oracle checks it."""
    cfg = W.MLA_DECODE_16K.with_(B=1, L=2049 * 64 + 40, n_splits=1, seed=63)
    q, k, _ = W.decode_inputs(cfg)
    for lam in (0.0, 1e-9):
        check_decode(cfg, q, k, None, lam, 1)
