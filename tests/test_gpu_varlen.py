"""Batched variable-length prefill (one threshold per sequence) on the GPU
against the fp64 oracle, and against the fixed-length kernel run on each
sequence alone."""

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_online_gb300 import binding as bs
from block_sparse_attention_online_gb300 import workloads as W
from tests.parity import check_outputs, compare_bits

pytestmark = pytest.mark.gpu


def run_varlen(cfg, q, k, v, cu, lams, causal=True):
    dev = torch.device("cuda")
    o, lse, bits = bs.attn_skip_prefill_varlen(q.to(dev), k.to(dev), v.to(dev), cu.to(dev),
                                               cfg.max_seqlen, lams.to(dev), causal)
    bs.attn_skip_last_device_error()
    n_t = -(-cfg.max_seqlen // 128)
    return o.float().cpu().numpy(), lse.cpu().numpy(), bs.unpack_bits(bits, n_t).numpy()


def check_varlen(cfg, q, k, v, cu, lams, causal=True, seqs=None):
    """Every sequence (or those in ``seqs``) against the oracle: bits exact
    outside the margin band, outputs within the bf16 tolerances; rows and
    bits of tiles a sequence does not have are untouched / zero."""
    o, lse, skip = run_varlen(cfg, q, k, v, cu, lams, causal)
    cu_np = cu.numpy()
    lam64 = lams.double().numpy()  # the fp32 values the kernel reads, widened
    n_t = skip.shape[2]
    seqs = range(cfg.n_seq) if seqs is None else seqs
    flips = 0
    for s in seqs:
        c0, c1 = int(cu_np[s]), int(cu_np[s + 1])
        T = c1 - c0
        nt = -(-T // 128)
        assert not skip[s, :, nt:].any() and not skip[s, :, :, nt:].any()
        if T == 0:
            continue
        qs, ks, vs = (x[c0:c1].transpose(0, 1)[None].contiguous() for x in (q, k, v))
        r = oracle.prefill(qs, ks, vs, cfg.scale, float(lam64[s]), 128, 128, causal)
        gs = skip[s:s + 1, :, :nt, :nt]
        n_bad, fl = compare_bits(gs, r["skip"], r["margin"], float(lam64[s]))
        assert n_bad == 0, f"sequence {s}: {n_bad} skip bits differ outside the margin band"
        if fl.any():
            flips += int(fl.sum())
            r = oracle.prefill(qs, ks, vs, cfg.scale, float(lam64[s]), 128, 128, causal,
                               force_skip=gs.astype(np.uint8))
        check_outputs(o[c0:c1].transpose(1, 0, 2), r["o"][0], lse[:, c0:c1], r["lse"][0], "bf16",
                      f"sequence {s} (T={T})")
    return skip, flips


LENS = (0, 1, 127, 128, 129, 300, 0, 2000, 4096, 777)


@pytest.mark.parametrize("causal", [True, False])
def test_varlen_mixed_lengths_per_sequence_lambda(causal):
    cfg = W.VarlenConfig("t", LENS, 8, 2, 128, sink_a=3.0, salient_a=1.5, seed=61)
    q, k, v, cu = W.varlen_inputs(cfg)
    lams = torch.tensor([0.0, 1e-3, 3e-2, 1e-4, 0.2, 1e-2, 0.5, 1e-3, 3e-3, 0.0],
                        dtype=torch.float32)
    skip, _ = check_varlen(cfg, q, k, v, cu, lams, causal)
    assert skip.sum() > 0
    assert not skip[0].any() and not skip[9].any()  # lambda = 0


def test_varlen_lambda_over_length():
    """lambda_s = a / L_s on the planted recipe: the threshold falls with the
    length as the page prescribes; every sequence matches the oracle."""
    cfg = W.VarlenConfig("t", (256, 512, 1024, 2048, 3000), 8, 2, 128, seed=62)
    q, k, v, cu = W.varlen_inputs(cfg)
    a = 2e-6
    lams = torch.tensor([min(a / L, 0.999) for L in cfg.lengths], dtype=torch.float32)
    skip, _ = check_varlen(cfg, q, k, v, cu, lams)
    assert skip.sum() > 0


def test_varlen_equals_the_fixed_length_kernel_per_sequence():
    """Each sequence of the packed batch gives bit for bit what
    attn_skip_prefill gives for it alone (same arithmetic, other layout)."""
    cfg = W.VarlenConfig("t", (1500, 128, 4000, 64, 2600), 32, 8, 128, seed=63)
    q, k, v, cu = W.varlen_inputs(cfg)
    lams = torch.tensor([1e-4, 0.0, 1e-6, 0.3, 1e-8], dtype=torch.float32)
    dev = torch.device("cuda")
    o, lse, bits = bs.attn_skip_prefill_varlen(q.to(dev), k.to(dev), v.to(dev), cu.to(dev),
                                               cfg.max_seqlen, lams.to(dev))
    bs.attn_skip_last_device_error()
    cu_np = cu.numpy()
    for s in range(cfg.n_seq):
        c0, c1 = int(cu_np[s]), int(cu_np[s + 1])
        qs, ks, vs = (x[c0:c1].transpose(0, 1)[None].contiguous().to(dev) for x in (q, k, v))
        o1, lse1, b1 = bs.attn_skip_prefill(qs, ks, vs, float(lams[s]), 128, 128, True)
        bs.attn_skip_last_device_error()
        nt = b1.shape[2]
        assert torch.equal(o[c0:c1].transpose(0, 1), o1[0])
        assert torch.equal(lse[:, c0:c1], lse1[0])
        assert torch.equal(bits[s, :, :nt, :b1.shape[3]], b1[0])


def test_varlen_full_size_workload():
    """The benchmark's batch: 16 sequences, 129 to 16384 tokens (65,536 in
    all), 32/8 heads, lambda_s = a / L_s; the short sequences against the
    oracle, all of them against the fixed-length kernel."""
    cfg = W.VARLEN_PREFILL_64K
    q, k, v, cu = W.varlen_inputs(cfg)
    a = 1e-4 * 4096
    lams = torch.tensor([min(a / L, 0.999) for L in cfg.lengths], dtype=torch.float32)
    short = [s for s in range(cfg.n_seq) if cfg.lengths[s] <= 1536]
    skip, _ = check_varlen(cfg, q, k, v, cu, lams, seqs=short)
    dev = torch.device("cuda")
    o, lse, bits = bs.attn_skip_prefill_varlen(q.to(dev), k.to(dev), v.to(dev), cu.to(dev),
                                               cfg.max_seqlen, lams.to(dev))
    bs.attn_skip_last_device_error()
    cu_np = cu.numpy()
    for s in range(cfg.n_seq):
        c0, c1 = int(cu_np[s]), int(cu_np[s + 1])
        qs, ks, vs = (x[c0:c1].transpose(0, 1)[None].contiguous().to(dev) for x in (q, k, v))
        o1, lse1, b1 = bs.attn_skip_prefill(qs, ks, vs, float(lams[s]), 128, 128, True)
        assert torch.equal(o[c0:c1].transpose(0, 1), o1[0]), f"sequence {s}"
        assert torch.equal(lse[:, c0:c1], lse1[0])
        assert torch.equal(bits[s, :, :b1.shape[2], :b1.shape[3]], b1[0])
    bs.attn_skip_last_device_error()
    assert skip.sum() > 0


def test_varlen_empty_batch_and_bad_device_arguments():
    dev = torch.device("cuda")
    z = torch.empty(0, 4, 128, dtype=torch.bfloat16, device=dev)
    zk = torch.empty(0, 2, 128, dtype=torch.bfloat16, device=dev)
    cu = torch.zeros(3, dtype=torch.int32, device=dev)
    lams = torch.zeros(2, dtype=torch.float32, device=dev)
    out = (torch.empty(0, 4, 128, dtype=torch.bfloat16, device=dev),
           torch.empty(4, 0, device=dev),
           torch.full(bs.varlen_bitmap_shape(2, 4, 256), -1, dtype=torch.int32, device=dev))
    bs.attn_skip_prefill_varlen(z, zk, zk, cu, 256, lams, out=out)  # total 0, max_seqlen 256
    bs.attn_skip_last_device_error()
    assert (out[2] == 0).all()
    # A length above max_seqlen and a lambda >= 1: the kernel treats the first
    # sequence as empty and the threshold as 0, and reports ATTN_EINVAL.
    cfg = W.VarlenConfig("t", (300, 200), 4, 2, 128, seed=64)
    q, k, v, cu = W.varlen_inputs(cfg)
    with pytest.raises(bs.AttnSkipError) as e:
        bs.attn_skip_prefill_varlen(q.to(dev), k.to(dev), v.to(dev), cu.to(dev), 256,
                                    torch.tensor([0.0, 1.5], device=dev))
        bs.attn_skip_last_device_error()
    assert e.value.status == bs.ATTN_EINVAL
    bs.attn_skip_last_device_error()  # cleared


@pytest.mark.parametrize("n_seq", [33, 150])
def test_varlen_many_sequences(n_seq):
    """More sequences than one warp holds (33) and than the registers cache
    (150): the general tile locator; empty sequences among them."""
    g = np.random.default_rng(n_seq)
    lens = tuple(int(x) for x in g.choice([0, 1, 64, 128, 129, 200, 383, 700], size=n_seq))
    cfg = W.VarlenConfig("t", lens, 4, 2, 128, sink_a=3.0, salient_a=1.5, seed=65)
    q, k, v, cu = W.varlen_inputs(cfg)
    lams = torch.tensor(g.choice([0.0, 1e-3, 3e-2], size=n_seq), dtype=torch.float32)
    check_varlen(cfg, q, k, v, cu, lams, seqs=range(0, n_seq, 7))
    dev = torch.device("cuda")
    o, lse, bits = bs.attn_skip_prefill_varlen(q.to(dev), k.to(dev), v.to(dev), cu.to(dev),
                                               cfg.max_seqlen, lams.to(dev))
    bs.attn_skip_last_device_error()
    cu_np = cu.numpy()
    for s in range(n_seq):
        c0, c1 = int(cu_np[s]), int(cu_np[s + 1])
        if c1 == c0:
            assert not bits[s].any()
            continue
        qs, ks, vs = (x[c0:c1].transpose(0, 1)[None].contiguous().to(dev) for x in (q, k, v))
        o1, lse1, b1 = bs.attn_skip_prefill(qs, ks, vs, float(lams[s]), 128, 128, True)
        assert torch.equal(o[c0:c1].transpose(0, 1), o1[0]), f"sequence {s}"
        assert torch.equal(lse[:, c0:c1], lse1[0])
        assert torch.equal(bits[s, :, :b1.shape[2], :b1.shape[3]], b1[0])
        assert not bits[s, :, b1.shape[2]:].any()
