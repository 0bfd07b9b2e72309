"""Pins of the batched variable-length prefill oracle (CPU only).

Each packed sequence is an independent causal prefill with its own threshold.
The pins reach the oracle through routes it does not use: torch's fp64 SDPA
on the sequence cut out of the packed tensors (a wrong offset, a transposed
token/head axis or a sequence bleeding into its neighbour fails it), the
closed-form softmax over each sequence's kept tokens, and the monotonicity of
the skip set in lambda.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from block_sparse_attention_online_gb300 import workloads as W
from tests.test_oracle import kept_token_mask, scores_full, softmax_rows

LENS = (0, 1, 127, 128, 129, 300, 0, 64)


def _small(temperate=False, lengths=LENS, Br=64):
    cfg = W.VarlenConfig("t", lengths, 4, 2, 32, dtype="f32", Br=Br, Bc=Br, seed=21)
    if temperate:
        cfg = cfg.with_(sink_a=3.0, salient_a=1.5)
    q, k, v, cu = W.varlen_inputs(cfg)
    return cfg, q, k, v, cu.numpy()


def _seq(x, cu, s):
    """[1, H, T_s, d] fp64 slice of a packed [total, H, d] tensor."""
    return x[cu[s]:cu[s + 1]].double().transpose(0, 1)[None]


def test_varlen_lambda0_is_sdpa_per_sequence():
    cfg, q, k, v, cu = _small()
    r = oracle.prefill_varlen(q, k, v, cu, cfg.scale, np.zeros(cfg.n_seq), cfg.Br, cfg.Bc, True)
    for s in range(cfg.n_seq):
        if cu[s + 1] == cu[s]:
            continue
        qs, ks, vs = _seq(q, cu, s), _seq(k, cu, s), _seq(v, cu, s)
        ks = ks.repeat_interleave(cfg.G, dim=1)
        vs = vs.repeat_interleave(cfg.G, dim=1)
        want = F.scaled_dot_product_attention(qs, ks, vs, is_causal=True, scale=cfg.scale)
        got = torch.from_numpy(r["o"][cu[s]:cu[s + 1]]).transpose(0, 1)[None]
        torch.testing.assert_close(got, want, rtol=1e-10, atol=1e-11)
        sc = cfg.scale * qs @ ks.transpose(-1, -2)
        T = qs.shape[2]
        sc = sc.masked_fill(~torch.tril(torch.ones(T, T, dtype=torch.bool)), float("-inf"))
        lse = torch.logsumexp(sc, dim=-1)[0]
        np.testing.assert_allclose(r["lse"][:, cu[s]:cu[s + 1]], lse.numpy(), rtol=1e-12,
                                   atol=1e-11)
    # no bit is set at lambda = 0; blocks a sequence does not have stay NaN
    assert r["skip"].sum() == 0
    assert np.isnan(r["margin"][0]).all()


@pytest.mark.parametrize("lams", [(1e-4, 1e-3, 3e-2, 1e-2, 0.2, 5e-2, 0.1, 1e-3),
                                  (0.3, 0.3, 0.3, 0.3, 0.3, 0.3, 0.3, 0.3)])
def test_varlen_output_is_softmax_over_each_sequences_kept_tokens(lams):
    cfg, q, k, v, cu = _small(temperate=True)
    r = oracle.prefill_varlen(q, k, v, cu, cfg.scale, np.float32(lams), cfg.Br, cfg.Bc, True)
    skipped = 0
    for s in range(cfg.n_seq):
        T = int(cu[s + 1] - cu[s])
        if T == 0:
            continue
        nt = -(-T // cfg.Br)
        qs, ks, vs = (_seq(x, cu, s).numpy() for x in (q, k, v))
        sc = scores_full(qs, ks, cfg.scale, True)
        km = kept_token_mask(r["skip"][s:s + 1, :, :nt, :nt], T, cfg.Br, cfg.Bc, True)
        p, lse = softmax_rows(np.where(km, sc, -np.inf))
        y = np.einsum("bhrc,bhce->bhre", p, np.repeat(vs, cfg.G, axis=1))
        np.testing.assert_allclose(r["o"][cu[s]:cu[s + 1]], y[0].transpose(1, 0, 2),
                                   rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(r["lse"][:, cu[s]:cu[s + 1]], lse[0], rtol=1e-12,
                                   atol=1e-11)
        skipped += int(r["skip"][s].sum())
        # nothing outside the sequence's own tiles and blocks
        assert r["skip"][s, :, nt:].sum() == 0 and r["skip"][s, :, :, nt:].sum() == 0
    assert skipped > 0


def test_varlen_larger_lambda_skips_a_superset():
    """Two copies of one sequence with thresholds 1e-3 and 3e-2: the same
    statistics, and the second skip set contains the first."""
    cfg, q, k, v, cu = _small(temperate=True, lengths=(300,))
    q2, k2, v2 = (torch.cat([x, x]) for x in (q, k, v))
    cu2 = np.array([0, 300, 600])
    r = oracle.prefill_varlen(q2, k2, v2, cu2, cfg.scale, np.float32([1e-3, 3e-2]), cfg.Br,
                              cfg.Bc, True)
    np.testing.assert_array_equal(r["margin"][0], r["margin"][1])
    a, b = r["skip"][0].astype(bool), r["skip"][1].astype(bool)
    assert (a <= b).all() and b.sum() > a.sum()


def test_varlen_generator_matches_per_sequence_draws():
    cfg = W.VarlenConfig("t", (70, 0, 200), 4, 2, 32, dtype="f32", seed=5)
    q, k, v, cu = W.varlen_inputs(cfg)
    assert cu.tolist() == [0, 70, 70, 270] and q.shape == (270, 4, 32)
    qs, ks, vs = W.prefill_inputs(cfg.sequence(2))
    assert torch.equal(q[70:270], qs[0].transpose(0, 1))
    assert torch.equal(v[70:270], vs[0].transpose(0, 1))
    assert not torch.equal(q[:70], qs[0, :, :70].transpose(0, 1))  # own seed per sequence
