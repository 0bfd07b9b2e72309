"""Seeded synthetic inputs for softmax-threshold block-skipping attention.

This module only draws numbers: it holds none of the attention arithmetic, so
both the CUDA path and the fp64 oracle may read what it produces.

Planted-salience recipe (one draw per KV head, independent across heads):

* ``u`` is a seeded random unit vector scaled to length ``sqrt(d)``;
* keys ``K_j = N(0, I) + a_j * u`` with ``a_0 = sink_a`` (an attention sink),
  ``a_j = salient_a`` on a seeded fraction of the positions ``1..T-1`` drawn
  without replacement, ``a_j = 0`` elsewhere;
* queries ``Q_i = N(0, I) + u`` (every query head of the group uses its KV
  head's ``u``), values ``V ~ N(0, 1)``;
* optional local band (long prefill): query tile ``t`` adds ``w_t`` and key
  block ``b`` adds ``band_a * (w_b + w_{b+1})``, so tile ``t`` sees about
  ``+band_a * sqrt(d)`` on the scores of blocks ``t-1`` and ``t`` (its 256
  nearest keys at 128-wide blocks).  The ``w`` are seeded ``N(0, I)`` draws
  made orthogonal to ``u``;
* bf16 configurations round every element to bf16 (round to nearest even).

Heavy-tailed score distributions of this kind stand in for the long-context
benchmarks the BLASST page evaluates on (RULER, LongBench), which are not
available here.  Each (tensor, batch, head) slice has its own generator keyed
by (seed, tensor tag, batch, head), so any head can be regenerated alone and
slices can be drawn in parallel.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

import torch

_TAGS = {"u": 1, "sal": 2, "k": 3, "v": 4, "q": 5, "w": 6, "santa": 7}


def _gen(seed: int, tag: str, b: int, h: int) -> torch.Generator:
    # A fixed mixing of the key into one 63-bit seed (splitmix64 finaliser).
    x = (seed * 0x9E3779B97F4A7C15 + _TAGS[tag] * 0xBF58476D1CE4E5B9
         + b * 0x94D049BB133111EB + h * 0xD6E8FEB86659FD93 + 0x632BE59BD9B4E019)
    x &= (1 << 64) - 1
    x ^= x >> 30
    x = (x * 0xBF58476D1CE4E5B9) & ((1 << 64) - 1)
    x ^= x >> 27
    x = (x * 0x94D049BB133111EB) & ((1 << 64) - 1)
    x ^= x >> 31
    return torch.Generator().manual_seed(x & ((1 << 63) - 1))


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    T: int
    d: int
    dtype: str  # "bf16" or "f32"
    Br: int = 128
    Bc: int = 128
    causal: bool = True
    salient_frac: float = 0.02
    sink_a: float = 6.0
    salient_a: float = 3.0
    band_a: float = 0.0
    seed: int = 1234

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def n_t(self) -> int:
        return -(-self.T // self.Br)

    @property
    def n_b(self) -> int:
        return -(-self.T // self.Bc)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def with_(self, **kw) -> "PrefillConfig":
        return replace(self, **kw)


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    L: int
    dk: int
    dv: int
    dtype: str
    Bc: int = 128
    n_splits: int = 8
    latent: bool = False  # V is the first dv columns of K (absorbed MLA)
    salient_frac: float = 0.02
    sink_a: float = 6.0
    salient_a: float = 3.0
    seed: int = 1234

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def n_b(self) -> int:
        return -(-self.L // self.Bc)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.dk)

    def with_(self, **kw) -> "DecodeConfig":
        return replace(self, **kw)


# The five workloads: shapes follow the attention layers of the models the
# BLASST page evaluates (Llama-3.1-8B GQA 32/8 heads, d=128; DeepSeek-style
# absorbed MLA with a 512+64 latent).
TINY_PREFILL = PrefillConfig("tiny_prefill_f32_T1024", 1, 1, 1, 1024, 64, "f32", seed=1234)
GQA_PREFILL_16K = PrefillConfig("gqa_prefill_bf16_T16384", 1, 32, 8, 16384, 128, "bf16", seed=1235)
GQA_DECODE_32K = DecodeConfig("gqa_decode_bf16_B16_L32768", 16, 32, 8, 32768, 128, 128, "bf16",
                              Bc=128, n_splits=8, seed=1236)
GQA_PREFILL_64K = PrefillConfig("gqa_prefill_bf16_T65536_band", 1, 32, 8, 65536, 128, "bf16",
                                salient_frac=0.01, band_a=2.0, seed=1237)
MLA_DECODE_16K = DecodeConfig("mla_decode_bf16_B32_L16384", 32, 128, 1, 16384, 576, 512, "bf16",
                              Bc=64, n_splits=16, latent=True, seed=1238)

CONFIGS = {c.name: c for c in (TINY_PREFILL, GQA_PREFILL_16K, GQA_DECODE_32K, GQA_PREFILL_64K,
                                MLA_DECODE_16K)}

# The same decode shape with weak salience (sink 1.2, salient keys 0.6): each
# head's attention spreads over hundreds of keys (the top key holds 5-65 % of
# the mass, 90 % of it sits on ~150-400 keys), the regime in which sampling
# the value rows is worth doing.  With the default salience the sink holds all
# but e^-30 of the mass and every sample lands on it.
SANTA_DECODE_32K = GQA_DECODE_32K.with_(name="santa_decode_bf16_B16_L32768", sink_a=1.2,
                                        salient_a=0.6, seed=1239)


@dataclass(frozen=True)
class VarlenConfig:
    """A batch of independent causal prefills of different lengths, packed
    token-major: q ``[total, Hq, d]``, k and v ``[total, Hkv, d]``, sequence
    ``s`` at tokens ``[cu[s], cu[s+1])``.  Sequence ``s`` is drawn with the
    planted-salience recipe of :class:`PrefillConfig` under its own seed."""
    name: str
    lengths: tuple
    Hq: int
    Hkv: int
    d: int
    dtype: str = "bf16"
    Br: int = 128
    Bc: int = 128
    causal: bool = True
    salient_frac: float = 0.02
    sink_a: float = 6.0
    salient_a: float = 3.0
    seed: int = 1240

    @property
    def n_seq(self) -> int:
        return len(self.lengths)

    @property
    def total(self) -> int:
        return int(sum(self.lengths))

    @property
    def max_seqlen(self) -> int:
        return int(max(self.lengths)) if self.lengths else 0

    @property
    def cu_seqlens(self) -> tuple:
        out = [0]
        for L in self.lengths:
            out.append(out[-1] + int(L))
        return tuple(out)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def sequence(self, s: int) -> PrefillConfig:
        return PrefillConfig(f"{self.name}[{s}]", 1, self.Hq, self.Hkv, int(self.lengths[s]),
                             self.d, self.dtype, self.Br, self.Bc, self.causal,
                             self.salient_frac, self.sink_a, self.salient_a, 0.0,
                             seed=self.seed + 101 * (s + 1))

    def with_(self, **kw) -> "VarlenConfig":
        return replace(self, **kw)


# Sixteen sequences from 129 to 16384 tokens (ragged lengths included), the
# Llama-3.1-8B attention shape; 65,536 tokens in all.
VARLEN_PREFILL_64K = VarlenConfig(
    "gqa_prefill_varlen_bf16_16seq_64k",
    (16384, 12000, 8192, 6144, 5000, 4096, 3163, 2731, 2048, 1536, 1500, 1024, 777, 512, 300,
     129), 32, 8, 128)


def _unit_u(seed: int, b: int, hk: int, d: int) -> torch.Tensor:
    u = torch.randn(d, generator=_gen(seed, "u", b, hk), dtype=torch.float64)
    return (u / u.norm() * math.sqrt(d)).to(torch.float32)


def _salience(seed: int, b: int, hk: int, T: int, frac: float, sink_a: float,
              salient_a: float) -> torch.Tensor:
    a = torch.zeros(T, dtype=torch.float32)
    if T > 0:
        a[0] = sink_a
    n_sal = int(round(frac * max(T - 1, 0)))
    if n_sal > 0:
        perm = torch.randperm(T - 1, generator=_gen(seed, "sal", b, hk))[:n_sal] + 1
        a[perm] = salient_a
    return a


def _band_vectors(seed: int, b: int, hk: int, n: int, d: int, u: torch.Tensor) -> torch.Tensor:
    w = torch.randn(n, d, generator=_gen(seed, "w", b, hk), dtype=torch.float32)
    un = u / u.norm()
    return w - (w @ un)[:, None] * un[None, :]


def _finish(x: torch.Tensor, dtype: str) -> torch.Tensor:
    return x.to(torch.bfloat16) if dtype == "bf16" else x.contiguous()


def prefill_inputs(cfg: PrefillConfig, heads=None):
    """Return ``(q, k, v)`` as CPU tensors in ``[B, H, T, d]`` layout.

    ``heads`` optionally restricts generation to a list of KV-head indices
    (the other heads are left as zeros); a restricted draw reproduces exactly
    the slices of a full draw.
    """
    B, Hq, Hkv, T, d, G = cfg.B, cfg.Hq, cfg.Hkv, cfg.T, cfg.d, cfg.G
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    q = torch.zeros(B, Hq, T, d, dtype=tdt)
    k = torch.zeros(B, Hkv, T, d, dtype=tdt)
    v = torch.zeros(B, Hkv, T, d, dtype=tdt)
    hks = range(Hkv) if heads is None else heads

    def one(job):
        b, hk = job
        u = _unit_u(cfg.seed, b, hk, d)
        a = _salience(cfg.seed, b, hk, T, cfg.salient_frac, cfg.sink_a, cfg.salient_a)
        kk = torch.randn(T, d, generator=_gen(cfg.seed, "k", b, hk)) + a[:, None] * u[None, :]
        band_q = None
        if cfg.band_a != 0.0:
            nb = cfg.n_b
            w = _band_vectors(cfg.seed, b, hk, nb + 1, d, u)
            wk = cfg.band_a * (w[:-1] + w[1:])  # [n_b, d]
            kk += wk.repeat_interleave(cfg.Bc, dim=0)[:T]
            band_q = w[: cfg.n_t].repeat_interleave(cfg.Br, dim=0)[:T]
        k[b, hk] = _finish(kk, cfg.dtype)
        v[b, hk] = _finish(torch.randn(T, d, generator=_gen(cfg.seed, "v", b, hk)), cfg.dtype)
        for g in range(G):
            h = hk * G + g
            qq = torch.randn(T, d, generator=_gen(cfg.seed, "q", b, h)) + u[None, :]
            if band_q is not None:
                qq += band_q
            q[b, h] = _finish(qq, cfg.dtype)

    jobs = [(b, hk) for b in range(B) for hk in hks]
    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, jobs))
    return q, k, v


def varlen_inputs(cfg: VarlenConfig):
    """Return ``(q, k, v, cu_seqlens)``: packed CPU tensors q ``[total, Hq, d]``,
    k and v ``[total, Hkv, d]`` and int32 ``cu_seqlens`` ``[n_seq + 1]``."""
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    q = torch.zeros(cfg.total, cfg.Hq, cfg.d, dtype=tdt)
    k = torch.zeros(cfg.total, cfg.Hkv, cfg.d, dtype=tdt)
    v = torch.zeros(cfg.total, cfg.Hkv, cfg.d, dtype=tdt)
    cu = cfg.cu_seqlens
    for s in range(cfg.n_seq):
        if cfg.lengths[s] == 0:
            continue
        qs, ks, vs = prefill_inputs(cfg.sequence(s))
        q[cu[s]:cu[s + 1]] = qs[0].transpose(0, 1)
        k[cu[s]:cu[s + 1]] = ks[0].transpose(0, 1)
        v[cu[s]:cu[s + 1]] = vs[0].transpose(0, 1)
    return q, k, v, torch.tensor(cu, dtype=torch.int32)


def decode_inputs(cfg: DecodeConfig, batches=None):
    """Return ``(q, k, v)``: q ``[B, Hq, dk]``, k ``[B, Hkv, L, dk]``.

    For a latent (MLA) configuration ``v`` is ``None``: the values are the
    first ``dv`` columns of ``k``.  ``batches`` restricts generation to a list
    of batch indices (others stay zero).
    """
    B, Hq, Hkv, L, dk, dv, G = cfg.B, cfg.Hq, cfg.Hkv, cfg.L, cfg.dk, cfg.dv, cfg.G
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    q = torch.zeros(B, Hq, dk, dtype=tdt)
    k = torch.zeros(B, Hkv, L, dk, dtype=tdt)
    v = None if cfg.latent else torch.zeros(B, Hkv, L, dv, dtype=tdt)
    bs = range(B) if batches is None else batches

    def one(job):
        b, hk = job
        u = _unit_u(cfg.seed, b, hk, dk)
        a = _salience(cfg.seed, b, hk, L, cfg.salient_frac, cfg.sink_a, cfg.salient_a)
        kk = torch.randn(L, dk, generator=_gen(cfg.seed, "k", b, hk)) + a[:, None] * u[None, :]
        k[b, hk] = _finish(kk, cfg.dtype)
        if v is not None:
            v[b, hk] = _finish(torch.randn(L, dv, generator=_gen(cfg.seed, "v", b, hk)), cfg.dtype)
        for g in range(G):
            h = hk * G + g
            qq = torch.randn(dk, generator=_gen(cfg.seed, "q", b, h)) + u
            q[b, h] = _finish(qq, cfg.dtype)

    jobs = [(b, hk) for b in bs for hk in range(Hkv)]
    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, jobs))
    return q, k, v


def decode_inputs_fp8(cfg: DecodeConfig, pow2_scales: bool = True):
    """The decode draws with an FP8 (E4M3) key/value cache: returns ``(q,
    k8, v8, k_scale, v_scale)`` with q bf16 ``[B, Hq, dk]``, k8 and v8 uint8
    E4M3 codes ``[B, Hkv, L, d]`` and fp32 scales ``[B, Hkv]``.  Each (sequence,
    KV head) slice of the bf16 draws is quantised with scale = amax / 448
    (rounded up to a power of two when ``pow2_scales``), codes = E4M3(x /
    scale) rounded to nearest even (torch's conversion)."""
    q, k, v = decode_inputs(cfg)

    def quant(x):
        xf = x.float()
        amax = xf.abs().amax(dim=(2, 3)).clamp_min(1e-30)
        sc = amax / 448.0
        if pow2_scales:
            sc = torch.exp2(torch.ceil(torch.log2(sc)))
        codes = (xf / sc[:, :, None, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        return codes.contiguous(), sc.to(torch.float32).contiguous()

    k8, ks = quant(k)
    v8, vs = quant(v)
    return q, k8, v8, ks, vs


# The GQA decode shape with the key/value cache in FP8 (E4M3) and one scale
# per (sequence, KV head) for keys and for values.
GQA_DECODE_FP8_32K = GQA_DECODE_32K.with_(name="gqa_decode_fp8_B16_L32768", seed=1241)


# Magnitudes of the E2M1 (FP4) codes 0..7; bit 3 is the sign.
E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _e2m1_codes(y: torch.Tensor) -> torch.Tensor:
    """E2M1 codes of y (saturating at 6), rounded to nearest, ties to the even
    code (mantissa bit 0)."""
    grid = torch.tensor(E2M1_GRID, dtype=torch.float32)
    a = y.abs().clamp(max=6.0).contiguous()
    lo = (torch.searchsorted(grid, a, right=True) - 1).clamp(0, 7)
    hi = (lo + 1).clamp(max=7)
    dlo, dhi = a - grid[lo], grid[hi] - a
    up = (hi != lo) & ((dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0)))
    idx = torch.where(up, hi, lo)
    sign = ((y < 0) & (idx > 0)).to(torch.int64) << 3
    return (idx | sign).to(torch.uint8)


def decode_inputs_nvfp4(cfg: DecodeConfig):
    """The decode draws with an NVFP4 key/value cache: returns ``(q, k4, v4,
    k_bs, v_bs, k_scale, v_scale)`` with q bf16 ``[B, Hq, dk]``; k4, v4 uint8
    ``[B, Hkv, L, d/2]`` holding two E2M1 codes per byte (element 2i in the
    low nibble); k_bs, v_bs uint8 E4M3 codes ``[B, Hkv, L, d/16]``, one scale
    per 16 consecutive elements of a row; k_scale, v_scale fp32 ``[B, Hkv]``.
    A row element is ``scale * E4M3(block scale) * E2M1(code)``.  Each
    (sequence, KV head) slice of the bf16 draws gets scale = amax / (6 * 448),
    each 16-element block the E4M3 code of (its amax / 6) / scale rounded up
    (no element exceeds the E2M1 range), each element the E2M1 code of
    x / (block scale * scale)."""
    q, k, v = decode_inputs(cfg)

    def quant(x):
        xf = x.float()
        B_, H_, L_, d_ = xf.shape
        blk = xf.reshape(B_, H_, L_, d_ // 16, 16)
        sc = (xf.abs().amax(dim=(2, 3)).clamp_min(1e-30) / (6.0 * 448.0))[:, :, None, None]
        want = (blk.abs().amax(-1) / 6.0) / sc  # in [0, 448]
        code = want.to(torch.float8_e4m3fn).view(torch.uint8)
        # rounded up to the next E4M3 value, so that no element exceeds 6
        up = code.view(torch.float8_e4m3fn).float() < want
        code = torch.where(up, (code + 1).clamp(max=0x7E), code)
        bs8 = code.view(torch.float8_e4m3fn)
        den = (bs8.float() * sc)[..., None]
        y = torch.where(den > 0, blk / den.clamp_min(1e-38), torch.zeros_like(blk))
        codes = _e2m1_codes(y).reshape(B_, H_, L_, d_)
        packed = codes[..., 0::2] | (codes[..., 1::2] << 4)
        return (packed.contiguous(), bs8.view(torch.uint8).contiguous(),
                sc[:, :, 0, 0].contiguous())

    k4, kbs, ks = quant(k)
    v4, vbs, vs = quant(v)
    return q, k4, v4, kbs, vbs, ks, vs


# The GQA decode shape with an NVFP4 key/value cache (E2M1 codes, one E4M3
# scale per 16 elements, one fp32 scale per (sequence, KV head)).
GQA_DECODE_NVFP4_32K = GQA_DECODE_32K.with_(name="gqa_decode_nvfp4_B16_L32768", seed=1243)


def santa_offsets(cfg: DecodeConfig, n_samples: int, mode: str, seed: int = 0) -> torch.Tensor:
    """Uniform draws in [0, 1) for the sampled decode (fp32, one generator per
    (sequence, query head)): ``[B, Hq]`` for the systematic sampler (one
    offset per head), ``[B, Hq, n_samples]`` for the stratified and i.i.d.
    samplers (one draw per sample).  ``seed`` selects another draw of the same
    workload (a new decode step)."""
    per = 1 if mode == "sys" else int(n_samples)
    u = torch.empty(cfg.B, cfg.Hq, per, dtype=torch.float32)
    for b in range(cfg.B):
        for h in range(cfg.Hq):
            u[b, h] = torch.rand(per, generator=_gen(cfg.seed + 7919 * seed, "santa", b, h),
                                 dtype=torch.float32)
    return u[:, :, 0].contiguous() if mode == "sys" else u


def temperate(cfg):
    """The same recipe with half-strength sink and salience (3 and 1.5), so
    outputs are true mixtures of many value rows and thresholds from 1e-3 to
    0.3 give intermediate block sparsity (a test-only variant)."""
    kw = dict(sink_a=3.0, salient_a=1.5)
    if isinstance(cfg, PrefillConfig) and cfg.band_a:
        kw["band_a"] = 1.0
    return cfg.with_(**kw)


def as_f32(x: torch.Tensor) -> torch.Tensor:
    """Exact fp32 copy of a bf16/f32 tensor (bf16 values are fp32-representable)."""
    return x.to(torch.float32).contiguous()
