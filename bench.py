"""Benchmark of softmax-threshold block-skipping attention on one GB300.

One step is one pass of the hot path over resident synthetic inputs:
  * causal GQA prefill, B=1, Hq=32, Hkv=8, d=128, T=16384, bf16, Br=Bc=128;
  * split-KV decode, B=16, Hq=32, Hkv=8, d=128, L=32768, bf16, Bc=128,
    8 splits, then the LSE merge;
both at the threshold that gives ~70 % block sparsity (stored in
tests/golden/lambdas.json, computed by the fp64 oracle alone).

The JSON line's ``value`` is prefill dense-equivalent TFLOP/s
(4 * d * Hq * T(T+1)/2 per call, i.e. the causal work of dense attention);
decode tokens/s and GB/s are in ``decode``.  Kernel durations come from CUDA
events on the launching stream; L2 is flushed (a 512 MB write) before every
timed launch.  ``--impl reference`` times the fp64 CPU oracle on a bounded
sample of the same prefill workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

from block_sparse_attention_online_gb300 import workloads as W  # noqa: E402

METRIC = "skip-softmax attn: prefill dense-equiv TFLOP/s, decode tok/s & GB/s @~70% skip"
PREFILL = W.GQA_PREFILL_16K
DECODE = W.GQA_DECODE_32K
MLA = W.MLA_DECODE_16K
LONG = W.GQA_PREFILL_64K
TARGET = "0.7"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CSRC = os.path.join(ROOT, "block_sparse_attention_online_gb300", "csrc")
# DRAM bytes (read + write) per launch from one ncu capture of the kernel at
# the bench's workload and threshold (summaries under profiles/).  Reported
# only while the kernel's source is the captured one.
NCU_TRAFFIC = {
    "prefill_tc_kernel": {
        "file": "prefill_tc.cu",
        "sha256": "860fc4c2ced66ea537075a7b808dfddaf5f8d87edf4acdfa1167f9d4e49a26b0",
        "bytes": 234510848 + 82156544},
    "decode_tc_kernel": {
        "file": "decode.cu",
        "sha256": "67c9de81d8f8ee7ddce7a6299cee4da7e507f86994a81d430c15461053d8a9e0",
        "bytes": 1396106752 + 4154112},
}


def ncu_traffic(kernel):
    import hashlib
    t = NCU_TRAFFIC[kernel]
    with open(os.path.join(CSRC, t["file"]), "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != t["sha256"]:
            return None
    return t["bytes"]


def lambdas():
    with open(os.path.join(ROOT, "tests", "golden", "lambdas.json")) as f:
        return json.load(f)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- work model --
def prefill_flops(cfg):
    """Dense-equivalent FLOPs of one causal prefill call, and executed FLOPs of
    the tile loop: every traversed (tile, block) pair runs QK^T (2*Br*Bc*d);
    kept pairs also run P.V (2*Br*Bc*d)."""
    dense = 4.0 * cfg.d * cfg.Hq * cfg.B * cfg.T * (cfg.T + 1) / 2
    per_pair = 2.0 * cfg.Br * cfg.Bc * cfg.d
    return dense, per_pair


def traversed_pairs(cfg):
    n_t = cfg.n_t
    per_head = sum(min(cfg.n_b, (min(cfg.T, (t + 1) * cfg.Br) - 1) // cfg.Bc + 1)
                   for t in range(n_t))
    return per_head * cfg.B * cfg.Hq


def decode_bytes(cfg, kept_blocks, total_blocks):
    """HBM bytes of one decode call: every K block, the V blocks of kept
    (b, KV head, split, block) units, the queries and the fp32 partials."""
    elt = 2
    kv_block = cfg.Bc * cfg.dk * elt
    v_block = cfg.Bc * cfg.dv * elt
    q = cfg.B * cfg.Hq * cfg.dk * elt
    part = cfg.B * cfg.Hq * cfg.n_splits * (cfg.dv + 1) * 4
    return total_blocks * kv_block + kept_blocks * v_block + q + part


MARGIN_BAND = 1e-3


def margin_blocks(mu, lam):
    """Traversed blocks whose statistic (from the kernel's statistics mode)
    lies within MARGIN_BAND of ln(lambda): the blocks whose skip bit fp32 and
    fp64 arithmetic may decide differently.  0 for lambda = 0."""
    if lam <= 0:
        return 0
    m = mu[~torch.isnan(mu)].double()
    return int(((m - math.log(lam)).abs() < MARGIN_BAND).sum())


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), float(f[3]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v == "Active"})
        loaded = [r for r in rows if r[2] > 300] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": rows[0][1],
                "power_w_max": max(r[2] for r in rows), "samples": len(rows), "reasons": reasons}


# ---------------------------------------------------------------- GPU arm --
def timed_launches(fn, n_warm, n_timed, flush, stream):
    """Durations (ms) of n_timed launches of fn, L2 flushed before each."""
    for _ in range(n_warm):
        fn()
    durs = []
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n_timed)]
    for i in range(n_timed):
        flush.zero_()
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    for a, b in ev:
        durs.append(a.elapsed_time(b))
    return durs


def run_gpu(args, rank, world):
    from block_sparse_attention_online_gb300 import binding as bs
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    lam = lambdas()
    pk, pk_kind = peaks()
    lp = {t: lam[PREFILL.name][t]["lambda"] for t in ("0.0", "0.5", "0.7", "0.85")
          if t in lam[PREFILL.name]}
    ld = {t: lam[DECODE.name][t]["lambda"] for t in ("0.0", "0.7")}

    # inputs resident in HBM
    q, k, v = W.prefill_inputs(PREFILL)
    dq, dk_, dv_ = (x.to(dev) for x in (q, k, v))
    qd, kd, vd = W.decode_inputs(DECODE)
    dqd, dkd, dvd = (x.to(dev) for x in (qd, kd, vd))
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    P = PREFILL
    po = torch.empty(P.B, P.Hq, P.T, P.d, dtype=torch.bfloat16, device=dev)
    plse = torch.empty(P.B, P.Hq, P.T, dtype=torch.float32, device=dev)
    pbits = torch.empty(bs.prefill_bitmap_shape(P.B, P.Hq, P.T, P.Br, P.Bc), dtype=torch.int32,
                        device=dev)
    D = DECODE
    op = torch.empty(D.B, D.Hq, D.n_splits, D.dv, dtype=torch.float32, device=dev)
    lpart = torch.empty(D.B, D.Hq, D.n_splits, dtype=torch.float32, device=dev)
    dbits = torch.empty(bs.decode_bitmap_shape(D.B, D.Hkv, D.L, D.Bc, D.n_splits),
                        dtype=torch.int32, device=dev)
    do = torch.empty(D.B, D.Hq, D.dv, dtype=torch.bfloat16, device=dev)
    dlse = torch.empty(D.B, D.Hq, dtype=torch.float32, device=dev)

    def prefill(lmb):
        return lambda: bs.attn_skip_prefill(dq, dk_, dv_, lmb, P.Br, P.Bc, True,
                                            out=(po, plse, pbits))

    def decode(lmb):
        return lambda: bs.attn_skip_decode(dqd, dkd, dvd, lmb, D.Bc, D.n_splits,
                                           out=(op, lpart, dbits))

    def combine():
        bs.attn_skip_decode_combine(op, lpart, out=(do, dlse))

    pairs = traversed_pairs(P)
    dense, per_pair = prefill_flops(P)
    n_b = -(-D.L // D.Bc)
    d_blocks = D.B * D.Hkv * n_b
    # each traversed block's statistic, for the margin-block counts
    p_mu = bs.attn_skip_prefill_margins(dq, dk_, P.Br, P.Bc, True).cpu()
    d_mu = bs.attn_skip_decode_margins(dqd, dkd, D.Bc, D.n_splits).cpu()

    # prefill sweep: lambda = 0 and the 50/70/85 % thresholds
    sweep = {}
    for t, lmb in lp.items():
        durs = timed_launches(prefill(lmb), args.warmup, args.steps, flush, stream)
        bits = bs.unpack_bits(pbits, P.n_b)
        skipped = int(bits.sum())
        kept = pairs - skipped
        executed = per_pair * (pairs + kept)
        ms = statistics.mean(durs)
        sweep[t] = {"lambda": lmb, "sparsity": skipped / pairs,
                    "margin_blocks": margin_blocks(p_mu, lmb), "ms": ms,
                    "dense_equiv_tflops": dense / ms / 1e9,
                    "executed_tflops": executed / ms / 1e9, "executed_flops": executed}
    for t in sweep:
        sweep[t]["speedup_vs_lambda0"] = sweep["0.0"]["ms"] / sweep[t]["ms"]
    dsweep = {}
    for t, lmb in ld.items():
        durs = timed_launches(decode(lmb), args.warmup, args.steps, flush, stream)
        cdurs = timed_launches(combine, args.warmup, args.steps, flush, stream)
        bits = bs.unpack_bits(dbits, -(-n_b // D.n_splits))
        skipped = int(bits.sum())
        kept = d_blocks - skipped
        byts = decode_bytes(D, kept, d_blocks)
        ms, cms = statistics.mean(durs), statistics.mean(cdurs)
        dsweep[t] = {"lambda": lmb, "sparsity": skipped / d_blocks,
                     "margin_blocks": margin_blocks(d_mu, lmb), "ms_decode": ms,
                     "ms_combine": cms, "tok_per_s": D.B / ((ms + cms) / 1e3),
                     "gbs": byts / ms / 1e6, "bytes": byts}
    for t in dsweep:
        dsweep[t]["speedup_vs_lambda0"] = ((dsweep["0.0"]["ms_decode"] + dsweep["0.0"]["ms_combine"])
                                          / (dsweep[t]["ms_decode"] + dsweep[t]["ms_combine"]))
    # per-head decisions at the group's ~70 % threshold: same value bytes
    # (a block is read when any head keeps it), more blocks left out per head
    hbits = torch.empty(bs.decode_bitmap_shape(D.B, D.Hq, D.L, D.Bc, D.n_splits),
                        dtype=torch.int32, device=dev)
    durs = timed_launches(
        lambda: bs.attn_skip_decode_per_head(dqd, dkd, dvd, ld[TARGET], D.Bc, D.n_splits,
                                             out=(op, lpart, hbits)),
        args.warmup, args.steps, flush, stream)
    dsweep["per_head_" + TARGET] = {
        "lambda": ld[TARGET], "ms_decode": statistics.mean(durs),
        "head_sparsity": float(bs.unpack_bits(hbits, -(-n_b // D.n_splits)).float().mean())}

    msweep = mla_sweep(args, bs, dev, stream, flush, lam)
    lsweep = long_prefill_sweep(args, bs, dev, stream, flush, lam, pk)
    calib = calibration(args, bs, dev, stream, flush, dq, dk_, dv_, dqd, dkd, lp, ld, pbits)
    blocks = block_set_sweep(args, bs, dev, stream, flush, dq, dk_, dv_, lp, po, plse, pbits)
    santa = santa_sweep(args, bs, dev, stream, flush)
    varlen = varlen_sweep(args, bs, dev, stream, flush)
    fp8 = fp8_decode_sweep(args, bs, dev, stream, flush, lam)
    nvfp4 = nvfp4_decode_sweep(args, bs, dev, stream, flush, lam)

    # ---- the timed region: K steps of the whole hot path at ~70 % ---------
    fp, fd = prefill(lp[TARGET]), decode(ld[TARGET])
    for _ in range(args.warmup):
        fp(); fd(); combine()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            fp()
            ev[i][1].record(stream)
            fd()
            ev[i][2].record(stream)
            combine()
            ev[i][3].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    p_ms = [e[0].elapsed_time(e[1]) for e in ev]
    d_ms = [e[1].elapsed_time(e[2]) for e in ev]
    c_ms = [e[2].elapsed_time(e[3]) for e in ev]
    step_ms = statistics.mean(a + b + c for a, b, c in zip(p_ms, d_ms, c_ms))
    p_avg, d_avg, c_avg = statistics.mean(p_ms), statistics.mean(d_ms), statistics.mean(c_ms)
    p_avg, d_avg, c_avg, step_ms = (max_over_ranks(x, world) for x in (p_avg, d_avg, c_avg,
                                                                         step_ms))
    s70 = sweep[TARGET]
    value = world * dense / p_avg / 1e9
    executed_tflops = s70["executed_flops"] / p_avg / 1e9
    dec = dsweep[TARGET]
    dec_gbs = dec["bytes"] / d_avg / 1e6

    # ---- end to end: pinned host buffers, copies inside the timed region --
    e2e = end_to_end(args, bs, dev, stream, q, k, v, lp[TARGET])
    # Any bounded wait that gave up anywhere in the run raises here.
    bs.attn_skip_last_device_error()

    peak_tf = pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    peak_hbm = pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{P.name}+{D.name}", "prefill": f"B{P.B} Hq{P.Hq} Hkv{P.Hkv} "
                   f"d{P.d} T{P.T} causal Br{P.Br} Bc{P.Bc}",
                   "decode": f"B{D.B} Hq{D.Hq} Hkv{D.Hkv} d{D.dk} L{D.L} Bc{D.Bc} "
                   f"splits{D.n_splits}", "target_sparsity": float(TARGET),
                   "l2": "flushed before every timed step (512 MB write)",
                   "parallelism": f"replicas x{world}"},
        "prefill": {"ms": round(p_avg, 4), "lambda": lp[TARGET],
                    "sparsity": round(s70["sparsity"], 4),
                    "margin_blocks": s70["margin_blocks"],
                    "dense_equiv_tflops": round(value / world, 2),
                    "executed_tflops": round(executed_tflops, 2),
                    "sweep": {t: {kk: (round(vv, 5) if isinstance(vv, float) and kk != "lambda"
                                       else vv)
                                  for kk, vv in s.items()} for t, s in sweep.items()}},
        "decode": {"ms": round(d_avg, 4), "ms_combine": round(c_avg, 4),
                   "lambda": ld[TARGET], "sparsity": round(dec["sparsity"], 4),
                   "margin_blocks": dec["margin_blocks"],
                   "tok_per_s": round(world * D.B / ((d_avg + c_avg) / 1e3), 1),
                   "gbs": round(dec_gbs, 1), "hbm_frac": round(dec_gbs / peak_hbm, 4),
                   "sweep": {t: {kk: (round(vv, 5) if isinstance(vv, float) and kk != "lambda"
                                      else vv)
                                 for kk, vv in s.items()} for t, s in dsweep.items()}},
        "roofline": {"bound": "tensor", "kernel": "prefill_tc_kernel",
                     "achieved": round(executed_tflops, 2), "peak": peak_tf,
                     "peak_kind": f"bf16 dense burst ({pk_kind})", "unit": "TFLOP/s",
                     "frac": round(executed_tflops / peak_tf, 4),
                     "frac_sustained": round(executed_tflops / pk.get(
                         "bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]), 4),
                     "traffic": ncu_traffic("prefill_tc_kernel"),
                     "algorithmic_bytes": int(P.B * P.Hq * P.T * P.d * 2 * 2
                                              + 2 * P.B * P.Hkv * P.T * P.d * 2)},
        "decode_roofline": {"bound": "hbm", "kernel": "decode_tc_kernel",
                            "achieved": round(dec_gbs, 1), "peak": peak_hbm, "unit": "GB/s",
                            "frac": round(dec_gbs / peak_hbm, 4),
                            "traffic": ncu_traffic("decode_tc_kernel"),
                            "algorithmic_bytes": dec["bytes"]},
        "mla_decode": msweep,
        "long_prefill": lsweep,
        "calibration": calib,
        "block_set": blocks,
        "santa_decode": santa,
        "varlen_prefill": varlen,
        "fp8_decode": fp8,
        "nvfp4_decode": nvfp4,
        "e2e": e2e,
        "device_errors": "none (device error word read after the run)",
        "gpu_launches": 3 * args.steps,  # prefill, decode, merge per timed step
        "clocks": clk.summary(),
    }
    return line


def mla_sweep(args, bs, dev, stream, flush, lam):
    """Absorbed-MLA decode (B=32, 128 heads, 576/512 latent, L=16384, Bc=64, 16
    splits) + merge at lambda = 0 and at the largest reachable sparsity."""
    M = MLA
    q, k, _ = W.decode_inputs(M)
    dq, dk_ = q.to(dev), k.to(dev)
    del q, k
    n_b = -(-M.L // M.Bc)
    units = M.B * n_b
    op = torch.empty(M.B, M.Hq, M.n_splits, M.dv, dtype=torch.float32, device=dev)
    lp = torch.empty(M.B, M.Hq, M.n_splits, dtype=torch.float32, device=dev)
    bits = torch.empty(bs.decode_bitmap_shape(M.B, 1, M.L, M.Bc, M.n_splits), dtype=torch.int32,
                       device=dev)
    o = torch.empty(M.B, M.Hq, M.dv, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(M.B, M.Hq, dtype=torch.float32, device=dev)
    out = {}
    mu = bs.attn_skip_decode_margins(dq, dk_, M.Bc, M.n_splits).cpu()
    for t in ("0.0", "max"):
        lmb = lam[M.name][t]["lambda"]

        def step():
            bs.attn_skip_decode(dq, dk_, None, lmb, M.Bc, M.n_splits, dv=M.dv,
                                out=(op, lp, bits))
            bs.attn_skip_decode_combine(op, lp, out=(o, lse))

        durs = timed_launches(step, args.warmup, args.steps, flush, stream)
        skipped = int(bs.unpack_bits(bits, -(-n_b // M.n_splits)).sum())
        kept = units - skipped
        ms = statistics.mean(durs)
        qk = 2.0 * M.Hq * M.Bc * M.dk * units          # every block
        pv = 2.0 * M.Hq * M.Bc * M.dv * kept           # kept blocks
        byts = M.B * M.L * M.dk * 2 + M.B * M.Hq * M.dk * 2 + op.numel() * 4 + lp.numel() * 4
        out[t] = {"lambda": lmb, "sparsity": round(skipped / units, 4),
                  "margin_blocks": margin_blocks(mu, lmb), "ms": round(ms, 4),
                  "tok_per_s": round(M.B / (ms / 1e3), 1), "gbs": round(byts / ms / 1e6, 1),
                  # the cluster kernel computes S = Q K^T once per block, so the
                  # executed products are the algorithmic ones
                  "algorithmic_tflops": round((qk + pv) / ms / 1e9, 2)}
    out["max"]["speedup_vs_lambda0"] = round(out["0.0"]["ms"] / out["max"]["ms"], 4)
    # Per-head decisions: lambda bisected (on the kernel's own bitmaps) for ~70 %
    # of the (head, block) pairs skipped; a block's values are still read when
    # any head keeps it.
    hbits = torch.empty(bs.decode_bitmap_shape(M.B, M.Hq, M.L, M.Bc, M.n_splits),
                        dtype=torch.int32, device=dev)
    bps = -(-n_b // M.n_splits)

    def head_sparsity(lmb):
        bs.attn_skip_decode_per_head(dq, dk_, None, lmb, M.Bc, M.n_splits, dv=M.dv,
                                     out=(op, lp, hbits))
        return float(bs.unpack_bits(hbits, bps).float().mean()) * (bps * M.n_splits) / n_b

    lo, hi = math.log(1e-8), math.log(0.999)
    for _ in range(14):
        mid = 0.5 * (lo + hi)
        if head_sparsity(math.exp(mid)) < float(TARGET):
            lo = mid
        else:
            hi = mid
    lmb = math.exp(hi)
    hs = head_sparsity(lmb)
    hb = bs.unpack_bits(hbits, bps).bool()
    all_skip = int(hb.all(dim=1).sum())  # blocks every head skipped

    def step_ph():
        bs.attn_skip_decode_per_head(dq, dk_, None, lmb, M.Bc, M.n_splits, dv=M.dv,
                                     out=(op, lp, hbits))
        bs.attn_skip_decode_combine(op, lp, out=(o, lse))

    ms = statistics.mean(timed_launches(step_ph, args.warmup, args.steps, flush, stream))
    out["per_head"] = {"lambda": lmb, "head_sparsity": round(hs, 4),
                       "block_sparsity": round(all_skip / units, 4), "ms": round(ms, 4),
                       "speedup_vs_lambda0": round(out["0.0"]["ms"] / ms, 4)}
    out["workload"] = (f"B{M.B} Hq{M.Hq} latent dk{M.dk} dv{M.dv} L{M.L} Bc{M.Bc} "
                       f"splits{M.n_splits}; 'max' = largest sparsity any lambda < 1 reaches")
    return out


def long_prefill_sweep(args, bs, dev, stream, flush, lam, pk):
    """Long causal GQA prefill (B=1, 32/8 heads, d=128, T=65536, 1 % salient
    keys plus the local band) at lambda = 0 and the 50/70/85 % thresholds."""
    C = LONG
    q, k, v = W.prefill_inputs(C)
    dq, dk_, dv_ = q.to(dev), k.to(dev), v.to(dev)
    del q, k, v
    o = torch.empty(C.B, C.Hq, C.T, C.d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(C.B, C.Hq, C.T, dtype=torch.float32, device=dev)
    bits = torch.empty(bs.prefill_bitmap_shape(C.B, C.Hq, C.T, C.Br, C.Bc), dtype=torch.int32,
                       device=dev)
    pairs = traversed_pairs(C)
    dense, per_pair = prefill_flops(C)
    peak_tf = pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    out = {"workload": f"{C.name}: B{C.B} Hq{C.Hq} Hkv{C.Hkv} d{C.d} T{C.T} causal "
                       f"Br{C.Br} Bc{C.Bc}; {C.salient_frac:.0%} salient keys, band "
                       f"+{C.band_a:g}*sqrt(d) on each tile's 256 nearest keys",
           "dense_equiv_flops": dense}
    mu = bs.attn_skip_prefill_margins(dq, dk_, C.Br, C.Bc, True).cpu()
    for t in ("0.0", "0.5", "0.7", "0.85"):
        lmb = lam[C.name][t]["lambda"]
        durs = timed_launches(
            lambda: bs.attn_skip_prefill(dq, dk_, dv_, lmb, C.Br, C.Bc, True,
                                         out=(o, lse, bits)),
            args.warmup, args.steps, flush, stream)
        skipped = int(bs.unpack_bits(bits, C.n_b).sum())
        executed = per_pair * (2 * pairs - skipped)
        ms = statistics.mean(durs)
        out[t] = {"lambda": lmb, "sparsity": round(skipped / pairs, 4),
                  "margin_blocks": margin_blocks(mu, lmb), "ms": round(ms, 4),
                  "dense_equiv_tflops": round(dense / ms / 1e9, 2),
                  "executed_tflops": round(executed / ms / 1e9, 2),
                  "executed_frac_of_peak": round(executed / ms / 1e9 / peak_tf, 4)}
    for t in ("0.5", "0.7", "0.85"):
        out[t]["speedup_vs_lambda0"] = round(out["0.0"]["ms"] / out[t]["ms"], 4)
    return out


def santa_sweep(args, bs, dev, stream, flush):
    """Sampled decode output (SANTA estimator, S = 128 samples per head, 16 key
    tiles) on the spread-attention decode inputs (B=16, 32/8 heads, L=32768),
    both samplers, against the exact decode (lambda = 0) of the same inputs."""
    C = W.SANTA_DECODE_32K
    S, n_tiles = 128, 16
    q, k, v = W.decode_inputs(C)
    dq, dk_, dv_ = q.to(dev), k.to(dev), v.to(dev)
    del q, k, v
    n_b = -(-C.L // 128)
    ns, nt = bs.attn_skip_santa_workspace(C.B, C.Hq, C.L, n_tiles)
    ws = (torch.empty(ns, dtype=torch.float32, device=dev),
          torch.empty(nt, dtype=torch.float32, device=dev))
    o = torch.empty(C.B, C.Hq, C.dv, dtype=torch.float32, device=dev)
    idx = torch.empty(C.B, C.Hq, S, dtype=torch.int32, device=dev)
    k_bytes = C.B * C.Hkv * C.L * C.dk * 2
    out = {"workload": f"{C.name}: B{C.B} Hq{C.Hq} Hkv{C.Hkv} d{C.dk} L{C.L}, sink 1.2, "
                       f"salient 0.6; S={S} samples per head, {n_tiles} key tiles"}
    for mode in ("sys", "strat", "iid"):
        u = W.santa_offsets(C, S, mode).to(dev)

        def step():
            bs.attn_skip_santa_decode(dq, dk_, dv_, S, mode, u, n_tiles=n_tiles, workspace=ws,
                                      out=o, idx_out=idx)

        durs = timed_launches(step, args.warmup, args.steps, flush, stream)
        ms = statistics.mean(durs)
        ix = idx.to("cpu").to(torch.int64)
        G = C.Hq // C.Hkv
        tiles_hit = sum(len(torch.unique(ix[b, h] // (C.L // n_tiles)))
                        for b in range(C.B) for h in range(C.Hq))
        rows = sum(len(torch.unique(ix[b, hk * G:(hk + 1) * G]))
                   for b in range(C.B) for hk in range(C.Hkv))
        byts = (k_bytes + C.B * C.Hq * n_b * 128 * 4                 # keys, stash write
                + tiles_hit * (n_b // n_tiles) * 128 * 4             # stash re-read
                + rows * C.dv * 2 + C.B * C.Hq * (C.dk * 2 + C.dv * 4))
        out[mode] = {"ms": round(ms, 4), "tok_per_s": round(C.B / (ms / 1e3), 1),
                     "gbs": round(byts / ms / 1e6, 1), "bytes": byts,
                     "value_rows_read": rows, "tiles_with_samples_frac":
                         round(tiles_hit / (C.B * C.Hq * n_tiles), 4)}
    # exact output of the same inputs: dense split-KV decode + merge
    op = torch.empty(C.B, C.Hq, C.n_splits, C.dv, dtype=torch.float32, device=dev)
    lpart = torch.empty(C.B, C.Hq, C.n_splits, dtype=torch.float32, device=dev)
    bits = torch.empty(bs.decode_bitmap_shape(C.B, C.Hkv, C.L, C.Bc, C.n_splits),
                       dtype=torch.int32, device=dev)
    do = torch.empty(C.B, C.Hq, C.dv, dtype=torch.bfloat16, device=dev)
    dlse = torch.empty(C.B, C.Hq, dtype=torch.float32, device=dev)

    def exact():
        bs.attn_skip_decode(dq, dk_, dv_, 0.0, C.Bc, C.n_splits, out=(op, lpart, bits))
        bs.attn_skip_decode_combine(op, lpart, out=(do, dlse))

    ms = statistics.mean(timed_launches(exact, args.warmup, args.steps, flush, stream))
    out["exact_decode_ms"] = round(ms, 4)
    for mode in ("sys", "strat"):
        out[mode]["speedup_vs_exact"] = round(ms / out[mode]["ms"], 4)
    return out


def fp8_decode_sweep(args, bs, dev, stream, flush, lam):
    """Decode over an FP8 (E4M3) key/value cache, the GQA decode shape (B=16,
    32/8 heads, L=32768, 8 splits), at lambda = 0 and the oracle's ~70 %
    threshold, decode + merge; bytes = key codes + kept value codes + Q +
    partials."""
    C = W.GQA_DECODE_FP8_32K
    q, k8, v8, ks, vs = W.decode_inputs_fp8(C)
    dq, dk8, dv8, dks, dvs = (x.to(dev) for x in (q, k8, v8, ks, vs))
    del q, k8, v8
    n_b = -(-C.L // C.Bc)
    blocks = C.B * C.Hkv * n_b
    op = torch.empty(C.B, C.Hq, C.n_splits, C.dv, dtype=torch.float32, device=dev)
    lpart = torch.empty(C.B, C.Hq, C.n_splits, dtype=torch.float32, device=dev)
    bits = torch.empty(bs.decode_bitmap_shape(C.B, C.Hkv, C.L, C.Bc, C.n_splits),
                       dtype=torch.int32, device=dev)
    o = torch.empty(C.B, C.Hq, C.dv, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(C.B, C.Hq, dtype=torch.float32, device=dev)
    out = {"workload": f"{C.name}: B{C.B} Hq{C.Hq} Hkv{C.Hkv} d{C.dk} L{C.L} Bc{C.Bc} "
                       f"splits{C.n_splits}, E4M3 codes, one scale per (sequence, KV head)"}
    for t in ("0.0", TARGET):
        lmb = lam[C.name][t]["lambda"]
        durs = timed_launches(
            lambda: bs.attn_skip_decode_fp8(dq, dk8, dv8, dks, dvs, lmb, C.Bc, C.n_splits,
                                            out=(op, lpart, bits)),
            args.warmup, args.steps, flush, stream)
        cdurs = timed_launches(lambda: bs.attn_skip_decode_combine(op, lpart, out=(o, lse)),
                               args.warmup, args.steps, flush, stream)
        skipped = int(bs.unpack_bits(bits, -(-n_b // C.n_splits)).sum())
        kept = blocks - skipped
        byts = (blocks + kept) * C.Bc * C.dk + C.B * C.Hq * C.dk * 2 + op.numel() * 4 * 2
        ms, cms = statistics.mean(durs), statistics.mean(cdurs)
        out[t] = {"lambda": lmb, "sparsity": round(skipped / blocks, 4), "ms_decode": round(ms, 4),
                  "ms_combine": round(cms, 4), "tok_per_s": round(C.B / ((ms + cms) / 1e3), 1),
                  "gbs": round(byts / ms / 1e6, 1), "bytes": byts}
    out[TARGET]["speedup_vs_lambda0"] = round(
        (out["0.0"]["ms_decode"] + out["0.0"]["ms_combine"])
        / (out[TARGET]["ms_decode"] + out[TARGET]["ms_combine"]), 4)
    return out


def nvfp4_decode_sweep(args, bs, dev, stream, flush, lam):
    """Decode over an NVFP4 key/value cache, the GQA decode shape (B=16,
    32/8 heads, L=32768, 8 splits), at lambda = 0 and the oracle's ~70 %
    threshold, decode + merge; bytes = key codes and block scales + kept
    value codes and block scales + Q + partials."""
    C = W.GQA_DECODE_NVFP4_32K
    inputs = [x.to(dev) for x in W.decode_inputs_nvfp4(C)]
    n_b = -(-C.L // C.Bc)
    blocks = C.B * C.Hkv * n_b
    op = torch.empty(C.B, C.Hq, C.n_splits, C.dv, dtype=torch.float32, device=dev)
    lpart = torch.empty(C.B, C.Hq, C.n_splits, dtype=torch.float32, device=dev)
    bits = torch.empty(bs.decode_bitmap_shape(C.B, C.Hkv, C.L, C.Bc, C.n_splits),
                       dtype=torch.int32, device=dev)
    o = torch.empty(C.B, C.Hq, C.dv, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(C.B, C.Hq, dtype=torch.float32, device=dev)
    block_bytes = C.Bc * (C.dk // 2 + C.dk // 16)  # codes + block scales
    out = {"workload": f"{C.name}: B{C.B} Hq{C.Hq} Hkv{C.Hkv} d{C.dk} L{C.L} Bc{C.Bc} "
                       f"splits{C.n_splits}, E2M1 codes, E4M3 scale per 16 elements, "
                       f"fp32 scale per (sequence, KV head)"}
    for t in ("0.0", TARGET):
        lmb = lam[C.name][t]["lambda"]
        durs = timed_launches(
            lambda: bs.attn_skip_decode_nvfp4(*inputs, lmb, C.Bc, C.n_splits,
                                              out=(op, lpart, bits)),
            args.warmup, args.steps, flush, stream)
        cdurs = timed_launches(lambda: bs.attn_skip_decode_combine(op, lpart, out=(o, lse)),
                               args.warmup, args.steps, flush, stream)
        skipped = int(bs.unpack_bits(bits, -(-n_b // C.n_splits)).sum())
        kept = blocks - skipped
        byts = (blocks + kept) * block_bytes + C.B * C.Hq * C.dk * 2 + op.numel() * 4 * 2
        ms, cms = statistics.mean(durs), statistics.mean(cdurs)
        out[t] = {"lambda": lmb, "sparsity": round(skipped / blocks, 4), "ms_decode": round(ms, 4),
                  "ms_combine": round(cms, 4), "tok_per_s": round(C.B / ((ms + cms) / 1e3), 1),
                  "gbs": round(byts / ms / 1e6, 1), "bytes": byts}
    out[TARGET]["speedup_vs_lambda0"] = round(
        (out["0.0"]["ms_decode"] + out["0.0"]["ms_combine"])
        / (out[TARGET]["ms_decode"] + out[TARGET]["ms_combine"]), 4)
    return out


def varlen_sweep(args, bs, dev, stream, flush):
    """Batched variable-length prefill (16 sequences, 129 to 16384 tokens,
    65,536 in all) with lambda_s = a / L_s.  ``a`` is calibrated in one pass
    for ~70 % sparsity of the whole batch: the statistics mode gives each
    traversed block's statistic mu, a block of sequence s is skipped when
    mu < ln(a) - ln(L_s), so ln(a) is placed between the shifted statistics
    mu + ln(L_s) around the target quantile.  Timed: the packed call at a / L_s
    and at lambda = 0, and the same work as one fixed-length call per sequence."""
    C = W.VARLEN_PREFILL_64K
    q, k, v, cu = W.varlen_inputs(C)
    dq, dk_, dv_, dcu = (x.to(dev) for x in (q, k, v, cu))
    cu_np = cu.numpy()
    seqs = []
    for s in range(C.n_seq):
        c0, c1 = int(cu_np[s]), int(cu_np[s + 1])
        seqs.append(tuple(x[c0:c1].transpose(0, 1)[None].contiguous().to(dev)
                          for x in (q, k, v)))
    del q, k, v
    shifted, pairs = [], 0
    for s, (qs, ks, _) in enumerate(seqs):
        mu = bs.attn_skip_prefill_margins(qs, ks, 128, 128, True).cpu().numpy().ravel()
        mu = mu[~np.isnan(mu)]
        pairs += mu.size
        shifted.append(mu[mu < 0] + math.log(C.lengths[s]))  # mu = 0 is never skipped
    x = np.sort(np.concatenate(shifted))
    kk = min(int(round(float(TARGET) * pairs)), x.size)
    ln_a = 0.5 * (x[kk - 1] + x[kk]) if kk < x.size else x[-1] + 1e-3
    a = math.exp(ln_a)
    lam = [min(a / L, math.nextafter(1.0, 0.0)) for L in C.lengths]
    dl = torch.tensor(lam, dtype=torch.float32, device=dev)
    dl0 = torch.zeros(C.n_seq, dtype=torch.float32, device=dev)
    o = torch.empty(C.total, C.Hq, C.d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(C.Hq, C.total, dtype=torch.float32, device=dev)
    bits = torch.empty(bs.varlen_bitmap_shape(C.n_seq, C.Hq, C.max_seqlen), dtype=torch.int32,
                       device=dev)
    out = {"workload": f"{C.name}: {C.n_seq} sequences, lengths {list(C.lengths)}, "
                       f"Hq{C.Hq} Hkv{C.Hkv} d{C.d} causal; lambda_s = a / L_s",
           "a": a}
    dense = sum(4.0 * C.d * C.Hq * L * (L + 1) / 2 for L in C.lengths)
    per_pair = 2.0 * 128 * 128 * C.d
    for name, lmb in (("0.0", dl0), ("a_over_L", dl)):
        durs = timed_launches(
            lambda: bs.attn_skip_prefill_varlen(dq, dk_, dv_, dcu, C.max_seqlen, lmb,
                                                out=(o, lse, bits)),
            args.warmup, args.steps, flush, stream)
        ms = statistics.mean(durs)
        skipped = int(bs.unpack_bits(bits, bits.shape[2]).sum())
        executed = per_pair * (2 * pairs - skipped)
        out[name] = {"ms": round(ms, 4), "sparsity": round(skipped / pairs, 4),
                     "dense_equiv_tflops": round(dense / ms / 1e9, 2),
                     "executed_tflops": round(executed / ms / 1e9, 2)}
    out["a_over_L"]["speedup_vs_lambda0"] = round(out["0.0"]["ms"] / out["a_over_L"]["ms"], 4)
    outs = [(torch.empty_like(qs), torch.empty(qs.shape[:3], dtype=torch.float32, device=dev),
             torch.empty(bs.prefill_bitmap_shape(1, C.Hq, qs.shape[2], 128, 128),
                         dtype=torch.int32, device=dev)) for qs, _, _ in seqs]

    def per_sequence():
        for (qs, ks, vs), ob, lm in zip(seqs, outs, lam):
            bs.attn_skip_prefill(qs, ks, vs, lm, 128, 128, True, out=ob)

    ms = statistics.mean(timed_launches(per_sequence, args.warmup, args.steps, flush, stream))
    out["per_sequence_calls_ms"] = round(ms, 4)
    out["a_over_L"]["speedup_vs_per_sequence_calls"] = round(ms / out["a_over_L"]["ms"], 4)
    return out


def infllm_like_set(P, topk, seed):
    """Per query tile: block 0 (init), the diagonal block and the one before
    (local), and `topk` blocks drawn at random from the rest of the causal
    range -- the shape of an InfLLM-V2 access set (SparDA page, section 2.1)."""
    g = torch.Generator().manual_seed(seed)
    allow = torch.zeros(P.B, P.Hq, P.n_t, P.n_b, dtype=torch.bool)
    allow[..., 0] = True
    for t in range(P.n_t):
        allow[:, :, t, t] = True
        if t > 0:
            allow[:, :, t, t - 1] = True
        if t > 2:
            r = torch.rand(P.B, P.Hq, t - 2, generator=g).argsort(-1)[..., :topk] + 1
            allow[:, :, t].scatter_(-1, r, True)
    return allow


def block_set_sweep(args, bs, dev, stream, flush, dq, dk_, dv_, lp, po, plse, pbits):
    """Prefill over an InfLLM-like block set (init + local + 16 top-k blocks per
    tile) alone (lambda = 0) and composed with the ~70 % threshold."""
    P = PREFILL
    allow = infllm_like_set(P, 16, seed=7)
    words = bs.pack_block_set(allow).to(dev)
    pairs_set = int(allow.sum())
    dense, per_pair = prefill_flops(P)
    out = {"set": "init + local + 16 top-k blocks per tile",
           "set_fraction_of_causal_pairs": round(pairs_set / traversed_pairs(P), 4)}
    for t in ("0.0", TARGET):
        lmb = lp[t]
        durs = timed_launches(
            lambda: bs.attn_skip_prefill_blocks(dq, dk_, dv_, lmb, words, P.Br, P.Bc, True,
                                                out=(po, plse, pbits)),
            args.warmup, args.steps, flush, stream)
        skipped = int(bs.unpack_bits(pbits, P.n_b).sum())
        ms = statistics.mean(durs)
        executed = per_pair * (2 * pairs_set - skipped)
        out[t] = {"lambda": lmb, "ms": round(ms, 4),
                  "threshold_sparsity_in_set": round(skipped / pairs_set, 4),
                  "executed_tflops": round(executed / ms / 1e9, 1),
                  "dense_equiv_tflops": round(dense / ms / 1e9, 1)}
    return out


def calibration(args, bs, dev, stream, flush, dq, dk_, dv_, dqd, dkd, lp, ld, pbits):
    """One-pass threshold calibration on the bench's workloads: the statistics
    pass of each kernel (no value load, exponential or P.V), the lambda it
    gives for the ~70 % target, and the sparsity a prefill at that lambda
    reaches; with --calibration-sweep, the exponential model
    lambda * L = alpha * exp(beta * s) fitted over prefill lengths 4K-64K."""
    P, D = PREFILL, DECODE
    pm = torch.empty(bs.prefill_margin_shape(P.B, P.Hq, P.T, P.Br, P.Bc), dtype=torch.float32,
                     device=dev)
    dm = torch.empty(bs.decode_margin_shape(D.B, D.Hkv, D.L, D.Bc, D.n_splits),
                     dtype=torch.float32, device=dev)
    pms = statistics.mean(timed_launches(
        lambda: bs.attn_skip_prefill_margins(dq, dk_, P.Br, P.Bc, True, out=pm),
        args.warmup, args.steps, flush, stream))
    dms = statistics.mean(timed_launches(
        lambda: bs.attn_skip_decode_margins(dqd, dkd, D.Bc, D.n_splits, out=dm),
        args.warmup, args.steps, flush, stream))
    lam_p = bs.attn_skip_lambda_for_sparsity(pm, float(TARGET))
    lam_d = bs.attn_skip_lambda_for_sparsity(dm, float(TARGET))
    bits = bs.attn_skip_prefill(dq, dk_, dv_, lam_p, P.Br, P.Bc, True)[2]
    trav = ~torch.isnan(pm.cpu())
    got = float(bs.unpack_bits(bits, P.n_b)[trav].float().mean())
    out = {"prefill_margins_ms": round(pms, 4), "decode_margins_ms": round(dms, 4),
           "prefill": {"lambda_from_margins": lam_p, "lambda_oracle": lp[TARGET],
                       "sparsity_reached": round(got, 4)},
           "decode": {"lambda_from_margins": lam_d, "lambda_oracle": ld[TARGET],
                      "sparsity_predicted": round(bs.attn_skip_sparsity_at(dm, lam_d), 4)}}
    if args.calibration_sweep:
        out["fit"] = calibration_fit(bs, dev)
    return out


def calibration_fit(bs, dev):
    """Section "校准算法" on synthetic inputs: statistics at T = 4K..64K (the
    16K prefill recipe at each length, 8/2 heads), points (lambda_j * L, s)
    for a lambda grid, the least-squares alpha, beta, and the sparsity the
    model's lambda = alpha * exp(beta * S) / L reaches at each length."""
    lengths = [4096, 8192, 16384, 32768, 65536]
    margins = {}
    for T in lengths:
        cfg = PREFILL.with_(T=T, Hq=8, Hkv=2, seed=4000 + T // 4096)
        q, k, _ = W.prefill_inputs(cfg)
        margins[T] = bs.attn_skip_prefill_margins(q.to(dev), k.to(dev), cfg.Br, cfg.Bc,
                                                  True).cpu()
    grid = [math.exp(x) for x in np.linspace(-30.0, -0.05, 60)]
    Ls, ss, lams = [], [], []
    for T in lengths:
        for lam in grid:
            s_ = bs.attn_skip_sparsity_at(margins[T], lam)
            if 0.2 <= s_ <= 0.9:
                Ls.append(T); ss.append(s_); lams.append(lam)
    alpha, beta = bs.attn_skip_fit_lambda_model(Ls, ss, lams)
    check = {}
    for S in (0.5, 0.7):
        check[str(S)] = {str(T): round(bs.attn_skip_sparsity_at(
            margins[T], bs.attn_skip_lambda_for_target(alpha, beta, S, T)), 4) for T in lengths}
    return {"alpha": alpha, "beta": beta, "points": len(Ls), "reached": check}


def max_over_ranks(x, world):
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def end_to_end(args, bs, dev, stream, q, k, v, lmb):
    """Prefill through the C ABI from pinned host buffers
    (attn_skip_prefill_from_host: the host->device copies of Q, K, V and the
    device->host copies of O and LSE, overlapped with the computation over
    groups of KV heads on two copy streams) inside the timed region of every
    step."""
    P = PREFILL
    hq, hk, hv = (x.pin_memory() for x in (q, k, v))
    ho = torch.empty(P.B, P.Hq, P.T, P.d, dtype=torch.bfloat16).pin_memory()
    hl = torch.empty(P.B, P.Hq, P.T, dtype=torch.float32).pin_memory()
    devbuf = tuple(torch.empty_like(x, device=dev) for x in (q, k, v)) + (
        torch.empty(P.B, P.Hq, P.T, P.d, dtype=torch.bfloat16, device=dev),
        torch.empty(P.B, P.Hq, P.T, dtype=torch.float32, device=dev),
        torch.empty(bs.prefill_bitmap_shape(P.B, P.Hq, P.T, P.Br, P.Bc), dtype=torch.int32,
                    device=dev))
    copy_streams = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))

    def step():
        bs.attn_skip_prefill_from_host(hq, hk, hv, lmb, devbuf, (ho, hl), P.Br, P.Bc, True,
                                       n_groups=8, stream=stream, copy_streams=copy_streams)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    dense, _ = prefill_flops(P)
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    return {"value": round(dense / ms / 1e9, 2), "unit": "TFLOP/s", "ms": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


# ------------------------------------------------------------ oracle (CPU) --
def oracle_sample_units(n_tiles):
    """The n_tiles longest causal tiles of query head 0 (a bounded sample of
    the prefill workload)."""
    P = PREFILL
    return list(range(P.n_t - n_tiles, P.n_t))


def oracle_prefill_rate(n_tiles, n_heads=1, q=None, k=None, v=None):
    """The fp64 oracle on the n_tiles longest causal tiles of the first n_heads
    query heads (KV heads 0 .. n_heads/G - 1) of the prefill workload."""
    import oracle
    P = PREFILL
    lam = lambdas()[P.name][TARGET]["lambda"]
    n_kv = max(1, -(-n_heads // P.G))
    if q is None:
        q, k, v = W.prefill_inputs(P.with_(Hq=n_kv * P.G, Hkv=n_kv))
    tiles = oracle_sample_units(n_tiles)
    units = [h * P.n_t + t for h in range(n_heads) for t in tiles]
    t0 = time.perf_counter()
    oracle.prefill(q, k, v, P.scale, lam, P.Br, P.Bc, True, units=units)
    dt = time.perf_counter() - t0
    dense = n_heads * sum(4.0 * P.d * tile_visible_pairs(P, t) for t in tiles)
    return dense / dt / 1e12, dt, min(oracle.num_threads(), len(units)), (q, k, v)


def tile_visible_pairs(P, t):
    """(row, key) pairs a causal tile attends to: sum of (r + 1) over its rows."""
    r0, r1 = t * P.Br, min(P.T, (t + 1) * P.Br)
    return (r1 * (r1 + 1) - r0 * (r0 + 1)) / 2


def cpu_baseline(n_heads=16):
    """The oracle on all tiles of the first n_heads query heads (about 15 s on
    16 cores)."""
    P = PREFILL
    rate, dt, cores, _ = oracle_prefill_rate(P.n_t, n_heads)
    return {"value": round(rate, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 oracle, prefill query heads 0-{n_heads - 1}, all {P.n_t} causal "
                      f"tiles of T={P.T} ({n_heads}/{P.Hq} of the workload) at the ~70% "
                      f"threshold, {dt:.1f} s"}


def run_reference(args):
    """The reference arm: the fp64 CPU oracle as it stands, each step a bounded
    sample (the 4 longest tiles of one query head) of the prefill workload."""
    n_tiles = 16
    rate, dt, cores, cache = oracle_prefill_rate(n_tiles)
    for _ in range(max(0, args.warmup - 1)):
        oracle_prefill_rate(n_tiles, 1, *cache)
    rates, times = [], []
    for _ in range(args.steps):
        r, t, _, _ = oracle_prefill_rate(n_tiles, 1, *cache)
        rates.append(r)
        times.append(t)
    value = statistics.mean(rates)
    sample = (f"fp64 oracle, prefill query head 0, the {n_tiles} longest causal tiles of "
              f"T={PREFILL.T} per step")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * statistics.mean(times), 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{PREFILL.name} (sampled tiles)",
                       "target_sparsity": float(TARGET)},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_profile_case(args):
    """Warm-up launches then one launch of a single kernel at the ~70 %
    threshold, for an ncu capture (prefill: the T=16384 workload, inputs 201 MB;
    decode: the B=16, L=32768 workload, 2.1 GB; mla: the absorbed-MLA decode,
    B=32, L=16384, 604 MB of latent rows, at lambda = 0)."""
    from block_sparse_attention_online_gb300 import binding as bs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lam = lambdas()
    if args.profile == "prefill":
        q, k, v = (x.to(dev) for x in W.prefill_inputs(PREFILL))
        lmb = lam[PREFILL.name][TARGET]["lambda"]
        fn = lambda: bs.attn_skip_prefill(q, k, v, lmb, PREFILL.Br, PREFILL.Bc, True)  # noqa: E731
    elif args.profile == "mla":
        q, k, _ = (x.to(dev) if x is not None else None for x in W.decode_inputs(MLA))
        lmb = lam[MLA.name]["0.0"]["lambda"]

        def fn():
            op, lp, _ = bs.attn_skip_decode(q, k, None, lmb, MLA.Bc, MLA.n_splits, dv=MLA.dv)
            bs.attn_skip_decode_combine(op, lp)
    elif args.profile == "nvfp4":
        C = W.GQA_DECODE_NVFP4_32K
        inputs = [x.to(dev) for x in W.decode_inputs_nvfp4(C)]
        lmb = lam[C.name][TARGET]["lambda"]

        def fn():
            op, lp, _ = bs.attn_skip_decode_nvfp4(*inputs, lmb, C.Bc, C.n_splits)
            bs.attn_skip_decode_combine(op, lp)
    elif args.profile == "fp8":
        C = W.GQA_DECODE_FP8_32K
        q, k8, v8, ks, vs = (x.to(dev) for x in W.decode_inputs_fp8(C))
        lmb = lam[C.name][TARGET]["lambda"]

        def fn():
            op, lp, _ = bs.attn_skip_decode_fp8(q, k8, v8, ks, vs, lmb, C.Bc, C.n_splits)
            bs.attn_skip_decode_combine(op, lp)
    else:
        q, k, v = (x.to(dev) for x in W.decode_inputs(DECODE))
        lmb = lam[DECODE.name][TARGET]["lambda"]

        def fn():
            op, lp, _ = bs.attn_skip_decode(q, k, v, lmb, DECODE.Bc, DECODE.n_splits)
            bs.attn_skip_decode_combine(op, lp)
    for _ in range(args.warmup + 1):
        fn()
    torch.cuda.synchronize()
    bs.attn_skip_last_device_error()
    print(json.dumps({"profile": args.profile, "launches": args.warmup + 1}))


def launch_plan(gpus, env, argv):
    """How to honour --gpus: ("run", world) when the process group matches it
    (torchrun's WORLD_SIZE, or one process for --gpus 1); ("relaunch", cmd)
    to start one process per GPU under torch.distributed.run when --gpus N > 1
    is given outside torchrun; ("error", why) when torchrun's world size and
    --gpus disagree."""
    if gpus < 1:
        return "error", f"--gpus must be at least 1 (got {gpus})"
    if "WORLD_SIZE" in env:
        world = int(env["WORLD_SIZE"])
        if world != gpus:
            return "error", f"--gpus {gpus} but WORLD_SIZE={world}"
        return "run", world
    if gpus == 1:
        return "run", 1
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={gpus}", "--master-addr", "127.0.0.1",
           "--master-port", env.get("MASTER_PORT", "29531"), os.path.abspath(__file__),
           *argv]
    return "relaunch", cmd


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--calibration-sweep", action="store_true",
                    help="also fit the threshold model over prefill lengths 4K-64K")
    ap.add_argument("--profile", choices=("prefill", "decode", "fp8", "nvfp4", "mla"),
                    help="only warm up and launch one kernel (for ncu captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    plan, what = launch_plan(args.gpus, os.environ, argv)
    if plan == "error":
        ap.error(what)
    if plan == "relaunch":
        sys.stdout.flush()
        os.execv(what[0], what)
    world = what
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    try:
        if args.profile:
            run_profile_case(args)
            return
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps(run_reference(args)), flush=True)
            return
        line = run_gpu(args, rank, world)
        if rank == 0:
            if not args.no_cpu_baseline:
                line["cpu_baseline"] = cpu_baseline()
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
