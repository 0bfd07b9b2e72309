"""Write ``lambdas.json``: per workload, the thresholds that give a target block
sparsity, computed by the fp64 oracle alone.

The skip decision of a (tile or split, block) pair is "tile statistic <
ln(lambda)", and the statistic does not depend on lambda or on earlier
decisions (the running max advances on skipped blocks too).  So one oracle run
at lambda = 0 gives the statistic of every traversed pair, and the sparsity at
any lambda is the fraction of statistics below ln(lambda).  For a target s we
take ln(lambda) halfway between the k-th and (k+1)-th smallest statistics,
k = round(s * n): the decision of every pair is then at least half a gap away
from the threshold.  The BLASST page recommends controlling sparsity rather
than lambda (section "固定阈值为什么不行"); this fixes lambda per workload.

Prefill workloads are sampled (a few query heads, all their tiles); the sample
is recorded next to each value.  Run:
    python tests/golden/make_lambdas.py [workload-name ...]
"""
import json
import math
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from block_sparse_attention_online_gb300 import workloads as W  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lambdas.json")
FP8 = {W.GQA_DECODE_FP8_32K.name: W.GQA_DECODE_FP8_32K}  # E4M3 cache workloads
NVFP4 = {W.GQA_DECODE_NVFP4_32K.name: W.GQA_DECODE_NVFP4_32K}  # NVFP4 cache workloads
TARGETS = (0.5, 0.7, 0.85)


def statistics(cfg):
    if isinstance(cfg, W.PrefillConfig):
        kv_heads = sorted({0, cfg.Hkv // 2, cfg.Hkv - 1}) if cfg.Hkv > 1 else [0]
        q, k, v = W.prefill_inputs(cfg, heads=kv_heads)
        units = [h * cfg.n_t + t for hk in kv_heads for h in [hk * cfg.G]
                 for t in range(cfg.n_t)]
        r = oracle.prefill(q, k, v, cfg.scale, 0.0, cfg.Br, cfg.Bc, cfg.causal, units=units)
        m = r["margin"].reshape(-1, cfg.n_b)[units]
        sample = f"query heads {[hk * cfg.G for hk in kv_heads]}, all {cfg.n_t} tiles"
    elif cfg.name in NVFP4:
        q, k4, v4, kbs, vbs, ks, vs = W.decode_inputs_nvfp4(cfg)
        r = oracle.decode_nvfp4(q, k4, v4, kbs, vbs, ks, vs, cfg.scale, 0.0, cfg.Bc,
                                cfg.n_splits)
        m = r["margin"]
        sample = "all (sequence, KV head, split) units"
    elif cfg.name in FP8:
        q, k8, v8, ks, vs = W.decode_inputs_fp8(cfg)
        r = oracle.decode_fp8(q, k8, v8, ks, vs, cfg.scale, 0.0, cfg.Bc, cfg.n_splits)
        m = r["margin"]
        sample = "all (sequence, KV head, split) units"
    else:
        q, k, v = W.decode_inputs(cfg)
        r = oracle.decode(q, k, v, cfg.scale, 0.0, cfg.Bc, cfg.n_splits, dv=cfg.dv)
        m = r["margin"]
        sample = "all (sequence, KV head, split) units"
    m = m[np.isfinite(m)]
    return np.sort(m), sample


def main(names):
    data = {}
    if os.path.exists(OUT):
        with open(OUT) as f:
            data = json.load(f)
    for name in names:
        cfg = W.CONFIGS[name] if name in W.CONFIGS else {**FP8, **NVFP4}[name]
        t0 = time.time()
        m, sample = statistics(cfg)
        entry = {"pairs": int(m.size), "sample": sample, "0.0": {"lambda": 0.0, "sparsity": 0.0}}
        for s in TARGETS:
            k = int(round(s * m.size))
            k = min(max(k, 1), m.size - 1)
            ln_lam = 0.5 * (m[k - 1] + m[k])
            if not ln_lam < 0:  # unreachable: too many blocks raise some row's max
                continue
            entry[str(s)] = {"lambda": math.exp(ln_lam), "ln_lambda": float(ln_lam),
                             "sparsity": float((m < ln_lam).mean()),
                             "gap": float(m[k] - m[k - 1])}
        # The largest reachable sparsity: ln(lambda) halfway between the largest
        # negative statistic and 0 (blocks with statistic 0 raise a row's max and
        # are never skipped, whatever lambda < 1).
        neg = m[m < 0]
        if neg.size:
            ln_lam = 0.5 * neg.max()
            entry["max"] = {"lambda": math.exp(ln_lam), "ln_lambda": float(ln_lam),
                            "sparsity": float((m < ln_lam).mean())}
        entry["seconds"] = round(time.time() - t0, 1)
        data[name] = entry
        print(name, json.dumps(entry))
        with open(OUT, "w") as f:
            json.dump(data, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main(sys.argv[1:] or [c for c in W.CONFIGS] + list(FP8) + list(NVFP4))
