"""Calibrates the query scale of the 128K-token long-context workload with the oracle: the scale s of
q = s N(0,1) for which the oracle fetches about 20% of L on average (eps = 0.02, delta = 0.05,
eta = 1/16, int8 sketch).  Writes long_context_query_scale.json beside this file.

    python tests/golden/calibrate_long_context.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from verified_kv_cache_gb300 import workloads  # noqa: E402


def fetched_fraction(scale, n=131072, kv_heads=2, rows_per_head=8, seed=5):
    w = workloads.qwen_layer_case(seed=3, n=n, n_kv=kv_heads, n_q=kv_heads * 4, n_needles=64, W=1, steps=1,
                                  sketch="int8", eta=1 / 16, eps=0.02, delta=0.05, query_mode="none")
    scores = workloads.synthetic_scores(kv_heads, n, seed=300)
    rng = np.random.default_rng(seed)
    out = []
    for h in range(kv_heads):
        _, _, _, r32 = oracle.waterfill(scores[h], w.n_sink, w.n_local, w.eta * n)
        flags = oracle.poisson_sample(r32, w.seed, h, 0, 0)
        codes, sc = oracle.sketch_int8(w.K[0, h])
        for _ in range(rows_per_head):
            q = scale * rng.standard_normal(w.d)
            te = oracle.logits_exact(q, w.K[0, h])
            ts = oracle.logits_int8(q, codes, sc)
            res = oracle.kvfetch_row(flags, r32, te, ts, w.eps, w.delta)
            out.append(res["kstar"] / res["n_l"])
    return float(np.mean(out))


def main():
    grid = [1.0, 1.1, 1.2, 1.3, 1.5]
    fr = {s: fetched_fraction(s) for s in grid}
    best = min(grid, key=lambda s: abs(fr[s] - 0.2))
    rec = {"target_fetched_fraction": 0.2, "scale": best, "fraction_at_scale": fr[best],
           "grid": {str(k): v for k, v in fr.items()},
           "recipe": "oracle kvfetch_row on 2 KV heads x 8 rows, n = 131072, synthetic scores seed 300, "
                     "q = scale * N(0,1) (seed 5), eps = 0.02, delta = 0.05, eta = 1/16, int8 sketch"}
    with open(os.path.join(HERE, "long_context_query_scale.json"), "w") as f:
        json.dump(rec, f, indent=1)
    print(rec)


if __name__ == "__main__":
    main()
