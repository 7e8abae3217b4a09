"""Seeded synthetic routing traces for the expert residency tiers.

A trace lists, for each step and MoE layer, the ascending distinct expert ids a call routes
to, plus a predicted id list for the lookahead prefetch.  Popularity is skewed: each layer
ranks its experts by a seeded permutation and draws them with weight (rank + 1) ** -skew
without replacement, so a few experts are hot and most are cold.  A predicted list keeps
each true id with probability `hit_rate` and otherwise puts a random other expert in its
place.  The measured one-layer-ahead predictability is 71.6% (README
"絕不為同一次硬碟讀取等待兩遍"), which is the default.  Inputs only: no policy
arithmetic lives here.
"""
import numpy as np


def routing_trace(seed, steps, n_layers, n_experts, per_call, skew=1.1, hit_rate=0.716):
    """-> (actual, predicted): lists [steps][n_layers] of ascending int32 arrays"""
    rng = np.random.default_rng(seed)
    weights = []
    for _ in range(n_layers):
        rank = rng.permutation(n_experts)
        w = (rank + 1.0) ** -skew
        weights.append(w / w.sum())
    actual, predicted = [], []
    for _ in range(steps):
        row_a, row_p = [], []
        for l in range(n_layers):
            ids = rng.choice(n_experts, size=per_call, replace=False, p=weights[l])
            keep = rng.random(per_call) < hit_rate
            others = np.setdiff1d(np.arange(n_experts), ids)
            wrong = rng.choice(others, size=min(int((~keep).sum()), others.size), replace=False)
            pred = np.concatenate([ids[keep], wrong])
            row_a.append(np.sort(ids).astype(np.int32))
            row_p.append(np.sort(pred).astype(np.int32))
        actual.append(row_a)
        predicted.append(row_p)
    return actual, predicted
