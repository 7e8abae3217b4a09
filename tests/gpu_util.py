"""Helpers shared by the GPU parity tests."""
import numpy as np


def normwise_rel(a, ref):
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.abs(np.asarray(a, dtype=np.float64) - ref).max() / np.abs(ref).max())


def to_np(t):
    return t.detach().cpu().numpy()


def stage_report(gpu, ora, keys):
    """{stage: (mismatching elements, total)} for every stage that differs bit-wise"""
    bad = {}
    for k in keys:
        g = np.ascontiguousarray(gpu[k])
        o = np.ascontiguousarray(ora[k])
        if g.shape != o.shape:
            bad[k] = ("shape", g.shape, o.shape)
            continue
        gb = g.view(np.uint8).reshape(g.size, -1) if g.size else g
        ob = o.view(np.uint8).reshape(o.size, -1) if o.size else o
        n = int((gb != ob).any(axis=1).sum()) if g.size else 0
        if n:
            bad[k] = (n, g.size)
    return bad
