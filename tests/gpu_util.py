"""Helpers shared by the GPU parity tests."""
import numpy as np


def normwise_rel(a, ref):
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.abs(np.asarray(a, dtype=np.float64) - ref).max() / np.abs(ref).max())


def to_np(t):
    return t.detach().cpu().numpy()
