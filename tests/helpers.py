"""Shared test helpers (no arithmetic of the method lives here)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def golden_dict(name):
    out = {}
    for parts in golden_lines(name):
        out.setdefault(parts[0], []).append(parts[1:])
    return out


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def max_abs_over_rms(a, ref):
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 1.0
    return float(np.max(np.abs(a - ref)) / max(rms, 1e-300)) if ref.size else 0.0
