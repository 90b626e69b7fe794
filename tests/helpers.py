"""Small shared helpers for the tests (no method arithmetic here)."""
import numpy as np


def rel_max_err(x, ref):
    """max |x - ref| / RMS(ref): the parity metric used throughout."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    if rms == 0.0:
        return float(np.max(np.abs(x - ref))) if x.size else 0.0
    return float(np.max(np.abs(x - ref)) / rms)


def rand_inputs(rng, T, dk, dv, *, H=1, B=1, g_lo=-5.0, g_hi=0.0, beta=None,
                normalise=True):
    """Random fp64 inputs [B, T, H, d] for oracle-side tests."""
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    if normalise:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    g = rng.uniform(g_lo, g_hi, size=(B, T, H, dk))
    if beta is None:
        b = rng.uniform(0.05, 0.95, size=(B, T, H))
    else:
        b = np.full((B, T, H), float(beta))
    return q, k, v, g, b
