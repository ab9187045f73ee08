"""Shared test helpers: the parity metric and small conversions."""
import numpy as np

# Tolerances (spec bar): bf16 outputs 2e-2, fp32 SSM state 1e-3, in the
# floored relative metric below.
TOL_BF16 = 2e-2
TOL_STATE = 1e-3


def bf16_to_f64(h) -> np.ndarray:
    h = np.ascontiguousarray(h).view(np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def floored_rel_err(got, ref, axis=None) -> float:
    """max_i |g_i - o_i| / max(|o_i|, rms(o)), rms over `axis` slices (all if None)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if axis is None:
        rms = np.sqrt(np.mean(ref * ref))
        den = np.maximum(np.abs(ref), rms)
    else:
        rms = np.sqrt(np.mean(ref * ref, axis=axis, keepdims=True))
        den = np.maximum(np.abs(ref), rms)
    den = np.where(den == 0, 1.0, den)
    return float(np.max(np.abs(got - ref) / den))


def state_rel_err(got_h, ref_h) -> float:
    """Floored relative error of an SSM state [..., H, P, N], rms per (sequence, head)."""
    return floored_rel_err(got_h, ref_h, axis=(-2, -1))
