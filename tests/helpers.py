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


# ---------------------------------------------------------------------------
# Rounding decisions.
#
# The layer rounds to bf16 at R3 (in_proj output), R4 (conv output), R5
# (gated-norm output) and R6 (layer output).  The GPU evaluates in fp32, the
# oracle in double; where an exact value lies within fp32 evaluation error of a
# bf16 rounding boundary the two may pick the neighbouring codes -- both are
# correct roundings.  Left alone, one flipped dt code moves dt by up to 2^-4
# relative and its head's state by several percent.  So the oracle follows the
# GPU's decisions (OracleLayer.run_decided): at each point it takes the GPU's
# code only where that code is a correct rounding of a value within the
# point's tolerance (times its sum of |terms|) of the oracle's own exact value,
# refuses every other difference, and still computes every value itself.  A
# test then requires zero refusals, the fp32 state within 1e-3 on every head,
# and bit-equal rings and positions.
#
# The GPU's codes are read back from the call's workspace: R3 and R4 always;
# R5 where the gated norm writes bf16 rows (tensor-core projections: decode of
# more than 8 rows, prefill of more than 8 tokens on the w8a16 arm); R6 (the
# output rows) together with R5 only, since R6's exact value depends on every
# R5 code.


def _rup(v, a):
    return (v + a - 1) // a * a


def _dd(d):
    di = d["nheads"] * d["head_dim"]
    dx = di + 2 * d["n_groups"] * d["d_state"]
    return di, dx, di + dx + d["nheads"]


def _u16(ws, off, rows, cols, sel=None):
    import torch
    t = ws[off: off + rows * cols * 2].view(torch.int16).view(rows, cols)
    if sel is not None:
        t = t[sel]
    return t.cpu().numpy().view(np.uint16)


def decode_candidates(ws, B, d, ring_after, pos_before, hidden_out, only=None):
    """Per batch row (or for the rows in `only`, others None), the GPU's codes
    of the last decode step: R3 (z, raw xBC from the ring slot just written,
    dt) and R4; R5 and R6 for B > 8."""
    di, dx, n_in = _dd(d)
    ldz = _rup(n_in, 8)
    L = d["d_conv"] - 1
    sel = list(range(B)) if only is None else list(only)
    o_zxu = _rup(B * d["hidden"] * 2, 256)
    zxu_s = _u16(ws, o_zxu, B, ldz, sel)
    o_y = o_zxu + _rup(B * ldz * 2, 256)
    o_g = o_y + _rup(B * di * 4, 256)
    g_s = _u16(ws, o_g, B, di, sel) if B > 8 else None
    zxu = {b: zxu_s[i] for i, b in enumerate(sel)}
    g = None if g_s is None else {b: g_s[i] for i, b in enumerate(sel)}
    out = []
    for b in range(B):
        if b not in zxu:
            out.append(None)
            continue
        r3 = np.empty(n_in, np.uint16)
        r3[:di] = zxu[b][:di]
        r3[di:di + dx] = ring_after[b][pos_before[b] % L]
        r3[di + dx:] = zxu[b][di + dx:n_in]
        c = {"R3": r3[None], "R4": zxu[b][None, di:di + dx].copy()}
        if g is not None:
            c["R5"] = g[b][None].copy()
            c["R6"] = np.asarray(hidden_out[b:b + 1], np.uint16).copy()
        out.append(c)
    return out


def prefill_candidates(ws, T, d, hidden_out, r5_available, a=0, b=None):
    """The GPU's codes of token rows a..b-1 of a (varlen) prefill of T rows:
    R3, R4, and R5 and R6 when the gated norm wrote bf16 rows (hidden_out:
    those rows' outputs)."""
    di, dx, n_in = _dd(d)
    b = T if b is None else b
    ldz = _rup(n_in, 8)
    o_zx = _rup(T * d["hidden"] * 2, 256)
    zx = _u16(ws, o_zx, T, ldz, slice(a, b))
    o_u = o_zx + _rup(T * ldz * 2, 256)
    u = _u16(ws, o_u, T, dx, slice(a, b))
    c = {"R3": zx[:, :n_in].copy(), "R4": u.copy()}
    if r5_available:
        o_y = o_u + _rup(T * dx * 2, 256)
        o_g = o_y + _rup(T * di * 4, 256)
        c["R5"] = _u16(ws, o_g, T, di, slice(a, b)).copy()
        c["R6"] = np.asarray(hidden_out, np.uint16).copy()
    return c


def rows(cand: dict, a: int, b: int) -> dict:
    """Rows a..b-1 of every candidate array."""
    return {k: v[a:b] for k, v in cand.items()}


class DecisionLog:
    """Sums the oracle's decision reports over tokens and sequences."""

    def __init__(self):
        self.taken = {}
        self.refused = {}
        self.worst = {}
        self.first = {}

    def add(self, rep: dict, where=None):
        for pt, r in rep.items():
            if pt == "hits":
                assert r == 0, f"dt clamp hit in the oracle at {where}"
                continue
            self.taken[pt] = self.taken.get(pt, 0) + r["taken"]
            self.refused[pt] = self.refused.get(pt, 0) + r["refused"]
            self.worst[pt] = max(self.worst.get(pt, 0.0), r["worst_taken"])
            if r["refused"] and pt not in self.first:
                self.first[pt] = (where, r["first_refused"], r["worst_refused"])

    def check(self):
        assert not any(self.refused.values()), f"GPU codes that are not correct roundings: {self.refused} {self.first}"
        return {"taken": dict(self.taken), "worst_excess": {k: float(v) for k, v in self.worst.items()}}


def check_state_all_heads(gpu_h, oracle_h, tol=TOL_STATE):
    """Floored relative error of every (sequence, head) slice of the state; all held to tol."""
    e = state_rel_err(gpu_h, oracle_h)
    assert e <= tol, f"state error {e} > {tol}"
    return e
