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
# R5 where a separate kernel writes the gated norm's rows (tensor-core
# projections: decode of more than 8 rows, prefill of more than 8 tokens on the
# w8a16 arm) -- bf16 rows as they are, and the f16 rows of an E4M3 out_proj
# (each prescaled by an exact power of two) unscaled and taken as the bf16
# codes they hold; R6 (the output rows) together with R5 only, since R6's
# exact value depends on every R5 code.


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


def _g_codes(ws, wm, rows, di, sel, g_f16):
    """The gated norm's rows as bf16 codes: read as they are (bf16), or as f16
    rows times their unscale (E4M3 out_proj; the second half of the unscale
    region), rounded to bf16 (exact for every value the f16 row holds in its
    normal range)."""
    import torch
    raw = _u16(ws, wm["g"], rows, di, sel)
    if not g_f16:
        return raw.copy()
    from oracle import oracle as orc
    us = ws[wm["unscale"]: wm["unscale"] + 2 * rows * 4].view(torch.float32)[rows:].cpu().numpy().astype(np.float64)
    us = us[sel] if sel is not None else us
    vals = raw.view(np.float16).astype(np.float64) * np.asarray(us).reshape(-1, 1)
    return orc.f64_array_to_bf16(vals)


def _u8(ws, off, rows, cols, sel=None):
    t = ws[off: off + rows * cols].view(rows, cols)
    if sel is not None:
        t = t[sel]
    return t.cpu().numpy()


def decode_candidates(ws, B, d, ring_after, pos_before, hidden_out, only=None, g_f16=False):
    """Per batch row (or for the rows in `only`, others None), the GPU's codes
    of the last decode step: R3 (z, raw xBC from the ring slot just written,
    dt) and R4; R5 and R6 for B > 8.  g_f16: the out_proj has E4M3 weights."""
    from mamba_ssm_layer_gb300 import abi
    di, dx, n_in = _dd(d)
    ldz = _rup(n_in, 8)
    L = d["d_conv"] - 1
    sel = list(range(B)) if only is None else list(only)
    wm = abi.m2_workspace_map(abi.dims_struct(d), abi.M2_WS_KIND_DECODE, B)
    zxu_s = _u16(ws, wm["zx"], B, ldz, sel)
    g_s = _g_codes(ws, wm, B, di, sel, g_f16) if B > 8 else None
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


def prefill_candidates(ws, cu, d, hidden_out, r5_available, a=0, b=None, w8a8=False, g_f16=False):
    """The GPU's codes of token rows a..b-1 of a (varlen) prefill over the
    sequences of cu: R3, R4, and R5 and R6 when a separate kernel wrote the
    gated norm's rows (hidden_out: those rows' outputs; g_f16: the out_proj has
    E4M3 weights).  W8A8 arm: the out_proj's E4M3 input codes and block scales
    ("Q5") and R6."""
    from mamba_ssm_layer_gb300 import abi
    di, dx, n_in = _dd(d)
    cu = [int(v) for v in cu]
    T = cu[-1]
    b = T if b is None else b
    kind = abi.M2_WS_KIND_PREFILL_W8A8 if w8a8 else abi.M2_WS_KIND_PREFILL
    wm = abi.m2_workspace_map(abi.dims_struct(d), kind, len(cu) - 1, cu)
    ldz = _rup(n_in, 8)
    zx = _u16(ws, wm["zx"], T, ldz, slice(a, b))
    u = _u16(ws, wm["u"], T, dx, slice(a, b))
    c = {"R3": zx[:, :n_in].copy(), "R4": u.copy()}
    if r5_available:
        c["R5"] = _g_codes(ws, wm, T, di, slice(a, b), g_f16)
        c["R6"] = np.asarray(hidden_out, np.uint16).copy()
    elif w8a8:
        import torch
        ldq = _rup(max(d["hidden"], di), 16)
        ldsq = _rup(T, 128)
        q = _u8(ws, wm["q8"], T, ldq, slice(a, b))[:, :di]
        sq = ws[wm["sq"]: wm["sq"] + (di // 128) * ldsq * 4].view(torch.float32).view(di // 128, ldsq)
        c["Q5"] = (q.copy(), sq[:, a:b].cpu().numpy().T.copy())
        c["R6"] = np.asarray(hidden_out, np.uint16).copy()
    return c


def rows(cand: dict, a: int, b: int) -> dict:
    """Rows a..b-1 of every candidate array (of each array of a tuple)."""
    return {k: (tuple(x[a:b] for x in v) if isinstance(v, tuple) else v[a:b]) for k, v in cand.items()}


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
                if r.get("diag") is not None:
                    self.diag = r["diag"]

    def check(self):
        if getattr(self, "diag", None) is not None:
            dg = self.diag
            own, cand = dg[256:384].astype(np.int64), dg[384:512].astype(np.int64)
            print("first refused Q5 block: candidate scale", dg[512], "own scale", dg[513])
            for i in range(128):
                print(f"  {i:3d} exact {dg[i]: .9e} scale {dg[128 + i]:.3e} own bf16 {own[i]:#06x} "
                      f"gpu e4m3 {cand[i]:#04x}")
        assert not any(self.refused.values()), f"GPU codes that are not correct roundings: {self.refused} {self.first}"
        return {"taken": dict(self.taken), "worst_excess": {k: float(v) for k, v in self.worst.items()}}


def check_state_all_heads(gpu_h, oracle_h, tol=TOL_STATE):
    """Floored relative error of every (sequence, head) slice of the state; all held to tol."""
    e = state_rel_err(gpu_h, oracle_h)
    assert e <= tol, f"state error {e} > {tol}"
    return e


# ---------------------------------------------------------------------------
# Guard bands: every device buffer the layer helpers allocate (states,
# workspaces, uploaded inputs and weights) sits between two 4 KB bands of a
# known byte pattern; after each GPU test the bands must be intact, so a
# kernel that writes past any of those buffers fails the test even where no
# compared output is hit.

GUARD = 4096
GUARD_BYTE = 0xA5


class GuardBands:
    def __init__(self):
        self.bufs = []

    def alloc(self, nbytes: int, device):
        import torch
        n = (nbytes + 255) // 256 * 256
        raw = torch.empty(n + 2 * GUARD, dtype=torch.uint8, device=device)
        raw[:GUARD].fill_(GUARD_BYTE)
        raw[GUARD + nbytes:].fill_(GUARD_BYTE)
        self.bufs.append((raw, nbytes))
        return raw[GUARD:GUARD + n]

    def check(self):
        import torch
        torch.cuda.synchronize()
        bad = []
        for raw, nbytes in self.bufs:
            lo = raw[:GUARD]
            hi = raw[GUARD + nbytes:]
            if bool((lo != GUARD_BYTE).any()) or bool((hi != GUARD_BYTE).any()):
                bad.append((raw.numel() - 2 * GUARD, nbytes))
        self.bufs.clear()
        assert not bad, f"writes past the end or before the start of {len(bad)} buffers: {bad[:5]}"
