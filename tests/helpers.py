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
# Rounding-decision analysis for multi-step layer runs.
#
# The layer rounds the in_proj outputs (R3) and the conv outputs (R4) to bf16.
# The GPU accumulates in fp32, the oracle in double; when an exact value lies
# within fp32 accumulation error of a bf16 rounding tie, the two sides may pick
# the two neighbouring bf16 codes -- both are correct roundings.  A flipped dt
# code moves dt by up to one bf16 ulp of dt_raw (<= 2^-4 relative for
# |dt_raw| < 16), and the SSM state of that head by up to ~6 %, decaying with
# prod(dA) afterwards.  The checks below therefore:
#   1. require every GPU/oracle code difference at R3 to be legitimate: the GPU
#      code is a correct rounding of a value within 2^-20 * sum|terms| of the
#      oracle's exact value (fp32 summation of K = 4096 terms errs by far less:
#      ~1e-9 * sum|terms| observed; a missing or wrong term would move the value
#      by ~sum|terms|/K = 2^-12 * sum|terms|); every R4 difference must be
#      legitimate in the same sense or within the propagated effect
#      sum_j |w_j| |dx_j| of R3 differences inside its conv window;
#   2. require the 1e-3 state bound for every head whose inputs saw no flip
#      that is still visible (residual decay weight >= 1e-3), and the derived
#      7e-2 bound for the (reported) heads that did.

FLIP_REL = 2.0 ** -20
FLIP_STATE_CAP = 7e-2


def _bf16_ord(c):
    c = np.asarray(c).astype(np.int64)
    return np.where(c & 0x8000, -(c & 0x7FFF), c)


def legit_flips(gpu_codes, exact, oracle_codes, abssum=None):
    """Indices where the codes differ, and whether each is legitimate: the GPU
    code must be the correct rounding of some value within FLIP_REL * sum|terms|
    of the exact value (its rounding interval meets that error interval).
    Under cancellation (|exact| << sum|terms|) that can be several ulps."""
    idx = np.nonzero(np.asarray(gpu_codes) != np.asarray(oracle_codes))[0]
    if idx.size == 0:
        return idx, np.ones(0, bool)
    g, e = np.asarray(gpu_codes)[idx], np.asarray(exact)[idx]
    scale = np.abs(e) if abssum is None else np.maximum(np.asarray(abssum)[idx], np.abs(e))
    gv = bf16_to_f64(g)
    half_ulp = 0.5 * np.spacing(np.abs(gv).astype(np.float32)).astype(np.float64) * 65536.0
    ok = np.abs(gv - e) <= half_ulp + FLIP_REL * scale
    return idx, ok


class FlipTracker:
    """Follows one sequence through decode / prefill tokens (see above)."""

    def __init__(self, dims, A_log, dt_bias, conv_w):
        self.H, self.P, self.N, self.G = dims["nheads"], dims["head_dim"], dims["d_state"], dims["n_groups"]
        self.L = dims["d_conv"] - 1
        self.d_inner = self.H * self.P
        self.d_xbc = self.d_inner + 2 * self.G * self.N
        self.A = np.exp(np.asarray(A_log, np.float64))
        self.dt_bias = np.asarray(dt_bias, np.float64)
        self.absw = np.abs(bf16_to_f64(conv_w)).reshape(self.d_xbc, self.L + 1)
        self.dx_hist = [np.zeros(self.d_xbc) for _ in range(self.L)]  # |R3 xBC differences| of past tokens
        self.taint_weight = np.zeros(self.H)  # residual weight of past taints per head
        self.n_r3 = 0
        self.n_r4 = 0
        self.bad = []

    def token(self, g3, e3, g4, e4):
        """g3: GPU R3 codes [n_in] (z | raw xBC | dt); e3: oracle (exact values,
        sums of |terms|); g4: GPU R4 codes [d_xbc]; e4: oracle (exact conv
        outputs, sums of |terms|)."""
        from oracle import oracle as orc
        di, dx, H, P, N, G = self.d_inner, self.d_xbc, self.H, self.P, self.N, self.G
        e3, a3 = e3
        e4, a4 = e4
        o3 = orc.f64_array_to_bf16(e3)
        idx3, ok3 = legit_flips(g3, e3, o3, a3)
        self.n_r3 += idx3.size
        self.bad += [("R3", int(i), int(g3[i]), int(o3[i]), float(e3[i]), float(a3[i])) for i in idx3[~ok3]]
        # the conv consumes the xBC codes of this and the previous L tokens;
        # a difference there propagates as sum_j |w_j| * |dx_j| (SiLU' <= 1.1)
        dxc = np.abs(bf16_to_f64(g3[di:di + dx]) - bf16_to_f64(o3[di:di + dx]))
        window = np.stack(self.dx_hist + [dxc], axis=1)           # [d_xbc][L+1], oldest first
        prop = 1.1 * np.sum(self.absw * window, axis=1)
        self.dx_hist = (self.dx_hist + [dxc])[-self.L:]
        o4 = orc.f64_array_to_bf16(e4)
        idx4, ok4 = legit_flips(g4, e4, o4, a4)
        self.n_r4 += idx4.size
        for i, ok in zip(idx4, ok4):
            if ok:
                continue
            gv = bf16_to_f64(g4[i:i + 1])[0]
            half_ulp = 0.5 * float(np.spacing(np.float32(abs(gv)))) * 65536.0
            if abs(gv - e4[i]) > half_ulp + FLIP_REL * max(a4[i], abs(e4[i])) + prop[i]:
                self.bad.append(("R4", int(i), int(g4[i]), int(o4[i]), float(e4[i]), float(prop[i])))
        # heads whose state inputs differ this token
        u_diff = set(int(i) for i in idx4)
        r3_diff = set(int(i) for i in idx3)
        tainted = np.zeros(H, bool)
        for hh in range(H):
            g = hh // (H // G)
            if (di + dx + hh) in r3_diff:
                tainted[hh] = True
                continue
            lo = hh * P
            if any(lo <= i < lo + P for i in u_diff):
                tainted[hh] = True
                continue
            b0, c0 = di + g * N, di + G * N + g * N
            if any(b0 <= i < b0 + N or c0 <= i < c0 + N for i in u_diff):
                tainted[hh] = True
        # decay this token (oracle dt), then add new taints at full weight
        dt_raw = bf16_to_f64(o3[di + dx: di + dx + H])
        dt = np.logaddexp(0.0, dt_raw + self.dt_bias)
        self.taint_weight = self.taint_weight * np.exp(-dt * self.A)
        self.taint_weight[tainted] = 1.0

    def check_state(self, gpu_h, oracle_h, tol=TOL_STATE):
        """Per-head floored relative error with the rules above; returns a report dict."""
        assert not self.bad, f"illegitimate rounding differences: {self.bad[:10]}"
        g = np.asarray(gpu_h, np.float64).reshape(self.H, self.P, self.N)
        o = np.asarray(oracle_h, np.float64).reshape(self.H, self.P, self.N)
        errs = np.array([floored_rel_err(g[h], o[h]) for h in range(self.H)])
        visible = self.taint_weight >= 1e-3
        strict = errs[~visible]
        assert strict.size == 0 or strict.max() <= tol, f"state err {strict.max()} > {tol} on an untainted head"
        assert errs.max() <= FLIP_STATE_CAP, f"state err {errs.max()} above the flip bound"
        return {"r3_flips": self.n_r3, "r4_diffs": self.n_r4, "heads_exempt": int(visible.sum()),
                "max_err_strict": float(strict.max()) if strict.size else 0.0, "max_err": float(errs.max())}
