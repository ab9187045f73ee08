"""CPU oracle for the Mamba-2 layer forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's ``cpu_baseline``
leg may import this module.  The product path (the CUDA library and its Python
binding) never touches it.  The arithmetic lives in ``m2_oracle.c`` (plain C,
IEEE double, bfloat16 rounding only at the layer's rounding points); this file
compiles it with gcc and marshals numpy arrays.  See the header of
``m2_oracle.c`` for the passage each function follows.

Every function here is pinned by ``tests/test_oracle_pins.py`` against library
routines, closed forms and invariants (no function is "parity unpinned").
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "m2_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/liboracle.so (gcc, OpenMP over rows)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC",
               "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            l = C.CDLL(build())
            d, u8, u16, f32, f64, i32, i64 = (C.c_double, C.c_uint8, C.c_uint16, C.c_float, C.c_double,
                                               C.c_int32, C.c_long)
            P = C.c_void_p
            l.or_e4m3_to_f64.argtypes = [u8]; l.or_e4m3_to_f64.restype = d
            l.or_bf16_to_f64.argtypes = [u16]; l.or_bf16_to_f64.restype = d
            l.or_f64_to_bf16.argtypes = [d]; l.or_f64_to_bf16.restype = u16
            l.or_softplus.argtypes = [d]; l.or_softplus.restype = d
            l.or_silu.argtypes = [d]; l.or_silu.restype = d
            l.or_init.argtypes = []
            l.or_rmsnorm.argtypes = [P, P, C.c_int, d, P]
            l.or_w8a16_gemv.argtypes = [P, C.c_int, P, P, C.c_int, C.c_int, P]
            l.or_bf16_gemv.argtypes = [P, C.c_int, P, C.c_int, C.c_int, P]
            l.or_conv1d_update.argtypes = [P, P, P, P, P, C.c_int, C.c_int, C.c_int, P]
            l.or_ssm_step.argtypes = [P, P, P, P, P, P, P, P, C.c_int, C.c_int, C.c_int, C.c_int, P, P]
            l.or_gated_rmsnorm.argtypes = [P, P, P, C.c_int, C.c_int, d, P]
            l.or_layer_token.argtypes = [P, P, P, P, P]; l.or_layer_token.restype = C.c_long
            l.or_layer_prefill.argtypes = [P, P, C.c_int, P, P, P]; l.or_layer_prefill.restype = C.c_long
            l.or_layer_prefill_traced.argtypes = [P, P, C.c_int, P, P, P, P, P, P, P]
            l.or_layer_prefill_traced.restype = C.c_long
            l.or_f64_to_bf16_array.argtypes = [P, P, C.c_long]
            l.or_f32_to_e4m3_sat.argtypes = [C.c_float]; l.or_f32_to_e4m3_sat.restype = u8
            l.or_act_quant.argtypes = [P, C.c_int, P, P]
            l.or_w8a8_gemv.argtypes = [P, P, P, P, C.c_int, C.c_int, P]
            l.or_w8a8_abs.argtypes = [P, P, P, P, C.c_int, C.c_int, P]
            l.or_proj_abs.argtypes = [C.c_int, P, P, P, C.c_int, C.c_int, P]
            l.or_conv1d_update_exact.argtypes = [P, P, P, P, P, C.c_int, C.c_int, C.c_int, P, P, P]
            l.or_bf16_round_interval.argtypes = [u16, C.POINTER(d), C.POINTER(d)]
            l.or_bf16_round_interval.restype = C.c_int
            l.or_decision_excess.argtypes = [u16, d, d]; l.or_decision_excess.restype = d
            l.or_layer_prefill_decided.argtypes = [P, P, C.c_int, P, P, P, C.POINTER(_OrDecisions)]
            l.or_layer_prefill_decided.restype = C.c_long
            l.or_init()
            _lib = l
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ scalars

def e4m3_to_f64(b: int) -> float:
    return lib().or_e4m3_to_f64(int(b))


def bf16_to_f64(h: int) -> float:
    return lib().or_bf16_to_f64(int(h))


def f64_to_bf16(v: float) -> int:
    return int(lib().or_f64_to_bf16(float(v)))


def softplus(v: float) -> float:
    return lib().or_softplus(float(v))


def silu(v: float) -> float:
    return lib().or_silu(float(v))


def bf16_array_to_f64(h: np.ndarray) -> np.ndarray:
    """Vector form of ``bf16_to_f64`` (the same bit reinterpretation)."""
    h = _c(h, np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_array_to_bf16(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().or_f64_to_bf16_array(_p(v), _p(out), v.size)
    return out


# ------------------------------------------------------------------ steps

def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """Step 1 on each row of x [M][K] (bf16 bits) -> bf16 bits."""
    x = _c(x, np.uint16); w = _c(w, np.uint16)
    x2 = x.reshape(-1, x.shape[-1])
    out = np.empty_like(x2)
    for m in range(x2.shape[0]):
        row = np.ascontiguousarray(x2[m]); o = np.empty_like(row)
        lib().or_rmsnorm(_p(row), _p(w), row.shape[0], float(eps), _p(o))
        out[m] = o
    return out.reshape(x.shape)


def w8a16_gemv(A: np.ndarray, W: np.ndarray, S: np.ndarray) -> np.ndarray:
    """out[m][n] = sum_k A[m][k] * E4M3(W[n][k]) * S[n/128][k/128], in double."""
    A = _c(A, np.uint16); W = _c(W, np.uint8); S = _c(S, np.uint16)
    M, K = A.shape
    N = W.shape[0]
    assert W.shape == (N, K) and S.shape == ((N + 127) // 128, (K + 127) // 128)
    out = np.empty((M, N), np.float64)
    lib().or_w8a16_gemv(_p(A), M, _p(W), _p(S), N, K, _p(out))
    return out


def bf16_gemv(A: np.ndarray, W: np.ndarray) -> np.ndarray:
    A = _c(A, np.uint16); W = _c(W, np.uint16)
    M, K = A.shape
    N = W.shape[0]
    out = np.empty((M, N), np.float64)
    lib().or_bf16_gemv(_p(A), M, _p(W), N, K, _p(out))
    return out


def conv1d_update(ring: np.ndarray, pos: int, x: np.ndarray, w: np.ndarray, b, silu_on: bool = True):
    """One token; returns (out bf16 [C], new ring).  ``pos`` is not advanced."""
    ring = _c(ring, np.uint16).copy()
    x = _c(x, np.uint16); w = _c(w, np.uint16)
    Cc = x.shape[0]
    dconv = w.shape[1]
    posa = np.array([pos], np.int32)
    out = np.empty(Cc, np.uint16)
    bp = _p(_c(b, np.uint16)) if b is not None else None
    lib().or_conv1d_update(_p(ring), _p(posa), _p(x), _p(w), bp, Cc, dconv, 1 if silu_on else 0, _p(out))
    return out, ring


def ssm_step(h: np.ndarray, x, Bm, Cm, dt_raw, A_log, D, dt_bias, G: int):
    """One sequence; h [H][P][N] (any float) -> (new h double, y double [H*P], clamp hits)."""
    h = _c(h, np.float64).copy()
    H, P, N = h.shape
    y = np.empty(H * P, np.float64)
    hits = C.c_long(0)
    args = [_c(x, np.uint16), _c(Bm, np.uint16), _c(Cm, np.uint16), _c(dt_raw, np.uint16),
            _c(A_log, np.float32), _c(D, np.float32), _c(dt_bias, np.float32)]
    lib().or_ssm_step(_p(h), *[_p(a) for a in args], H, P, N, G, _p(y), C.byref(hits))
    return h, y, hits.value


def gated_rmsnorm(y: np.ndarray, z: np.ndarray, w: np.ndarray, group: int, eps: float) -> np.ndarray:
    y = _c(y, np.float64); z = _c(z, np.uint16); w = _c(w, np.uint16)
    out = np.empty(y.shape[0], np.uint16)
    lib().or_gated_rmsnorm(_p(y), _p(z), _p(w), y.shape[0], int(group), float(eps), _p(out))
    return out


def f32_to_e4m3_sat(v: float) -> int:
    """fp32 -> E4M3FN code, round to nearest even, saturating to +-448."""
    return int(lib().or_f32_to_e4m3_sat(float(np.float32(v))))


def act_quant(a_bits: np.ndarray):
    """One bf16 row [K] -> (E4M3 codes [K], fp32 block scales [ceil(K/128)]) of the W8A8 arm."""
    a = _c(a_bits, np.uint16)
    K = a.shape[0]
    q = np.empty(K, np.uint8)
    s = np.empty((K + 127) // 128, np.float32)
    lib().or_act_quant(_p(a), K, _p(q), _p(s))
    return q, s


def proj_abs(a: np.ndarray, W: np.ndarray, S=None) -> np.ndarray:
    """sum_k |a[k] * W~[n][k]| of one bf16 row a against E4M3 W with bf16 block
    scales S (or bf16 W when S is None)."""
    a = _c(a, np.uint16)
    N, K = W.shape
    out = np.empty(N, np.float64)
    if S is None:
        lib().or_proj_abs(2, _p(_c(W, np.uint16)), None, _p(a), N, K, _p(out))
    else:
        lib().or_proj_abs(1, _p(_c(W, np.uint8)), _p(_c(S, np.uint16)), _p(a), N, K, _p(out))
    return out


def w8a8_abs(q: np.ndarray, sa: np.ndarray, W: np.ndarray, S: np.ndarray) -> np.ndarray:
    """The W8A8 product's sum of |terms| for one quantized row."""
    q = _c(q, np.uint8); sa = _c(sa, np.float32); W = _c(W, np.uint8); S = _c(S, np.uint16)
    N, K = W.shape
    out = np.empty(N, np.float64)
    lib().or_w8a8_abs(_p(q), _p(sa), _p(W), _p(S), N, K, _p(out))
    return out


def conv1d_update_exact(ring: np.ndarray, pos: int, x: np.ndarray, w: np.ndarray, b, silu_on: bool = True):
    """As conv1d_update, also returning the unrounded outputs and their sums of |terms|."""
    ring = np.array(ring, np.uint16, copy=True, order="C")
    L1, Cc = ring.shape
    dconv = L1 + 1
    out = np.empty(Cc, np.uint16)
    ex = np.empty(Cc, np.float64)
    ab = np.empty(Cc, np.float64)
    p = np.array([pos], np.int32)
    bb = None if b is None else _p(_c(b, np.uint16))
    lib().or_conv1d_update_exact(_p(ring), _p(p), _p(_c(x, np.uint16)), _p(_c(w, np.uint16)), bb, Cc, dconv,
                                 1 if silu_on else 0, _p(out), _p(ex), _p(ab))
    return out, ring, ex, ab


def bf16_round_interval(code: int):
    """[lo, hi]: the reals that round to the bf16 code (None for NaN / infinity)."""
    lo, hi = C.c_double(), C.c_double()
    if not lib().or_bf16_round_interval(int(code), C.byref(lo), C.byref(hi)):
        return None
    return lo.value, hi.value


def decision_excess(code: int, exact: float, scale: float) -> float:
    """Distance of `exact` from the rounding interval of `code`, over `scale`."""
    return float(lib().or_decision_excess(int(code), float(exact), float(scale)))


def w8a8_gemv(q: np.ndarray, sa: np.ndarray, W: np.ndarray, S: np.ndarray) -> np.ndarray:
    """W8A8 product of one quantized row with E4M3 W [N][K] and bf16 block scales S (double)."""
    q = _c(q, np.uint8); sa = _c(sa, np.float32); W = _c(W, np.uint8); S = _c(S, np.uint16)
    N, K = W.shape
    out = np.empty(N, np.float64)
    lib().or_w8a8_gemv(_p(q), _p(sa), _p(W), _p(S), N, K, _p(out))
    return out


# ------------------------------------------------------------------ layer

class _OrDecisions(C.Structure):
    _fields_ = [("cand", C.c_void_p * 4), ("ld", C.c_long * 4), ("tol", C.c_double * 4),
                ("taken", C.c_long * 4), ("refused", C.c_long * 4), ("worst_taken", C.c_double * 4),
                ("worst_refused", C.c_double * 4), ("first_refused", C.c_long * 4),
                ("q5_codes", C.c_void_p), ("q5_scales", C.c_void_p), ("q5_ld", C.c_long), ("q5_lds", C.c_long),
                ("q5_taken", C.c_long), ("q5_refused", C.c_long), ("q5_first_refused", C.c_long),
                ("r5_trace", C.c_void_p), ("q5_diag", C.c_void_p)]


# Rounding points whose decisions the oracle can follow, and the relative
# tolerance of each (times the point's sum of |terms|):
#   R3 in_proj output, R4 conv output, R6 layer output: fp32 summation of at
#   most 16384 terms errs by far less than 2^-20 of their sum of |terms|; a
#   dropped or wrong term moves a value by about 2^-12 of it or more.
#   R5 gated-norm output: y comes from the fp32 state, whose own bar is 1e-3;
#   2^-12 of y's sum of |terms| is four times tighter than that bar.
POINTS = ("R3", "R4", "R5", "R6")
DECISION_TOL = {"R3": 2.0 ** -20, "R4": 2.0 ** -20, "R5": 2.0 ** -12, "R6": 2.0 ** -20}


class _OrLayer(C.Structure):
    _fields_ = [("hidden", C.c_int), ("H", C.c_int), ("P", C.c_int), ("N", C.c_int), ("G", C.c_int),
                ("dconv", C.c_int), ("gnorm_group", C.c_int), ("eps_in", C.c_double),
                ("eps_gated", C.c_double), ("norm_w", C.c_void_p), ("in_fmt", C.c_int),
                ("in_w", C.c_void_p), ("in_s", C.c_void_p), ("conv_w", C.c_void_p),
                ("conv_b", C.c_void_p), ("A_log", C.c_void_p), ("D", C.c_void_p),
                ("dt_bias", C.c_void_p), ("gnorm_w", C.c_void_p), ("out_fmt", C.c_int),
                ("out_w", C.c_void_p), ("out_s", C.c_void_p), ("act_fp8", C.c_int)]


class OracleLayer:
    """Holds one layer's weights (numpy, as the generator made them) for the oracle.

    ``layer`` is the dict returned by ``mamba_ssm_layer_gb300.synth.make_layer``.
    """

    def __init__(self, layer: dict, act_fp8: bool = False):
        """act_fp8: the E4M3 projections take FP8 activations (the W8A8 arm)."""
        d = layer["dims"]
        self.dims = d
        keep = {}
        for k in ("norm_w", "in_w", "in_s", "conv_w", "conv_b", "A_log", "D", "dt_bias", "gnorm_w",
                  "out_w", "out_s"):
            v = layer.get(k)
            keep[k] = None if v is None else np.ascontiguousarray(v)
        self._keep = keep
        s = _OrLayer()
        s.hidden, s.H, s.P, s.N, s.G, s.dconv = (d["hidden"], d["nheads"], d["head_dim"], d["d_state"],
                                                  d["n_groups"], d["d_conv"])
        s.gnorm_group = d.get("gnorm_group", d["nheads"] * d["head_dim"])
        s.eps_in, s.eps_gated = d["eps"], d["eps"]
        s.in_fmt = 1 if layer["in_fmt"] == "fp8" else 2
        s.out_fmt = 1 if layer["out_fmt"] == "fp8" else 2
        s.act_fp8 = 1 if act_fp8 else 0
        for k, v in keep.items():
            setattr(s, k, None if v is None else v.ctypes.data)
        self._s = s

    def new_state(self):
        d = self.dims
        d_xbc = d["nheads"] * d["head_dim"] + 2 * d["n_groups"] * d["d_state"]
        h = np.zeros((d["nheads"], d["head_dim"], d["d_state"]), np.float64)
        ring = np.zeros((d["d_conv"] - 1, d_xbc), np.uint16)
        pos = np.zeros(1, np.int32)
        return h, ring, pos

    def run(self, hidden: np.ndarray, h: np.ndarray, ring: np.ndarray, pos: np.ndarray) -> int:
        """Run T = hidden.shape[0] tokens sequentially (in place); returns clamp hits."""
        assert hidden.dtype == np.uint16 and hidden.flags["C_CONTIGUOUS"]
        assert h.dtype == np.float64 and ring.dtype == np.uint16 and pos.dtype == np.int32
        T = hidden.shape[0]
        return lib().or_layer_prefill(C.byref(self._s), _p(hidden), T, _p(h), _p(ring), _p(pos))

    def run_decided(self, hidden, h, ring, pos, cand: dict, tol: dict | None = None, r5_trace=None) -> dict:
        """Run T = hidden.shape[0] tokens (in place) following, at each rounding
        point named in `cand` ("R3": [T][n_in], "R4": [T][d_xbc], "R5":
        [T][d_inner], "R6": [T][hidden] bf16 codes), every candidate code that
        is a correct rounding of a value within tol * (sum of |terms|) of the
        oracle's exact value; any other difference is refused and counted, and
        the oracle keeps its own code there.  "Q5" (W8A8 arm): a pair (E4M3
        codes [T][d_inner], fp32 block scales [T][d_inner/128]) of the
        out_proj's quantized input, taken per 128-block where it is what the
        quantization makes of legitimate R5 decisions.  Returns per point the
        taken and refused counts, the worst excess of each, and the first
        refused index."""
        assert hidden.dtype == np.uint16 and hidden.flags["C_CONTIGUOUS"]
        tol = dict(DECISION_TOL, **(tol or {}))
        T = hidden.shape[0]
        dec = _OrDecisions()
        keep = []
        for i, pt in enumerate(POINTS):
            c = cand.get(pt)
            dec.tol[i] = tol[pt]
            dec.first_refused[i] = -1
            if c is None:
                continue
            c = np.ascontiguousarray(c, np.uint16).reshape(T, -1)
            keep.append(c)
            dec.cand[i] = c.ctypes.data
            dec.ld[i] = c.shape[1]
        dec.q5_first_refused = -1
        diag = np.zeros(514, np.float64)
        dec.q5_diag = diag.ctypes.data
        if r5_trace is not None:
            assert r5_trace.dtype == np.uint16 and r5_trace.flags["C_CONTIGUOUS"] and r5_trace.shape[0] == T
            dec.r5_trace = r5_trace.ctypes.data
        if cand.get("Q5") is not None:
            qc = np.ascontiguousarray(cand["Q5"][0], np.uint8).reshape(T, -1)
            qs = np.ascontiguousarray(cand["Q5"][1], np.float32).reshape(T, -1)
            keep += [qc, qs]
            dec.q5_codes, dec.q5_scales = qc.ctypes.data, qs.ctypes.data
            dec.q5_ld, dec.q5_lds = qc.shape[1], qs.shape[1]
        hits = lib().or_layer_prefill_decided(C.byref(self._s), _p(hidden), T, _p(h), _p(ring), _p(pos),
                                              C.byref(dec))
        q5 = {"Q5": {"taken": dec.q5_taken, "refused": dec.q5_refused, "worst_taken": 0.0, "worst_refused": 0.0,
                     "first_refused": dec.q5_first_refused,
                     "diag": diag if dec.q5_refused else None}} if cand.get("Q5") is not None else {}
        return {"hits": hits, **q5,
                **{pt: {"taken": dec.taken[i], "refused": dec.refused[i], "worst_taken": dec.worst_taken[i],
                        "worst_refused": dec.worst_refused[i], "first_refused": dec.first_refused[i]}
                   for i, pt in enumerate(POINTS) if cand.get(pt) is not None}}

    def run_traced(self, hidden, h, ring, pos):
        """As run(), also returning the unrounded in_proj outputs [T][n_in] and conv
        outputs [T][d_xbc] (the values rounded to bf16 at R3 and R4), and the
        sums of |terms| of each (the scale of any evaluation's rounding error)."""
        assert hidden.dtype == np.uint16 and hidden.flags["C_CONTIGUOUS"]
        d = self.dims
        d_inner = d["nheads"] * d["head_dim"]
        d_xbc = d_inner + 2 * d["n_groups"] * d["d_state"]
        n_in = d_inner + d_xbc + d["nheads"]
        T = hidden.shape[0]
        zx = np.empty((T, n_in), np.float64)
        u = np.empty((T, d_xbc), np.float64)
        zxa = np.empty((T, n_in), np.float64)
        ua = np.empty((T, d_xbc), np.float64)
        hits = lib().or_layer_prefill_traced(C.byref(self._s), _p(hidden), T, _p(h), _p(ring), _p(pos), _p(zx),
                                             _p(u), _p(zxa), _p(ua))
        return hits, (zx, zxa), (u, ua)
