"""ctypes binding of libmamba2_gb300.so (include/mamba2.h).

Argument marshalling only: the functions here take integer device pointers (or
torch tensors, whose ``data_ptr()`` is passed) and a CUDA stream handle, and
call the C entry points of the same names.  Every step of the layer runs in the
library's CUDA kernels; there is no fallback.  If the library has not been
built, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmamba2_gb300.so")

M2_OK = 0
M2_ERR_ARG = -1
M2_ERR_FORMAT = -2
M2_ERR_WORKSPACE = -3
M2_ERR_LAUNCH = -4
M2_ERR_UNSUPPORTED = -5
M2_ERR_ALIGN = -6
M2_ERR_DEVICE = -7
M2_ERR_TIMEOUT = -8
M2_ERR_SCRATCH = -9
M2_NOALLOC_SCRATCH_BYTES = 8 << 20

M2_W_FP8_BLOCK128 = 1
M2_W_BF16 = 2

# Every entry point include/mamba2.h declares (checked by the host tests).
EXPORTS = ("m2_strerror", "m2_validate", "m2_workspace_bytes", "mamba2_layer_decode", "mamba2_layer_prefill",
           "mamba2_layer_decode_noalloc", "mamba2_layer_decode_prefetch", "mamba2_layer_prefill_varlen",
           "m2_workspace_bytes_varlen",
           "mamba2_layer_prefill_varlen_w8a8", "w8a8_gemm", "m2_w8a8_workspace_bytes",
           "w8a16_gemv", "conv1d_update", "mamba2_ssm_step", "m2_device_status", "m2_launch_count",
           "m2_trace_begin", "m2_trace_end", "m2_kernel_name", "m2_kernel_count", "m2_set_fused_decode", "m2_copy",
           "m2_set_wait_limit", "m2_wait_check", "m2_workspace_map")


class M2Dims(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("nheads", C.c_int32), ("head_dim", C.c_int32), ("d_state", C.c_int32),
                ("n_groups", C.c_int32), ("d_conv", C.c_int32), ("eps_in", C.c_float), ("eps_gated", C.c_float),
                ("gnorm_group", C.c_int32)]


class M2Weight(C.Structure):
    _fields_ = [("w", C.c_void_p), ("scale", C.c_void_p), ("n", C.c_int32), ("k", C.c_int32), ("fmt", C.c_int32)]


class M2Layer(C.Structure):
    _fields_ = [("norm_w", C.c_void_p), ("in_proj", M2Weight), ("conv_w", C.c_void_p), ("conv_b", C.c_void_p),
                ("A_log", C.c_void_p), ("D", C.c_void_p), ("dt_bias", C.c_void_p), ("gnorm_w", C.c_void_p),
                ("out_proj", M2Weight)]


class M2Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status} ({strerror(status)})")
        self.status = status


_lock = threading.Lock()
_lib = None


def lib():
    """Load the library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                                   "(there is no CPU fallback)")
            try:
                import torch  # noqa: F401  (loads the CUDA runtime the library links against)
            except Exception:
                pass
            l = C.CDLL(LIB_PATH)
            P, I32, SZ = C.c_void_p, C.c_int32, C.c_size_t
            l.m2_strerror.argtypes = [C.c_int]; l.m2_strerror.restype = C.c_char_p
            l.m2_validate.argtypes = [C.POINTER(M2Dims), C.POINTER(M2Layer)]; l.m2_validate.restype = C.c_int
            l.m2_workspace_bytes.argtypes = [C.POINTER(M2Dims), I32, I32]; l.m2_workspace_bytes.restype = SZ
            l.mamba2_layer_decode.argtypes = [C.POINTER(M2Dims), C.POINTER(M2Layer), P, I32, P, P, P, P, SZ, P]
            l.mamba2_layer_decode.restype = C.c_int
            l.mamba2_layer_decode_noalloc.argtypes = [C.POINTER(M2Dims), C.POINTER(M2Layer), P, I32, P, P, P, P]
            l.mamba2_layer_decode_noalloc.restype = C.c_int
            l.mamba2_layer_decode_prefetch.argtypes = [C.POINTER(M2Dims), C.POINTER(M2Layer), P, I32, P, P, P, P, SZ,
                                                       P, SZ, P]
            l.mamba2_layer_decode_prefetch.restype = C.c_int
            l.mamba2_layer_prefill.argtypes = [C.POINTER(M2Dims), C.POINTER(M2Layer), P, I32, P, P, P, P, SZ, P]
            l.mamba2_layer_prefill.restype = C.c_int
            l.mamba2_layer_prefill_varlen.argtypes = [C.POINTER(M2Dims), C.POINTER(M2Layer), P, I32,
                                                      C.POINTER(C.c_int32), P, P, P, P, SZ, P]
            l.mamba2_layer_prefill_varlen.restype = C.c_int
            l.mamba2_layer_prefill_varlen_w8a8.argtypes = l.mamba2_layer_prefill_varlen.argtypes
            l.mamba2_layer_prefill_varlen_w8a8.restype = C.c_int
            l.m2_workspace_bytes_varlen.argtypes = [C.POINTER(M2Dims), I32, I32]
            l.m2_workspace_bytes_varlen.restype = SZ
            l.w8a8_gemm.argtypes = [P, P, P, P, I32, I32, I32, P, SZ, P]; l.w8a8_gemm.restype = C.c_int
            l.m2_w8a8_workspace_bytes.argtypes = [I32, I32]; l.m2_w8a8_workspace_bytes.restype = SZ
            l.w8a16_gemv.argtypes = [P, P, P, P, I32, I32, I32, P]; l.w8a16_gemv.restype = C.c_int
            l.conv1d_update.argtypes = [P, P, P, I32, P, P, P, I32, I32, I32, I32, P]; l.conv1d_update.restype = C.c_int
            l.mamba2_ssm_step.argtypes = [P, P, P, P, P, I32, P, P, P, P, I32, I32, I32, I32, I32, P]
            l.mamba2_ssm_step.restype = C.c_int
            l.m2_device_status.argtypes = [C.c_int]; l.m2_device_status.restype = C.c_int
            l.m2_launch_count.argtypes = []; l.m2_launch_count.restype = C.c_int64
            l.m2_trace_begin.argtypes = [I32]; l.m2_trace_begin.restype = C.c_int
            l.m2_trace_end.argtypes = [C.POINTER(C.c_double), C.POINTER(C.c_int32), I32]
            l.m2_trace_end.restype = C.c_int
            l.m2_kernel_name.argtypes = [I32]; l.m2_kernel_name.restype = C.c_char_p
            l.m2_kernel_count.argtypes = []; l.m2_kernel_count.restype = I32
            l.m2_set_fused_decode.argtypes = [C.c_int]; l.m2_set_fused_decode.restype = C.c_int
            l.m2_copy.argtypes = [P, P, C.c_size_t, P]; l.m2_copy.restype = C.c_int
            l.m2_set_wait_limit.argtypes = [C.c_int64]; l.m2_set_wait_limit.restype = C.c_int
            l.m2_wait_check.argtypes = [P, P, P]; l.m2_wait_check.restype = C.c_int
            l.m2_workspace_map.argtypes = [C.POINTER(M2Dims), I32, I32, C.POINTER(C.c_int32), C.POINTER(SZ), I32]
            l.m2_workspace_map.restype = C.c_int
            _lib = l
    return _lib


def strerror(status: int) -> str:
    try:
        return lib().m2_strerror(int(status)).decode()
    except Exception:
        return "?"


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream  # torch.cuda.Stream


def _check(fn: str, st: int) -> int:
    if st != M2_OK:
        raise M2Error(fn, st)
    return st


def dims_struct(d: dict) -> M2Dims:
    d_inner = d["nheads"] * d["head_dim"]
    return M2Dims(d["hidden"], d["nheads"], d["head_dim"], d["d_state"], d["n_groups"], d["d_conv"],
                  float(d.get("eps", 1e-5)), float(d.get("eps", 1e-5)), int(d.get("gnorm_group", d_inner)))


def weight_struct(w, s, n: int, k: int, fmt: int) -> M2Weight:
    return M2Weight(_ptr(w), _ptr(s), n, k, fmt)


# ------------------------------------------------------------------ entry points

def m2_validate(dims: M2Dims, layer: M2Layer) -> int:
    return lib().m2_validate(C.byref(dims), C.byref(layer))


def m2_workspace_bytes(dims: M2Dims, max_batch: int, max_tokens: int) -> int:
    return lib().m2_workspace_bytes(C.byref(dims), max_batch, max_tokens)


def mamba2_layer_decode(dims, layer, hidden, B, ssm_state, conv_state, conv_pos, ws, ws_bytes, stream=None,
                        check=True) -> int:
    st = lib().mamba2_layer_decode(C.byref(dims), C.byref(layer), _ptr(hidden), B, _ptr(ssm_state),
                                   _ptr(conv_state), _ptr(conv_pos), _ptr(ws), ws_bytes, _stream(stream))
    return _check("mamba2_layer_decode", st) if check else st


M2_PREFETCH_MAX_BYTES = 96 << 20


def mamba2_layer_decode_prefetch(dims, layer, hidden, B, ssm_state, conv_state, conv_pos, ws, ws_bytes, prefetch,
                                 prefetch_bytes, stream=None, check=True) -> int:
    """Decode step with a hint: [prefetch, prefetch + prefetch_bytes) is pulled toward L2 during the out_proj."""
    st = lib().mamba2_layer_decode_prefetch(C.byref(dims), C.byref(layer), _ptr(hidden), B, _ptr(ssm_state),
                                            _ptr(conv_state), _ptr(conv_pos), _ptr(ws), ws_bytes, _ptr(prefetch),
                                            prefetch_bytes, _stream(stream))
    return _check("mamba2_layer_decode_prefetch", st) if check else st


def mamba2_layer_decode_noalloc(dims, layer, hidden, B, ssm_state, conv_state, conv_pos, stream=None,
                                check=True) -> int:
    """Decode step with the library's built-in scratch instead of a workspace
    (for callers that cannot allocate device memory; see include/mamba2.h)."""
    st = lib().mamba2_layer_decode_noalloc(C.byref(dims), C.byref(layer), _ptr(hidden), B, _ptr(ssm_state),
                                           _ptr(conv_state), _ptr(conv_pos), _stream(stream))
    return _check("mamba2_layer_decode_noalloc", st) if check else st


def mamba2_layer_prefill(dims, layer, hidden, T, ssm_state, conv_state, conv_pos, ws, ws_bytes, stream=None,
                         check=True) -> int:
    st = lib().mamba2_layer_prefill(C.byref(dims), C.byref(layer), _ptr(hidden), T, _ptr(ssm_state),
                                    _ptr(conv_state), _ptr(conv_pos), _ptr(ws), ws_bytes, _stream(stream))
    return _check("mamba2_layer_prefill", st) if check else st


def mamba2_layer_prefill_varlen(dims, layer, hidden, cu_seqlens, ssm_state, conv_state, conv_pos, ws, ws_bytes,
                                stream=None, check=True) -> int:
    """cu_seqlens: host sequence of nseq + 1 token offsets."""
    cu = (C.c_int32 * len(cu_seqlens))(*[int(v) for v in cu_seqlens])
    st = lib().mamba2_layer_prefill_varlen(C.byref(dims), C.byref(layer), _ptr(hidden), len(cu_seqlens) - 1, cu,
                                           _ptr(ssm_state), _ptr(conv_state), _ptr(conv_pos), _ptr(ws), ws_bytes,
                                           _stream(stream))
    return _check("mamba2_layer_prefill_varlen", st) if check else st


def mamba2_layer_prefill_varlen_w8a8(dims, layer, hidden, cu_seqlens, ssm_state, conv_state, conv_pos, ws,
                                     ws_bytes, stream=None, check=True) -> int:
    """The W8A8 arm of the varlen prefill (FP8 activations into the E4M3 projections)."""
    cu = (C.c_int32 * len(cu_seqlens))(*[int(v) for v in cu_seqlens])
    st = lib().mamba2_layer_prefill_varlen_w8a8(C.byref(dims), C.byref(layer), _ptr(hidden), len(cu_seqlens) - 1,
                                                cu, _ptr(ssm_state), _ptr(conv_state), _ptr(conv_pos), _ptr(ws),
                                                ws_bytes, _stream(stream))
    return _check("mamba2_layer_prefill_varlen_w8a8", st) if check else st


def m2_workspace_bytes_varlen(dims: M2Dims, max_seqs: int, max_total_tokens: int) -> int:
    return lib().m2_workspace_bytes_varlen(C.byref(dims), max_seqs, max_total_tokens)


def w8a8_gemm(A, W, S, out, M, N, K, ws, ws_bytes, stream=None, check=True) -> int:
    st = lib().w8a8_gemm(_ptr(A), _ptr(W), _ptr(S), _ptr(out), M, N, K, _ptr(ws), ws_bytes, _stream(stream))
    return _check("w8a8_gemm", st) if check else st


def m2_w8a8_workspace_bytes(M: int, K: int) -> int:
    return lib().m2_w8a8_workspace_bytes(M, K)


def w8a16_gemv(A, W, S, out, M, N, K, stream=None, check=True) -> int:
    st = lib().w8a16_gemv(_ptr(A), _ptr(W), _ptr(S), _ptr(out), M, N, K, _stream(stream))
    return _check("w8a16_gemv", st) if check else st


def conv1d_update(conv_state, conv_pos, x, ld_x, w, bias, out, B, Cc, d_conv, silu=1, stream=None,
                  check=True) -> int:
    st = lib().conv1d_update(_ptr(conv_state), _ptr(conv_pos), _ptr(x), ld_x, _ptr(w), _ptr(bias), _ptr(out), B,
                             Cc, d_conv, silu, _stream(stream))
    return _check("conv1d_update", st) if check else st


def mamba2_ssm_step(h, x, Bm, Cm, dt_raw, ld_in, A_log, D, dt_bias, y, B, H, P, N, G, stream=None,
                    check=True) -> int:
    st = lib().mamba2_ssm_step(_ptr(h), _ptr(x), _ptr(Bm), _ptr(Cm), _ptr(dt_raw), ld_in, _ptr(A_log), _ptr(D),
                               _ptr(dt_bias), _ptr(y), B, H, P, N, G, _stream(stream))
    return _check("mamba2_ssm_step", st) if check else st


def m2_copy(dst, src, nbytes: int, stream=None, check=True) -> int:
    """Kernel copy between device tensors and/or pinned host tensors (stays in the PDL launch chain)."""
    st = lib().m2_copy(_ptr(dst), _ptr(src), nbytes, _stream(stream))
    return _check("m2_copy", st) if check else st


def m2_device_status(clear: bool = False) -> int:
    return lib().m2_device_status(1 if clear else 0)


def m2_launch_count() -> int:
    return lib().m2_launch_count()


def m2_set_fused_decode(enable: bool) -> bool:
    """Single-launch batch-1 decode step (True) or the kernel chain (False, the default); returns the previous setting."""
    return bool(lib().m2_set_fused_decode(1 if enable else 0))


def m2_set_wait_limit(cycles: int, check=True) -> int:
    """Limit of the in-kernel pipeline waits on the current device (SM clock cycles; <= 0: the default)."""
    st = lib().m2_set_wait_limit(int(cycles))
    return _check("m2_set_wait_limit", st) if check else st


def m2_wait_check(probe, out, stream=None, check=True) -> int:
    """Timeout-path check: a kernel waits on a barrier nothing signals (see include/mamba2.h)."""
    st = lib().m2_wait_check(_ptr(probe), _ptr(out), _stream(stream))
    return _check("m2_wait_check", st) if check else st


M2_WS_KIND_DECODE, M2_WS_KIND_PREFILL, M2_WS_KIND_PREFILL_W8A8 = 0, 1, 2
WS_REGIONS = ("xn", "zx", "u", "y", "g", "q8", "sq", "unscale")


def m2_workspace_map(dims, kind: int, n: int, cu_seqlens=None) -> dict:
    """Byte offsets of a call's workspace regions ({name: offset}; regions the call does not use are left out)."""
    k = len(WS_REGIONS)
    out = (C.c_size_t * k)()
    cu = None
    if cu_seqlens is not None:
        arr = (C.c_int32 * len(cu_seqlens))(*[int(v) for v in cu_seqlens])
        cu = C.cast(arr, C.POINTER(C.c_int32))
    _check("m2_workspace_map", lib().m2_workspace_map(C.byref(dims), kind, n, cu, out, k))
    none = (1 << (8 * C.sizeof(C.c_size_t))) - 1
    return {name: out[i] for i, name in enumerate(WS_REGIONS) if out[i] != none}


def kernel_names() -> list[str]:
    l = lib()
    return [l.m2_kernel_name(i).decode() for i in range(l.m2_kernel_count())]


def trace_begin(capacity: int) -> None:
    _check("m2_trace_begin", lib().m2_trace_begin(capacity))


def trace_end() -> dict:
    """Stop tracing; returns {kernel name: (total ms, launches)} for kernels that ran."""
    l = lib()
    n = l.m2_kernel_count()
    ms = (C.c_double * n)()
    cnt = (C.c_int32 * n)()
    st = l.m2_trace_end(ms, cnt, n)
    if st < 0:
        raise M2Error("m2_trace_end", st)
    names = kernel_names()
    return {names[i]: (ms[i], cnt[i]) for i in range(n) if cnt[i] > 0}
