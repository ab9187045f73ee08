"""Device-side holders for one Mamba-2 layer and its per-sequence state.

PyTorch provides the device memory and the stream; every computation is one of
the C entry points in ``abi``.  Host arrays (numpy, bf16 as uint16 bits) are
uploaded once.
"""
from __future__ import annotations

import numpy as np
import torch

from . import abi


# Optional device allocator: a callable (nbytes, device) -> uint8 tensor of at
# least nbytes, 256-byte aligned.  None: torch's allocator.  Tests install one
# that surrounds every buffer with guard bands.
_ALLOC = None


def set_allocator(fn):
    """Route this module's device buffers through fn (None restores torch's); returns the previous one."""
    global _ALLOC
    prev, _ALLOC = _ALLOC, fn
    return prev


def _empty(shape, dtype, device) -> torch.Tensor:
    if _ALLOC is None:
        return torch.empty(shape, dtype=dtype, device=device)
    n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
    return _ALLOC(max(n, 1), device)[:n].view(dtype).view(shape)


def _zeros(shape, dtype, device) -> torch.Tensor:
    return _empty(shape, dtype, device).zero_()


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    """Upload a numpy array (uint16 bf16 bits stay int16-typed bit patterns)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16))
    elif a.dtype == np.uint8:
        t = torch.from_numpy(a)
    else:
        t = torch.from_numpy(a)
    if _ALLOC is None:
        return t.to(device)
    out = _empty(tuple(t.shape), t.dtype, device)
    out.copy_(t)
    return out


def bits_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint16)


class DeviceLayer:
    """One layer's parameters on the device plus the ctypes structs that point at them."""

    def __init__(self, layer: dict, device="cuda"):
        d = layer["dims"]
        self.dims_dict = d
        self.dims = abi.dims_struct(d)
        d_inner = d["nheads"] * d["head_dim"]
        self.d_inner = d_inner
        self.d_xbc = d_inner + 2 * d["n_groups"] * d["d_state"]
        self.n_in = d_inner + self.d_xbc + d["nheads"]
        self.t = {k: to_dev(layer[k], device) for k in ("norm_w", "in_w", "conv_w", "conv_b", "A_log", "D", "dt_bias",
                                                         "gnorm_w", "out_w")}
        for k in ("in_s", "out_s"):
            self.t[k] = None if layer.get(k) is None else to_dev(layer[k], device)
        fi = abi.M2_W_FP8_BLOCK128 if layer["in_fmt"] == "fp8" else abi.M2_W_BF16
        fo = abi.M2_W_FP8_BLOCK128 if layer["out_fmt"] == "fp8" else abi.M2_W_BF16
        t = self.t
        self.struct = abi.M2Layer(
            t["norm_w"].data_ptr(),
            abi.weight_struct(t["in_w"], t["in_s"], self.n_in, d["hidden"], fi),
            t["conv_w"].data_ptr(), t["conv_b"].data_ptr(), t["A_log"].data_ptr(), t["D"].data_ptr(),
            t["dt_bias"].data_ptr(), t["gnorm_w"].data_ptr(),
            abi.weight_struct(t["out_w"], t["out_s"], d["hidden"], d_inner, fo))

    def new_state(self, B: int, device="cuda"):
        d = self.dims_dict
        h = _zeros((B, d["nheads"], d["head_dim"], d["d_state"]), torch.float32, device)
        ring = _zeros((B, d["d_conv"] - 1, self.d_xbc), torch.int16, device)
        pos = _zeros((B,), torch.int32, device)
        return h, ring, pos

    def workspace(self, max_batch: int, max_tokens: int, device="cuda") -> torch.Tensor:
        n = abi.m2_workspace_bytes(self.dims, max_batch, max_tokens)
        return _empty((max(n, 256),), torch.uint8, device)

    # Bytes of the next layer's in_proj pulled toward L2 during a step's
    # out_proj (decode(..., ahead=...)).  Measured on the 8B-like layer at batch
    # 1, with the SSM step's 10 MB out_proj prefetch: 8 MB of the 76 MB matrix
    # gave the shortest step (30.06 against 30.26 us without a hint; 12 MB
    # 30.19, 16 MB 30.36); more competes with the step's own traffic.
    AHEAD_BYTES = 8 << 20

    def decode(self, hidden: torch.Tensor, state, ws: torch.Tensor, stream=None, ahead=None) -> None:
        """One decode step.  ahead: the DeviceLayer decoded next on this stream;
        the first AHEAD_BYTES of its in_proj weights are pulled toward L2 during
        this step's out_proj (a hint: the results do not change)."""
        h, ring, pos = state
        B = hidden.shape[0]
        s = stream if stream is not None else torch.cuda.current_stream()
        if ahead is None:
            abi.mamba2_layer_decode(self.dims, self.struct, hidden, B, h, ring, pos, ws, ws.numel(), s)
        else:
            w = ahead.t["in_w"]
            n = min(w.numel() * w.element_size(), self.AHEAD_BYTES)
            abi.mamba2_layer_decode_prefetch(self.dims, self.struct, hidden, B, h, ring, pos, ws, ws.numel(), w, n, s)

    def workspace_varlen(self, max_seqs: int, max_total_tokens: int, device="cuda") -> torch.Tensor:
        n = abi.m2_workspace_bytes_varlen(self.dims, max_seqs, max_total_tokens)
        return _empty((max(n, 256),), torch.uint8, device)

    def prefill_varlen(self, hidden: torch.Tensor, cu_seqlens, state, ws: torch.Tensor, stream=None,
                       w8a8: bool = False) -> None:
        """hidden [T][hidden]: rows cu_seqlens[i] .. cu_seqlens[i+1]-1 belong to sequence i of `state`
        (h [n][H][P][N], ring [n][d_conv-1][d_xbc], pos [n]).  w8a8: the FP8-activation arm."""
        h, ring, pos = state
        fn = abi.mamba2_layer_prefill_varlen_w8a8 if w8a8 else abi.mamba2_layer_prefill_varlen
        fn(self.dims, self.struct, hidden, list(cu_seqlens), h, ring, pos, ws, ws.numel(),
           stream if stream is not None else torch.cuda.current_stream())

    def prefill(self, hidden: torch.Tensor, state, ws: torch.Tensor, stream=None) -> None:
        h, ring, pos = state
        T = hidden.shape[0]
        abi.mamba2_layer_prefill(self.dims, self.struct, hidden, T, h, ring, pos, ws, ws.numel(),
                                 stream if stream is not None else torch.cuda.current_stream())
