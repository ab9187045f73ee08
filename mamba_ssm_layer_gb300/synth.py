"""Seeded synthetic inputs for the Mamba-2 layer (weights, states, hidden rows).

This module holds the input recipe only: random draws with fixed seeds, and the
FP8 weight encoding done with PyTorch's own dtype casts (a library routine).
It contains none of the layer's arithmetic and is shared by the tests, the
benchmark and the smoke check.

Distributions (all seeded by ``numpy.random.default_rng([workload, layer, tensor])``):
  projection weights  fp32 N(0, 1/sqrt(K)), then either
                      * E4M3 per 128x128 block: s = bf16(amax/448),
                        q = e4m3(clamp(w/s, -448, 448)) (torch RNE cast; an
                        all-zero block gets s = 0, q = 0; partial edge blocks use
                        only their in-range elements), or
                      * bf16 (round to nearest even).
  hidden              N(0, 1) -> bf16
  A_log               U(log 1, log 16)              fp32
  dt_bias             inverse softplus of dt0, dt0 ~ logU(1e-3, 1e-1), fp32
  D                   N(1, 0.1)                     fp32
  conv weight / bias  N(0, 0.5) / N(0, 0.1)         bf16
  norm weights        1 + N(0, 0.1)                 bf16
"""
from __future__ import annotations

import math

import numpy as np
import torch

# Named workloads: layer shapes of the two layer sizes used throughout.
TINY = dict(name="tiny", hidden=256, nheads=8, head_dim=32, d_state=16, n_groups=1, d_conv=4, eps=1e-5)
NEMOTRON_H_8B = dict(name="nemotron_h_8b_like", hidden=4096, nheads=128, head_dim=64, d_state=128,
                     n_groups=8, d_conv=4, eps=1e-5)

# Workload ids used as the first seed component.
WL_TINY_DECODE = 0
WL_8B_DECODE_B1 = 1
WL_8B_DECODE_B64 = 2
WL_8B_PREFILL_1K = 3
WL_8B_STACK8 = 4

_T_NORM, _T_IN_W, _T_CONV_W, _T_CONV_B, _T_ALOG, _T_D, _T_DT, _T_GNORM, _T_OUT_W, _T_HIDDEN = range(10)


def derived(d: dict) -> dict:
    d_inner = d["nheads"] * d["head_dim"]
    d_xbc = d_inner + 2 * d["n_groups"] * d["d_state"]
    n_in = d_inner + d_xbc + d["nheads"]
    return dict(d_inner=d_inner, d_xbc=d_xbc, n_in=n_in)


def _rng(*key) -> np.random.Generator:
    return np.random.default_rng([int(k) for k in key])


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def quantize_fp8_block128(w: np.ndarray):
    """fp32 [N][K] -> (E4M3 bytes [N][K], bf16 scale bits [ceil(N/128)][ceil(K/128)])."""
    N, K = w.shape
    nb, kb = (N + 127) // 128, (K + 127) // 128
    pad = np.zeros((nb * 128, kb * 128), np.float32)
    pad[:N, :K] = w
    amax = np.abs(pad.reshape(nb, 128, kb, 128)).max(axis=(1, 3)).astype(np.float32)
    s_bits = to_bf16_bits(amax / np.float32(448.0))
    s = torch.from_numpy(s_bits.view(np.int16)).view(torch.bfloat16).float()  # exact widening
    s_full = s.repeat_interleave(128, 0).repeat_interleave(128, 1)[:N, :K]
    wt = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32))
    safe = torch.where(s_full > 0, s_full, torch.ones_like(s_full))
    q = torch.where(s_full > 0, wt / safe, torch.zeros_like(wt)).clamp_(-448.0, 448.0)
    qb = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    return qb, s_bits


def make_weight(N: int, K: int, fmt: str, *key):
    w = _rng(*key).standard_normal((N, K), dtype=np.float32) * np.float32(1.0 / math.sqrt(K))
    if fmt == "fp8":
        return quantize_fp8_block128(w)
    if fmt == "bf16":
        return to_bf16_bits(w), None
    raise ValueError(fmt)


def make_layer(dims: dict, workload: int, layer: int = 0, in_fmt: str = "fp8", out_fmt: str = "fp8") -> dict:
    """All parameters of one layer as numpy arrays (bf16 as uint16 bits)."""
    dd = derived(dims)
    H, hid, d_inner, d_xbc, n_in = dims["nheads"], dims["hidden"], dd["d_inner"], dd["d_xbc"], dd["n_in"]
    key = (workload, layer)
    out = dict(dims=dict(dims), in_fmt=in_fmt, out_fmt=out_fmt)
    out["norm_w"] = to_bf16_bits(1.0 + 0.1 * _rng(*key, _T_NORM).standard_normal(hid))
    out["in_w"], out["in_s"] = make_weight(n_in, hid, in_fmt, *key, _T_IN_W)
    out["conv_w"] = to_bf16_bits(0.5 * _rng(*key, _T_CONV_W).standard_normal((d_xbc, dims["d_conv"])))
    out["conv_b"] = to_bf16_bits(0.1 * _rng(*key, _T_CONV_B).standard_normal(d_xbc))
    out["A_log"] = _rng(*key, _T_ALOG).uniform(math.log(1.0), math.log(16.0), H).astype(np.float32)
    out["D"] = (1.0 + 0.1 * _rng(*key, _T_D).standard_normal(H)).astype(np.float32)
    dt0 = np.exp(_rng(*key, _T_DT).uniform(math.log(1e-3), math.log(1e-1), H))
    out["dt_bias"] = (dt0 + np.log(-np.expm1(-dt0))).astype(np.float32)  # softplus^-1(dt0)
    out["gnorm_w"] = to_bf16_bits(1.0 + 0.1 * _rng(*key, _T_GNORM).standard_normal(d_inner))
    out["out_w"], out["out_s"] = make_weight(hid, d_inner, out_fmt, *key, _T_OUT_W)
    return out


def make_hidden(rows: int, hidden: int, *key) -> np.ndarray:
    """N(0,1) bf16 hidden rows [rows][hidden]; key = (workload, stream id, step)."""
    return to_bf16_bits(_rng(*key, _T_HIDDEN).standard_normal((rows, hidden)))


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# Eight-layer stack of the 8B-like layer: layers 2 and 5 (0-based) carry BF16
# projections, the others E4M3; 16 sequences with prompt lengths drawn from the
# integers 64..512 inclusive, then 256 batched decode steps with fresh hidden
# rows each step (outputs are not fed back).
STACK8 = dict(n_layers=8, bf16_layers=(2, 5), n_seqs=16, prompt_min=64, prompt_max=512, decode_steps=256)
_S_PROMPT_LEN, _S_PROMPT, _S_DECODE = 100, 101, 102


def stack_layers(dims: dict = NEMOTRON_H_8B, spec: dict = STACK8) -> list[dict]:
    out = []
    for l in range(spec["n_layers"]):
        fmt = "bf16" if l in spec["bf16_layers"] else "fp8"
        out.append(make_layer(dims, WL_8B_STACK8, l, fmt, fmt))
    return out


def stack_prompt_lengths(spec: dict = STACK8) -> np.ndarray:
    return _rng(WL_8B_STACK8, _S_PROMPT_LEN).integers(spec["prompt_min"], spec["prompt_max"] + 1, spec["n_seqs"])


def stack_prompt(seq: int, T: int, hidden: int) -> np.ndarray:
    return make_hidden(T, hidden, WL_8B_STACK8, _S_PROMPT, seq)


def stack_decode_rows(step: int, n_seqs: int, hidden: int) -> np.ndarray:
    return make_hidden(n_seqs, hidden, WL_8B_STACK8, _S_DECODE, step)
