"""A stack of Mamba-2 layers run back to back (the hidden rows of one layer's
output are the next layer's input), with per-layer, per-sequence state.

Prefill runs one sequence at a time through every layer; decode advances all
sequences one token through every layer.  Every computation is a C entry point
(``mamba2_layer_prefill`` / ``mamba2_layer_decode``) on one stream.
"""
from __future__ import annotations

import torch

from . import abi
from .layer import DeviceLayer, _empty


class DeviceStack:
    def __init__(self, layers: list[dict], device="cuda"):
        self.layers = [DeviceLayer(l, device) for l in layers]
        self.device = device

    def new_state(self, B: int):
        """Per layer: (h [B,H,P,N] fp32, ring [B,d_conv-1,d_xbc] bf16 bits, pos [B] int32), zeroed."""
        return [dl.new_state(B, self.device) for dl in self.layers]

    def workspace(self, max_batch: int, max_tokens: int, max_seqs: int = 1) -> torch.Tensor:
        """Workspace for decode of max_batch sequences, single-sequence prefill of
        max_tokens, and varlen prefill of max_seqs sequences with max_tokens rows."""
        n = max(max(abi.m2_workspace_bytes(dl.dims, max_batch, max_tokens),
                    abi.m2_workspace_bytes_varlen(dl.dims, max_seqs, max_tokens)) for dl in self.layers)
        return _empty((max(n, 256),), torch.uint8, self.device)

    def prefill(self, hidden: torch.Tensor, states, seq: int, ws: torch.Tensor, stream=None) -> None:
        """hidden [T, hidden] bf16 bits of sequence `seq`, transformed in place by every layer."""
        for dl, (h, ring, pos) in zip(self.layers, states):
            dl.prefill(hidden, (h[seq], ring[seq], pos[seq:seq + 1]), ws, stream)

    def prefill_varlen(self, hidden: torch.Tensor, cu_seqlens, states, ws: torch.Tensor, stream=None) -> None:
        """hidden [T, hidden]: all sequences' prompt rows (sequence i at rows
        cu_seqlens[i] .. cu_seqlens[i+1]-1), through every layer in one call per layer."""
        for dl, st in zip(self.layers, states):
            dl.prefill_varlen(hidden, cu_seqlens, st, ws, stream)

    def decode(self, hidden: torch.Tensor, states, ws: torch.Tensor, stream=None) -> None:
        """hidden [B, hidden]: one token of each of the B sequences, in place
        through every layer; each layer's out_proj pulls part of the next
        layer's in_proj weights toward L2 (the last layer's: the first one's,
        for the next token)."""
        n = len(self.layers)
        for i, (dl, st) in enumerate(zip(self.layers, states)):
            dl.decode(hidden, st, ws, stream, ahead=self.layers[(i + 1) % n])
