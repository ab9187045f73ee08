"""GPU parity of the eight-layer stack workload at full size: 8 layers of the
8B-like layer (layers 2 and 5 with BF16 projections), 16 sequences with prompts
of 64..512 tokens prefilled through every layer in one varlen call per layer,
then 256 batched decode steps (the batched decode runs the tensor-core
projections, M = 16).

The oracle follows one sampled sequence (the one with the shortest prompt)
through the stack as the GPU ran it: every prompt row and all 256 decode
steps, layer by layer.  At every layer it takes the GPU's bf16 codes at the
rounding points R3..R6 where each is a correct rounding of a value within
tolerance of the oracle's own exact value (tests/helpers.py), refuses any
other difference, and computes every value itself; each layer's input is the
previous layer's output so decided.  Sequences are independent, so the
sampled sequence's outputs and states are the oracle's quantities.

Bars: no refused decision anywhere; every layer's fp32 state within 1e-3 on
every head; rings bit-equal; positions exact; outputs within 2e-2.
"""
import numpy as np
import pytest
import torch

from mamba_ssm_layer_gb300 import abi, synth
from mamba_ssm_layer_gb300.layer import bits_u16, to_dev
from mamba_ssm_layer_gb300.stack import DeviceStack
from oracle import oracle as orc
from tests.helpers import (TOL_BF16, DecisionLog, bf16_to_f64, check_state_all_heads, decode_candidates,
                           floored_rel_err, prefill_candidates)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from __graft_entry__ import build
    build()
    abi.m2_device_status(clear=True)
    yield
    assert abi.m2_device_status() == abi.M2_OK


def test_stack8_prefill_and_256_decode_steps_sampled_sequence():
    spec, d = synth.STACK8, synth.NEMOTRON_H_8B
    hid = d["hidden"]
    layers = synth.stack_layers(d, spec)
    lens = synth.stack_prompt_lengths(spec)
    S, steps, nl = spec["n_seqs"], spec["decode_steps"], spec["n_layers"]
    samp = int(np.argmin(lens))
    T = int(lens[samp])
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    a, b = int(cu[samp]), int(cu[samp + 1])

    stk = DeviceStack(layers)
    st = stk.new_state(S)
    ws = stk.workspace(S, int(cu[-1]), S)
    ols = [orc.OracleLayer(l) for l in layers]
    ost = [ol.new_state() for ol in ols]
    logs = [DecisionLog() for _ in range(nl)]

    # ---- prefill: all 16 prompts in one varlen call per layer
    xall = to_dev(np.concatenate([synth.stack_prompt(s, int(lens[s]), hid) for s in range(S)]))
    x_or = synth.stack_prompt(samp, T, hid)  # the oracle's row block of the sampled sequence
    for l, dl in enumerate(stk.layers):
        dl.prefill_varlen(xall, cu, st[l], ws)
        torch.cuda.synchronize()
        got = bits_u16(xall[a:b])
        cand = prefill_candidates(ws, cu, d, got, r5_available=True, a=a, b=b,
                                  g_f16=layers[l]["out_fmt"] == "fp8")
        logs[l].add(ols[l].run_decided(x_or, *ost[l], cand), ("prefill", l))
        assert floored_rel_err(bf16_to_f64(got), bf16_to_f64(x_or), axis=-1) <= TOL_BF16, l
    # ---- 256 decode steps of all 16 sequences
    worst = 0.0
    for k in range(steps):
        x = to_dev(synth.stack_decode_rows(k, S, hid))
        row = np.ascontiguousarray(synth.stack_decode_rows(k, S, hid)[samp:samp + 1])
        for l, dl in enumerate(stk.layers):
            pos_before = st[l][2].cpu().numpy().copy()
            dl.decode(x, st[l], ws)
            torch.cuda.synchronize()
            got = bits_u16(x[samp:samp + 1])
            ring = {samp: bits_u16(st[l][1][samp:samp + 1])[0]}
            cand = decode_candidates(ws, S, d, ring, pos_before, np.repeat(got, S, axis=0), only=[samp],
                                     g_f16=layers[l]["out_fmt"] == "fp8")[samp]
            logs[l].add(ols[l].run_decided(row, *ost[l], cand), ("decode", k, l))
            worst = max(worst, floored_rel_err(bf16_to_f64(got), bf16_to_f64(row), axis=-1))
    assert abi.m2_device_status() == abi.M2_OK

    errs = []
    for l in range(nl):
        rep = logs[l].check()
        errs.append(check_state_all_heads(st[l][0][samp].cpu().numpy(), ost[l][0]))
        assert np.array_equal(bits_u16(st[l][1][samp]), ost[l][1]), l
        assert np.array_equal(st[l][2].cpu().numpy(), lens.astype(np.int32) + steps), l  # every sequence
        assert int(ost[l][2][0]) == T + steps
        print(f"stack8 layer {l}: state {errs[-1]:.2e} decisions {rep}")
    assert worst <= TOL_BF16
    print("stack8: worst output", worst, "worst state", max(errs))
