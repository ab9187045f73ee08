"""The single-launch batch-1 decode step against the kernel chain it replaces.

Both forms run the same row groups, per-group MMA work and fixed-order
reductions, so every output must be bit-identical: the hidden rows, the fp32
SSM state, the conv ring and the positions, step after step, from the same
seeded inputs.  (The chain, the default form, is held to the oracle by the parity
tests; through this bit-identity the fused step is too.)
"""
import numpy as np
import pytest
import torch

from mamba_ssm_layer_gb300 import abi, synth
from mamba_ssm_layer_gb300.layer import DeviceLayer, bits_u16, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from __graft_entry__ import build
    build()
    abi.m2_device_status(clear=True)
    prev = abi.m2_set_fused_decode(False)
    yield
    abi.m2_set_fused_decode(prev)
    assert abi.m2_device_status() == abi.M2_OK


def _run(dl, fused: bool, steps: int, hid: int, wl: int):
    abi.m2_set_fused_decode(fused)
    st = dl.new_state(1)
    ws = dl.workspace(1, 0)
    outs = []
    for k in range(steps):
        x = to_dev(synth.make_hidden(1, hid, wl, 7, k))
        dl.decode(x, st, ws)
        outs.append(bits_u16(x))
    torch.cuda.synchronize()
    assert abi.m2_device_status() == abi.M2_OK
    return np.concatenate(outs), [t.cpu().numpy() for t in st]


def _kernels_of_one_step(dl, hid, wl):
    abi.m2_set_fused_decode(True)
    st = dl.new_state(1)
    ws = dl.workspace(1, 0)
    x = to_dev(synth.make_hidden(1, hid, wl, 7, 0))
    dl.decode(x, st, ws)
    torch.cuda.synchronize()
    abi.trace_begin(64)
    dl.decode(x, st, ws)
    return abi.trace_end()


@pytest.mark.parametrize("dims,wl,fmt,steps", [
    (synth.TINY, synth.WL_TINY_DECODE, "fp8", 12),
    (synth.NEMOTRON_H_8B, synth.WL_8B_DECODE_B1, "fp8", 6),
    (synth.NEMOTRON_H_8B, synth.WL_8B_STACK8, "bf16", 4),
])
def test_fused_step_bit_identical_to_chain(dims, wl, fmt, steps):
    lay = synth.make_layer(dims, wl, 0, fmt, fmt)
    dl = DeviceLayer(lay)
    hid = dims["hidden"]
    tr = _kernels_of_one_step(dl, hid, wl)
    assert set(tr) == {"decode_step_fused"}, tr
    o_f, s_f = _run(dl, True, steps, hid, wl)
    o_c, s_c = _run(dl, False, steps, hid, wl)
    assert np.array_equal(o_f, o_c)
    for a, b in zip(s_f, s_c):  # SSM state (fp32 bits), conv ring, positions
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    assert np.array_equal(s_f[2], np.full(1, steps, np.int32))


def test_fused_step_one_launch_per_step_and_chain_three():
    lay = synth.make_layer(synth.NEMOTRON_H_8B, synth.WL_8B_DECODE_B1)
    dl = DeviceLayer(lay)
    st = dl.new_state(1)
    ws = dl.workspace(1, 0)
    x = to_dev(synth.make_hidden(1, 4096, synth.WL_8B_DECODE_B1, 7, 0))
    for fused, want in ((True, 1), (False, 3)):
        abi.m2_set_fused_decode(fused)
        n0 = abi.m2_launch_count()
        for _ in range(5):
            dl.decode(x, st, ws)
        torch.cuda.synchronize()
        assert abi.m2_launch_count() - n0 == 5 * want
    abi.m2_set_fused_decode(False)
