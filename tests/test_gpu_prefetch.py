"""The prefetching decode (mamba2_layer_decode_prefetch): a hint that pulls a
byte range -- the next layer's first in_proj weights -- toward L2 during the
step's out_proj.  It must not change any result: outputs, states, rings and
positions are bit-identical to mamba2_layer_decode over several steps that
alternate two layers (each step hinting the other), at batch 1 and 4.  A range
outside one device allocation is refused before anything is launched."""
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
    yield
    assert abi.m2_device_status() == abi.M2_OK


@pytest.mark.parametrize("B", [1, 4])
def test_prefetch_hint_leaves_results_bit_identical(B):
    d = synth.NEMOTRON_H_8B
    layers = [DeviceLayer(synth.make_layer(d, synth.WL_8B_DECODE_B1)),
              DeviceLayer(synth.make_layer(d, synth.WL_8B_DECODE_B64))]
    ws = layers[0].workspace(B, 0)
    runs = []
    for hinted in (False, True):
        states = [dl.new_state(B) for dl in layers]
        x = to_dev(synth.make_hidden(B, d["hidden"], 31, B, 0))
        rows = []
        n0 = abi.m2_launch_count()
        for k in range(6):
            i = k % 2
            layers[i].decode(x, states[i], ws, ahead=layers[1 - i] if hinted else None)
            rows.append(bits_u16(x))
        torch.cuda.synchronize()
        launches = abi.m2_launch_count() - n0
        runs.append((np.concatenate(rows), [s[0].cpu().numpy() for s in states],
                     [bits_u16(s[1]) for s in states], [s[2].cpu().numpy() for s in states], launches))
    plain, hinted = runs
    assert np.array_equal(plain[0], hinted[0])
    for a, b in zip(plain[1] + plain[2] + plain[3], hinted[1] + hinted[2] + hinted[3]):
        assert np.array_equal(a, b)
    assert plain[4] == hinted[4]  # the hint adds no launch


def test_prefetch_range_outside_one_allocation_is_refused():
    d = synth.NEMOTRON_H_8B
    dl = DeviceLayer(synth.make_layer(d, synth.WL_8B_DECODE_B1))
    ws = dl.workspace(1, 0)
    h, ring, pos = dl.new_state(1)
    x = to_dev(synth.make_hidden(1, d["hidden"], 32, 0, 0))
    small = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    n0 = abi.m2_launch_count()
    st = abi.mamba2_layer_decode_prefetch(dl.dims, dl.struct, x, 1, h, ring, pos, ws, ws.numel(), small, 2 << 20,
                                          check=False)
    assert st == abi.M2_ERR_ARG
    assert abi.m2_launch_count() == n0
    before = bits_u16(x).copy()
    st = abi.mamba2_layer_decode_prefetch(dl.dims, dl.struct, x, 1, h, ring, pos, ws, ws.numel(), small, 1 << 20)
    torch.cuda.synchronize()
    assert st == abi.M2_OK and not np.array_equal(bits_u16(x), before)
