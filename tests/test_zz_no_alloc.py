"""The no-allocation decode entry point, through the C ABI.

mamba2_layer_decode_noalloc serves callers that cannot allocate device memory
when they need it (a plug-in inside a host that reserved all device memory for
its own pool, or a latency-critical loop that must not enter the allocator).
It uses a fixed scratch array built into the library instead of a workspace.
This test checks, on two calls in a row, that it produces what
mamba2_layer_decode produces (same tolerance as the other layer tests), and
that a request larger than the built-in scratch is refused.  The file is
collected last so that a stop-at-first-failure run has run every other test.
"""
import numpy as np
import pytest
import torch

from mamba_ssm_layer_gb300 import abi, synth
from mamba_ssm_layer_gb300.layer import DeviceLayer, bits_u16, to_dev
from tests.helpers import TOL_BF16, TOL_STATE, bf16_to_f64, floored_rel_err, state_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from __graft_entry__ import build
    build()


@pytest.mark.parametrize("dims,wl,B", [(synth.TINY, synth.WL_TINY_DECODE, 3),
                                       (synth.NEMOTRON_H_8B, synth.WL_8B_DECODE_B1, 1),
                                       # tensor-core projections, k-split partials in the built-in array
                                       (synth.NEMOTRON_H_8B, synth.WL_8B_DECODE_B64, 16),
                                       # the largest batch the built-in array holds for this layer
                                       (synth.NEMOTRON_H_8B, synth.WL_8B_DECODE_B64, 88)])
def test_noalloc_decode_matches_workspace_decode(dims, wl, B):
    lay = synth.make_layer(dims, wl)
    dl = DeviceLayer(lay)
    st_ref = dl.new_state(B)
    st_new = dl.new_state(B)
    ws = dl.workspace(B, 0)
    for step in range(2):  # two calls in a row: the scratch keeps the last call's contents
        hid = synth.make_hidden(B, dims["hidden"], wl, 77, step)
        x_ref, x_new = to_dev(hid), to_dev(hid)
        abi.mamba2_layer_decode(dl.dims, dl.struct, x_ref, B, st_ref[0], st_ref[1], st_ref[2], ws, ws.numel(),
                                torch.cuda.current_stream())
        abi.mamba2_layer_decode_noalloc(dl.dims, dl.struct, x_new, B, st_new[0], st_new[1], st_new[2],
                                        torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert floored_rel_err(bf16_to_f64(bits_u16(x_new)), bf16_to_f64(bits_u16(x_ref)), axis=-1) <= TOL_BF16
        assert state_rel_err(st_new[0].cpu().numpy(), st_ref[0].cpu().numpy()) <= TOL_STATE
        assert np.array_equal(bits_u16(st_new[1]), bits_u16(st_ref[1]))
        assert torch.equal(st_new[2], st_ref[2])
    assert abi.m2_device_status() == abi.M2_OK


def test_noalloc_rejects_batches_beyond_the_scratch():
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE)
    dl = DeviceLayer(lay)
    B = 1
    while abi.m2_workspace_bytes(dl.dims, B, 0) <= abi.M2_NOALLOC_SCRATCH_BYTES:
        B += 1
    assert abi.m2_workspace_bytes(dl.dims, B - 1, 0) <= abi.M2_NOALLOC_SCRATCH_BYTES
    launches = abi.m2_launch_count()
    st = abi.mamba2_layer_decode_noalloc(dl.dims, dl.struct, 1 << 20, B, 1 << 20, 1 << 20, 1 << 20, check=False)
    assert st == abi.M2_ERR_SCRATCH
    assert abi.m2_launch_count() == launches
