"""m2_copy, the staging copy kernel: bytes arrive exactly between device and
page-locked host memory in either direction, pageable host memory is refused
before any launch, and a host-staged decode loop built on it gives the same
bits as one staged with the runtime's copies."""
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


@pytest.mark.parametrize("nbytes", [16, 8192, 3 * 65536 + 48])
def test_copy_bytes_exact_all_directions(nbytes):
    rng = np.random.default_rng(nbytes)
    src = torch.from_numpy(rng.integers(0, 256, nbytes, dtype=np.uint8)).pin_memory()
    dev = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    dev2 = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    n0 = abi.m2_launch_count()
    abi.m2_copy(dev, src, nbytes)     # host -> device
    abi.m2_copy(dev2, dev, nbytes)    # device -> device
    abi.m2_copy(back, dev2, nbytes)   # device -> host
    torch.cuda.synchronize()
    assert abi.m2_launch_count() - n0 == 3
    assert torch.equal(back, src)


def test_copy_refuses_pageable_and_misaligned():
    dev = torch.zeros(64, dtype=torch.uint8, device="cuda")
    pageable = torch.zeros(64, dtype=torch.uint8)
    n0 = abi.m2_launch_count()
    assert abi.m2_copy(dev, pageable, 64, check=False) == abi.M2_ERR_ARG
    assert abi.m2_copy(dev, dev[1:].data_ptr(), 48, check=False) == abi.M2_ERR_ALIGN
    assert abi.m2_copy(dev, dev, 40, check=False) == abi.M2_ERR_ALIGN
    assert abi.m2_launch_count() == n0


def test_host_staged_decode_loop_matches_runtime_copies():
    lay = synth.make_layer(synth.NEMOTRON_H_8B, synth.WL_8B_DECODE_B1)
    dl = DeviceLayer(lay)
    ws = dl.workspace(1, 0)
    hin = [torch.from_numpy(synth.make_hidden(1, 4096, 9, 9, i).view(np.int16)).pin_memory() for i in range(6)]
    outs = {}
    for form in ("runtime", "kernel"):
        st = dl.new_state(1)
        dev = torch.empty((1, 4096), dtype=torch.int16, device="cuda")
        host_out = [torch.empty((1, 4096), dtype=torch.int16).pin_memory() for _ in hin]
        for i, h in enumerate(hin):
            if form == "runtime":
                dev.copy_(h, non_blocking=True)
                dl.decode(dev, st, ws)
                host_out[i].copy_(dev, non_blocking=True)
            else:
                abi.m2_copy(dev, h, 8192)
                dl.decode(dev, st, ws)
                abi.m2_copy(host_out[i], dev, 8192)
        torch.cuda.synchronize()
        outs[form] = (np.stack([o.numpy() for o in host_out]), st[0].cpu().numpy())
    assert np.array_equal(outs["runtime"][0], outs["kernel"][0])
    assert np.array_equal(outs["runtime"][1].view(np.uint8), outs["kernel"][1].view(np.uint8))


def test_copy_refuses_a_range_past_the_allocation():
    # a size no allocation holds: refused on the host before any launch, in
    # either direction and for device and page-locked host memory alike
    dev = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    pinned = torch.zeros(4096, dtype=torch.uint8).pin_memory()
    huge = 1 << 44
    n0 = abi.m2_launch_count()
    assert abi.m2_copy(dev, pinned, huge, check=False) == abi.M2_ERR_ARG
    assert abi.m2_copy(pinned, dev, huge, check=False) == abi.M2_ERR_ARG
    assert abi.m2_copy(dev, dev, huge, check=False) == abi.M2_ERR_ARG
    assert abi.m2_launch_count() == n0
    # in range: still copies
    pinned[:] = torch.arange(4096, dtype=torch.int32).to(torch.uint8)
    abi.m2_copy(dev, pinned, 4096)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), pinned)
