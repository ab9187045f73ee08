"""Bounded in-kernel waits: a wait that runs out records M2_ERR_TIMEOUT, the
kernel still waits for the copies and tensor-core work it issued, frees its
tensor memory and returns, and the device stays usable.

The failure is made without a fault: a barrier that nothing signals
(m2_wait_check), or a pipeline wait limit far below what a healthy pipeline
needs (m2_set_wait_limit), so that waits give up on valid inputs.  After each
case the limit is restored and the same kernels must again match the oracle.
"""
import numpy as np
import pytest
import torch

from mamba_ssm_layer_gb300 import abi, synth
from mamba_ssm_layer_gb300.layer import DeviceLayer, bits_u16, to_dev
from oracle import oracle as orc
from tests.helpers import bf16_to_f64, floored_rel_err

pytestmark = pytest.mark.gpu

TOL_UNIT = 2.0 ** -8


@pytest.fixture(scope="module", autouse=True)
def _built():
    from __graft_entry__ import build
    build()
    abi.m2_device_status(clear=True)
    yield
    abi.m2_set_wait_limit(0)
    abi.m2_device_status(clear=True)


@pytest.fixture(autouse=True)
def _restore_limit():
    yield
    abi.m2_set_wait_limit(0)


def _gemv_case(M, N, K, seed):
    rng = np.random.default_rng(seed)
    W, S = synth.quantize_fp8_block128((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))
    A = synth.to_bf16_bits(rng.standard_normal((M, K)))
    return A, W, S


def _w8a16(A, W, S):
    M, K = A.shape
    N = W.shape[0]
    out = torch.zeros((M, N), dtype=torch.int16, device="cuda")
    abi.w8a16_gemv(to_dev(A), to_dev(W), to_dev(S), out, M, N, K)
    return out


def _w8a8(A, W, S):
    M, K = A.shape
    N = W.shape[0]
    ws = torch.empty(abi.m2_w8a8_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    out = torch.zeros((M, N), dtype=torch.int16, device="cuda")
    abi.w8a8_gemm(to_dev(A), to_dev(W), to_dev(S), out, M, N, K, ws, ws.numel())
    return out


def test_wait_check_times_out_and_leaves_the_device_usable():
    probe = torch.arange(4, dtype=torch.int32, device="cuda") * 0x01010101 + 0x12345678
    out = torch.zeros(4, dtype=torch.int32, device="cuda")
    abi.m2_device_status(clear=True)
    abi.m2_set_wait_limit(200_000)  # about 0.1 ms
    abi.m2_wait_check(probe, out)
    assert abi.m2_device_status() == abi.M2_ERR_TIMEOUT
    assert torch.equal(out, probe)  # the copy in flight was waited for before the kernel returned
    abi.m2_device_status(clear=True)
    assert abi.m2_device_status() == abi.M2_OK
    abi.m2_set_wait_limit(0)
    # tensor memory was freed: the tensor-core GEMM allocates it on every SM
    A, W, S = _gemv_case(130, 1000, 4096, 3)
    out = _w8a16(A, W, S)
    torch.cuda.synchronize()
    assert abi.m2_device_status() == abi.M2_OK
    assert floored_rel_err(bf16_to_f64(bits_u16(out)), orc.w8a16_gemv(A, W, S)) <= TOL_UNIT


def test_wait_check_rejects_unaligned_pointers():
    buf = torch.zeros(16, dtype=torch.int32, device="cuda")
    n0 = abi.m2_launch_count()
    assert abi.m2_wait_check(buf.data_ptr() + 4, buf, check=False) == abi.M2_ERR_ALIGN
    assert abi.m2_wait_check(None, buf, check=False) == abi.M2_ERR_ARG
    assert abi.m2_launch_count() == n0


# (M, N, K): decode GEMV on warp MMA, CUDA-core GEMV (K > 8192), tcgen05 GEMM (64- and 128-token tiles)
CASES = [(1, 18560, 4096), (4, 129, 16384), (40, 552, 1024), (130, 1000, 4096)]


def test_real_kernels_time_out_cleanly_under_a_one_cycle_limit():
    # every wait that is not complete on its first poll gives up at once (the
    # first weight stage of any kernel is still in flight when its consumers
    # first look), so each kernel takes its timeout exit: stop the pipeline,
    # wait for its own copies and MMAs, free tensor memory, return
    data = [_gemv_case(M, N, K, M + N) for M, N, K in CASES]
    q8 = _gemv_case(70, 552, 512, 11)
    # each kernel runs once first: the first launch of a kernel in a process
    # starts its roles late (its code is not yet loaded near the SM), so its
    # consumers' first polls can find the data already landed and no wait
    # runs out
    for A, W, S in data:
        _w8a16(A, W, S)
    _w8a8(*q8)
    torch.cuda.synchronize()
    abi.m2_device_status(clear=True)
    abi.m2_set_wait_limit(1)
    for i, (A, W, S) in enumerate(data):
        _w8a16(A, W, S)
        torch.cuda.synchronize()
        assert abi.m2_device_status(clear=True) == abi.M2_ERR_TIMEOUT, CASES[i]
    _w8a8(*q8)
    torch.cuda.synchronize()
    assert abi.m2_device_status(clear=True) == abi.M2_ERR_TIMEOUT
    abi.m2_set_wait_limit(0)
    for A, W, S in data:
        out = _w8a16(A, W, S)
        torch.cuda.synchronize()
        assert floored_rel_err(bf16_to_f64(bits_u16(out)), orc.w8a16_gemv(A, W, S)) <= TOL_UNIT, A.shape
    out = _w8a8(*q8)
    torch.cuda.synchronize()
    A, W, S = q8
    ref = np.stack([orc.w8a8_gemv(*orc.act_quant(A[m]), W, S) for m in range(A.shape[0])])
    assert floored_rel_err(bf16_to_f64(bits_u16(out)), bf16_to_f64(orc.f64_array_to_bf16(ref)), axis=-1) <= 2e-2
    assert abi.m2_device_status() == abi.M2_OK


def test_fused_decode_grid_barrier_realigns_after_timeouts():
    # The single-launch step synchronises its CTAs through one device-wide
    # arrival counter.  Under a one-cycle limit its grid barriers give up (the
    # CTAs reach them microseconds apart); every CTA still arrives once per
    # barrier, so the next launches line up again and give the chain's results
    # bit for bit.
    lay = synth.make_layer(synth.NEMOTRON_H_8B, synth.WL_8B_DECODE_B1)
    dl = DeviceLayer(lay)
    ws = dl.workspace(1, 0)
    prev = abi.m2_set_fused_decode(True)
    try:
        junk = dl.new_state(1)
        abi.m2_device_status(clear=True)
        abi.m2_set_wait_limit(1)
        for k in range(3):
            dl.decode(to_dev(synth.make_hidden(1, 4096, 5, 5, k)), junk, ws)
        torch.cuda.synchronize()
        st = abi.m2_device_status(clear=True)
        assert st == abi.M2_ERR_TIMEOUT, st
        abi.m2_set_wait_limit(0)
        outs = {}
        for fused in (True, False):
            abi.m2_set_fused_decode(fused)
            s = dl.new_state(1)
            rows = []
            for k in range(4):
                x = to_dev(synth.make_hidden(1, 4096, 6, 6, k))
                dl.decode(x, s, ws)
                rows.append(bits_u16(x))
            torch.cuda.synchronize()
            outs[fused] = (np.concatenate(rows), s[0].cpu().numpy(), bits_u16(s[1]), s[2].cpu().numpy())
        for a, b in zip(outs[True], outs[False]):
            assert np.array_equal(a, b)
        assert abi.m2_device_status() == abi.M2_OK
    finally:
        abi.m2_set_fused_decode(prev)
