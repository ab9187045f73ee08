"""Host-only checks of the C ABI: the library loads, exports every declared
entry point, and rejects bad arguments before launching anything.  No GPU."""
import ctypes as C
import os
import re

import pytest

from mamba_ssm_layer_gb300 import abi, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from __graft_entry__ import build
    build()
    return abi.lib()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z][A-Za-z0-9_]*)\s*\(", src, re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "mamba2_layer_decode" in names and "w8a16_gemv" in names and len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert set(abi.EXPORTS) <= set(names)


def test_strerror_and_kernel_names(lib):
    assert abi.strerror(0) == "ok"
    assert "workspace" in abi.strerror(abi.M2_ERR_WORKSPACE)
    names = abi.kernel_names()
    assert "gemv_fp8" in names and len(names) == lib.m2_kernel_count()


def _dims(**over):
    d = dict(synth.NEMOTRON_H_8B)
    d.update(over)
    return abi.dims_struct(d)


def test_workspace_bytes(lib):
    d = _dims()
    a = abi.m2_workspace_bytes(d, 1, 0)
    b = abi.m2_workspace_bytes(d, 64, 0)
    c = abi.m2_workspace_bytes(d, 0, 1024)
    assert 0 < a < b and c > b
    # xn + zxu + y + g per row, each 256-aligned
    assert a >= 4096 * 2 + 18560 * 2 + 8192 * 4 + 8192 * 2
    bad = _dims(d_state=96)
    assert abi.m2_workspace_bytes(bad, 1, 1) == 0


FAKE = 1 << 20  # a 16-byte-aligned non-null "device" address; never dereferenced


def _layer(in_fmt=abi.M2_W_FP8_BLOCK128, in_scale=FAKE, n_in=18560, out_n=4096, align=0):
    return abi.M2Layer(FAKE, abi.M2Weight(FAKE + align, in_scale, n_in, 4096, in_fmt), FAKE, FAKE, FAKE, FAKE, FAKE,
                       FAKE, abi.M2Weight(FAKE, FAKE, out_n, 8192, abi.M2_W_FP8_BLOCK128))


def test_validate_accepts_good_layer(lib):
    assert abi.m2_validate(_dims(), _layer()) == abi.M2_OK


@pytest.mark.parametrize("case,expect", [
    (dict(layer=dict(in_fmt=7)), abi.M2_ERR_FORMAT),
    (dict(layer=dict(in_scale=None)), abi.M2_ERR_FORMAT),
    (dict(layer=dict(in_fmt=abi.M2_W_BF16)), abi.M2_ERR_FORMAT),   # bf16 with a scale grid
    (dict(layer=dict(n_in=18559)), abi.M2_ERR_ARG),
    (dict(layer=dict(out_n=4095)), abi.M2_ERR_ARG),
    (dict(layer=dict(align=8)), abi.M2_ERR_ALIGN),
    (dict(dims=dict(nheads=127)), abi.M2_ERR_ARG),                 # H % G
    (dict(dims=dict(d_state=96)), abi.M2_ERR_UNSUPPORTED),
    (dict(dims=dict(d_conv=1)), abi.M2_ERR_UNSUPPORTED),
    (dict(dims=dict(hidden=4100)), abi.M2_ERR_UNSUPPORTED),
    (dict(dims=dict(gnorm_group=1000)), abi.M2_ERR_UNSUPPORTED),
])
def test_validate_rejects(lib, case, expect):
    d = _dims(**case.get("dims", {}))
    L = _layer(**case.get("layer", {}))
    assert abi.m2_validate(d, L) == expect


def test_entry_points_reject_before_launch(lib):
    # These return before touching the device: no GPU is needed to run them.
    launches0 = abi.m2_launch_count()
    d, L = _dims(), _layer()
    ws_need = abi.m2_workspace_bytes(d, 2, 0)
    st = abi.mamba2_layer_decode(d, L, FAKE, 2, FAKE, FAKE, FAKE, FAKE, ws_need - 1, check=False)
    assert st == abi.M2_ERR_WORKSPACE
    st = abi.mamba2_layer_decode(d, L, FAKE, 0, FAKE, FAKE, FAKE, FAKE, ws_need, check=False)
    assert st == abi.M2_ERR_ARG
    st = abi.mamba2_layer_decode(d, L, FAKE + 2, 2, FAKE, FAKE, FAKE, FAKE, ws_need, check=False)
    assert st == abi.M2_ERR_ALIGN
    st = abi.mamba2_layer_decode(d, L, FAKE, 2, FAKE, FAKE, FAKE, FAKE + 16, ws_need, check=False)
    assert st == abi.M2_ERR_WORKSPACE  # workspace must be 256-byte aligned
    # the L2 hint of the prefetching decode: checked first, then the decode's own checks
    st = abi.mamba2_layer_decode_prefetch(d, L, FAKE, 2, FAKE, FAKE, FAKE, FAKE, ws_need, FAKE + 8, 4096, check=False)
    assert st == abi.M2_ERR_ALIGN
    st = abi.mamba2_layer_decode_prefetch(d, L, FAKE, 2, FAKE, FAKE, FAKE, FAKE, ws_need, FAKE,
                                          abi.M2_PREFETCH_MAX_BYTES + 16, check=False)
    assert st == abi.M2_ERR_ARG
    st = abi.mamba2_layer_decode_prefetch(d, L, FAKE, 2, FAKE, FAKE, FAKE, FAKE, ws_need - 1, FAKE, 0, check=False)
    assert st == abi.M2_ERR_WORKSPACE  # no hint: exactly mamba2_layer_decode
    st = abi.mamba2_layer_prefill(d, L, FAKE, 5, FAKE, FAKE, None, FAKE, 1 << 30, check=False)
    assert st == abi.M2_ERR_ARG
    bad = _layer(in_fmt=3)
    st = abi.mamba2_layer_prefill(d, bad, FAKE, 5, FAKE, FAKE, FAKE, FAKE, 1 << 30, check=False)
    assert st == abi.M2_ERR_FORMAT
    assert abi.w8a16_gemv(FAKE, FAKE, FAKE, FAKE, 1, 10, 24, check=False) == abi.M2_ERR_UNSUPPORTED
    assert abi.w8a16_gemv(None, FAKE, FAKE, FAKE, 1, 10, 32, check=False) == abi.M2_ERR_ARG
    assert abi.w8a16_gemv(FAKE, FAKE + 4, FAKE, FAKE, 1, 10, 32, check=False) == abi.M2_ERR_ALIGN
    assert abi.conv1d_update(FAKE, FAKE, FAKE, 8, FAKE, FAKE, FAKE, 1, 8, 9, check=False) == abi.M2_ERR_UNSUPPORTED
    assert abi.conv1d_update(FAKE, FAKE, FAKE, 4, FAKE, FAKE, FAKE, 1, 8, 4, check=False) == abi.M2_ERR_ARG
    assert abi.mamba2_ssm_step(FAKE, FAKE, FAKE, FAKE, FAKE, 64, FAKE, FAKE, FAKE, FAKE, 1, 8, 8, 48, 1,
                               check=False) == abi.M2_ERR_UNSUPPORTED
    assert abi.mamba2_ssm_step(FAKE, FAKE, FAKE, FAKE, FAKE, 64, FAKE, FAKE, FAKE, FAKE, 1, 8, 8, 16, 3,
                               check=False) == abi.M2_ERR_ARG
    assert abi.m2_copy(None, FAKE, 16, check=False) == abi.M2_ERR_ARG
    assert abi.m2_copy(FAKE, FAKE + 8, 16, check=False) == abi.M2_ERR_ALIGN
    assert abi.m2_copy(FAKE, FAKE, 24, check=False) == abi.M2_ERR_ALIGN
    assert abi.m2_copy(FAKE, FAKE, 0, check=False) == abi.M2_OK  # nothing to copy
    assert abi.m2_launch_count() == launches0  # nothing was launched by any of the above


def _rup(v, a):
    return (v + a - 1) // a * a


def test_w8a8_workspace_follows_documented_layout(lib):
    # codes [M][rup16(K)] bytes, then at the next 256-byte boundary the fp32
    # scales [K/128][rup128(M)], the whole rounded up to 256 bytes
    for M, K in [(9, 256), (70, 512), (1024, 4096), (130, 8192)]:
        want = _rup(M * _rup(K, 16), 256) + _rup((K // 128) * _rup(M, 128) * 4, 256)
        assert abi.m2_w8a8_workspace_bytes(M, K) == want, (M, K)
    assert abi.m2_w8a8_workspace_bytes(0, 128) == 0


def test_varlen_workspace_and_rejections_before_launch(lib):
    d, L = _dims(), _layer()
    w1 = abi.m2_workspace_bytes_varlen(d, 1, 1024)
    assert 0 < w1 <= abi.m2_workspace_bytes_varlen(d, 16, 1024) < abi.m2_workspace_bytes_varlen(d, 16, 2048)
    assert w1 >= abi.m2_workspace_bytes(d, 0, 1024)  # plus the W8A8 arm's codes and scales
    assert abi.m2_workspace_bytes_varlen(_dims(d_state=96), 1, 64) == 0
    launches0 = abi.m2_launch_count()
    for cu in ([1, 5], [0, 5, 3], [0, 0]):
        st = abi.mamba2_layer_prefill_varlen(d, L, FAKE, cu, FAKE, FAKE, FAKE, FAKE, 1 << 34, check=False)
        assert st == abi.M2_ERR_ARG, cu
    # the W8A8 arm needs more than 8 token rows (tensor-core projections)
    st = abi.mamba2_layer_prefill_varlen_w8a8(d, L, FAKE, [0, 3, 8], FAKE, FAKE, FAKE, FAKE, 1 << 34, check=False)
    assert st == abi.M2_ERR_UNSUPPORTED
    need = abi.m2_workspace_bytes_varlen(d, 2, 300)
    st = abi.mamba2_layer_prefill_varlen(d, L, FAKE, [0, 100, 300], FAKE, FAKE, FAKE, FAKE, need // 2, check=False)
    assert st == abi.M2_ERR_WORKSPACE
    # the W8A8 product as a unit
    assert abi.w8a8_gemm(FAKE, FAKE, FAKE, FAKE, 8, 256, 256, FAKE, 1 << 30, check=False) == abi.M2_ERR_UNSUPPORTED
    assert abi.w8a8_gemm(FAKE, FAKE, FAKE, FAKE, 64, 256, 200, FAKE, 1 << 30, check=False) == abi.M2_ERR_UNSUPPORTED
    small = abi.m2_w8a8_workspace_bytes(64, 256) - 1
    assert abi.w8a8_gemm(FAKE, FAKE, FAKE, FAKE, 64, 256, 256, FAKE, small, check=False) == abi.M2_ERR_WORKSPACE
    assert abi.m2_launch_count() == launches0


def test_fused_decode_toggle_is_host_only(lib):
    # the batch-1 single-launch step is off by default; the setter returns the previous value
    assert abi.m2_set_fused_decode(True) is False
    assert abi.m2_set_fused_decode(False) is True
    assert abi.m2_set_fused_decode(False) is False
