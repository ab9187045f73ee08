"""GPU parity of the W8A8 arm (FP8 activations into the E4M3 projections;
tcgen05 kind::f8f6f4) against the oracle's W8A8 definition.

Integer work is bit-exact: the activation codes and block scales (an integer
decision taken in fp32 on both sides), and the whole product when every partial
sum is an exactly representable integer.  Layer results follow the
single-layer bar (2e-2 on bf16 outputs; the oracle follows the GPU's
legitimate rounding decisions and every head's fp32 state meets 1e-3)."""
import numpy as np
import pytest
import torch

from mamba_ssm_layer_gb300 import abi, synth
from mamba_ssm_layer_gb300.layer import DeviceLayer, bits_u16, to_dev
from oracle import oracle as orc
from tests.helpers import TOL_BF16, DecisionLog, bf16_to_f64, check_state_all_heads, floored_rel_err, prefill_candidates

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from __graft_entry__ import build
    build()
    abi.m2_device_status(clear=True)
    yield
    assert abi.m2_device_status() == abi.M2_OK


def _rup(v, a):
    return (v + a - 1) // a * a


def _w8a8(A, W, S):
    M, K = A.shape
    N = W.shape[0]
    ws = torch.empty(abi.m2_w8a8_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    out = torch.zeros((M, N), dtype=torch.int16, device="cuda")
    abi.w8a8_gemm(to_dev(A), to_dev(W), to_dev(S), out, M, N, K, ws, ws.numel())
    torch.cuda.synchronize()
    ldq = _rup(K, 16)
    off = _rup(M * ldq, 256)
    q = ws[:M * ldq].view(M, ldq).cpu().numpy()[:, :K]
    sq = ws[off:off + (K // 128) * _rup(M, 128) * 4].view(torch.float32).view(K // 128, _rup(M, 128)).cpu().numpy()
    return bits_u16(out), q, sq[:, :M].T.copy()


@pytest.mark.parametrize("M,N,K", [(9, 300, 256), (70, 552, 512), (130, 1000, 4096)])
def test_w8a8_codes_scales_bit_exact_and_product(M, N, K):
    rng = np.random.default_rng(M * 7 + K)
    A = synth.to_bf16_bits((rng.standard_normal((M, K)) * np.exp(rng.uniform(-2, 2, (M, 1)))).astype(np.float32))
    A[0, 128:256] = 0  # a zero block
    W, S = synth.quantize_fp8_block128((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))
    got, q, sq = _w8a8(A, W, S)
    ref = np.empty((M, N))
    for m in range(M):
        qo, so = orc.act_quant(A[m])
        assert np.array_equal(q[m], qo), m          # codes: integer decisions, bit-exact
        assert np.array_equal(sq[m], so), m         # fp32 scales, bit-exact
        ref[m] = orc.w8a8_gemv(qo, so, W, S)
    err = floored_rel_err(bf16_to_f64(got), bf16_to_f64(orc.f64_array_to_bf16(ref)), axis=-1)
    assert err <= TOL_BF16, err


# (40, 384, 512): 64-token tiles.  (300, 4900, 512): 256-token tiles, the second
# one ragged, over 39 weight tiles, without a k split (the call has no
# partials buffer).
@pytest.mark.parametrize("M,N,K", [(40, 384, 512), (300, 4900, 512)])
def test_w8a8_product_exact_on_integer_operands(M, N, K):
    # every block holds one 448 (so its scale is 1 and its codes are the values),
    # the rest small integers; weights small integers; power-of-two weight scales:
    # all partial sums are exact integers, so the bf16 result is the oracle's bit for bit
    rng = np.random.default_rng(5)
    a = rng.integers(-8, 9, (M, K)).astype(np.float32)
    a[:, ::128] = 448.0
    A = synth.to_bf16_bits(a)
    wv = rng.integers(-8, 9, (N, K)).astype(np.float32)
    W = torch.from_numpy(wv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    S = synth.to_bf16_bits(np.exp2(rng.integers(-8, -2, (-(-N // 128), K // 128))).astype(np.float32))
    got, _, _ = _w8a8(A, W, S)
    ref = np.stack([orc.w8a8_gemv(*orc.act_quant(A[m]), W, S) for m in range(M)])
    assert np.array_equal(got, orc.f64_array_to_bf16(ref))


def _w8a8_prefill_case(lay, T, key):
    d = lay["dims"]
    hd = d["hidden"]
    dl = DeviceLayer(lay)
    ol = orc.OracleLayer(lay, act_fp8=True)
    st = dl.new_state(1)
    ost = ol.new_state()
    hid = synth.make_hidden(T, hd, *key)
    x = to_dev(hid)
    ws = dl.workspace_varlen(1, T)
    dl.prefill_varlen(x, [0, T], st, ws, w8a8=True)
    torch.cuda.synchronize()
    got = bits_u16(x)
    # the E4M3 out_proj takes codes and scales (no bf16 gated-norm rows): the
    # oracle judges those per 128-block, then the outputs (R6)
    cand = prefill_candidates(ws, [0, T], d, got, r5_available=False, w8a8=True)
    ref = hid.copy()
    log = DecisionLog()
    log.add(ol.run_decided(ref, *ost, cand), "prefill")
    rep = log.check()
    err = floored_rel_err(bf16_to_f64(got), bf16_to_f64(ref), axis=-1)
    e_h = check_state_all_heads(st[0][0].cpu().numpy(), ost[0])
    assert err <= TOL_BF16, err
    assert np.array_equal(bits_u16(st[1])[0], ost[1])
    assert int(st[2][0]) == T
    print("w8a8 prefill parity", T, err, "state", e_h, rep)


@pytest.mark.parametrize("T", [9, 129, 300])
def test_w8a8_prefill_tiny(T):
    _w8a8_prefill_case(synth.make_layer(synth.TINY, synth.WL_TINY_DECODE), T, (synth.WL_TINY_DECODE, 90, T))


def test_w8a8_prefill_8b_layer_1024_tokens():
    _w8a8_prefill_case(synth.make_layer(synth.NEMOTRON_H_8B, synth.WL_8B_PREFILL_1K), 1024,
                       (synth.WL_8B_PREFILL_1K, 91, 0))


def test_w8a8_rejects_small_blocks():
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE)
    dl = DeviceLayer(lay)
    st = dl.new_state(1)
    x = to_dev(synth.make_hidden(8, 256, 1, 1, 1))
    ws = dl.workspace_varlen(1, 8)
    code = abi.mamba2_layer_prefill_varlen_w8a8(dl.dims, dl.struct, x, [0, 8], *st, ws, ws.numel(), check=False)
    assert code == abi.M2_ERR_UNSUPPORTED
