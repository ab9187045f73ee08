"""GPU parity: every C entry point against the CPU oracle on the same seeded
inputs.  Integer work (E4M3 decode, block-scale index, ring slots, positions)
is compared bit-exactly; floating point in the floored relative metric of
tests/helpers.py with the stated tolerances.  Layer runs follow the GPU's
legitimate rounding decisions in the oracle (tests/helpers.py) and hold the
fp32 state of every head to 1e-3."""
import numpy as np
import pytest
import torch

from mamba_ssm_layer_gb300 import abi, synth
from mamba_ssm_layer_gb300.layer import DeviceLayer, bits_u16, to_dev
from oracle import oracle as orc
from tests.helpers import (TOL_BF16, TOL_STATE, DecisionLog, bf16_to_f64, check_state_all_heads, decode_candidates,
                           floored_rel_err, prefill_candidates, rows, state_rel_err)

pytestmark = pytest.mark.gpu

# Unit ops round one fp32 result to bf16: half an ulp (2^-9) plus fp32
# summation-order error; 2^-8 bounds it.
TOL_UNIT = 2.0 ** -8


@pytest.fixture(scope="module", autouse=True)
def _built():
    from __graft_entry__ import build
    build()
    abi.m2_device_status(clear=True)
    yield
    assert abi.m2_device_status() == abi.M2_OK


def _sync():
    torch.cuda.synchronize()


# ------------------------------------------------------------------ GEMV

def _rand_fp8(N, K, seed):
    rng = np.random.default_rng(seed)
    return synth.quantize_fp8_block128((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))


@pytest.mark.parametrize("M", [1, 3, 16, 30, 70])
def test_gemv_one_hot_is_bit_exact(M):
    # one-hot activations with power-of-two scales: out = E4M3(W[n,k]) * S exactly
    N, K = 300, 448
    rng = np.random.default_rng(21)
    W = rng.integers(0, 256, (N, K), dtype=np.uint8)
    W[(W & 0x7F) == 0x7F] = 0x41
    nb, kb = 3, 4
    S = synth.to_bf16_bits(np.exp2(np.arange(nb * kb).reshape(nb, kb) % 7 - 3.0))
    ks = [0, 127, 128, 200, 255, 256, 383, 447][: max(M, 1) * 2]
    for trial in range(2):
        A = np.zeros((M, K), np.uint16)
        sel = [ks[(trial * M + m) % len(ks)] for m in range(M)]
        for m, k in enumerate(sel):
            A[m, k] = 0x3F80
        out = torch.zeros((M, N), dtype=torch.int16, device="cuda")
        dA, dW, dS = to_dev(A), to_dev(W), to_dev(S)
        abi.w8a16_gemv(dA, dW, dS, out, M, N, K)
        _sync()
        ref = orc.f64_array_to_bf16(orc.w8a16_gemv(A, W, S))
        assert np.array_equal(bits_u16(out), ref)


@pytest.mark.parametrize("M,N,K", [(1, 552, 256), (3, 300, 448), (1, 18560, 4096), (2, 4096, 8192),
                                   (5, 1000, 4096), (4, 129, 16384),
                                   # tensor-core GEMM (M > 8): ragged M / N / K tiles, token
                                   # tiles of 16, 32, 64 and 128
                                   (9, 300, 448), (24, 1000, 4096), (64, 552, 256), (130, 1000, 4096),
                                   (200, 256, 8192)])
def test_gemv_matches_oracle(M, N, K):
    W, S = _rand_fp8(N, K, N + K)
    A = synth.to_bf16_bits(np.random.default_rng(M).standard_normal((M, K)))
    out = torch.zeros((M, N), dtype=torch.int16, device="cuda")
    abi.w8a16_gemv(to_dev(A), to_dev(W), to_dev(S), out, M, N, K)
    _sync()
    ref = orc.w8a16_gemv(A, W, S)
    assert floored_rel_err(bf16_to_f64(bits_u16(out)), ref) <= TOL_UNIT


# ------------------------------------------------------------------ conv

def test_conv_update_ring_and_pos_bit_exact():
    # counter inputs and one-hot taps (no SiLU, no bias): every output is an
    # earlier input, so ring slots and positions are checked bit-exactly
    B, Cc, dconv, steps = 3, 40, 4, 7
    ring = torch.zeros((B, dconv - 1, Cc), dtype=torch.int16, device="cuda")
    pos = torch.tensor([0, 2, 5], dtype=torch.int32, device="cuda")
    ring_o = [np.zeros((dconv - 1, Cc), np.uint16) for _ in range(B)]
    pos_o = [0, 2, 5]
    w = np.zeros((Cc, dconv), np.float32)
    for c in range(Cc):
        w[c, c % dconv] = 1.0
    wb = synth.to_bf16_bits(w)
    dw = to_dev(wb)
    for t in range(steps):
        x = synth.to_bf16_bits(np.arange(B * Cc, dtype=np.float32).reshape(B, Cc) % 97 + t * 100)
        out = torch.zeros((B, Cc), dtype=torch.int16, device="cuda")
        abi.conv1d_update(ring, pos, to_dev(x), Cc, dw, None, out, B, Cc, dconv, 0)
        _sync()
        for b in range(B):
            ref, ring_o[b] = orc.conv1d_update(ring_o[b], pos_o[b], x[b], wb, None, False)
            pos_o[b] += 1
            assert np.array_equal(bits_u16(out)[b], ref)
            assert np.array_equal(bits_u16(ring)[b], ring_o[b])
        assert pos.cpu().tolist() == pos_o


def test_conv_update_matches_oracle_with_silu_and_view():
    B, Cc, dconv, ld = 2, 1000, 4, 1200
    rng = np.random.default_rng(3)
    wb = synth.to_bf16_bits(0.5 * rng.standard_normal((Cc, dconv)))
    bb = synth.to_bf16_bits(0.1 * rng.standard_normal(Cc))
    ring = torch.zeros((B, dconv - 1, Cc), dtype=torch.int16, device="cuda")
    pos = torch.zeros(B, dtype=torch.int32, device="cuda")
    ring_o = [np.zeros((dconv - 1, Cc), np.uint16) for _ in range(B)]
    for t in range(5):
        xw = synth.to_bf16_bits(rng.standard_normal((B, ld)))
        out = torch.zeros((B, Cc), dtype=torch.int16, device="cuda")
        abi.conv1d_update(ring, pos, to_dev(xw), ld, to_dev(wb), to_dev(bb), out, B, Cc, dconv, 1)
        _sync()
        for b in range(B):
            ref, ring_o[b] = orc.conv1d_update(ring_o[b], t, xw[b, :Cc], wb, bb, True)
            assert floored_rel_err(bf16_to_f64(bits_u16(out)[b]), bf16_to_f64(ref)) <= TOL_UNIT
            assert np.array_equal(bits_u16(ring)[b], ring_o[b])


# ------------------------------------------------------------------ SSM step

@pytest.mark.parametrize("B,H,P,N,G", [(3, 8, 32, 16, 2), (1, 128, 64, 128, 8), (2, 4, 20, 64, 1), (2, 6, 8, 32, 3)])
def test_ssm_step_matches_oracle(B, H, P, N, G):
    rng = np.random.default_rng(B * 100 + N)
    ld = H * P + 2 * G * N + H + 4
    ld += (-ld) % 4
    A_log = rng.uniform(0, np.log(16), H).astype(np.float32)
    D = (1 + 0.1 * rng.standard_normal(H)).astype(np.float32)
    dt0 = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), H))
    dtb = (dt0 + np.log(-np.expm1(-dt0))).astype(np.float32)
    h0 = rng.standard_normal((B, H, P, N)).astype(np.float32)
    dh = torch.from_numpy(h0).cuda()
    hs = [h0[b].astype(np.float64) for b in range(B)]
    for step in range(3):
        buf = synth.to_bf16_bits(rng.standard_normal((B, ld)))
        dbuf = to_dev(buf)
        y = torch.zeros((B, H * P), dtype=torch.float32, device="cuda")
        xo, bo, co, do = 0, H * P, H * P + G * N, H * P + 2 * G * N
        abi.mamba2_ssm_step(dh, dbuf[:, xo:], dbuf[:, bo:], dbuf[:, co:], dbuf[:, do:], ld, to_dev(A_log), to_dev(D),
                            to_dev(dtb), y, B, H, P, N, G)
        _sync()
        for b in range(B):
            hs[b], yo, hits = orc.ssm_step(hs[b], buf[b, xo:xo + H * P], buf[b, bo:bo + G * N],
                                           buf[b, co:co + G * N], buf[b, do:do + H], A_log, D, dtb, G)
            assert hits == 0
            assert state_rel_err(dh[b].cpu().numpy(), hs[b]) <= 1e-5
            assert floored_rel_err(y[b].cpu().numpy(), yo) <= 1e-5


# ------------------------------------------------------------------ layer

def _run_decode(lay, B, steps, seqs_checked, hidden_key, warm=0):
    """Decode `warm + steps` steps of B sequences on the GPU; follow sequences
    `seqs_checked` with the oracle (taking the GPU's legitimate rounding
    decisions, refusing any other difference), checking every output row, and
    every head of the final state, bit-equal rings and positions."""
    dl = DeviceLayer(lay)
    ol = orc.OracleLayer(lay)
    d = lay["dims"]
    st = dl.new_state(B)
    ws = dl.workspace(B, 0)
    ost = {b: ol.new_state() for b in seqs_checked}
    log = DecisionLog()
    hd = d["hidden"]
    worst_out = 0.0
    for t in range(warm + steps):
        hid = synth.make_hidden(B, hd, *hidden_key, t)
        x = to_dev(hid)
        pos_before = st[2].cpu().numpy().copy()
        dl.decode(x, st, ws)
        _sync()
        got = bits_u16(x)
        cand = decode_candidates(ws, B, d, bits_u16(st[1]), pos_before, got, g_f16=lay["out_fmt"] == "fp8")
        for b in seqs_checked:
            ref = np.ascontiguousarray(hid[b:b + 1])
            log.add(ol.run_decided(ref, *ost[b], cand[b]), (t, b))
            if t >= warm:
                worst_out = max(worst_out, floored_rel_err(bf16_to_f64(got[b]), bf16_to_f64(ref[0])))
    rep = log.check()
    h = st[0].cpu().numpy()
    errs = []
    for b in seqs_checked:
        errs.append(check_state_all_heads(h[b], ost[b][0]))
        assert np.array_equal(bits_u16(st[1])[b], ost[b][1])  # ring: the (checked) R3 codes
        assert int(st[2][b]) == int(ost[b][2][0]) == warm + steps
    assert worst_out <= TOL_BF16
    print("decode parity", B, steps, worst_out, "state", max(errs), rep)
    return worst_out


def test_decode_tiny_16_steps():
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE)
    _run_decode(lay, 1, 16, [0], (synth.WL_TINY_DECODE, 0))


def test_decode_tiny_batch_and_batch_invariance():
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE)
    _run_decode(lay, 5, 6, [0, 3, 4], (synth.WL_TINY_DECODE, 1))
    # a sequence's result does not depend on the batch it is decoded in
    # (batches that fit one GEMV pass use identical per-row arithmetic)
    dl = DeviceLayer(lay)
    hid = synth.make_hidden(3, 256, 9, 9, 9)
    outs = []
    for B in (1, 3):
        st = dl.new_state(B)
        ws = dl.workspace(B, 0)
        x = to_dev(hid[:B])
        for _ in range(3):
            dl.decode(x, st, ws)
        _sync()
        outs.append(bits_u16(x)[0])
    assert np.array_equal(outs[0], outs[1])


def test_decode_8b_layer_b1_128_steps():
    lay = synth.make_layer(synth.NEMOTRON_H_8B, synth.WL_8B_DECODE_B1)
    _run_decode(lay, 1, 128, [0], (synth.WL_8B_DECODE_B1, 0))


def test_decode_8b_layer_b64_sampled():
    # 64 sequences, 32 warm-up steps + 64 steps; the oracle follows 2 of them
    lay = synth.make_layer(synth.NEMOTRON_H_8B, synth.WL_8B_DECODE_B64)
    _run_decode(lay, 64, 64, [0, 37], (synth.WL_8B_DECODE_B64, 0), warm=32)


def _prefill_case(lay, T, warm_decode, key):
    """Decode `warm_decode` tokens, then prefill T tokens; compare with the oracle
    (the prefill of T tokens is T sequential decode steps by definition)."""
    dl = DeviceLayer(lay)
    ol = orc.OracleLayer(lay)
    d = lay["dims"]
    hd = d["hidden"]
    st = dl.new_state(1)
    ws = dl.workspace(1, T)
    ost = ol.new_state()
    log = DecisionLog()
    for t in range(warm_decode):
        hid = synth.make_hidden(1, hd, *key, 1000 + t)
        x = to_dev(hid)
        pos_before = st[2].cpu().numpy().copy()
        dl.decode(x, st, ws)
        _sync()
        cand = decode_candidates(ws, 1, d, bits_u16(st[1]), pos_before, bits_u16(x))
        log.add(ol.run_decided(hid, *ost, cand[0]), ("decode", t))
    hid = synth.make_hidden(T, hd, *key, 0)
    x = to_dev(hid)
    dl.prefill(x, (st[0][0], st[1][0], st[2][:1]), ws)
    _sync()
    got = bits_u16(x)
    cand = prefill_candidates(ws, [0, T], d, got, r5_available=T > 8, g_f16=lay["out_fmt"] == "fp8")
    ref = hid.copy()
    log.add(ol.run_decided(ref, *ost, cand), "prefill")
    rep = log.check()
    err = floored_rel_err(bf16_to_f64(got), bf16_to_f64(ref), axis=-1)
    assert err <= TOL_BF16, err
    e_h = check_state_all_heads(st[0][0].cpu().numpy(), ost[0])
    assert np.array_equal(bits_u16(st[1])[0], ost[1])
    assert int(st[2][0]) == warm_decode + T
    print("prefill parity", T, err, "state", e_h, rep)
    return err


@pytest.mark.parametrize("T,warm", [(1, 0), (3, 2), (5, 0), (127, 1), (128, 0), (129, 3), (300, 2)])
def test_prefill_tiny(T, warm):
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE)
    _prefill_case(lay, T, warm, (synth.WL_TINY_DECODE, 5))


def test_prefill_split_equals_whole():
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE)
    dl = DeviceLayer(lay)
    hid = synth.make_hidden(200, 256, 7, 7, 7)
    ws = dl.workspace(1, 200)
    st1 = dl.new_state(1)
    a = to_dev(hid)
    dl.prefill(a, (st1[0][0], st1[1][0], st1[2][:1]), ws)
    st2 = dl.new_state(1)
    b1, b2 = to_dev(hid[:77]), to_dev(hid[77:])
    dl.prefill(b1, (st2[0][0], st2[1][0], st2[2][:1]), ws)
    dl.prefill(b2, (st2[0][0], st2[1][0], st2[2][:1]), ws)
    _sync()
    whole = bf16_to_f64(bits_u16(a))
    split = bf16_to_f64(np.concatenate([bits_u16(b1), bits_u16(b2)]))
    assert floored_rel_err(split, whole, axis=-1) <= TOL_BF16
    assert state_rel_err(st2[0].cpu().numpy(), st1[0].cpu().numpy()) <= TOL_STATE
    assert np.array_equal(bits_u16(st1[1]), bits_u16(st2[1]))
    assert int(st1[2][0]) == int(st2[2][0]) == 200


def test_prefill_8b_layer_1024_tokens():
    lay = synth.make_layer(synth.NEMOTRON_H_8B, synth.WL_8B_PREFILL_1K)
    _prefill_case(lay, 1024, 0, (synth.WL_8B_PREFILL_1K, 0))


# ------------------------------------------------------------------ bf16 weights

def _bf16_layer():
    return synth.make_layer(synth.TINY, synth.WL_TINY_DECODE, layer=2, in_fmt="bf16", out_fmt="bf16")


@pytest.mark.parametrize("B", [1, 5, 16])
def test_decode_tiny_bf16_weights(B):
    # the unquantised projections of a mixed-precision checkpoint: warp-MMA GEMV
    # for B <= 8, tensor-core GEMM above
    _run_decode(_bf16_layer(), B, 6, sorted({0, B - 1}), (synth.WL_TINY_DECODE, 31))


@pytest.mark.parametrize("T", [7, 129])
def test_prefill_tiny_bf16_weights(T):
    _prefill_case(_bf16_layer(), T, 2, (synth.WL_TINY_DECODE, 32))


def test_decode_tiny_b16_tensor_core_path():
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE)
    _run_decode(lay, 16, 5, [0, 9, 15], (synth.WL_TINY_DECODE, 33))


@pytest.mark.parametrize("dims,wl", [(synth.TINY, synth.WL_TINY_DECODE), (synth.NEMOTRON_H_8B, synth.WL_8B_DECODE_B64)])
def test_decode_equal_rows_give_bit_equal_results(dims, wl):
    # every reduction runs in a fixed order, so sequences with equal inputs and
    # states give bit-equal outputs and states, on the GEMV (B = 4) and the
    # tensor-core (B = 16) projections alike
    lay = synth.make_layer(dims, wl)
    dl = DeviceLayer(lay)
    hd = dims["hidden"]
    for B in (4, 16):
        st = dl.new_state(B)
        ws = dl.workspace(B, 0)
        for k in range(6):
            x = to_dev(np.repeat(synth.make_hidden(1, hd, 77, 0, k), B, axis=0))
            dl.decode(x, st, ws)
            got = bits_u16(x)
            assert np.array_equal(got, np.repeat(got[:1], B, axis=0)), (B, k)
        h = st[0].cpu().numpy()
        assert np.array_equal(h, np.repeat(h[:1], B, axis=0)), B


def test_prefill_8b_layer_40_tokens_k_split():
    # 40 tokens: the tensor-core GEMM takes 64-token tiles and splits the
    # out_proj's k range over work items (fp32 partials summed in split order)
    lay = synth.make_layer(synth.NEMOTRON_H_8B, synth.WL_8B_PREFILL_1K)
    _prefill_case(lay, 40, 0, (synth.WL_8B_PREFILL_1K, 40))
