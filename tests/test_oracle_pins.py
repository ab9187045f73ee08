"""Pins of the CPU oracle to things other than itself (library routines, closed
forms, special cases, brute force).  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from mamba_ssm_layer_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def torch_e4m3_to_f64(b: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(b, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def torch_bf16_bits(v32: np.ndarray) -> np.ndarray:
    return synth.to_bf16_bits(v32)


def bf(h):
    return orc.bf16_array_to_f64(h)


# ------------------------------------------------------------------ E4M3

def test_e4m3_all_256_match_library_cast():
    ours = np.array([orc.e4m3_to_f64(b) for b in range(256)])
    ref = torch_e4m3_to_f64(np.arange(256, dtype=np.uint8))
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(ours[m], ref[m])
    # signed zero
    assert math.copysign(1.0, orc.e4m3_to_f64(0x80)) == -1.0


def test_e4m3_ocp_special_values():
    with open(os.path.join(GOLDEN, "e4m3_ocp_special_values.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) >= 10
    for hexb, val in rows:
        got = orc.e4m3_to_f64(int(hexb, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_e4m3_roundtrip_through_library_encoder():
    # every finite code decodes to a value that the library encoder maps back to it
    codes = np.array([b for b in range(256) if b not in (0x7F, 0xFF)], np.uint8)
    vals = np.array([orc.e4m3_to_f64(int(b)) for b in codes], np.float32)
    back = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # 0x80 (-0.0) re-encodes as 0x80; all codes must survive
    assert np.array_equal(back, codes)


# ------------------------------------------------------------------ bf16

def test_bf16_rne_matches_library_on_float32_values():
    rng = np.random.default_rng(7)
    exps = rng.integers(-140, 128, 20000)
    mant = rng.random(20000) + 1.0
    v = (mant * np.exp2(exps.astype(np.float64))).astype(np.float32)
    v *= np.where(rng.random(20000) < 0.5, -1, 1).astype(np.float32)
    # add exact ties and near-ties around 1.0
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -(1 + 2 ** -8),
                     2 ** -130 * 1.5, 3.0e38, 3.39e38, 3.4028e38, 0.0, -0.0], np.float32)
    v = np.concatenate([v, ties])
    ours = np.array([orc.f64_to_bf16(float(x)) for x in v], np.uint16)
    assert np.array_equal(ours, torch_bf16_bits(v))


def test_bf16_rounds_double_once():
    # 1 + 2^-8 + 2^-40 lies just above the tie between 1 and 1+2^-7: one rounding
    # gives 1+2^-7 (0x3F81); rounding through float32 first would give 1.0.
    assert orc.f64_to_bf16(1 + 2 ** -8 + 2 ** -40) == 0x3F81
    assert orc.f64_to_bf16(1 + 2 ** -8) == 0x3F80
    assert orc.f64_to_bf16(1 + 3 * 2 ** -8) == 0x3F82
    assert orc.f64_to_bf16(float("inf")) == 0x7F80
    assert orc.f64_to_bf16(-float("inf")) == 0xFF80
    assert math.isnan(orc.bf16_to_f64(orc.f64_to_bf16(float("nan"))))
    # bf16 -> double is the exact widening of the top 16 bits of a float32
    for h in (0x3F80, 0xBF80, 0x7F7F, 0x0001, 0x8001, 0x4049):
        f = np.array([h << 16], np.uint32).view(np.float32)[0]
        assert orc.bf16_to_f64(h) == float(f)


# ------------------------------------------------------------------ scalars

def test_softplus_and_silu_special_values():
    assert orc.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-15)
    assert orc.softplus(30.0) == 30.0
    assert orc.softplus(-30.0) == pytest.approx(math.exp(-30.0), rel=1e-12)
    # library: torch softplus (beta 1, threshold 20: identity above 20)
    for v in np.linspace(-25, 25, 101):
        ref = torch.nn.functional.softplus(torch.tensor(float(v), dtype=torch.float64)).item()
        assert orc.softplus(float(v)) == pytest.approx(ref, rel=1e-13, abs=1e-300)
        if v <= 20:
            assert orc.softplus(float(v)) == pytest.approx(float(np.logaddexp(0.0, v)), rel=1e-13)
    assert orc.silu(0.0) == 0.0
    assert orc.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    assert abs(orc.silu(-40.0)) < 1e-15
    for v in np.linspace(-10, 10, 41):
        ref = torch.nn.functional.silu(torch.tensor(float(v), dtype=torch.float64)).item()
        assert orc.silu(float(v)) == pytest.approx(ref, rel=1e-14, abs=1e-300)


# ------------------------------------------------------------------ GEMV

def _dequant_library(W, S, N, K):
    """Dequantise with the library's E4M3 cast and an explicit 2-D scale lookup."""
    wf = torch_e4m3_to_f64(W)
    sf = bf(S)
    n_idx = np.arange(N)[:, None] // 128
    k_idx = np.arange(K)[None, :] // 128
    return wf * sf[n_idx, k_idx]


@pytest.mark.parametrize("M,N,K", [(1, 552, 256), (3, 300, 448), (2, 129, 128)])
def test_w8a16_gemv_matches_library_matmul(M, N, K):
    rng = np.random.default_rng(M * 1000 + N)
    W, S = synth.quantize_fp8_block128((rng.standard_normal((N, K)) / math.sqrt(K)).astype(np.float32))
    A = synth.to_bf16_bits(rng.standard_normal((M, K)))
    ref = torch.from_numpy(bf(A)) @ torch.from_numpy(_dequant_library(W, S, N, K)).T
    got = orc.w8a16_gemv(A, W, S)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_w8a16_block_scale_index_brute_force():
    # one-hot activations pick one weight column; distinct power-of-two scales
    # per block make the product exact, so the block index is checked bit-exactly
    N, K = 300, 448
    nb, kb = 3, 4
    rng = np.random.default_rng(3)
    W = rng.integers(0, 256, (N, K), dtype=np.uint8)
    W[(W & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    S = synth.to_bf16_bits(np.exp2(np.arange(nb * kb).reshape(nb, kb) - 5.0))
    for k in (0, 127, 128, 255, 256, 383, 384, 447):
        A = np.zeros((1, K), np.uint16)
        A[0, k] = 0x3F80  # 1.0
        got = orc.w8a16_gemv(A, W, S)[0]
        for n in range(N):
            expect = orc.e4m3_to_f64(int(W[n, k])) * 2.0 ** ((n // 128) * kb + (k // 128) - 5)
            assert got[n] == expect, (n, k)


def test_bf16_gemv_matches_library_matmul():
    rng = np.random.default_rng(11)
    N, K = 200, 320
    W = synth.to_bf16_bits(rng.standard_normal((N, K)) / math.sqrt(K))
    A = synth.to_bf16_bits(rng.standard_normal((2, K)))
    ref = torch.from_numpy(bf(A)) @ torch.from_numpy(bf(W)).T
    np.testing.assert_allclose(orc.bf16_gemv(A, W), ref.numpy(), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ conv

def _run_conv(xs, w, b, pos0=0, silu=False, ring=None):
    Cc = xs.shape[1]
    L = w.shape[1] - 1
    ring = np.zeros((L, Cc), np.uint16) if ring is None else ring
    outs = []
    for t in range(xs.shape[0]):
        o, ring = orc.conv1d_update(ring, pos0 + t, xs[t], w, b, silu)
        outs.append(o)
    return np.array(outs), ring


@pytest.mark.parametrize("dconv", [2, 3, 4, 6])
def test_conv_matches_zero_padded_direct_convolution(dconv):
    # small integers keep every value exact, so the comparison is exact
    rng = np.random.default_rng(5 + dconv)
    T, Cc = 11, 7
    x = rng.integers(-8, 9, (T, Cc)).astype(np.float32)
    w = rng.integers(-3, 4, (Cc, dconv)).astype(np.float32)
    b = rng.integers(-4, 5, Cc).astype(np.float32)
    outs, _ = _run_conv(synth.to_bf16_bits(x), synth.to_bf16_bits(w), synth.to_bf16_bits(b))
    # library: causal depthwise conv1d with left zero padding (cross-correlation)
    xt = torch.from_numpy(x.T.astype(np.float64))[None]  # [1, C, T]
    ref = torch.nn.functional.conv1d(torch.nn.functional.pad(xt, (dconv - 1, 0)),
                                     torch.from_numpy(w.astype(np.float64))[:, None, :],
                                     torch.from_numpy(b.astype(np.float64)), groups=Cc)[0].T.numpy()
    assert np.array_equal(bf(outs), ref)


def test_conv_impulse_returns_taps_in_time_reversed_order():
    Cc, dconv = 3, 4
    w = np.array([[1, 2, 3, 4], [5, 6, 7, 8], [-1, -2, -3, -4]], np.float32)
    x = np.zeros((6, Cc), np.float32)
    x[0] = 1.0
    outs, _ = _run_conv(synth.to_bf16_bits(x), synth.to_bf16_bits(w), None)
    got = bf(outs)
    for t in range(4):
        assert np.array_equal(got[t], w[:, dconv - 1 - t])
    assert np.all(got[4:] == 0)


@pytest.mark.parametrize("pos0,dconv", [(0, 4), (1, 4), (2, 4), (5, 4), (1000, 4), (3, 2), (7, 3), (11, 6)])
def test_conv_ring_slots_and_positions_counter(pos0, dconv):
    # x_t = t+1 (exact); a one-hot tap j returns the token d_conv-1-j steps back
    Cc, T = 2, 9
    x = np.tile(np.arange(1, T + 1, dtype=np.float32)[:, None], (1, Cc))
    for j in range(dconv):
        w = np.zeros((Cc, dconv), np.float32)
        w[:, j] = 1.0
        outs, ring = _run_conv(synth.to_bf16_bits(x), synth.to_bf16_bits(w), None, pos0=pos0)
        lag = dconv - 1 - j
        expect = np.array([t + 1 - lag if t - lag >= 0 else 0 for t in range(T)], np.float64)
        assert np.array_equal(bf(outs)[:, 0], expect)
        # after T tokens, the ring holds the last d_conv-1 tokens at slots (pos0+t) mod (d_conv-1)
        L = dconv - 1
        for t in range(T - L, T):
            assert bf(ring)[(pos0 + t) % L, 0] == t + 1


def test_conv_silu_and_bias():
    x = synth.to_bf16_bits(np.array([[0.5, -1.0]], np.float32))
    w = synth.to_bf16_bits(np.array([[0, 0, 0, 2.0], [0, 0, 0, 1.0]], np.float32))
    b = synth.to_bf16_bits(np.array([0.25, 1.0], np.float32))
    o, _ = orc.conv1d_update(np.zeros((3, 2), np.uint16), 0, x[0], w, b, True)
    pre = np.array([0.5 * 2 + 0.25, -1.0 + 1.0])
    ref = torch.nn.functional.silu(torch.from_numpy(pre)).numpy()
    assert bf(o)[1] == 0.0
    assert abs(bf(o)[0] - ref[0]) <= 2 ** -8 * abs(ref[0])


# ------------------------------------------------------------------ SSM

def _ssm_inputs(rng, H, P, N, G, zeroB=False, zeroC=False):
    x = synth.to_bf16_bits(rng.standard_normal(H * P))
    Bm = synth.to_bf16_bits(np.zeros(G * N) if zeroB else rng.standard_normal(G * N))
    Cm = synth.to_bf16_bits(np.zeros(G * N) if zeroC else rng.standard_normal(G * N))
    dt = synth.to_bf16_bits(rng.standard_normal(H))
    return x, Bm, Cm, dt


def test_ssm_unrolled_closed_form():
    # h_T = (prod_r dA_r) h_0 + sum_s (prod_{r>s} dA_r) dt_s x_s B_s ;  y_t = C_t.h_t + D x_t
    rng = np.random.default_rng(9)
    H, P, N, G, T = 2, 2, 2, 1, 8
    A_log = np.array([0.3, 1.7], np.float32)
    D = np.array([1.1, 0.9], np.float32)
    dtb = np.array([-2.0, -4.0], np.float32)
    h0 = rng.standard_normal((H, P, N))
    h = h0.copy()
    steps = [_ssm_inputs(rng, H, P, N, G) for _ in range(T)]
    ys = []
    for s in steps:
        h, y, hits = orc.ssm_step(h, *s, A_log, D, dtb, G)
        ys.append(y)
        assert hits == 0
    dts = np.array([np.logaddexp(0.0, bf(s[3]) + dtb.astype(np.float64)) for s in steps])  # [T][H]
    dA = np.exp(dts * -np.exp(A_log.astype(np.float64)))                                   # [T][H]
    for hh in range(H):
        for p in range(P):
            for n in range(N):
                for t_end in range(1, T + 1):
                    val = np.prod(dA[:t_end, hh]) * h0[hh, p, n]
                    for s in range(t_end):
                        x = bf(steps[s][0])[hh * P + p]
                        val += np.prod(dA[s + 1:t_end, hh]) * dts[s, hh] * x * bf(steps[s][1])[n]
                    if t_end == T:
                        assert h[hh, p, n] == pytest.approx(val, rel=1e-12, abs=1e-14)
                # y at the last step from the closed-form state
    t = T - 1
    for hh in range(H):
        for p in range(P):
            yv = sum(bf(steps[t][2])[n] * h[hh, p, n] for n in range(N)) + D[hh] * bf(steps[t][0])[hh * P + p]
            assert ys[t][hh * P + p] == pytest.approx(yv, rel=1e-12, abs=1e-14)


def test_ssm_special_cases():
    rng = np.random.default_rng(10)
    H, P, N, G = 4, 3, 5, 2
    A_log = rng.uniform(0, math.log(16), H).astype(np.float32)
    D = rng.standard_normal(H).astype(np.float32)
    dtb = rng.uniform(-6, -2, H).astype(np.float32)
    h0 = rng.standard_normal((H, P, N))
    # B = 0: pure decay by exp(dt*A)
    x, Bm, Cm, dt = _ssm_inputs(rng, H, P, N, G, zeroB=True)
    h1, y, _ = orc.ssm_step(h0, x, Bm, Cm, dt, A_log, D, dtb, G)
    dtv = np.logaddexp(0.0, bf(dt) + dtb)
    decay = np.exp(-dtv * np.exp(A_log.astype(np.float64)))
    np.testing.assert_allclose(h1, h0 * decay[:, None, None], rtol=1e-14)
    # C = 0: y = D x
    x, Bm, Cm, dt = _ssm_inputs(rng, H, P, N, G, zeroC=True)
    _, y, _ = orc.ssm_step(h0, x, Bm, Cm, dt, A_log, D, dtb, G)
    np.testing.assert_allclose(y, np.repeat(D.astype(np.float64), P) * bf(x), rtol=1e-15)
    # group map: heads h use group h // (H/G) -> B of group 1 only reaches heads 2,3
    x = synth.to_bf16_bits(np.ones(H * P))
    Bm = synth.to_bf16_bits(np.concatenate([np.zeros(N), np.ones(N)]))
    h1, _, _ = orc.ssm_step(np.zeros((H, P, N)), x, Bm, Bm, dt, A_log, D, dtb, G)
    assert np.all(h1[:2] == 0) and np.all(h1[2:] > 0)


def test_ssm_constant_input_geometric_series():
    H, P, N, G, T = 1, 1, 1, 1, 50
    A_log = np.array([math.log(3.0)], np.float32)
    D = np.zeros(1, np.float32)
    dtb = np.array([-3.0], np.float32)
    x = synth.to_bf16_bits(np.array([0.75]))
    Bm = synth.to_bf16_bits(np.array([1.25]))
    dt = synth.to_bf16_bits(np.array([0.5]))
    h = np.zeros((1, 1, 1))
    for _ in range(T):
        h, _, _ = orc.ssm_step(h, x, Bm, Bm, dt, A_log, D, dtb, G)
    dtv = float(np.logaddexp(0.0, 0.5 - 3.0))
    a = math.exp(-dtv * math.exp(float(A_log[0])))  # A_log is stored as float32
    expect = dtv * 0.75 * 1.25 * (1 - a ** T) / (1 - a)
    assert h[0, 0, 0] == pytest.approx(expect, rel=1e-13)


def test_ssm_dt_clamp_never_binds_on_workload_distribution():
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE)
    rng = np.random.default_rng(1)
    H = synth.TINY["nheads"]
    hits = 0
    for _ in range(20):
        x, Bm, Cm, dt = _ssm_inputs(rng, H, 32, 16, 1)
        _, _, n = orc.ssm_step(np.zeros((H, 32, 16)), x, Bm, Cm, dt, lay["A_log"], lay["D"], lay["dt_bias"], 1)
        hits += n
    assert hits == 0
    # and the clamp does bind where it should
    big = synth.to_bf16_bits(np.full(H, 3.0e9))
    _, _, n = orc.ssm_step(np.zeros((H, 32, 16)), x, Bm, Cm, big, lay["A_log"], lay["D"],
                           np.zeros(H, np.float32), 1)
    assert n == H


# ------------------------------------------------------------------ norms

def test_rmsnorm_constant_vector_and_library():
    K = 64
    x = synth.to_bf16_bits(np.full((1, K), -3.0))
    w = synth.to_bf16_bits(np.full(K, 1.5))
    out = orc.rmsnorm(x, w, 0.0)
    assert np.all(bf(out) == -1.5)
    rng = np.random.default_rng(2)
    x = synth.to_bf16_bits(rng.standard_normal((3, K)))
    w = synth.to_bf16_bits(1 + 0.1 * rng.standard_normal(K))
    ref = torch.nn.functional.rms_norm(torch.from_numpy(bf(x)), (K,), torch.from_numpy(bf(w)), eps=1e-5)
    got = bf(orc.rmsnorm(x, w, 1e-5))
    np.testing.assert_allclose(got, ref.numpy(), rtol=2 ** -8)


def test_gated_rmsnorm_special_cases_and_library():
    rng = np.random.default_rng(4)
    d = 96
    y = rng.standard_normal(d)
    w = synth.to_bf16_bits(1 + 0.1 * rng.standard_normal(d))
    assert np.all(bf(orc.gated_rmsnorm(y, np.zeros(d, np.uint16), w, d, 1e-5)) == 0)
    z = synth.to_bf16_bits(rng.standard_normal(d) * 2)
    for group in (d, 32):
        got = bf(orc.gated_rmsnorm(y, z, w, group, 1e-5))
        yt = torch.from_numpy(y).reshape(-1, group)
        ref = torch.nn.functional.rms_norm(yt, (group,), eps=1e-5).reshape(-1) * torch.from_numpy(bf(w))
        ref = ref * torch.nn.functional.silu(torch.from_numpy(bf(z)))
        np.testing.assert_allclose(got, ref.numpy(), rtol=2 ** -8, atol=1e-30)
    # the norm is over y alone: scaling z does not change the normaliser
    c = np.full(d, 2.0)
    out = bf(orc.gated_rmsnorm(c, synth.to_bf16_bits(np.full(d, 30.0)), synth.to_bf16_bits(np.ones(d)), d, 0.0))
    assert np.all(out == 30.0)


# ------------------------------------------------------------------ layer

def _tiny_layer(**over):
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE)
    lay.update(over)
    return lay


def test_layer_zero_out_proj_scales_is_identity():
    lay = _tiny_layer()
    lay["out_s"] = np.zeros_like(lay["out_s"])
    L = orc.OracleLayer(lay)
    h, ring, pos = L.new_state()
    hid = synth.make_hidden(4, 256, 0, 0, 0)
    out = hid.copy()
    L.run(out, h, ring, pos)
    assert np.array_equal(out, hid)
    assert pos[0] == 4 and np.any(h != 0)


def test_layer_zero_in_proj_scales_closed_form():
    # all in_proj outputs are 0: z = 0 gates the output to 0 (out = hidden),
    # u = silu(conv bias) for every token, dt = softplus(dt_bias)
    lay = _tiny_layer()
    lay["in_s"] = np.zeros_like(lay["in_s"])
    L = orc.OracleLayer(lay)
    h, ring, pos = L.new_state()
    hid = synth.make_hidden(3, 256, 0, 0, 1)
    out = hid.copy()
    L.run(out, h, ring, pos)
    assert np.array_equal(out, hid)
    assert np.all(ring == 0)
    d_inner, N, H, P = 256, 16, 8, 32
    u = torch.nn.functional.silu(torch.from_numpy(bf(lay["conv_b"]))).numpy()
    u = bf(synth.to_bf16_bits(u))  # R4 (float64 -> float32 -> bf16 is exact-safe here within 1 ulp)
    x, Bm = u[:d_inner], u[d_inner:d_inner + N]
    dt = np.logaddexp(0.0, lay["dt_bias"].astype(np.float64))
    a = np.exp(-dt * np.exp(lay["A_log"].astype(np.float64)))
    expect = (dt * (1 + a + a * a))[:, None, None] * x.reshape(H, P)[:, :, None] * Bm[None, None, :]
    np.testing.assert_allclose(h, expect, rtol=1e-2)


def test_prefill_is_sequential_decode_and_splits():
    lay = _tiny_layer()
    L = orc.OracleLayer(lay)
    hid = synth.make_hidden(10, 256, 0, 0, 2)
    a = hid.copy(); st_a = L.new_state(); L.run(a, *st_a)
    b = hid.copy(); st_b = L.new_state()
    b1 = np.ascontiguousarray(b[:4]); b2 = np.ascontiguousarray(b[4:])
    L.run(b1, *st_b); L.run(b2, *st_b)
    assert np.array_equal(a, np.concatenate([b1, b2]))
    for x, y in zip(st_a, st_b):
        assert np.array_equal(x, y)


def test_layer_composition_against_library_pipeline():
    """One token through the tiny layer vs a float64 pipeline of library routines
    (torch rms_norm, matmul on library-dequantised weights, conv1d, silu), with the
    same bf16 rounding points; the SSM step uses the unrolled form from zero state."""
    lay = _tiny_layer()
    L = orc.OracleLayer(lay)
    h, ring, pos = L.new_state()
    hid = synth.make_hidden(1, 256, 0, 0, 3)
    out = hid.copy()
    L.run(out, h, ring, pos)

    d = synth.TINY; dd = synth.derived(d)
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    rb = lambda v: t(bf(synth.to_bf16_bits(np.asarray(v, np.float64).astype(np.float32))))
    xn = rb(torch.nn.functional.rms_norm(t(bf(hid)), (256,), t(bf(lay["norm_w"])), eps=1e-5).numpy())
    Win = t(_dequant_library(lay["in_w"], lay["in_s"], dd["n_in"], 256))
    zx = rb((xn @ Win.T).numpy())[0]
    z, xbc, dtr = zx[:dd["d_inner"]], zx[dd["d_inner"]:dd["d_inner"] + dd["d_xbc"]], zx[-d["nheads"]:]
    cw = t(bf(lay["conv_w"]))
    conv = torch.nn.functional.conv1d(torch.nn.functional.pad(xbc[None, :, None], (3, 0)), cw[:, None, :],
                                      t(bf(lay["conv_b"])), groups=dd["d_xbc"])[0, :, 0]
    u = rb(torch.nn.functional.silu(conv).numpy())
    H, P, N = 8, 32, 16
    x, Bm, Cm = u[:256].reshape(H, P), u[256:272], u[272:288]
    dt = torch.nn.functional.softplus(dtr + t(lay["dt_bias"]))
    hs = (dt[:, None, None] * x[:, :, None] * Bm[None, None, :])  # from zero state
    y = (hs * Cm).sum(-1) + t(lay["D"])[:, None] * x
    g = torch.nn.functional.rms_norm(y.reshape(1, -1), (256,), t(bf(lay["gnorm_w"])), eps=1e-5)[0]
    g = rb((g * torch.nn.functional.silu(z)).numpy())
    Wout = t(_dequant_library(lay["out_w"], lay["out_s"], 256, 256))
    ref = t(bf(hid))[0] + Wout @ g
    np.testing.assert_allclose(bf(out)[0], ref.numpy(), rtol=2e-2, atol=2e-2)
    np.testing.assert_allclose(h, hs.numpy(), rtol=1e-2, atol=1e-6)


# ------------------------------------------------------------------ W8A8 arm

def _torch_e4m3_codes(v32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v32, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_e4m3_quantizer_matches_library_cast_in_range():
    rng = np.random.default_rng(40)
    v = np.concatenate([
        rng.uniform(-448, 448, 20000), rng.uniform(-1, 1, 20000) * 2.0 ** -6,   # normals, subnormals
        np.ldexp(rng.integers(-16, 16, 2000).astype(np.float64), -10),        # exact ties in the subnormal range
        (np.arange(8, 16) + 0.5)[None, :].repeat(16, 0).ravel() * np.ldexp(1.0, np.repeat(np.arange(-6, 10), 8) - 3),
        [0.0, -0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10]]).astype(np.float32)
    v = v[np.abs(v) <= 448.0]
    ours = np.array([orc.f32_to_e4m3_sat(x) for x in v], np.uint8)
    assert np.array_equal(ours, _torch_e4m3_codes(v))


def test_e4m3_quantizer_saturates():
    for x in (448.5, 464.0, 1e6, np.float32(3.4e38)):
        assert orc.f32_to_e4m3_sat(x) == 0x7E
        assert orc.f32_to_e4m3_sat(-x) == 0xFE


def test_activation_quantization_blocks():
    rng = np.random.default_rng(41)
    a32 = (rng.standard_normal(300) * np.exp(rng.uniform(-3, 3, 300))).astype(np.float32)
    a32[128:256] = 0.0                                  # an all-zero block
    a = synth.to_bf16_bits(a32)
    q, s = orc.act_quant(a)
    av = bf(a).astype(np.float32)
    for b, (k0, k1) in enumerate([(0, 128), (128, 256), (256, 300)]):
        amax = np.float32(np.abs(av[k0:k1]).max())
        if amax == 0:
            assert s[b] == 0 and np.all(q[k0:k1] == 0)
            continue
        inv = np.float32(448.0) / amax
        assert s[b] == amax / np.float32(448.0)
        assert np.array_equal(q[k0:k1], _torch_e4m3_codes(av[k0:k1] * inv))
        # the block maximum maps to +-448 exactly
        assert np.abs(np.array([orc.e4m3_to_f64(c) for c in q[k0:k1]])).max() == 448.0


def test_w8a8_gemv_matches_library_matmul():
    rng = np.random.default_rng(42)
    N, K = 260, 300
    W, S = synth.quantize_fp8_block128((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))
    q = rng.integers(0, 256, K, dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x30
    sa = rng.uniform(0.1, 2.0, 3).astype(np.float32)
    ours = orc.w8a8_gemv(q, sa, W, S)
    qa = torch_e4m3_to_f64(q) * np.repeat(sa.astype(np.float64), 128)[:K]
    Wd = torch_e4m3_to_f64(W) * np.repeat(np.repeat(bf(S), 128, 0), 128, 1)[:N, :K]
    np.testing.assert_allclose(ours, Wd @ qa, rtol=1e-12, atol=1e-12)


def test_w8a8_layer_zero_out_proj_scales_is_identity_and_close_to_w8a16():
    lay = _tiny_layer()
    hid = synth.make_hidden(5, 256, 0, 0, 4)
    outs = []
    for fp8a in (False, True):
        L = orc.OracleLayer(lay, act_fp8=fp8a)
        h, ring, pos = L.new_state()
        out = hid.copy()
        L.run(out, h, ring, pos)
        outs.append(bf(out))
    # FP8 activations change the result by about the E4M3 step (2^-4 relative per term)
    d = np.abs(outs[1] - outs[0]).max() / np.abs(outs[0]).max()
    assert 0.0 < d < 0.1
    lay2 = dict(lay)
    lay2["out_s"] = np.zeros_like(lay["out_s"])
    L = orc.OracleLayer(lay2, act_fp8=True)
    h, ring, pos = L.new_state()
    out = hid.copy()
    L.run(out, h, ring, pos)
    assert np.array_equal(out, hid)
