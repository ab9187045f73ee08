"""CPU pins of the oracle's decision-following mode (OracleLayer.run_decided)
and of the sums of |terms| that scale its tolerances.

run_decided lets the oracle take another evaluation's bf16 code at a rounding
point only where that code is a correct rounding of a value within tolerance
of the oracle's own exact value.  These tests pin: the rounding interval of a
code against the library's bf16 cast; the |terms| sums against float64 numpy
sums; that no candidates, or the oracle's own codes as candidates, change
nothing; that a near-tie neighbour is taken; and that wrong codes -- a code a
few ulps off, or every code an evaluation that dropped one term would give --
are refused while the oracle keeps its own."""
import numpy as np
import pytest
import torch

from mamba_ssm_layer_gb300 import synth
from oracle import oracle as orc


def _bf16_cast(v):
    """Library rounding of float32-representable values to bf16 codes."""
    t = torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("code", [0x0000, 0x0001, 0x007F, 0x0080, 0x3F80, 0x3F81, 0x4000, 0x7F7E, 0x8000, 0xBF80,
                                  0xC123, 0x1234, 0x7F7F])
def test_round_interval_matches_the_library_cast(code):
    lo, hi = orc.bf16_round_interval(code)
    assert lo < orc.bf16_to_f64(code) < hi or (code & 0x7FFF) == 0
    width = hi - lo
    inside = [lo + width * f for f in (1 / 64, 1 / 2, 63 / 64)]
    got = _bf16_cast(inside)
    assert np.all((got & 0x7FFF) == (code & 0x7FFF)), (hex(code), got)
    if (code & 0x7FFF) not in (0, 0x7F7F):
        out = _bf16_cast([lo - width / 64, hi + width / 64])
        assert np.all(out != code)


def test_round_interval_of_nan_and_inf_is_none():
    for c in (0x7F80, 0xFF80, 0x7FC0):
        assert orc.bf16_round_interval(c) is None
        assert orc.decision_excess(c, 1.0, 1.0) == np.inf


def test_decision_excess_is_distance_over_scale():
    lo, hi = orc.bf16_round_interval(0x3F80)  # 1.0: [1 - 2^-9, 1 + 2^-8]
    assert (lo, hi) == (1 - 2 ** -9, 1 + 2 ** -8)
    assert orc.decision_excess(0x3F80, 1.0 + 2 ** -8, 1.0) == 0.0
    assert orc.decision_excess(0x3F80, 1.0 + 2 ** -7, 4.0) == pytest.approx(2 ** -8 / 4.0, rel=1e-15)
    assert orc.decision_excess(0x3F80, 1.0 - 2 ** -8, 1.0) == pytest.approx(2 ** -9, rel=1e-15)


def test_proj_abs_matches_a_float64_sum():
    rng = np.random.default_rng(4)
    N, K = 300, 448
    W, S = synth.quantize_fp8_block128((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))
    a = synth.to_bf16_bits(rng.standard_normal(K))
    wd = torch.from_numpy(W).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    sd = np.repeat(np.repeat(orc.bf16_array_to_f64(S), 128, 0), 128, 1)[:N, :K]
    ref = np.sum(np.abs(orc.bf16_array_to_f64(a)[None, :] * wd * sd), axis=1)
    assert np.allclose(orc.proj_abs(a, W, S), ref, rtol=1e-12, atol=0)
    Wb = synth.to_bf16_bits(rng.standard_normal((N, K)))
    refb = np.sum(np.abs(orc.bf16_array_to_f64(a)[None, :] * orc.bf16_array_to_f64(Wb)), axis=1)
    assert np.allclose(orc.proj_abs(a, Wb), refb, rtol=1e-12, atol=0)


def test_w8a8_abs_matches_a_float64_sum():
    rng = np.random.default_rng(5)
    N, K = 260, 384
    W, S = synth.quantize_fp8_block128((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))
    a = synth.to_bf16_bits(rng.standard_normal(K))
    q, sa = orc.act_quant(a)
    qd = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    wd = torch.from_numpy(W).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    sd = orc.bf16_array_to_f64(S)
    ref = np.zeros(N)
    for b in range(K // 128):
        part = np.sum(np.abs(qd[None, b * 128:(b + 1) * 128] * wd[:, b * 128:(b + 1) * 128]), axis=1)
        ref += np.abs(sa[b] * sd[np.arange(N) // 128, b]) * part
    assert np.allclose(orc.w8a8_abs(q, sa, W, S), ref, rtol=1e-12, atol=0)


def test_conv_exact_and_abs_match_a_direct_convolution():
    rng = np.random.default_rng(6)
    Cc, dconv, pos = 50, 4, 5
    L = dconv - 1
    ring = synth.to_bf16_bits(rng.standard_normal((L, Cc)))
    x = synth.to_bf16_bits(rng.standard_normal(Cc))
    w = synth.to_bf16_bits(0.5 * rng.standard_normal((Cc, dconv)))
    b = synth.to_bf16_bits(0.1 * rng.standard_normal(Cc))
    out, ring2, ex, ab = orc.conv1d_update_exact(ring, pos, x, w, b)
    win = np.stack([orc.bf16_array_to_f64(ring[(pos + j) % L]) for j in range(L)] + [orc.bf16_array_to_f64(x)], 1)
    wd, bd = orc.bf16_array_to_f64(w), orc.bf16_array_to_f64(b)
    pre = bd + np.sum(wd * win, axis=1)
    assert np.allclose(ex, pre / (1 + np.exp(-pre)), rtol=1e-14, atol=1e-300)
    assert np.allclose(ab, np.abs(bd) + np.sum(np.abs(wd * win), axis=1), rtol=1e-14, atol=0)
    assert np.array_equal(out, orc.f64_array_to_bf16(ex))
    assert np.array_equal(ring2[pos % L], x)


def _tiny():
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE)
    return lay, orc.OracleLayer(lay)


def _run(ol, hid, cand=None):
    st = ol.new_state()
    h = hid.copy()
    rep = ol.run_decided(h, *st, cand or {}) if cand is not None else ol.run(h, *st)
    return h, st, rep


def _same(a, b):
    (ha, sa, _), (hb, sb, _) = a, b
    return (np.array_equal(ha, hb) and np.array_equal(sa[0], sb[0]) and np.array_equal(sa[1], sb[1])
            and np.array_equal(sa[2], sb[2]))


def test_no_candidates_and_own_codes_change_nothing():
    lay, ol = _tiny()
    hid = synth.make_hidden(6, 256, 40, 0, 0)
    plain = _run(ol, hid)
    assert _same(plain, _run(ol, hid, {}))
    st = ol.new_state()
    h = hid.copy()
    _, (e3, _), (e4, _) = ol.run_traced(h, *st)
    own = {"R3": orc.f64_array_to_bf16(e3), "R4": orc.f64_array_to_bf16(e4), "R6": plain[0]}
    dec = _run(ol, hid, own)
    assert _same(plain, dec)
    for pt in ("R3", "R4", "R6"):
        assert dec[2][pt]["taken"] == 0 and dec[2][pt]["refused"] == 0


def test_wrong_codes_are_refused_and_the_oracle_keeps_its_own():
    lay, ol = _tiny()
    hid = synth.make_hidden(4, 256, 41, 0, 0)
    plain = _run(ol, hid)
    st = ol.new_state()
    _, (e3, _), _ = ol.run_traced(hid.copy(), *st)
    own = orc.f64_array_to_bf16(e3)
    bad = own.copy()
    n_in = bad.shape[1]
    for t, i in [(0, n_in - 1), (1, 3), (3, 300)]:  # a dt, a z and an x code, three ulps off
        bad[t, i] = bad[t, i] + 3
    dec = _run(ol, hid, {"R3": bad})
    assert dec[2]["R3"]["refused"] == 3 and dec[2]["R3"]["taken"] == 0
    assert dec[2]["R3"]["first_refused"] == n_in - 1
    assert _same(plain, dec)


def test_a_near_tie_neighbour_is_taken():
    lay, ol = _tiny()
    hid = synth.make_hidden(8, 256, 42, 0, 0)
    st = ol.new_state()
    _, (e3, a3), _ = ol.run_traced(hid.copy(), *st)
    own = orc.f64_array_to_bf16(e3)
    # the other code across each value's nearest rounding boundary, and its excess
    flat_e, flat_a, flat_o = e3.ravel(), a3.ravel(), own.ravel()
    vals = orc.bf16_array_to_f64(flat_o)
    step = np.where((flat_e > vals) == (flat_o < 0x8000), 1, -1).astype(np.int64)
    nb = (flat_o.astype(np.int64) + step).astype(np.uint16)
    ex = np.array([orc.decision_excess(int(c), float(e), float(max(a, abs(e))))
                   for c, e, a in zip(nb, flat_e, flat_a)])
    i_take = int(np.argmin(ex))
    assert ex[i_take] <= orc.DECISION_TOL["R3"]
    i_refuse = int(np.argmax(np.where(ex > 4 * orc.DECISION_TOL["R3"], -ex, -np.inf)))
    cand = flat_o.copy()
    cand[i_take] = nb[i_take]
    cand[i_refuse] = nb[i_refuse]
    dec = _run(ol, hid, {"R3": cand.reshape(own.shape)})
    assert dec[2]["R3"]["taken"] == 1 and dec[2]["R3"]["refused"] == 1
    assert dec[2]["R3"]["first_refused"] == i_refuse


def test_codes_of_an_evaluation_that_drops_a_term_are_refused():
    # the mistake the tolerance must catch: an in_proj that misses its last
    # k term; every code that mistake changes has to be refused
    lay, ol = _tiny()
    d = lay["dims"]
    hid = synth.make_hidden(1, 256, 43, 0, 0)
    st = ol.new_state()
    _, (e3, _), _ = ol.run_traced(hid.copy(), *st)
    xn = orc.rmsnorm(hid, lay["norm_w"], d["eps"])[0]
    K = d["hidden"]
    wd = torch.from_numpy(lay["in_w"][:, K - 1].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    sd = orc.bf16_array_to_f64(lay["in_s"][np.arange(wd.shape[0]) // 128, (K - 1) // 128])
    term = orc.bf16_array_to_f64(xn[K - 1:K])[0] * wd * sd
    wrong = orc.f64_array_to_bf16(e3[0] - term)[None]
    n_diff = int(np.sum(wrong != orc.f64_array_to_bf16(e3)))
    assert n_diff > 10
    dec = _run(ol, hid, {"R3": wrong})
    assert dec[2]["R3"]["refused"] == n_diff and dec[2]["R3"]["taken"] == 0


def test_w8a8_quantized_inputs_no_decision_gives_are_refused():
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE)
    ol = orc.OracleLayer(lay, act_fp8=True)
    d = lay["dims"]
    di = d["nheads"] * d["head_dim"]
    hid = synth.make_hidden(3, 256, 44, 0, 0)
    st = ol.new_state()
    plain = hid.copy()
    ol.run(plain, *st)
    # candidates that no legitimate R5 decision gives, in every block: all
    # refused, and the result equals the plain run
    bad_q = np.full((3, di), 0x38, np.uint8)            # every code 1.0
    bad_s = np.full((3, di // 128), 1.0, np.float32)    # scale 1: amax 448, not these rows'
    st2 = ol.new_state()
    h2 = hid.copy()
    rep = ol.run_decided(h2, *st2, {"Q5": (bad_q, bad_s)})
    assert rep["Q5"]["refused"] == 3 * (di // 128) and rep["Q5"]["taken"] == 0
    assert rep["Q5"]["first_refused"] == 0
    assert np.array_equal(h2, plain) and np.array_equal(st2[0], st[0])


def test_w8a8_quantized_inputs_of_legitimate_r5_decisions_are_taken():
    # the own quantization as candidates changes nothing; the quantization of
    # gated-norm rows with one legitimate near-tie flip is taken (its block
    # only), and gives the same result as taking that flip at R5 itself
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE)
    ol = orc.OracleLayer(lay, act_fp8=True)
    d = lay["dims"]
    di = d["nheads"] * d["head_dim"]
    T = 6
    hid = synth.make_hidden(T, 256, 45, 0, 0)

    def run(cand, trace=False):
        st = ol.new_state()
        h = hid.copy()
        tr = np.zeros((T, di), np.uint16) if trace else None
        rep = ol.run_decided(h, *st, cand, r5_trace=tr)
        return h, st, rep, tr

    def quant(rows):
        q = np.zeros((T, di), np.uint8)
        s = np.zeros((T, di // 128), np.float32)
        for t in range(T):
            q[t], s[t] = orc.act_quant(rows[t])
        return q, s

    h0, st0, _, r5 = run({}, trace=True)
    h1, st1, rep1, _ = run({"Q5": quant(r5)})
    assert rep1["Q5"]["taken"] == 0 and rep1["Q5"]["refused"] == 0
    assert np.array_equal(h0, h1) and np.array_equal(st0[0], st1[0])
    # flip one R5 code of token 2 to its neighbour: try elements until the R5
    # decision takes it and the flip changes that block's quantization
    for i in range(di):
        r5f = r5.copy()
        mag, sgn = int(r5[2, i]) & 0x7FFF, int(r5[2, i]) & 0x8000
        if mag in (0, 0x7F7F):
            continue
        for step in (1, -1):
            r5f[2, i] = sgn | (mag + step)
            ha, sta, repa, _ = run({"R5": r5f})
            qf = quant(r5f)
            if repa["R5"]["taken"] != 1 or np.array_equal(qf[0][2], quant(r5)[0][2]):
                continue
            hb, stb, repb, _ = run({"Q5": qf})
            assert repb["Q5"]["taken"] == 1 and repb["Q5"]["refused"] == 0
            assert np.array_equal(ha, hb)  # the same decision, taken at R5 or at its quantization
            return
    pytest.fail("no legitimate R5 neighbour changes a quantized block")
