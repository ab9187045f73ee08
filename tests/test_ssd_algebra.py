"""The chunked (state-space dual) form of the SSM recurrence, written out in
float64 numpy, equals T sequential oracle decode steps.  CPU only.

This checks the algebra the prefill scan kernels implement (intra-chunk
decay-weighted C B^T products, per-chunk states, a sequential pass over chunk
states, the inter-chunk term exp(cumsum) C h_in) against the oracle's plain
recurrence (source listing nemotron_mamba2.rs, `ssm_decode`; the SSD chunked
prefill scan row of its kernel table).  It shares no code with the CUDA path.
"""
import numpy as np
import pytest

from oracle import oracle as orc
from mamba_ssm_layer_gb300 import synth


def _softplus(v):
    return np.where(v > 20.0, v, np.log1p(np.exp(np.minimum(v, 20.0))))


def chunked_scan(h0, x, Bm, Cm, dt_raw, A_log, D, dt_bias, G, Q):
    """h0 [H,P,N]; x [T,H,P]; Bm, Cm [T,G,N]; dt_raw [T,H] (float64 values)."""
    T, H, P = x.shape
    N = Bm.shape[2]
    A = -np.exp(A_log.astype(np.float64))
    dt = np.clip(_softplus(dt_raw + dt_bias.astype(np.float64)), 1e-9, 1e9)
    grp = np.arange(H) // (H // G)
    y = np.zeros((T, H, P))
    h = h0.copy()
    for c0 in range(0, T, Q):
        sl = slice(c0, min(T, c0 + Q))
        q = sl.stop - sl.start
        a = dt[sl] * A                       # [q, H]
        cs = np.cumsum(a, axis=0)            # inclusive
        xc, bc, cc, dtc = x[sl], Bm[sl][:, grp], Cm[sl][:, grp], dt[sl]
        # intra-chunk: y_t += sum_{s<=t} (C_t.B_s) exp(cs_t - cs_s) dt_s x_s
        cb = np.einsum("thn,shn->hts", cc, bc)
        seg = cs.T[:, :, None] - cs.T[:, None, :]           # [H, t, s]
        mask = np.tril(np.ones((q, q), bool))
        L = np.where(mask, cb * np.exp(np.where(mask, seg, 0.0)), 0.0) * dtc.T[:, None, :]
        y[sl] += np.einsum("hts,shp->thp", L, xc)
        # inter-chunk: exp(cs_t) C_t h_in
        y[sl] += np.exp(cs)[:, :, None] * np.einsum("thn,hpn->thp", cc, h)
        y[sl] += D.astype(np.float64)[None, :, None] * xc
        # chunk state
        w = np.exp(cs[-1][None, :] - cs) * dtc                # [q, H]
        dH = np.einsum("sh,shp,shn->hpn", w, xc, bc)
        h = np.exp(cs[-1])[:, None, None] * h + dH
    return h, y


@pytest.mark.parametrize("T,Q", [(1, 128), (5, 4), (37, 8), (300, 128)])
def test_chunked_form_matches_sequential_oracle(T, Q):
    H, P, N, G = 4, 8, 16, 2
    rng = np.random.default_rng([T, Q])
    bits = lambda shape, s: synth.to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * s)
    x, Bm, Cm = bits((T, H * P), 1.0), bits((T, G * N), 0.5), bits((T, G * N), 0.5)
    dt_raw = bits((T, H), 1.0)
    A_log = rng.uniform(0.0, np.log(16.0), H).astype(np.float32)
    D = rng.standard_normal(H).astype(np.float32)
    dt_bias = rng.uniform(-4.0, 0.0, H).astype(np.float32)
    h0 = rng.standard_normal((H, P, N))
    # oracle: T sequential steps
    h = h0.copy()
    y_seq = np.zeros((T, H * P))
    for t in range(T):
        h, y_seq[t], _ = orc.ssm_step(h, x[t], Bm[t], Cm[t], dt_raw[t], A_log, D, dt_bias, G)
    f = orc.bf16_array_to_f64
    h_ch, y_ch = chunked_scan(h0, f(x).reshape(T, H, P), f(Bm).reshape(T, G, N), f(Cm).reshape(T, G, N),
                              f(dt_raw).reshape(T, H), A_log, D, dt_bias, G, Q)
    np.testing.assert_allclose(h_ch, h, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(y_ch.reshape(T, H * P), y_seq, rtol=1e-10, atol=1e-10)


def test_chunked_form_detects_a_dropped_inter_chunk_term():
    """A chunked scan without the exp(cs) C h_in term must not pass (guards the test above)."""
    T, H, P, N, G = 20, 2, 4, 8, 1
    rng = np.random.default_rng(7)
    x = rng.standard_normal((T, H, P)); Bm = rng.standard_normal((T, G, N)); Cm = rng.standard_normal((T, G, N))
    dt_raw = rng.standard_normal((T, H)); A_log = np.zeros(H, np.float32); D = np.zeros(H, np.float32)
    dt_bias = np.zeros(H, np.float32); h0 = rng.standard_normal((H, P, N))
    _, y1 = chunked_scan(h0, x, Bm, Cm, dt_raw, A_log, D, dt_bias, G, 4)
    _, y2 = chunked_scan(np.zeros_like(h0), x, Bm, Cm, dt_raw, A_log, D, dt_bias, G, 4)
    _, y3 = chunked_scan(h0, x, Bm, Cm, dt_raw, A_log, D, dt_bias, G, T)
    assert np.abs(y1 - y2).max() > 1e-3          # the carried state matters
    np.testing.assert_allclose(y1, y3, rtol=1e-10, atol=1e-10)  # chunk length does not
