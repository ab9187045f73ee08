"""GPU parity of the varlen prefill (several sequences of different lengths in
one call per kernel; K-token decode of n sequences is the equal-length case)
against the oracle, sequence by sequence: each sequence's prefill is by
definition its T_i sequential decode steps, so the oracle runs them on that
sequence's own state.  Rounding decisions and states are checked as in the
single-sequence tests (tests/helpers.py): the oracle follows the GPU's
legitimate decisions, refuses none, and every head's state meets 1e-3."""
import numpy as np
import pytest
import torch

from mamba_ssm_layer_gb300 import abi, synth
from mamba_ssm_layer_gb300.layer import DeviceLayer, bits_u16, to_dev
from oracle import oracle as orc
from tests.helpers import (TOL_BF16, TOL_STATE, DecisionLog, bf16_to_f64, check_state_all_heads, decode_candidates,
                           floored_rel_err, prefill_candidates, rows, state_rel_err)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from __graft_entry__ import build
    build()
    abi.m2_device_status(clear=True)
    yield
    assert abi.m2_device_status() == abi.M2_OK


def _varlen_case(lay, lens, warm, key, w8a8=False):
    """`warm` batched decode steps of all sequences, then one varlen prefill of
    lens[i] tokens per sequence (w8a8: on the FP8-activation arm, against the
    oracle's W8A8 layer); every sequence checked against the oracle."""
    d = lay["dims"]
    hd = d["hidden"]
    n = len(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    dl = DeviceLayer(lay)
    ol = orc.OracleLayer(lay)
    olp = orc.OracleLayer(lay, act_fp8=True) if w8a8 else ol  # the prefill's definition
    st = dl.new_state(n)
    ost = [ol.new_state() for _ in range(n)]
    log = DecisionLog()
    wsd = dl.workspace(n, 0)
    for t in range(warm):
        hid = synth.make_hidden(n, hd, *key, 1000 + t)
        x = to_dev(hid)
        pos_before = st[2].cpu().numpy().copy()
        dl.decode(x, st, wsd)
        torch.cuda.synchronize()
        cand = decode_candidates(wsd, n, d, bits_u16(st[1]), pos_before, bits_u16(x), g_f16=lay["out_fmt"] == "fp8")
        for i in range(n):
            log.add(ol.run_decided(np.ascontiguousarray(hid[i:i + 1]), *ost[i], cand[i]), ("decode", t, i))
    hid = synth.make_hidden(T, hd, *key, 0)
    x = to_dev(hid)
    ws = dl.workspace_varlen(n, T)
    dl.prefill_varlen(x, cu, st, ws, w8a8=w8a8)
    torch.cuda.synchronize()
    assert abi.m2_device_status() == abi.M2_OK
    got = bits_u16(x)
    # the gated norm writes bf16 rows on the tensor-core path, except on the
    # W8A8 arm with an E4M3 out_proj (codes and scales instead)
    r5 = T > 8 and not (w8a8 and lay["out_fmt"] == "fp8")
    cand = prefill_candidates(ws, cu, d, got, r5_available=r5, w8a8=w8a8, g_f16=lay["out_fmt"] == "fp8")
    worst = 0.0
    errs = []
    h = st[0].cpu().numpy()
    ring = bits_u16(st[1])
    for i in range(n):
        a, b = int(cu[i]), int(cu[i + 1])
        ref = hid[a:b].copy()
        if b > a:
            log.add(olp.run_decided(ref, *ost[i], rows(cand, a, b)), ("prefill", i))
            worst = max(worst, floored_rel_err(bf16_to_f64(got[a:b]), bf16_to_f64(ref), axis=-1))
        errs.append(check_state_all_heads(h[i], ost[i][0]))
        assert np.array_equal(ring[i], ost[i][1]), i
        assert int(st[2][i]) == warm + (b - a), i  # positions: integer work
    rep = log.check()
    assert worst <= TOL_BF16, worst
    print("varlen parity", lens, worst, "state", max(errs), rep)
    return dl, st, hid, cu


def test_varlen_tiny_mixed_lengths_with_empty_sequence():
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE)
    _varlen_case(lay, [5, 0, 130, 1, 127, 128, 3], 2, (synth.WL_TINY_DECODE, 70))


def test_varlen_w8a8_tiny_mixed_lengths():
    # the W8A8 arm over a varlen batch: per-token activation blocks ignore
    # sequence boundaries; an empty and a one-token sequence included
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE)
    _varlen_case(lay, [9, 1, 130, 0, 40], 2, (synth.WL_TINY_DECODE, 74), w8a8=True)


def test_varlen_tiny_bf16_weights():
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE, layer=2, in_fmt="bf16", out_fmt="bf16")
    _varlen_case(lay, [9, 200, 4], 1, (synth.WL_TINY_DECODE, 71))


def test_k_token_decode_8b_layer():
    # speculative-verify shape: 4 sequences x 4 tokens after 3 ordinary decode steps
    lay = synth.make_layer(synth.NEMOTRON_H_8B, synth.WL_8B_DECODE_B64)
    _varlen_case(lay, [4, 4, 4, 4], 3, (synth.WL_8B_DECODE_B64, 72))


def test_varlen_8b_layer_chunk_boundaries():
    lay = synth.make_layer(synth.NEMOTRON_H_8B, synth.WL_8B_PREFILL_1K)
    _varlen_case(lay, [200, 1, 129], 0, (synth.WL_8B_PREFILL_1K, 73))


def test_varlen_equals_separate_prefills():
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE)
    lens = [70, 3, 129]
    cu = np.concatenate([[0], np.cumsum(lens)])
    hid = synth.make_hidden(int(cu[-1]), 256, 8, 8, 8)
    dl = DeviceLayer(lay)
    st1 = dl.new_state(len(lens))
    x = to_dev(hid)
    dl.prefill_varlen(x, cu, st1, dl.workspace_varlen(len(lens), int(cu[-1])))
    st2 = dl.new_state(len(lens))
    ws = dl.workspace(1, int(max(lens)))
    outs = []
    for i in range(len(lens)):
        xi = to_dev(hid[cu[i]:cu[i + 1]])
        dl.prefill(xi, (st2[0][i], st2[1][i], st2[2][i:i + 1]), ws)
        outs.append(xi)
    torch.cuda.synchronize()
    sep = np.concatenate([bits_u16(o) for o in outs])
    assert floored_rel_err(bf16_to_f64(bits_u16(x)), bf16_to_f64(sep), axis=-1) <= TOL_BF16
    assert state_rel_err(st1[0].cpu().numpy(), st2[0].cpu().numpy()) <= TOL_STATE
    assert np.array_equal(st1[2].cpu().numpy(), st2[2].cpu().numpy())


def test_varlen_rejects_bad_offsets():
    lay = synth.make_layer(synth.TINY, synth.WL_TINY_DECODE)
    dl = DeviceLayer(lay)
    st = dl.new_state(2)
    x = to_dev(synth.make_hidden(4, 256, 1, 1, 1))
    ws = dl.workspace_varlen(2, 4)
    n0 = abi.m2_launch_count()
    for cu in ([1, 2, 4], [0, 3, 2], [0, 0, 0]):
        st_code = abi.mamba2_layer_prefill_varlen(dl.dims, dl.struct, x, cu, *st, ws, ws.numel(), check=False)
        assert st_code == abi.M2_ERR_ARG, cu
    assert abi.m2_launch_count() == n0
