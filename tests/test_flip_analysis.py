"""CPU checks of the rounding-decision analysis used by the GPU layer tests:
it must accept a flip at a bf16 tie and reject any other code difference."""
import numpy as np

from mamba_ssm_layer_gb300 import synth
from oracle import oracle as orc
from tests.helpers import FlipTracker, legit_flips


def test_legit_flip_accepts_near_tie_only():
    # exact value 1 + 2^-8 (+ tiny): the tie between bf16 1.0 and 1.0078125
    e = np.array([1 + 2 ** -8 + 2 ** -30, 1 + 2 ** -8 + 2 ** -11, 3.0, 1e-6, 1e-6])
    a = np.array([1.0, 1.0, 3.0, 40.0, 40.0])  # sums of |terms|
    o = orc.f64_array_to_bf16(e)
    g = o.copy()
    g[0] = 0x3F80          # the other neighbour of a near-tie: legitimate
    g[1] = 0x3F80          # exact value a quarter of an ulp from the tie: not
    g[2] = 0x4041          # adjacent code but 3.0 is exact: not
    g[3] = orc.f64_to_bf16(1e-6 + 3e-8)   # cancellation: 40 * 2^-20 = 3.8e-5 of slack: legitimate
    g[4] = orc.f64_to_bf16(1e-6 + 1e-4)   # far outside the slack: not
    idx, ok = legit_flips(g, e, o, a)
    assert list(idx) == [0, 1, 2, 3, 4] and list(ok) == [True, False, False, True, False]


def test_tracker_flags_bad_differences_and_taints():
    d = synth.TINY
    dd = synth.derived(d)
    rng = np.random.default_rng(0)
    A_log = np.zeros(d["nheads"], np.float32)
    dtb = np.zeros(d["nheads"], np.float32)
    tr = FlipTracker(d, A_log, dtb, np.zeros((dd['d_xbc'], d['d_conv']), np.uint16))
    e3 = rng.standard_normal(dd["n_in"])
    e4 = rng.standard_normal(dd["d_xbc"])
    g3, g4 = orc.f64_array_to_bf16(e3), orc.f64_array_to_bf16(e4)
    a3, a4 = np.abs(e3), np.abs(e4)
    tr.token(g3, (e3, a3), g4, (e4, a4))
    assert tr.bad == [] and tr.taint_weight.max() == 0
    # a wrong dt code (not at a tie) is reported
    g3b = g3.copy()
    g3b[-1] ^= 0x0001
    tr.token(g3b, (e3, a3), g4, (e4, a4))
    assert tr.bad and tr.bad[0][0] == "R3"
