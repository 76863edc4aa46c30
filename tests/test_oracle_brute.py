"""The C oracle against an independently written NumPy brute force of the whole layer
(tests/brute_layer.py: its own MX decode, its own bf16 rounding, dense per-row evaluation).

Both evaluate the same arithmetic in f64 with the same rounding points, so every bf16 stage
must agree bit for bit (a difference needs two f64 sums of different order to straddle a
bf16 rounding midpoint: odds ~1e-13 per value), the KV records byte for byte, the top-k
exactly, and the unrounded f64 outputs to ~1e-12.  A dropped term, a wrong sign, a wrong
index map or a transposed operand in either restatement fails here.  Workloads: the tiny
layer (one row), a mid-size layer with ragged tiles and a pad row, a narrow layer with a
300-key window, 256 experts and routed_scale 2.5, and non-causal variants of the first two.
"""
import numpy as np
import pytest

import gen
from tests import brute_layer as brute
from tests.helpers import np_inputs

BF16_STAGES = ["xn", "qkv", "q_latn", "kvn", "q", "o", "oa", "h", "u", "t_s", "t_r", "out"]

CASES = [("tiny", {}), ("small_r11", {}), ("wide_r9", {}),
         ("tiny", dict(causal=0, swa_width=20)), ("small_r11", dict(causal=0, swa_width=30))]


def _case(name, overrides):
    spec, w, st = gen.make_workload(name)
    spec = dict(spec, **overrides)
    wn, sn = np_inputs(w, st)
    return spec, wn, sn


@pytest.mark.parametrize("name,overrides", CASES,
                         ids=[f"{n}{'-noncausal' if o else ''}" for n, o in CASES])
def test_oracle_equals_independent_brute_force(orc, name, overrides):
    spec, wn, sn = _case(name, overrides)
    ref = orc.layer(spec, wn, sn)
    assert ref["rc"] == 0
    bf = brute.layer(spec, wn, sn)
    for k in BF16_STAGES:
        a, b = np.asarray(ref[k]), np.asarray(bf[k])
        assert a.shape == b.shape, k
        bad = np.count_nonzero(a != b)
        assert bad == 0, f"{k}: {bad} of {a.size} bf16 values differ"
    assert np.array_equal(ref["cache"], bf["cache"]), "KV records"
    assert np.array_equal(ref["logits"], bf["logits"]), "f32 router logits"
    assert np.array_equal(ref["topk_idx"], bf["topk_idx"]), "top-k experts"
    np.testing.assert_allclose(ref["topk_w"], bf["topk_w"], rtol=1e-12, atol=0)
    np.testing.assert_allclose(ref["probs"], bf["probs"], rtol=1e-12, atol=1e-300)
    for k in ("y_s", "y_r"):
        a, b = np.asarray(ref[k], np.float64), np.asarray(bf[k], np.float64)
        assert np.linalg.norm(a - b) <= 1e-12 * np.linalg.norm(b), k
    # the case is not vacuous: live rows attend, route and change the residual stream
    live = np.asarray(sn["positions"]) >= 0
    assert np.abs(brute.bf16_value(bf["o"][live])).max() > 0
    assert (bf["topk_idx"][live] >= 0).all()
    assert np.count_nonzero(bf["out"][live] != np.asarray(sn["x"])[live]) > 0.5 * bf["out"][live].size


def test_brute_force_rounding_and_decode_pins():
    """The brute force's own helpers against values fixed by the formats' definitions."""
    # bf16 round-to-nearest-even: 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> 1 (even);
    # 1 + 3 * 2^-8 ties between 1 + 2^-7 and 1 + 2^-6 -> 1 + 2^-6 (even); just above a tie
    # rounds up; the sign is kept
    v = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -30, -3.0, 0.0])
    got = brute.bf16_value(brute.bf16_rne(v))
    np.testing.assert_array_equal(got, [1.0, 1 + 2.0 ** -6, 1 + 2.0 ** -7, -3.0, 0.0])
    # e2m1 (OCP MX v1.0): code 0x7 = 6, 0x1 = 0.5 (subnormal), 0xA = -1, 0xF = -6; element
    # 2i in the low nibble
    w = brute.dequant_mxfp4(np.array([[0x17, 0xFA] + [0] * 14], np.uint8),
                            np.array([[127]], np.uint8))
    np.testing.assert_array_equal(w[0, :4], [6.0, 0.5, -1.0, -6.0])
    # e4m3: 0x7E = 448, 0x08 = 2^-6, 0x01 = 2^-9 (subnormal), 0xB8 = -1; E8M0 130 = 8
    np.testing.assert_array_equal(brute.e4m3_value(np.array([0x7E, 0x08, 0x01, 0xB8])),
                                  [448.0, 2.0 ** -6, 2.0 ** -9, -1.0])
    assert brute.e8m0_value(130) == 8.0 and brute.e8m0_value(127) == 1.0
    # MXFP8 block indexing: scale [n/32][k/32]
    codes = np.full((64, 64), 0x38, np.uint8)            # 1.0 everywhere
    s = np.array([[127, 128], [129, 130]], np.uint8)
    d = brute.dequant_mxfp8(codes, s)
    assert d[0, 0] == 1 and d[0, 40] == 2 and d[40, 0] == 4 and d[63, 63] == 8
