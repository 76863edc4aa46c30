"""Pins for the oracle's FFN launch (the MoE half fed by an attention output).

The residual h = bf16(x + a) is pinned by closed forms (a = 0 gives x; a = -x gives an
all-zero layer; x and a commute), the MoE half by the whole-layer oracle, whose own pins
hold it to the stage functions: with x set to the layer's residual and a = 0, the FFN
launch must reproduce the layer's routing, expert outputs and output bit for bit.
"""
import numpy as np
import pytest

import gen
from tests.helpers import bf16_f64, np_inputs

_FFN_KEYS = ["ffn_norm", "router", "sh_gu", "sh_gu_s", "sh_d", "sh_d_s", "ex_gu", "ex_gu_s",
             "ex_d", "ex_d_s"]


@pytest.fixture(scope="module")
def small():
    spec, w, st = gen.make_workload("small_r11")
    a = gen.make_attn_out(spec, st, seed=5)
    wn, sn = np_inputs(w, st)
    return spec, wn, sn, np_inputs({"a": a}, {})[0]["a"]


def test_residual_is_rounded_sum(orc, small):
    spec, w, st, a = small
    tr = orc.ffn_layer(spec, w, st["x"], a, st["positions"])
    h = orc.bf16_round_array(bf16_f64(st["x"]) + bf16_f64(a))  # the f64 sum of two bf16 is exact
    assert np.array_equal(tr["h"], h)
    assert np.array_equal(tr["u"], orc.rmsnorm(h, w["ffn_norm"], spec["eps"]))


def test_equals_layer_moe_half(orc, small):
    spec, w, st, _ = small
    lay = orc.layer(spec, w, st)
    valid = np.asarray(st["positions"]) >= 0
    tr = orc.ffn_layer(spec, w, lay["h"], np.zeros_like(lay["h"]), st["positions"])
    assert np.array_equal(tr["h"], lay["h"])
    for k in ("u", "logits", "topk_idx", "topk_w", "t_s", "y_s", "t_r", "y_r"):
        assert np.array_equal(tr[k], lay[k]), k
    assert np.array_equal(tr["out"][valid], lay["out"][valid])
    assert np.array_equal(tr["out"][~valid], lay["h"][~valid])  # pad rows give back x


def test_opposite_inputs_cancel(orc, small):
    spec, w, st, _ = small
    x = st["x"]
    tr = orc.ffn_layer(spec, w, x, x ^ np.uint16(0x8000), st["positions"])
    valid = np.asarray(st["positions"]) >= 0
    assert not bf16_f64(tr["h"]).any()
    assert not bf16_f64(tr["out"][valid]).any()
    assert np.array_equal(tr["out"][~valid], x[~valid])


def test_inputs_commute(orc, small):
    spec, w, st, a = small
    one = orc.ffn_layer(spec, w, st["x"], a, st["positions"])
    two = orc.ffn_layer(spec, w, a, st["x"], st["positions"])
    valid = np.asarray(st["positions"]) >= 0
    assert np.array_equal(one["h"], two["h"])
    assert np.array_equal(one["out"][valid], two["out"][valid])
    assert np.array_equal(two["out"][~valid], a[~valid])


def test_zero_experts_give_residual(orc, small):
    spec, w, st, a = small
    w0 = dict(w)
    w0["sh_gu"] = np.zeros_like(w["sh_gu"])
    w0["ex_gu"] = np.zeros_like(w["ex_gu"])
    tr = orc.ffn_layer(spec, w0, st["x"], a, st["positions"])
    valid = np.asarray(st["positions"]) >= 0
    assert np.array_equal(tr["out"][valid], tr["h"][valid])
    assert not tr["y_s"].any() and not tr["y_r"].any()


def test_reads_only_ffn_weights(orc, small):
    spec, w, st, a = small
    full = orc.ffn_layer(spec, w, st["x"], a, st["positions"])
    only = orc.ffn_layer(spec, {k: w[k] for k in _FFN_KEYS}, st["x"], a, st["positions"])
    assert np.array_equal(full["out"], only["out"])


def test_forced_routing(orc, small):
    spec, w, st, a = small
    tr = orc.ffn_layer(spec, w, st["x"], a, st["positions"])
    same = orc.ffn_layer(spec, w, st["x"], a, st["positions"], force_idx=tr["topk_idx"])
    assert np.array_equal(same["out"], tr["out"])
